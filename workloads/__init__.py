"""Seeded synthetic inputs for the ragged sparse-attention decode step.

This module is the only code shared by the CPU oracle and the GPU path. It
draws random numbers and stores them in the types the step consumes; it holds
none of the step's arithmetic (no scoring, selection or attention).

Shapes follow the DeepSeek-V4 joint-decode rows of mlx-native
(`src/ops/deepseek_rows.rs`, structs `DeepSeekIndexerRow` and
`DeepSeekSparseAttentionRow`; `src/shaders/deepseek_rows.metal`, constants
IDX_HEADS/IDX_DIM/IDX_TOPK and DS_HEADS/DS_DIM):

* indexer query  qI [R, 64, 128] bf16, head weights wI [R, 64] fp32,
  indexer keys   KI_r [L_r, 128] bf16, one cache per row;
* attention query qA [R, 64, 512] bf16, shared KV KV_r [L_r, 512] bf16
  (used as both K and V), sinks fp32 [64] (shared) or [R, 64] (per row);
* per-row table {kv_len, width = min(512, kv_len), index_offset, q_row}.

Recipe (one ``numpy.random.default_rng(seed)`` per workload): values are
drawn in fp32 and rounded to bf16 with round-to-nearest-even. Per row the
draw order is qI, KI, wI, qA, KV; sinks are drawn after all rows.

bf16 tensors are returned as ``uint16`` bit patterns; converting them to a
wider float is exact and left to the consumer.
"""

from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np

HEADS = 64
INDEX_DIM = 128
KV_DIM = 512
TOP_K = 512
MAX_ROWS = 8


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact widening)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass
class Row:
    kv_len: int
    width: int
    index_offset: int
    q_row: int


@dataclasses.dataclass
class Workload:
    name: str
    seed: int
    rows: List[Row]
    q_index: np.ndarray          # uint16 [Q, 64, 128] bf16 bits
    w_index: np.ndarray          # float32 [Q, 64]
    keys: List[np.ndarray]       # uint16 [L_r, 128] per row
    q_attn: np.ndarray           # uint16 [Q, 64, 512]
    kv: List[np.ndarray]         # uint16 [L_r, 512] per row
    sinks: np.ndarray            # float32 [64] (shared) or [Q, 64] (per q_row)
    scale: float
    integer_valued: bool = False

    @property
    def num_rows(self) -> int:
        return len(self.rows)

    @property
    def sinks_row_stride(self) -> int:
        return 0 if self.sinks.ndim == 1 else HEADS

    @property
    def index_elements(self) -> int:
        return max(r.index_offset + r.width for r in self.rows)

    def algorithmic_bytes(self) -> int:
        """Bytes one decode step must move: indexer keys + selected KV + q + out.

        Per row: 256*L (keys) + 1024*W (gathered KV rows) + 16384 (qI) +
        65536 (qA) + 65536 (output); weights, sinks and indices excluded.
        """
        return sum(256 * r.kv_len + 1024 * r.width + 16384 + 65536 + 65536 for r in self.rows)

    def row_sinks(self, e: int) -> np.ndarray:
        r = self.rows[e]
        return self.sinks if self.sinks.ndim == 1 else self.sinks[r.q_row]

    def subset(self, entries: List[int]) -> "Workload":
        """The same caches and queries, with a table of only `entries` (in order)."""
        return dataclasses.replace(
            self,
            rows=[self.rows[e] for e in entries],
            keys=[self.keys[e] for e in entries],
            kv=[self.kv[e] for e in entries],
        )


def _normal_bf16(rng, shape, std=1.0):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x = x * np.float32(std)
    return bf16_bits(x)


def _int_bf16(rng, shape):
    return bf16_bits(rng.integers(-3, 3, endpoint=True, size=shape).astype(np.float32))


def _table(kv_lens):
    rows, off = [], 0
    for e, L in enumerate(kv_lens):
        w = min(TOP_K, L)
        rows.append(Row(kv_len=int(L), width=int(w), index_offset=off, q_row=e))
        off += TOP_K
    return rows


def make_workload(name: str, seed: int, kv_lens, *, integer: bool = False,
                  prototypes: bool = False, per_row_sinks: bool = True,
                  sink_overrides: Optional[dict] = None) -> Workload:
    """Draw one workload. `kv_lens` may be a list, or a callable rng -> list."""
    rng = np.random.default_rng(seed)
    if callable(kv_lens):
        kv_lens = kv_lens(rng)
    kv_lens = [int(L) for L in kv_lens]
    R = len(kv_lens)
    protos = _normal_bf16(rng, (64, INDEX_DIM)) if prototypes else None
    qI = np.empty((R, HEADS, INDEX_DIM), np.uint16)
    wI = np.empty((R, HEADS), np.float32)
    qA = np.empty((R, HEADS, KV_DIM), np.uint16)
    keys, kv = [], []
    for e, L in enumerate(kv_lens):
        if integer:
            qI[e] = _int_bf16(rng, (HEADS, INDEX_DIM))
            keys.append(_int_bf16(rng, (L, INDEX_DIM)))
            wI[e] = rng.integers(-3, 3, endpoint=True, size=HEADS).astype(np.float32)
            qA[e] = _int_bf16(rng, (HEADS, KV_DIM))
            kv.append(_int_bf16(rng, (L, KV_DIM)))
        else:
            qI[e] = _normal_bf16(rng, (HEADS, INDEX_DIM))
            if prototypes:
                pick = rng.integers(0, 64, size=L)
                base = bits_to_f32(protos)[pick]
                noise = rng.standard_normal(size=(L, INDEX_DIM), dtype=np.float32) * np.float32(1e-3)
                keys.append(bf16_bits(base + noise))
            else:
                keys.append(_normal_bf16(rng, (L, INDEX_DIM)))
            wI[e] = rng.standard_normal(size=HEADS, dtype=np.float32) / np.float32(8.0)
            qA[e] = _normal_bf16(rng, (HEADS, KV_DIM))
            kv.append(_normal_bf16(rng, (L, KV_DIM)))
    if per_row_sinks:
        sinks = rng.standard_normal(size=(R, HEADS), dtype=np.float32)
        for e, value in (sink_overrides or {}).items():
            sinks[e, :] = np.float32(value)
    else:
        sinks = rng.standard_normal(size=HEADS, dtype=np.float32)
    return Workload(name=name, seed=seed, rows=_table(kv_lens), q_index=qI, w_index=wI,
                    keys=keys, q_attn=qA, kv=kv, sinks=sinks,
                    scale=1.0 / math.sqrt(KV_DIM), integer_valued=integer)


CONFIG_NAMES = [
    "1x2048",
    "4x{300,512,1000,4096}-int",
    "8xU[4096,65536]",
    "8x131072",
    "8x{1,17,511,512,513,32768,65536,262144}-edge",
]

CONFIG4_LENS = [1, 17, 511, 512, 513, 32768, 65536, 262144]


def config2_lens(rng) -> List[int]:
    return [int(x) for x in rng.integers(4096, 65536, endpoint=True, size=8)]


def config(i: int) -> Workload:
    """The five benchmark workloads (index 0..4)."""
    if i == 0:
        return make_workload(CONFIG_NAMES[0], 0, [2048], per_row_sinks=False)
    if i == 1:
        return make_workload(CONFIG_NAMES[1], 1, [300, 512, 1000, 4096], integer=True,
                             per_row_sinks=False)
    if i == 2:
        return make_workload(CONFIG_NAMES[2], 2, config2_lens)
    if i == 3:
        return make_workload(CONFIG_NAMES[3], 3, [131072] * 8)
    if i == 4:
        # kv_len 511 (entry 2) gets sinks +20, kv_len 32768 (entry 5) gets -20.
        return make_workload(CONFIG_NAMES[4], 4, CONFIG4_LENS, prototypes=True,
                             sink_overrides={2: 20.0, 5: -20.0})
    raise ValueError(f"no config {i}")


def config_kv_lens(i: int) -> List[int]:
    """Row lengths of config i without drawing the tensors."""
    if i == 0:
        return [2048]
    if i == 1:
        return [300, 512, 1000, 4096]
    if i == 2:
        return config2_lens(np.random.default_rng(2))
    if i == 3:
        return [131072] * 8
    if i == 4:
        return list(CONFIG4_LENS)
    raise ValueError(f"no config {i}")


def draw_queries(wl: Workload, seed: int):
    """Another set of queries for the same caches, drawn with the workload's recipe:
    (q_index uint16 [Q,64,128], w_index float32 [Q,64], q_attn uint16 [Q,64,512])."""
    rng = np.random.default_rng(seed)
    Q = wl.q_index.shape[0]
    if wl.integer_valued:
        qI = _int_bf16(rng, (Q, HEADS, INDEX_DIM))
        wI = rng.integers(-3, 3, endpoint=True, size=(Q, HEADS)).astype(np.float32)
        qA = _int_bf16(rng, (Q, HEADS, KV_DIM))
    else:
        qI = _normal_bf16(rng, (Q, HEADS, INDEX_DIM))
        wI = rng.standard_normal(size=(Q, HEADS), dtype=np.float32) / np.float32(8.0)
        qA = _normal_bf16(rng, (Q, HEADS, KV_DIM))
    return qI, wI, qA


def draw_index_queries(wl: Workload, seed: int, count: int):
    """`count` indexer queries for the same caches (several consecutive queries
    per row), drawn with the workload's recipe: (q_index uint16 [count,64,128],
    w_index float32 [count,64])."""
    rng = np.random.default_rng(seed)
    if wl.integer_valued:
        qI = _int_bf16(rng, (count, HEADS, INDEX_DIM))
        wI = rng.integers(-3, 3, endpoint=True, size=(count, HEADS)).astype(np.float32)
    else:
        qI = _normal_bf16(rng, (count, HEADS, INDEX_DIM))
        wI = rng.standard_normal(size=(count, HEADS), dtype=np.float32) / np.float32(8.0)
    return qI, wI


# ---------------------------------------------------------------------------
# Stand-alone stage inputs (scores for the top-k stage, indices for attention)
# ---------------------------------------------------------------------------

def random_scores(seed: int, kv_lens, *, ties: bool = False, nonfinite: bool = False,
                  signed_zeros: bool = False, crowd=None) -> List[np.ndarray]:
    """fp32 score rows for the top-k stage alone.

    ties: draw from a small set of values so that exact ties are frequent.
    nonfinite: sprinkle NaN / +-Inf entries. signed_zeros: mix -0.0 and +0.0.
    crowd: per row, a number m of scores, at random positions, that share the
    top 11 bits of their order key (values 1 + k/4096, k < 1024, so with ties),
    above the rest of the row (uniform in [0, 0.5)): the best ones are all in
    one crowded bin of a top-11-bit histogram.
    """
    rng = np.random.default_rng(seed)
    out = []
    for e, L in enumerate(kv_lens):
        if crowd is not None:
            s = rng.uniform(0.0, 0.5, size=L).astype(np.float32)
            m = min(int(crowd[e]), L)
            at = rng.choice(L, size=m, replace=False)
            s[at] = (1.0 + rng.integers(0, 1024, size=m) / 4096.0).astype(np.float32)
        elif ties:
            s = rng.integers(-20, 20, size=L).astype(np.float32) * np.float32(0.25)
        else:
            s = rng.standard_normal(size=L, dtype=np.float32)
        if signed_zeros:
            z = rng.random(L) < 0.3
            s[z] = np.where(rng.random(int(z.sum())) < 0.5, np.float32(-0.0), np.float32(0.0))
        if nonfinite:
            bad = rng.random(L) < 0.05
            choice = rng.integers(0, 3, size=int(bad.sum()))
            s[bad] = np.array([np.nan, np.inf, -np.inf], np.float32)[choice]
        out.append(s)
    return out


def random_indices(seed: int, rows: List[Row], *, sentinel_frac: float = 0.0,
                   bad_rows=(), unique: bool = True) -> np.ndarray:
    """int32 index buffer for the attention stage alone.

    Each row gets `width` indices into [0, kv_len) (distinct when `unique`),
    a fraction replaced by the -1 sentinel; rows listed in `bad_rows` get one
    out-of-range index.
    """
    rng = np.random.default_rng(seed)
    n = max(r.index_offset + r.width for r in rows)
    idx = np.full(n, -7, np.int32)
    for e, r in enumerate(rows):
        if unique:
            sel = rng.permutation(r.kv_len)[: r.width]
        else:
            sel = rng.integers(0, r.kv_len, size=r.width)
        sel = sel.astype(np.int32)
        if sentinel_frac > 0:
            sel[rng.random(r.width) < sentinel_frac] = -1
        if e in bad_rows:
            sel[rng.integers(0, r.width)] = np.int32(r.kv_len + 5)
        idx[r.index_offset: r.index_offset + r.width] = sel
    return idx
