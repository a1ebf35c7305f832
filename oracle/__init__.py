"""CPU fp64 oracle for the ragged DeepSeek sparse-attention decode step.

TEST INFRASTRUCTURE ONLY. Only the test-suite, the smoke check of
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import this
package. The product path (the CUDA library and its Python binding) never
calls it, and this package imports nothing from the product path.

Every function is a plain, slow, direct statement of what the prior art
computes, in float64. The prior art is the mlx-native crate (0.18-0.21):
Metal kernels in ``src/shaders/deepseek_rows.metal`` and their host dispatch
in ``src/ops/deepseek_rows.rs``. Each function names the kernel it follows.

Readings taken where the pages leave a step open (each also listed in the
design notes):

* Every key of a row is valid (no causal cut): the decode row table has no
  position, and width = min(512, kv_len). ``indexer_score_causal`` and
  ``topk_causal`` carry the positioned variant.
* The indexer stages q and K as fp16 on the prior art's hardware; here the
  bf16 inputs are used exactly (fp64 products, no fp16 rounding).
* A value that the fp32 kernels would see as non-finite is treated as
  non-finite here too: a score, logit, denominator or output whose fp64 value
  lies beyond the largest finite fp32 magnitude counts as overflowed.
* Output order of top-k is best first: score descending, then lower index.
  Ties compare with IEEE ``==`` (so -0.0 ties +0.0).
* The sink has no value row: it enters the softmax max and denominator only.
* bf16 output rounding is round-to-nearest-even (``round_bf16``).
"""

from __future__ import annotations

import math
from typing import Dict, List, Tuple

import numpy as np

FLT_MAX = float(np.finfo(np.float32).max)
TOP_K = 512


# ---------------------------------------------------------------------------
# Input decoding
# ---------------------------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def _fp32_finite(x) -> np.ndarray:
    """True where x is finite and within the fp32 range."""
    x = np.asarray(x, dtype=np.float64)
    return np.isfinite(x) & (np.abs(x) <= FLT_MAX)


# ---------------------------------------------------------------------------
# (1) Lightning-indexer score
# deepseek_rows.metal, "Lightning indexer score and deterministic top-512",
# kernel deepseek_indexer_score_mma_rows_bf16: per key, per head the q.k dot
# product, ReLU, times the head weight, summed over the heads; a non-finite
# score (or a masked key) is stored as -inf.
# ---------------------------------------------------------------------------

def indexer_score(q: np.ndarray, w: np.ndarray, keys: np.ndarray) -> np.ndarray:
    """s[j] = sum_h w[h] * max(0, sum_d q[h, d] * keys[j, d]), float64.

    q [H, D], w [H], keys [L, D] (float64). Non-finite results become -inf.
    """
    q = np.asarray(q, np.float64)
    w = np.asarray(w, np.float64)
    keys = np.asarray(keys, np.float64)
    with np.errstate(invalid="ignore", over="ignore"):
        dots = keys @ q.T                       # [L, H]: dots[j, h] = q_h . k_j
        relu = np.where(dots > 0.0, dots, 0.0)  # max(0, x); NaN propagates below
        relu = np.where(np.isnan(dots), np.nan, relu)
        s = relu @ w                            # [L]
    return np.where(_fp32_finite(s), s, -np.inf)


def indexer_score_causal(q, w, keys, start_pos: int, ratio: int = 4) -> np.ndarray:
    """Positioned variant: keys at or past valid_count = min(L, (start_pos+1)//ratio)
    are masked to -inf (score_mma kernel, valid_count of its one-query loop)."""
    s = indexer_score(q, w, keys)
    valid = min(len(keys), (int(start_pos) + 1) // int(ratio))
    s = s.copy()
    s[valid:] = -np.inf
    return s


# ---------------------------------------------------------------------------
# (2) Deterministic top-k
# deepseek_rows.metal, index_rows_better (the total order), kernels
# deepseek_indexer_topk_block/merge/finalize_rows_i32: best `width` indices,
# score descending then lower index first; non-finite scores never selected;
# unfilled slots are -1.
# ---------------------------------------------------------------------------

def topk(scores: np.ndarray, width: int) -> np.ndarray:
    """First `width` indices of the finite scores ordered by (-score, index).

    Slots beyond the number of finite scores hold -1. int32 [width].
    """
    s = np.asarray(scores, np.float64)
    cand = np.nonzero(_fp32_finite(s))[0]
    # lexsort: last key is primary. -s ascending == s descending (-0.0 and
    # +0.0 compare equal, so they tie and fall back to the index).
    order = cand[np.lexsort((cand, -s[cand]))]
    out = np.full(int(width), -1, dtype=np.int32)
    n = min(int(width), len(order))
    out[:n] = order[:n]
    return out


def topk_causal(scores, start_pos: int, offset: int = 0, ratio: int = 4,
                width: int = TOP_K) -> np.ndarray:
    """topk_finalize: slot < min(valid_count, 512) and a filled index -> index + offset,
    else -1; valid_count = min(kv_len, (start_pos + 1) // ratio)."""
    s = np.asarray(scores, np.float64).copy()
    valid = min(len(s), (int(start_pos) + 1) // int(ratio))
    s[valid:] = -np.inf
    idx = topk(s, width)
    out = np.full(int(width), -1, np.int32)
    for slot in range(int(width)):
        if slot < min(valid, width) and idx[slot] >= 0:
            out[slot] = idx[slot] + int(offset)
    return out


def indexer_topk_queries(q, w, keys, start_pos: int, offset: int = 0, ratio: int = 4,
                         width: int = TOP_K) -> Tuple[np.ndarray, np.ndarray]:
    """Several consecutive queries of one row (the score kernel's query loop,
    deepseek_indexer_score_mma_rows_bf16): query j (q[j], w[j]) sits at position
    start_pos + j, so its causal count is min(L, (start_pos + j + 1) // ratio).
    Reading for the selection: each query takes its own top-`width` with the
    finalize rule at its own count (the pages' top-k kernels take query 0 only).
    Returns scores [Q, L] and indices int32 [Q, width]."""
    q = np.asarray(q, np.float64)
    w = np.asarray(w, np.float64)
    nq = q.shape[0]
    scores = np.empty((nq, len(keys)))
    out = np.empty((nq, int(width)), np.int32)
    for j in range(nq):
        scores[j] = indexer_score_causal(q[j], w[j], keys, int(start_pos) + j, ratio)
        out[j] = topk_causal(scores[j], int(start_pos) + j, offset, ratio, width)
    return scores, out


# ---------------------------------------------------------------------------
# (3)+(4) Gather and sink-softmax sparse attention
# deepseek_rows.metal, "Sparse attention (selected shared-KV rows with learned
# sinks)", kernels deepseek_sparse_attention_score_rows_bf16 and
# deepseek_sparse_attention_reduce_rows_bf16.
# ---------------------------------------------------------------------------

def sparse_attention(q: np.ndarray, kv: np.ndarray, indices: np.ndarray,
                     sinks: np.ndarray, scale: float) -> Tuple[np.ndarray, np.ndarray]:
    """Sink-softmax attention of each head over the selected KV rows.

    q [H, F], kv [L, F] (float64), indices int [W], sinks [H], scale > 0.
    Returns (out [H, F] float64, invalid [H] bool).

    Per head h (score kernel, then reduce kernel):
      slot t with index -1 is skipped (logit -inf, no value);
      an index < -1 or >= L poisons every head (its logit is NaN);
      a non-finite q[h] or KV element on a selected row poisons the head;
      logit l_t = scale * q[h] . kv[idx_t]; an overflowed logit poisons it;
      m = max(sink_h, max_t l_t); den = exp(sink_h - m) + sum_t exp(l_t - m);
      out[h] = sum_t exp(l_t - m) * kv[idx_t] / den.
    A poisoned head, a non-finite sink, a non-finite max or den <= 0 gives a
    zero head ("fail closed"); a non-finite output element is zeroed alone.
    """
    q = np.asarray(q, np.float64)
    kv = np.asarray(kv, np.float64)
    sinks = np.asarray(sinks, np.float64)
    idx = np.asarray(indices, np.int64)
    H, F = q.shape
    L = kv.shape[0]
    out = np.zeros((H, F), np.float64)
    invalid = np.zeros(H, bool)

    bad_index = bool(np.any((idx < -1) | (idx >= L)))
    live = idx[(idx >= 0) & (idx < L)]              # selected rows, slot order
    rows = kv[live] if len(live) else np.zeros((0, F))
    rows_finite = bool(np.all(np.isfinite(rows)))
    with np.errstate(invalid="ignore", over="ignore"):
        for h in range(H):
            sink = sinks[h]
            if not _fp32_finite(sink) or bad_index:
                invalid[h] = True
                continue
            if len(live) and (not rows_finite or not np.all(np.isfinite(q[h]))):
                invalid[h] = True
                continue
            logits = scale * (rows @ q[h])                 # [W_live]
            if not np.all(_fp32_finite(logits)):
                invalid[h] = True
                continue
            m = max(sink, float(np.max(logits))) if len(logits) else sink
            e = np.exp(logits - m)
            den = math.exp(sink - m) + float(np.sum(e))
            if not (_fp32_finite(den) and den > 0.0):
                invalid[h] = True
                continue
            o = (e @ rows) / den if len(live) else np.zeros(F)
            out[h] = np.where(_fp32_finite(o), o, 0.0)
    return out, invalid


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 (ties to even); float64 result.

    bf16 keeps 8 significant bits: the spacing at |x| in [2^e, 2^(e+1)) is
    2^(e-7). Used only to display the oracle's result at the output type.
    """
    x = np.asarray(x, np.float64)
    out = np.zeros_like(x)
    nz = (x != 0) & np.isfinite(x)
    e = np.floor(np.log2(np.abs(x[nz])))
    e = np.maximum(e, -126.0)                      # bf16 subnormal spacing 2^-133
    ulp = np.exp2(e - 7.0)
    out[nz] = np.rint(x[nz] / ulp) * ulp           # rint: ties to even
    out[~np.isfinite(x)] = x[~np.isfinite(x)]
    return out


# ---------------------------------------------------------------------------
# (5) Learned KV compressor, one decode token per row
# deepseek_rows.metal, kernel deepseek_compressor_rows_bf16 (the append
# branch of deepseek_compressor_bf16 at one token, no cache write), dispatched
# by dispatch_deepseek_compressor_rows.
# ---------------------------------------------------------------------------

COMPRESSOR_SHAPES = ((4, 128), (4, 512), (128, 512))  # supported (ratio, head_dim)


def compress_kv(kv, score, ape, norm, kv_state, score_state, start_pos: int, ratio: int, head_dim: int,
                eps: float):
    """One token of the learned KV compressor for one row.

    With coff = 2 when ratio == 4 (overlapping windows) and 1 otherwise, and
    P = coff * head_dim features per token:
      kv, score  fp32 [P]           the token's projected values and scores
      ape        fp32 [ratio, P]    position bias added to the score
      norm       fp32 [head_dim]    RMSNorm weight
      kv_state, score_state  fp32 [coff * ratio, P]  the row's window (not modified)
    Returns (out [head_dim] float64 holding bf16 values, new kv_state, new score_state).

    The state is kept in fp32 as the pages keep it (the score + ape sum is an
    fp32 add); the pooling and the norm run in float64, with the pages' bf16
    rounding of the pooled value and of the output.
    1. The token (position start_pos, token = start_pos mod ratio) is written
       to state row (ratio if overlapping else 0) + token: its kv (0 where not
       finite) and score + ape (NaN where either is not finite).
    2. When start_pos + 1 is a multiple of ratio the block is complete: each
       feature f softmax-pools the window's values with its scores over the
       window's rows (2 ratio rows when overlapping: the first ratio rows read
       feature f, the last ratio rows feature head_dim + f), the pooled value
       is rounded to bf16, and the row is RMS-normalised and scaled by norm:
         out = bf16(c * norm / sqrt(mean(c^2) + eps)).
       A NaN or +inf score, a non-finite value, pooled value or norm, or a
       non-finite sum or result zeroes the whole row ("fail closed").
       Overlapping windows then move the current block into the previous rows
       (whether or not the row was zeroed).
    3. Otherwise the output is zero.
    """
    ratio, head_dim = int(ratio), int(head_dim)
    overlap = ratio == 4
    coff = 2 if overlap else 1
    proj = coff * head_dim
    kv32 = np.asarray(kv, np.float32).reshape(proj)
    with np.errstate(invalid="ignore", over="ignore"):
        s32 = np.asarray(score, np.float32).reshape(proj) + np.asarray(ape, np.float32).reshape(ratio, proj)[
            int(start_pos) % ratio]
    kv_new = np.array(kv_state, np.float32).reshape(coff * ratio, proj)
    sc_new = np.array(score_state, np.float32).reshape(coff * ratio, proj)
    slot = (ratio if overlap else 0) + int(start_pos) % ratio
    v_ok = np.isfinite(kv32)
    kv_new[slot] = np.where(v_ok, kv32, np.float32(0.0))
    sc_new[slot] = np.where(v_ok & np.isfinite(s32), s32, np.float32(np.nan))

    out = np.zeros(head_dim)
    if (int(start_pos) + 1) % ratio != 0:
        return out, kv_new, sc_new

    items = coff * ratio
    feat = np.arange(head_dim)
    # Row i of the window reads feature f, or head_dim + f for the current block
    # of an overlapping window.
    src = np.where((np.arange(items)[:, None] >= ratio) & overlap, head_dim + feat[None, :], feat[None, :])
    S = sc_new.astype(np.float64)[np.arange(items)[:, None], src]   # [items, head_dim]
    V = kv_new.astype(np.float64)[np.arange(items)[:, None], src]
    nrm = np.asarray(norm, np.float64).reshape(head_dim)
    bad = np.isnan(S).any(0) | (S == np.inf).any(0) | ~np.isfinite(V).all(0)
    with np.errstate(invalid="ignore", over="ignore", divide="ignore"):
        m = np.max(np.where(np.isnan(S), -np.inf, S), axis=0)
        w = np.exp(S - m[None, :])
        pooled = (w * V).sum(0) / w.sum(0)
    bad |= ~_fp32_finite(pooled) | ~np.isfinite(nrm)
    c = round_bf16(np.where(_fp32_finite(pooled), pooled, 0.0))
    ss = float(np.sum(c * c))
    if not bad.any() and _fp32_finite(ss):
        scale = 1.0 / math.sqrt(ss / head_dim + float(eps))
        with np.errstate(invalid="ignore", over="ignore"):
            y = c * scale * nrm
        if math.isfinite(scale) and _fp32_finite(y).all():
            out = round_bf16(y)
    if overlap:
        kv_new[:ratio] = kv_new[ratio:].copy()
        sc_new[:ratio] = sc_new[ratio:].copy()
    return out, kv_new, sc_new


# ---------------------------------------------------------------------------
# The whole decode step over a row table
# ---------------------------------------------------------------------------

def decode_row(qI, wI, keys, qA, kv, sinks, scale, width) -> Dict[str, np.ndarray]:
    """One row: scores -> top-width indices -> sink attention (all float64)."""
    s = indexer_score(qI, wI, keys)
    idx = topk(s, width)
    out, invalid = sparse_attention(qA, kv, idx, sinks, scale)
    return {"scores": s, "indices": idx, "out": out, "invalid": invalid}


def decode(workload, entries=None) -> List[Dict[str, np.ndarray]]:
    """Run `decode_row` for each table entry of a `workloads.Workload`.

    Caches are decoded one row at a time; only the selected KV rows are
    widened to float64.
    """
    res = []
    ents = range(workload.num_rows) if entries is None else entries
    for e in ents:
        r = workload.rows[e]
        qI = bf16_to_f64(workload.q_index[r.q_row])
        wI = np.asarray(workload.w_index[r.q_row], np.float64)
        keys = bf16_to_f64(workload.keys[e][: r.kv_len])
        s = indexer_score(qI, wI, keys)
        idx = topk(s, r.width)
        kv = _LazyRows(workload.kv[e], r.kv_len)
        qA = bf16_to_f64(workload.q_attn[r.q_row])
        out, invalid = sparse_attention_rows(qA, kv, idx, workload.row_sinks(e), workload.scale)
        res.append({"scores": s, "indices": idx, "out": out, "invalid": invalid})
    return res


class _LazyRows:
    """A bf16 [L, F] cache viewed as float64 rows on demand (avoids widening all of it)."""

    def __init__(self, bits, L):
        self.bits = bits
        self.L = int(L)
        self.shape = (self.L, bits.shape[1])

    def take(self, idx):
        return bf16_to_f64(self.bits[np.asarray(idx, np.int64)])


def sparse_attention_rows(q, kv_rows: "_LazyRows", indices, sinks, scale):
    """`sparse_attention` on a lazily widened cache: only in-range selected rows
    are read; the rest of the rule set is identical."""
    idx = np.asarray(indices, np.int64)
    L = kv_rows.L
    ok = (idx >= 0) & (idx < L)
    # Build a compact cache of the rows referenced, re-indexed in slot order.
    uniq, inv = np.unique(idx[ok], return_inverse=True)
    compact = kv_rows.take(uniq) if len(uniq) else np.zeros((0, kv_rows.shape[1]))
    remap = idx.copy()
    remap[ok] = inv
    # Out-of-range indices keep their "bad" status against the compact length.
    remap[~ok & (idx != -1)] = -2
    return sparse_attention(q, compact, remap, sinks, scale)
