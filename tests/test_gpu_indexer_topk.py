"""GPU parity of the positioned indexer + causal top-512 (ds_rows_indexer_topk)
against the CPU oracle (indexer_score_causal, topk_causal), through the C-ABI.

Positions are chosen so that every case of the finalize rule appears: all keys
valid, a causal cut inside the cache, fewer than 512 valid keys (-1 fill), no
valid key at all, and offsets added to the emitted indices.
"""

import functools

import numpy as np
import pytest
import torch

import deepseek_sparse_attention_ragged_gb300 as ds
import oracle
import workloads
from workloads.device import to_device

from parity import check_topk, score_bound

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    ds.build()
    ds.load()


@functools.lru_cache(maxsize=None)
def cfg(i):
    return workloads.config(i)


@functools.lru_cache(maxsize=None)
def cfg_dev(i):
    return to_device(cfg(i), "cuda")


def positioned_rows(wl, valid, offsets):
    """IndexerRow per entry: start_pos = 4 valid - 1 (valid 0: start_pos 2)."""
    rows = []
    for e, r in enumerate(wl.rows):
        v = valid[e]
        start = 4 * v - 1 if v > 0 else 2
        rows.append(ds.IndexerRow(r.kv_len, start, offsets[e], r.q_row, 512 * e))
    return rows


def run(wl, dev, rows, entries=None):
    entries = list(range(len(rows))) if entries is None else entries
    out = torch.full((512 * len(wl.rows),), -7, dtype=torch.int32, device="cuda")
    sel = [rows[e] for e in entries]
    ws = ds.indexer_topk_workspace(sel, "cuda")
    ds.ds_rows_indexer_topk(sel, dev.q_index, dev.w_index, [dev.keys[e] for e in entries], out, workspace_t=ws)
    torch.cuda.synchronize()
    assert ds.workspace_status(ws) == 0
    return out.cpu().numpy()


def reference(wl, e, row):
    r = wl.rows[e]
    q = oracle.bf16_to_f64(wl.q_index[r.q_row])
    w = wl.w_index[r.q_row].astype(np.float64)
    keys = oracle.bf16_to_f64(wl.keys[e])
    s = oracle.indexer_score_causal(q, w, keys, row.start_pos)
    return s, oracle.topk_causal(s, row.start_pos, offset=row.offset), score_bound(q, w, keys)


def test_integer_config_bit_exact():
    # kv_len 300, 512, 1000, 4096: all valid (< 512: -1 fill), none valid, a cut, all valid.
    wl, dev = cfg(1), cfg_dev(1)
    rows = positioned_rows(wl, [300, 0, 600, 4096], [5, 0, 1000, 123456])
    got = run(wl, dev, rows)
    for e, row in enumerate(rows):
        _, ref, _ = reference(wl, e, row)
        np.testing.assert_array_equal(got[512 * e: 512 * e + 512], ref, err_msg=f"row {e}")
    assert (got[512:1024] == -1).all()  # no valid key
    assert (got[300:512] == -1).all() and (got[:300] >= 5).all()


def test_float_config_near_ties_only():
    wl, dev = cfg(2), cfg_dev(2)
    lens = [r.kv_len for r in wl.rows]
    valid = [lens[0], lens[1] // 3, 513, 511, lens[4], 1, lens[6] - 1, 2048]
    offs = [0, 17, 4096, 0, 99999, 3, 0, 1 << 20]
    rows = positioned_rows(wl, valid, offs)
    got = run(wl, dev, rows)
    for e, row in enumerate(rows):
        s, ref, T = reference(wl, e, row)
        g = got[512 * e: 512 * e + 512].astype(np.int64)
        # Slots past the valid keys are -1; filled slots carry the offset.
        n = min(valid[e], 512)
        assert (g[n:] == -1).all(), f"row {e}: fill"
        assert (g[:n] >= row.offset).all(), f"row {e}: offset"
        g0 = np.where(g >= 0, g - row.offset, -1)
        r0 = np.where(ref >= 0, ref.astype(np.int64) - row.offset, -1)
        assert (g0[:n] < valid[e]).all(), f"row {e}: index past the causal count"
        check_topk(g0, r0, s, 512, T=T, what=f"row {e}")


def test_joint_equals_single_row():
    wl, dev = cfg(2), cfg_dev(2)
    lens = [r.kv_len for r in wl.rows]
    rows = positioned_rows(wl, [l // 2 + 7 for l in lens], [e * 1000 for e in range(8)])
    joint = run(wl, dev, rows)
    for e in range(8):
        single = run(wl, dev, rows, entries=[e])  # writes at the row's own output_offset
        np.testing.assert_array_equal(single[512 * e: 512 * e + 512], joint[512 * e: 512 * e + 512],
                                      err_msg=f"row {e}")


def test_all_valid_equals_unpositioned_stages():
    """With every key valid and offset 0, the positioned call is bitwise the
    indexer-score + top-k stages (same scores, same selection)."""
    wl, dev = cfg(2), cfg_dev(2)
    rows = positioned_rows(wl, [r.kv_len for r in wl.rows], [0] * 8)
    got = run(wl, dev, rows)
    stride = max(r.kv_len for r in wl.rows)
    scores = torch.empty((wl.num_rows, stride), dtype=torch.float32, device="cuda")
    ds.ds_rows_indexer_score(dev.rows, dev.q_index, dev.w_index, dev.keys, scores, stride)
    idx = torch.full((wl.index_elements,), -7, dtype=torch.int32, device="cuda")
    ds.ds_rows_topk(dev.rows, scores, stride, idx, ds.workspace(dev.rows))
    torch.cuda.synchronize()
    ref = idx.cpu().numpy()
    for e, r in enumerate(wl.rows):
        np.testing.assert_array_equal(got[512 * e: 512 * e + r.width],
                                      ref[r.index_offset: r.index_offset + r.width], err_msg=f"row {e}")
