"""GPU parity of the multi-query positioned indexer + causal top-512
(ds_rows_indexer_topk_queries) against the CPU oracle (indexer_topk_queries),
through the C-ABI.

Entry e's queries j < Q use query rows e*Q + j and positions start_pos + j, so
their causal counts step inside a run; runs of 1-4 queries share key tiles on
the tensor cores, and Q = 5, 8, 12 cross from one run of four to the next.
"""

import functools

import numpy as np
import pytest
import torch

import deepseek_sparse_attention_ragged_gb300 as ds
import oracle
import workloads
from workloads.device import bf16_tensor, to_device

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


@functools.lru_cache(maxsize=None)
def queries(i, count, seed):
    qI, wI = workloads.draw_index_queries(cfg(i), seed, count)
    return qI, wI, bf16_tensor(qI, "cuda"), torch.from_numpy(np.ascontiguousarray(wI)).to("cuda")


def table(wl, Q, starts, offsets):
    return [ds.IndexerRow(r.kv_len, starts[e], offsets[e], e * Q, 512 * Q * e) for e, r in enumerate(wl.rows)]


def run(i, Q, rows, seed, entries=None):
    wl, dev = cfg(i), cfg_dev(i)
    _, _, q, w = queries(i, len(wl.rows) * Q, seed)
    entries = list(range(len(rows))) if entries is None else entries
    out = torch.full((512 * Q * len(wl.rows),), -7, dtype=torch.int32, device="cuda")
    sub = [rows[e] for e in entries]
    ws = ds.indexer_topk_workspace(sub, "cuda", Q)
    ds.ds_rows_indexer_topk_queries(sub, Q, q, w, [dev.keys[e] for e in entries], out, workspace_t=ws)
    torch.cuda.synchronize()
    assert ds.workspace_status(ws) == 0
    return out.cpu().numpy().reshape(len(wl.rows), Q, 512)


def reference(i, Q, e, row, seed):
    wl = cfg(i)
    qI, wI, _, _ = queries(i, len(wl.rows) * Q, seed)
    q = oracle.bf16_to_f64(qI[e * Q: e * Q + Q])
    w = wI[e * Q: e * Q + Q].astype(np.float64)
    keys = oracle.bf16_to_f64(wl.keys[e])
    s, idx = oracle.indexer_topk_queries(q, w, keys, row.start_pos, offset=row.offset)
    return s, idx, [score_bound(q[j], w[j], keys) for j in range(Q)]


@pytest.mark.parametrize("Q", [2, 3, 4, 5, 8, 12])
def test_integer_config_bit_exact(Q):
    # kv_len 300, 512, 1000, 4096. Counts: all valid, none then one valid,
    # a cut stepping across the 128-key tile edge (127..129), a cut deep inside.
    wl = cfg(1)
    starts = [4 * 300 - Q, 2, 507, 4 * 3000 - 1]
    rows = table(wl, Q, starts, [5, 0, 1000, 123456])
    got = run(1, Q, rows, seed=500 + Q)
    for e, row in enumerate(rows):
        _, ref, _ = reference(1, Q, e, row, 500 + Q)
        np.testing.assert_array_equal(got[e], ref, err_msg=f"row {e}")


@pytest.mark.parametrize("Q", [3, 8])
def test_float_config_near_ties_only(Q):
    wl = cfg(2)
    lens = [r.kv_len for r in wl.rows]
    starts = [4 * lens[0] - Q, 4 * (lens[1] // 3), 4 * 513 - 2, 4 * 511, 4 * lens[4] - Q - 40, 3,
              4 * lens[6] - Q, 4 * 2048 + 1]
    offs = [0, 17, 4096, 0, 99999, 3, 0, 1 << 20]
    rows = table(wl, Q, starts, offs)
    got = run(2, Q, rows, seed=600 + Q)
    for e, row in enumerate(rows):
        s, ref, T = reference(2, Q, e, row, 600 + Q)
        for j in range(Q):
            valid = min(row.kv_len, (row.start_pos + j + 1) // 4)
            g = got[e, j].astype(np.int64)
            n = min(valid, 512)
            assert (g[n:] == -1).all(), f"row {e} query {j}: fill"
            assert (g[:n] >= row.offset).all(), f"row {e} query {j}: offset"
            g0 = np.where(g >= 0, g - row.offset, -1)
            r0 = np.where(ref[j] >= 0, ref[j].astype(np.int64) - row.offset, -1)
            assert (g0[:n] < valid).all(), f"row {e} query {j}: index past the causal count"
            check_topk(g0, r0, s[j], 512, T=T[j], what=f"row {e} query {j}")


@pytest.mark.parametrize("Q", [4, 5])
def test_each_query_equals_the_one_query_call(Q):
    """Query j of the multi-query call is bitwise the positioned indexer of
    start_pos + j on query row q_row + j: a query's scores do not depend on
    the other queries that share its key tiles."""
    wl, dev = cfg(2), cfg_dev(2)
    lens = [r.kv_len for r in wl.rows]
    starts = [2 * l + 11 for l in lens]
    rows = table(wl, Q, starts, [e * 1000 for e in range(8)])
    got = run(2, Q, rows, seed=700 + Q)
    _, _, q, w = queries(2, len(wl.rows) * Q, 700 + Q)
    for j in range(Q):
        one = [ds.IndexerRow(r.kv_len, r.start_pos + j, r.offset, r.q_row + j, 512 * e)
               for e, r in enumerate(rows)]
        out = torch.full((512 * len(wl.rows),), -7, dtype=torch.int32, device="cuda")
        ws = ds.indexer_topk_workspace(one, "cuda")
        ds.ds_rows_indexer_topk(one, q, w, dev.keys, out, workspace_t=ws)
        torch.cuda.synchronize()
        assert ds.workspace_status(ws) == 0
        single = out.cpu().numpy().reshape(len(wl.rows), 512)
        np.testing.assert_array_equal(got[:, j], single, err_msg=f"query {j}")


def test_joint_equals_single_row_and_full_table():
    # 8 rows x 8 queries: 64 (row, query) pairs, the most one call takes.
    wl = cfg(2)
    Q = 8
    lens = [r.kv_len for r in wl.rows]
    rows = table(wl, Q, [l + 3 for l in lens], [7] * 8)
    joint = run(2, Q, rows, seed=800)
    for e in (0, 5):
        single = run(2, Q, rows, seed=800, entries=[e])  # writes at the row's own output_offset
        np.testing.assert_array_equal(single[e], joint[e], err_msg=f"row {e}")
