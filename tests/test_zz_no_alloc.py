"""The workspace-free top-k entry point, checked against the ordinary one.

ds_rows_topk_static exists for callers that cannot allocate device memory when
they run the top-k stage (allocation-free graph or real-time code, or code that
cannot reach the device allocator). It keeps its scratch in one array inside
the library, so these tests call it twice in a row, on different scores, to
show that each call starts from a clean state. They compare every result with
ds_rows_topk through the C-ABI, and with the oracle's stable sort on scores
with exact ties and non-finite values; the indices are integers, so they must
be equal. The status word it keeps in the library reads 0 after each call. One
test captures the call in a CUDA graph and replays it on new scores.

This file sorts last so that a run stopping at the first failure has already
run every other test.
"""

import numpy as np
import pytest
import torch

import deepseek_sparse_attention_ragged_gb300 as ds
import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    ds.build()
    ds.load()


def _scores(seed, lens, **kw):
    rows_s = workloads.random_scores(seed, lens, **kw)
    stride = max(lens)
    host = np.full((len(lens), stride), np.nan, np.float32)
    for e, s in enumerate(rows_s):
        host[e, : len(s)] = s
    return torch.from_numpy(host).cuda(), stride


def test_static_scratch_topk_matches_workspace_topk_twice():
    lens = [131072, 40000, 513, 1, 9000, 70000, 2048, 300]
    rows = [workloads.Row(L, min(512, L), 512 * e, e) for e, L in enumerate(lens)]
    ws = ds.workspace(rows)
    for call, kw in enumerate([dict(), dict(ties=True, nonfinite=True)]):
        scores, stride = _scores(71 + call, lens, **kw)
        want = torch.full((512 * len(lens),), -7, dtype=torch.int32, device="cuda")
        got = torch.full_like(want, -9)
        ds.ds_rows_topk(rows, scores, stride, want, ws)
        ds.ds_rows_topk_static(rows, scores, stride, got)
        assert ds.topk_static_status() == 0
        assert ds.workspace_status(ws) == 0
        for r in rows:
            sl = slice(r.index_offset, r.index_offset + r.width)
            assert torch.equal(got[sl], want[sl]), f"call {call}, row kv_len {r.kv_len}"


def test_static_scratch_topk_matches_the_oracle_twice():
    lens = [4096, 1000, 512, 300, 1]
    rows = [workloads.Row(L, min(512, L), 512 * e, e) for e, L in enumerate(lens)]
    for call in range(2):
        scores, stride = _scores(91 + call, lens, ties=True, nonfinite=True)
        got = torch.full((512 * len(lens),), -9, dtype=torch.int32, device="cuda")
        ds.ds_rows_topk_static(rows, scores, stride, got)
        assert ds.topk_static_status() == 0
        host, g = scores.cpu().numpy(), got.cpu().numpy()
        for e, r in enumerate(rows):
            want = oracle.topk(host[e, : r.kv_len], r.width)
            np.testing.assert_array_equal(g[r.index_offset: r.index_offset + r.width], want,
                                          err_msg=f"call {call}, row kv_len {r.kv_len}")


def test_static_scratch_topk_replays_from_a_cuda_graph():
    """The stated use: a warm-up call (it looks up the array), then the call
    captured in a CUDA graph and replayed after the scores change in place.
    Each replay's indices equal the oracle's, and the status reads 0."""
    lens = [70000, 4096, 513, 300]
    rows = [workloads.Row(L, min(512, L), 512 * e, e) for e, L in enumerate(lens)]
    scores, stride = _scores(101, lens, ties=True, nonfinite=True)
    got = torch.full((512 * len(lens),), -9, dtype=torch.int32, device="cuda")
    ds.ds_rows_topk_static(rows, scores, stride, got)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        ds.ds_rows_topk_static(rows, scores, stride, got)
    for seed in (102, 103):
        new, _ = _scores(seed, lens, ties=seed == 103, nonfinite=seed == 103)
        scores.copy_(new)
        got.fill_(-9)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert ds.topk_static_status() == 0
        host, g = scores.cpu().numpy(), got.cpu().numpy()
        for e, r in enumerate(rows):
            want = oracle.topk(host[e, : r.kv_len], r.width)
            np.testing.assert_array_equal(g[r.index_offset: r.index_offset + r.width], want,
                                          err_msg=f"replay with seed {seed}, row kv_len {r.kv_len}")


def test_static_scratch_topk_rejects_too_many_rows():
    rows = [workloads.Row(16, 16, 16 * e, e) for e in range(9)]
    scores = torch.zeros((9, 16), dtype=torch.float32, device="cuda")
    idx = torch.zeros((9 * 16,), dtype=torch.int32, device="cuda")
    with pytest.raises(ds.DsRowsError, match="rows must be 1..=8"):
        ds.ds_rows_topk_static(rows, scores, 16, idx)
