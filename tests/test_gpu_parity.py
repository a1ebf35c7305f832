"""GPU parity: every stage and the fused decode step against the CPU oracle,
through the C-ABI, on the five benchmark workloads and stand-alone stage inputs.
"""

import dataclasses
import functools

import numpy as np
import pytest
import torch

import deepseek_sparse_attention_ragged_gb300 as ds
import oracle
import workloads
from workloads.device import bf16_tensor, to_device

from parity import (check_out, check_scores, check_topk, check_topk_consistent, score_bound)

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
def cfg_ref(i):
    return oracle.decode(cfg(i))


def _row_inputs(wl, e):
    r = wl.rows[e]
    q = oracle.bf16_to_f64(wl.q_index[r.q_row])
    w = wl.w_index[r.q_row].astype(np.float64)
    keys = oracle.bf16_to_f64(wl.keys[e])
    return q, w, keys


def run_decode(dev, rows=None, indices=True, invalid=True, stream=None):
    """The decode of `rows` (all of dev's by default) into NaN-, -7- and
    7-filled out, indices and invalid buffers; the workspace's status word must
    read 0 afterwards (no bounded wait gave up, no selection check failed)."""
    rows = dev.rows if rows is None else rows
    nq = max(r.q_row for r in dev.rows) + 1
    out = torch.full((nq, 64, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    n_idx = max(r.index_offset + r.width for r in dev.rows)
    idx = torch.full((n_idx,), -7, dtype=torch.int32, device="cuda") if indices else None
    inv = torch.full((nq, 64), 7, dtype=torch.int32, device="cuda") if invalid else None
    keys = [dev.keys[dev.rows.index(r)] for r in rows]
    kv = [dev.kv[dev.rows.index(r)] for r in rows]
    ws = ds.workspace(rows)
    ds.ds_rows_decode(rows, dev.q_index, dev.w_index, keys, dev.q_attn, kv, dev.sinks, dev.sinks_row_stride,
                      dev.scale, out, indices=idx, invalid=inv, workspace_t=ws, stream=stream)
    torch.cuda.synchronize()
    assert ds.workspace_status(ws) == 0
    return out, idx, inv


def untouched_indices(idx, rows):
    """Every index slot outside the rows' [index_offset, index_offset + width)
    ranges still holds the -7 fill (no write past a row's width)."""
    mask = np.ones(idx.shape[0], bool)
    for r in rows:
        mask[r.index_offset: r.index_offset + r.width] = False
    return np.all(idx[mask] == -7)


# ---------------------------------------------------------------------------
# (1) indexer scores
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("i", [0, 1, 2, 3, 4])
def test_indexer_scores(i):
    wl, dev = cfg(i), cfg_dev(i)
    stride = max(r.kv_len for r in wl.rows)
    scores = torch.full((wl.num_rows, stride), float("nan"), dtype=torch.float32, device="cuda")
    ds.ds_rows_indexer_score(dev.rows, dev.q_index, dev.w_index, dev.keys, scores, stride)
    torch.cuda.synchronize()
    got = scores.cpu().numpy()
    for e, r in enumerate(wl.rows):
        q, w, keys = _row_inputs(wl, e)
        ref = cfg_ref(i)[e]["scores"]
        check_scores(got[e, : r.kv_len], ref, score_bound(q, w, keys), exact=wl.integer_valued,
                     what=f"cfg{i} row{e}")
        assert np.isnan(got[e, r.kv_len:]).all(), "wrote past kv_len"


# ---------------------------------------------------------------------------
# (2) top-k on generated scores (bit-exact: fp32 inputs, exact comparisons)
# ---------------------------------------------------------------------------

TOPK_CASES = {
    "normal": dict(lens=[1, 17, 511, 512, 513, 8191, 8193, 40000], kw={}),
    "ties": dict(lens=[300, 1000, 9000, 70000], kw=dict(ties=True)),
    "nonfinite": dict(lens=[20, 600, 9000, 33000], kw=dict(nonfinite=True)),
    "zeros": dict(lens=[513, 5000, 16385], kw=dict(signed_zeros=True, ties=True)),
    "long": dict(lens=[262144, 131072, 3], kw={}),
    # The threshold bin holds m candidates: held in registers, 4, 5, 9 or 12
    # per thread (m <= 2048, 2560, 4608, 6144), then refined from the gathered
    # candidates and sorted by index (m > 6144), and refined from the full row
    # (one CTA's slice has more than 2048).
    "crowded": dict(lens=[20000, 40000, 50000, 60000, 100000, 120000, 70000, 30000],
                    kw=dict(crowd=(1500, 3000, 3800, 5000, 10000, 60000, 4500, 2400))),
}


def _bin_of_120(L, seed):
    """Scores whose 512th best falls among 120 distinct values that share the
    top 22 bits of their order key (1.0f plus 0..119 ulps): the refinement
    ends with a threshold bin of 120 elements, ranked directly."""
    rng = np.random.default_rng(seed)
    s = -1.0 - rng.random(L).astype(np.float32)          # far below
    top = rng.permutation(L)[:450 + 120]
    s[top[:450]] = 10.0 + rng.random(450).astype(np.float32)  # certain winners
    s[top[450:]] = (np.uint32(0x3F800000) + rng.permutation(120).astype(np.uint32)).view(np.float32)
    return s


def test_topk_direct_ranking_of_a_full_bin():
    lens = [4096, 70000]
    rows = [workloads.Row(L, 512, 512 * e, e) for e, L in enumerate(lens)]
    stride = max(lens)
    host = np.full((len(lens), stride), np.nan, np.float32)
    for e, L in enumerate(lens):
        host[e, :L] = _bin_of_120(L, 7 + e)
    scores = torch.from_numpy(host).cuda()
    idx = torch.full((512 * len(lens),), -7, dtype=torch.int32, device="cuda")
    ws = ds.workspace(rows)
    ds.ds_rows_topk(rows, scores, stride, idx, ws)
    torch.cuda.synchronize()
    assert ds.workspace_status(ws) == 0
    got = idx.cpu().numpy()
    for e, L in enumerate(lens):
        want = oracle.topk(host[e, :L], 512)
        np.testing.assert_array_equal(got[512 * e: 512 * e + 512], want, err_msg=f"row {e}")


@pytest.mark.parametrize("case", sorted(TOPK_CASES))
def test_topk_exact(case):
    spec = TOPK_CASES[case]
    lens = spec["lens"]
    rows = [workloads.Row(L, min(512, L), 512 * e, e) for e, L in enumerate(lens)]
    rows_s = workloads.random_scores(31 + len(case), lens, **spec["kw"])
    stride = max(lens)
    host = np.full((len(lens), stride), np.nan, np.float32)
    for e, s in enumerate(rows_s):
        host[e, : len(s)] = s
    scores = torch.from_numpy(host).cuda()
    idx = torch.full((512 * len(lens),), -7, dtype=torch.int32, device="cuda")
    ws = ds.workspace(rows)
    ds.ds_rows_topk(rows, scores, stride, idx, ws)
    torch.cuda.synchronize()
    assert ds.workspace_status(ws) == 0
    got = idx.cpu().numpy()
    for e, r in enumerate(rows):
        ref = oracle.topk(rows_s[e].astype(np.float64), r.width)
        np.testing.assert_array_equal(got[r.index_offset: r.index_offset + r.width], ref, err_msg=f"row {e}")
    assert untouched_indices(got, rows)


def test_topk_equal_scores_slow_path():
    """All-equal scores on a row longer than the candidate list: the threshold bin
    overflows, the row is refined from its full score array, and the lowest
    indices win."""
    lens = [40000, 70000]
    rows = [workloads.Row(L, 512, 512 * e, e) for e, L in enumerate(lens)]
    host = np.full((2, 70000), 1.5, np.float32)
    host[1, 12345] = 2.0
    host[1, 50000:50010] = np.nan
    scores = torch.from_numpy(host).cuda()
    idx = torch.full((1024,), -7, dtype=torch.int32, device="cuda")
    ds.ds_rows_topk(rows, scores, 70000, idx, ds.workspace(rows))
    got = idx.cpu().numpy()
    np.testing.assert_array_equal(got[:512], np.arange(512))
    np.testing.assert_array_equal(got[512:], oracle.topk(host[1].astype(np.float64), 512))


def test_topk_fewer_finite_than_width():
    L = 700
    s = np.full(L, -np.inf, np.float32)
    s[[5, 600, 33]] = [1.0, 3.0, 1.0]
    rows = [workloads.Row(L, 512, 0, 0)]
    idx = torch.full((512,), -7, dtype=torch.int32, device="cuda")
    ds.ds_rows_topk(rows, torch.from_numpy(s).cuda(), L, idx, ds.workspace(rows))
    got = idx.cpu().numpy()
    assert got[:3].tolist() == [600, 5, 33]
    assert np.all(got[3:] == -1)


# ---------------------------------------------------------------------------
# (3)+(4) attention on generated indices
# ---------------------------------------------------------------------------

ATTN_CASES = {
    "unique": dict(sentinel_frac=0.0),
    "sentinels": dict(sentinel_frac=0.3),
    "duplicates": dict(unique=False),
    "bad_rows": dict(sentinel_frac=0.1, bad_rows=(1,)),
}


@pytest.mark.parametrize("case", sorted(ATTN_CASES))
def test_sparse_attn(case):
    wl = workloads.make_workload("attn", 41, [600, 5000, 33, 1], per_row_sinks=True)
    rows = [workloads.Row(r.kv_len, w, r.index_offset, r.q_row) for r, w in zip(wl.rows, [512, 300, 33, 1])]
    dev = to_device(wl)
    idx_h = workloads.random_indices(43, rows, **ATTN_CASES[case])
    idx = torch.from_numpy(idx_h).cuda()
    out = torch.full((4, 64, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    inv = torch.full((4, 64), 7, dtype=torch.int32, device="cuda")
    ws = ds.workspace(rows)
    ds.ds_rows_sparse_attn(rows, dev.q_attn, dev.sinks, 64, idx, dev.scale, out, dev.kv, invalid=inv,
                           workspace_t=ws)
    torch.cuda.synchronize()
    assert ds.workspace_status(ws) == 0
    got = out.float().cpu().numpy()
    ginv = inv.cpu().numpy()
    for e, r in enumerate(rows):
        sel = idx_h[r.index_offset: r.index_offset + r.width]
        ref, rinv = oracle.sparse_attention_rows(oracle.bf16_to_f64(wl.q_attn[r.q_row]),
                                                 oracle._LazyRows(wl.kv[e], r.kv_len), sel,
                                                 wl.sinks[r.q_row], wl.scale)
        np.testing.assert_array_equal(ginv[r.q_row], rinv.astype(np.int32), err_msg=f"row {e} flags")
        check_out(got[r.q_row], ref, what=f"{case} row {e}")


def test_sparse_attn_shared_sinks_and_dense_closed_form():
    """width == kv_len with every row selected and sink -3e38 (exp underflows):
    dense softmax attention; sinks shared (stride 0)."""
    L = 96
    wl = workloads.make_workload("dense", 44, [L], per_row_sinks=False)
    dev = to_device(wl)
    rows = [workloads.Row(L, L, 0, 0)]
    idx = torch.arange(L, dtype=torch.int32, device="cuda")
    sinks = torch.full((64,), -3.0e38, dtype=torch.float32, device="cuda")
    out = torch.empty((1, 64, 512), dtype=torch.bfloat16, device="cuda")
    ds.ds_rows_sparse_attn(rows, dev.q_attn, sinks, 0, idx, dev.scale, out, dev.kv)
    q = oracle.bf16_to_f64(wl.q_attn[0])
    kv = oracle.bf16_to_f64(wl.kv[0])
    logits = wl.scale * q @ kv.T
    p = np.exp(logits - logits.max(axis=1, keepdims=True))
    dense = (p / p.sum(axis=1, keepdims=True)) @ kv
    check_out(out.float().cpu().numpy()[0], dense, what="dense")


# ---------------------------------------------------------------------------
# the fused decode step
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("i", [0, 1, 2, 3, 4])
def test_decode(i):
    wl, dev = cfg(i), cfg_dev(i)
    out, idx, inv = run_decode(dev)
    got = out.float().cpu().numpy()
    gidx = idx.cpu().numpy()
    ginv = inv.cpu().numpy()
    swaps = 0
    for e, r in enumerate(wl.rows):
        ref = cfg_ref(i)[e]
        q, w, keys = _row_inputs(wl, e)
        sel = gidx[r.index_offset: r.index_offset + r.width]
        swaps += check_topk(sel, ref["indices"], ref["scores"], r.width, exact=wl.integer_valued,
                            T=score_bound(q, w, keys), what=f"cfg{i} row{e}")
        if set(sel.tolist()) == set(ref["indices"].tolist()):
            expect, rinv = ref["out"], ref["invalid"]
        else:
            # A near-tie swap (allowed above): the attention of the selected set,
            # already validated against the oracle's scores, is the expected value.
            expect, rinv = oracle.sparse_attention_rows(oracle.bf16_to_f64(wl.q_attn[r.q_row]),
                                                        oracle._LazyRows(wl.kv[e], r.kv_len), sel,
                                                        wl.row_sinks(e), wl.scale)
        np.testing.assert_array_equal(ginv[r.q_row], rinv.astype(np.int32))
        check_out(got[r.q_row], expect, what=f"cfg{i} row{e}")
    assert untouched_indices(gidx, wl.rows), "an index was written outside a row's [offset, offset + width)"
    print(f"cfg{i}: near-tie swaps {swaps}")


@pytest.mark.parametrize("i", [1, 4])
def test_decode_canaries_around_outputs(i):
    """Entries on odd query rows (even rows belong to no entry) and index ranges
    with gaps between them: the gaps keep their -7 fill, the unowned query rows
    of out and invalid keep their NaN and 7 fills, and every entry's results
    are bitwise those of the decode on the workload's own dense layout."""
    wl, dev = cfg(i), cfg_dev(i)
    R = wl.num_rows
    rows = [workloads.Row(r.kv_len, r.width, 640 * e + 7, 2 * e + 1) for e, r in enumerate(wl.rows)]

    def spread(t):
        out = torch.zeros((2 * R,) + tuple(t.shape[1:]), dtype=t.dtype, device="cuda")
        out[1::2] = t
        return out

    sinks = spread(dev.sinks) if dev.sinks_row_stride else dev.sinks
    moved = dataclasses.replace(dev, rows=rows, q_index=spread(dev.q_index), w_index=spread(dev.w_index),
                                q_attn=spread(dev.q_attn), sinks=sinks)
    out, idx, inv = run_decode(moved)
    ref_out, ref_idx, ref_inv = run_decode(dev)
    got_idx = idx.cpu().numpy()
    assert untouched_indices(got_idx, rows)
    for e, (r, r0) in enumerate(zip(rows, wl.rows)):
        assert torch.equal(out[r.q_row].view(torch.int16), ref_out[r0.q_row].view(torch.int16)), f"row {e} out"
        assert torch.equal(inv[r.q_row], ref_inv[r0.q_row]), f"row {e} invalid"
        assert torch.equal(idx[r.index_offset: r.index_offset + r.width],
                           ref_idx[r0.index_offset: r0.index_offset + r0.width]), f"row {e} indices"
    assert torch.isnan(out[0::2].float()).all(), "a query row no entry owns was written"
    assert bool((inv[0::2] == 7).all()), "an invalid row no entry owns was written"


@pytest.mark.parametrize("i", [0, 1, 2, 3, 4])
def test_joint_equals_single_row(i):
    """Row r of a joint launch is bitwise equal to a launch of row r alone."""
    dev = cfg_dev(i)
    out, idx, _ = run_decode(dev)
    for e, r in enumerate(dev.rows):
        o1, i1, _ = run_decode(dev, rows=[r])
        assert torch.equal(o1[r.q_row].view(torch.int16), out[r.q_row].view(torch.int16)), f"row {e} out"
        assert torch.equal(i1[r.index_offset: r.index_offset + r.width],
                           idx[r.index_offset: r.index_offset + r.width]), f"row {e} indices"


def test_decode_stages_agree():
    """decode == indexer_score -> topk -> sparse_attn, bitwise. The decode's
    indices output equals ds_rows_topk's (best first); both attentions sum over
    the selected rows in ascending index order, so the stand-alone attention of
    those indices is the decode's output bit for bit. The top-k is exactly the
    top-width of the GPU's own scores."""
    wl, dev = cfg(2), cfg_dev(2)
    out, idx, _ = run_decode(dev)
    stride = max(r.kv_len for r in wl.rows)
    scores = torch.empty((wl.num_rows, stride), dtype=torch.float32, device="cuda")
    ds.ds_rows_indexer_score(dev.rows, dev.q_index, dev.w_index, dev.keys, scores, stride)
    idx2 = torch.full_like(idx, -7)
    ds.ds_rows_topk(dev.rows, scores, stride, idx2, ds.workspace(dev.rows))
    torch.cuda.synchronize()
    assert torch.equal(idx, idx2)
    out2 = torch.full_like(out, float("nan"))
    ds.ds_rows_sparse_attn(dev.rows, dev.q_attn, dev.sinks, dev.sinks_row_stride, idx2, dev.scale, out2, dev.kv)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    s = scores.cpu().numpy()
    for e, r in enumerate(wl.rows):
        check_topk_consistent(idx2.cpu().numpy()[r.index_offset: r.index_offset + r.width], s[e, : r.kv_len],
                              r.width)


def test_decode_repeatable_and_on_side_stream():
    dev = cfg_dev(0)
    a, ia, _ = run_decode(dev)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b, ib, _ = run_decode(dev, stream=s)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(ia, ib)


def test_decode_without_optional_outputs():
    dev = cfg_dev(0)
    a, ia, _ = run_decode(dev)
    b, _, _ = run_decode(dev, indices=False, invalid=False)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ---------------------------------------------------------------------------
# fail-closed data
# ---------------------------------------------------------------------------

def test_fail_closed_decode():
    wl = workloads.make_workload("fail", 51, [700, 900, 300], per_row_sinks=True)
    wl.q_attn[0, 5, 17] = 0x7FC0                       # NaN in row 0, head 5
    wl.sinks[1, 9] = np.inf                            # row 1 head 9 sink
    dev = to_device(wl)
    out, idx, inv = run_decode(dev)
    ginv = inv.cpu().numpy()
    got = out.float().cpu().numpy()
    ref = oracle.decode(wl)
    for e, r in enumerate(wl.rows):
        np.testing.assert_array_equal(ginv[r.q_row], ref[e]["invalid"].astype(np.int32))
        check_out(got[r.q_row], ref[e]["out"], what=f"row {e}")
    assert ginv[0, 5] == 1 and np.all(got[0, 5] == 0)
    assert ginv[1, 9] == 1 and np.all(got[1, 9] == 0)
    assert ginv[2].sum() == 0


def test_fail_closed_kv_and_keys():
    """A non-finite KV element on a selected row zeroes every head of the row;
    a non-finite indexer key is never selected."""
    wl = workloads.make_workload("fail2", 52, [800, 800], per_row_sinks=True)
    ref0 = oracle.decode(wl)
    j = int(ref0[0]["indices"][3])
    wl.kv[0][j, 100] = 0x7F80                          # +Inf
    best = int(ref0[1]["indices"][0])
    wl.keys[1][best, 7] = 0x7FC0                       # NaN key: excluded from top-k
    dev = to_device(wl)
    out, idx, inv = run_decode(dev)
    ref = oracle.decode(wl)
    assert best not in ref[1]["indices"].tolist()
    gidx = idx.cpu().numpy()
    assert best not in gidx[512:1024].tolist()
    assert np.all(inv.cpu().numpy()[0] == 1)
    assert np.all(out[0].float().cpu().numpy() == 0)
    check_out(out[1].float().cpu().numpy(), ref[1]["out"], what="row 1")


def test_decode_full_size_in_the_bench_launch_configuration():
    """The bench's launch configuration on the full 8 x 131072 workload: four
    consecutive decode steps (four query sets) captured in one CUDA graph on a
    side stream and replayed. Every step's output and indices are bitwise those
    of the same step run eagerly, and step 0 run eagerly is the decode that
    test_decode checks against the oracle."""
    wl, dev = cfg(3), cfg_dev(3)
    qsets = [(dev.q_index, dev.w_index, dev.q_attn)]
    for i in range(3):
        qI, wI, qA = workloads.draw_queries(wl, 1000 + i)
        qsets.append((bf16_tensor(qI, "cuda"), torch.from_numpy(wI).cuda(), bf16_tensor(qA, "cuda")))
    n_idx = max(r.index_offset + r.width for r in dev.rows)
    outs = [torch.full((8, 64, 512), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    idxs = [torch.full((n_idx,), -7, dtype=torch.int32, device="cuda") for _ in range(4)]
    ws = ds.workspace(dev.rows)
    s = torch.cuda.Stream()

    def step(i):
        qI, wI, qA = qsets[i]
        ds.ds_rows_decode(dev.rows, qI, wI, dev.keys, qA, dev.kv, dev.sinks, dev.sinks_row_stride, dev.scale,
                          outs[i], indices=idxs[i], workspace_t=ws, stream=s)

    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for i in range(4):
            step(i)
    s.synchronize()
    eager = [(o.clone(), x.clone()) for o, x in zip(outs, idxs)]
    for o, x in zip(outs, idxs):
        o.fill_(float("nan"))
        x.fill_(-7)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(4):
            step(i)
    with torch.cuda.stream(s):
        g.replay()
        g.replay()
    s.synchronize()
    for i in range(4):
        assert torch.equal(outs[i].view(torch.int16), eager[i][0].view(torch.int16)), f"step {i} out"
        assert torch.equal(idxs[i], eager[i][1]), f"step {i} indices"
    ref0, idx0, _ = run_decode(dev)
    assert torch.equal(ref0.view(torch.int16), eager[0][0].view(torch.int16))
    assert torch.equal(idx0, eager[0][1])


def test_indexer_identical_keys_identical_scores():
    """Copies of one key placed at other tiles, other lanes of a tile and in a
    ragged last tile score bitwise the same: a key's score depends only on its
    data and the query."""
    wl = cfg(4)
    dev = cfg_dev(4)
    copies = {4: {0: [300, 133, 512]},                # kv_len 513: key 512 is alone in the last tile
              6: {3: [130, 4097, 65535], 1000: [1, 20000, 65408], 40000: [129, 777, 60000]}}  # kv_len 65536
    rows, keys = [], []
    for n, (e, moves) in enumerate(copies.items()):
        r = wl.rows[e]
        k = wl.keys[e].copy()
        for src, dsts in moves.items():
            k[dsts] = k[src]
        rows.append(workloads.Row(r.kv_len, r.width, 512 * n, r.q_row))
        keys.append(bf16_tensor(k, "cuda"))
    stride = max(r.kv_len for r in rows)
    scores = torch.empty((len(rows), stride), dtype=torch.float32, device="cuda")
    ds.ds_rows_indexer_score(rows, dev.q_index, dev.w_index, keys, scores, stride)
    torch.cuda.synchronize()
    got = scores.cpu().numpy().view(np.uint32)
    for n, (e, moves) in enumerate(copies.items()):
        for src, dsts in moves.items():
            np.testing.assert_array_equal(got[n, dsts], np.full(len(dsts), got[n, src], dtype=np.uint32),
                                          err_msg=f"row {e}, copies of key {src}")
