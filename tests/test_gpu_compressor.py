"""GPU parity of the learned KV compressor (ds_rows_compress_kv) against the
CPU oracle (oracle.compress_kv), through the C-ABI: the state buffers bit for
bit, the output within two bf16 ulps (the pooled value is rounded to bf16 on
both sides, from fp32 here and fp64 there, so a rounding tie may fall either
way; the RMS scale and the final rounding add no more).
"""

import numpy as np
import pytest
import torch

import deepseek_sparse_attention_ragged_gb300 as ds
import oracle

pytestmark = pytest.mark.gpu

SHAPES = [(4, 128), (4, 512), (128, 512)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    ds.build()
    ds.load()


def _inputs(rng, rows, ratio, head_dim):
    coff = 2 if ratio == 4 else 1
    P = coff * head_dim
    f = lambda *sh: rng.standard_normal(sh).astype(np.float32)
    return dict(kv=f(rows, P), score=f(rows, P), ape=f(ratio, P), norm=(1.0 + 0.1 * f(head_dim)).astype(np.float32),
                kv_state=[f(coff * ratio, P) for _ in range(rows)],
                score_state=[f(coff * ratio, P) for _ in range(rows)])


def _run(a, pos, ratio, head_dim, eps=1e-6, rows=None):
    rows = list(range(len(pos))) if rows is None else rows
    cu = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    ks = [cu(a["kv_state"][e]) for e in rows]
    ss = [cu(a["score_state"][e]) for e in rows]
    out = torch.full((len(rows), head_dim), float("nan"), dtype=torch.bfloat16, device="cuda")
    ds.ds_rows_compress_kv(ks, ss, [pos[e] for e in rows], cu(a["kv"][rows]), cu(a["score"][rows]), cu(a["ape"]),
                           cu(a["norm"]), ratio, head_dim, eps, out)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), [k.cpu().numpy() for k in ks], [s.cpu().numpy() for s in ss]


def _ref(a, e, pos, ratio, head_dim, eps=1e-6):
    return oracle.compress_kv(a["kv"][e], a["score"][e], a["ape"], a["norm"], a["kv_state"][e],
                              a["score_state"][e], pos, ratio, head_dim, eps)


def _check(out, ks, ss, ref, what):
    o_ref, k_ref, s_ref = ref
    np.testing.assert_array_equal(ks, k_ref, err_msg=f"{what}: kv_state")
    assert np.array_equal(np.isnan(ss), np.isnan(s_ref)), f"{what}: score_state NaN pattern"
    np.testing.assert_array_equal(np.nan_to_num(ss), np.nan_to_num(s_ref), err_msg=f"{what}: score_state")
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(o_ref), 1e-30))) - 7.0)
    err = np.abs(out - o_ref)
    assert (err <= 2 * ulp + 1e-30).all(), f"{what}: output off by {float((err / (ulp + 1e-30)).max())} ulp"
    assert np.array_equal(out == 0, o_ref == 0) or (np.abs(o_ref[out == 0]) <= 2 * ulp[out == 0]).all()


@pytest.mark.parametrize("ratio,head_dim", SHAPES)
def test_one_token_mixed_positions(ratio, head_dim):
    rng = np.random.default_rng(ratio + head_dim)
    a = _inputs(rng, 8, ratio, head_dim)
    # Rows that complete a block and rows in the middle of one.
    pos = [ratio - 1, 2 * ratio - 1, ratio * 7 + 3, 1, ratio * 1000 - 1, ratio + 1, 5 * ratio - 1, 2]
    out, ks, ss = _run(a, pos, ratio, head_dim)
    for e in range(8):
        _check(out[e], ks[e], ss[e], _ref(a, e, pos[e], ratio, head_dim), f"row {e} pos {pos[e]}")
        if (pos[e] + 1) % ratio:
            assert not out[e].any()


@pytest.mark.parametrize("ratio,head_dim", SHAPES)
def test_consecutive_tokens_through_blocks(ratio, head_dim):
    """Tokens one after another (the state carries over, windows shift)."""
    rng = np.random.default_rng(7 * ratio + head_dim)
    rows = 3
    a = _inputs(rng, rows, ratio, head_dim)
    state_k = [k.copy() for k in a["kv_state"]]
    state_s = [s.copy() for s in a["score_state"]]
    start = [1, ratio - 2, 3 * ratio]
    steps = 2 * ratio + 3 if ratio == 4 else ratio + 2
    for step in range(steps):
        b = _inputs(rng, rows, ratio, head_dim)
        b["kv_state"], b["score_state"], b["ape"], b["norm"] = state_k, state_s, a["ape"], a["norm"]
        pos = [p + step for p in start]
        out, ks, ss = _run(b, pos, ratio, head_dim)
        for e in range(rows):
            ref = _ref(b, e, pos[e], ratio, head_dim)
            _check(out[e], ks[e], ss[e], ref, f"step {step} row {e}")
        state_k, state_s = ks, ss


@pytest.mark.parametrize("what", ["kv_nan_read_half", "norm_inf", "state_score_inf", "kv_nan_unread_half",
                                  "norm_all_max", "norm_big_finite"])
def test_fail_closed(what):
    """A bad input zeroes its row (or every row, for the shared norm). With a
    norm of fp32's largest value every output overflows, so the rows are
    zeroed; a norm of 5e37 makes the kernel compare the outputs' flags across
    the cluster, though none overflows."""
    rng = np.random.default_rng(11)
    ratio, head_dim = 4, 512
    a = _inputs(rng, 2, ratio, head_dim)
    if what == "kv_nan_read_half":
        a["kv"][0, head_dim + 9] = np.nan
    elif what == "norm_inf":
        a["norm"][9] = np.inf
    elif what == "state_score_inf":
        a["score_state"][0][2, 9] = np.inf
    elif what == "norm_all_max":
        a["norm"][:] = np.finfo(np.float32).max
    elif what == "norm_big_finite":
        a["norm"][9] = np.float32(5e37)
    else:
        a["kv"][0, 9] = np.nan          # first half: only read by the next block
    pos = [7, 7]
    out, ks, ss = _run(a, pos, ratio, head_dim)
    for e in range(2):
        _check(out[e], ks[e], ss[e], _ref(a, e, pos[e], ratio, head_dim), f"{what} row {e}")
    if what in ("kv_nan_read_half", "state_score_inf"):
        assert not out[0].any() and out[1].any()
    elif what in ("norm_inf", "norm_all_max"):
        assert not out.any()
    elif what == "norm_big_finite":
        assert out[0].any() and out[1].any()
    else:
        assert out[0].any()


@pytest.mark.parametrize("what", ["kv_nan", "window_score_inf", "window_score_nan", "window_kv_inf", "norm_inf",
                                  "norm_all_max", "norm_big_finite"])
def test_fail_closed_ratio128(what):
    """The same rules on the (128, 512) path, whose pooling reduces over warps
    through shared memory: a bad token value, window score or window value
    zeroes its row only, a bad norm zeroes every row."""
    rng = np.random.default_rng(12)
    ratio, head_dim = 128, 512
    a = _inputs(rng, 2, ratio, head_dim)
    if what == "kv_nan":
        a["kv"][0, 300] = np.nan                   # the token's own row, feature 300
    elif what == "window_score_inf":
        a["score_state"][0][37, 5] = np.inf
    elif what == "window_score_nan":
        a["score_state"][0][126, 511] = np.nan
    elif what == "window_kv_inf":
        a["kv_state"][0][64, 200] = -np.inf
    elif what == "norm_inf":
        a["norm"][100] = np.inf
    elif what == "norm_all_max":
        a["norm"][:] = np.finfo(np.float32).max
    else:
        a["norm"][100] = np.float32(5e37)
    pos = [127, 255]                               # both complete a block; tokens 127 and 127
    out, ks, ss = _run(a, pos, ratio, head_dim)
    for e in range(2):
        _check(out[e], ks[e], ss[e], _ref(a, e, pos[e], ratio, head_dim), f"{what} row {e}")
    if what in ("norm_inf", "norm_all_max"):
        assert not out.any()
    elif what == "norm_big_finite":
        assert out[0].any() and out[1].any()
    else:
        assert not out[0].any() and out[1].any()


@pytest.mark.parametrize("ratio,head_dim", SHAPES)
def test_joint_equals_single_row(ratio, head_dim):
    rng = np.random.default_rng(3 * ratio + head_dim)
    a = _inputs(rng, 8, ratio, head_dim)
    pos = [ratio * (e + 2) - 1 for e in range(8)]
    joint = _run(a, pos, ratio, head_dim)
    for e in (0, 5, 7):
        single = _run(a, pos, ratio, head_dim, rows=[e])
        np.testing.assert_array_equal(single[0][0], joint[0][e])
        np.testing.assert_array_equal(single[1][0], joint[1][e])
