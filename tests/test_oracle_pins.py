"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each pin is a hand-derived fixture (tests/golden), a closed form, an identity
of the mathematics, exact integer arithmetic or a brute force on tiny inputs.
The last group plants plausible mistakes in copies of the oracle functions and
checks that some pin catches each one.
"""

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.special

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# Indexer score
# ---------------------------------------------------------------------------

def test_indexer_golden():
    g = _golden("indexer_tiny.json")
    s = oracle.indexer_score(np.array(g["q"], float), np.array(g["w"]), np.array(g["keys"], float))
    assert s.tolist() == g["scores"]


def _indexer_exact(q, w, keys):
    """Exact rational brute force with Python integers / Fractions and loops."""
    out = []
    for k in keys:
        total = Fraction(0)
        for h in range(len(q)):
            dot = Fraction(0)
            for d in range(len(k)):
                dot += Fraction(q[h][d]) * Fraction(k[d])
            total += Fraction(w[h]) * max(dot, Fraction(0))
        out.append(total)
    return out


def test_indexer_integer_inputs_exact():
    rng = np.random.default_rng(11)
    q = rng.integers(-3, 4, size=(5, 7))
    w = rng.integers(-3, 4, size=5)
    keys = rng.integers(-3, 4, size=(9, 7))
    exact = _indexer_exact(q.tolist(), w.tolist(), keys.tolist())
    s = oracle.indexer_score(q.astype(float), w.astype(float), keys.astype(float))
    assert [Fraction(x) for x in s] == exact


def test_indexer_relu_identity():
    """relu(x) - relu(-x) = x, so s(q) - s(-q) = sum_h w_h (q_h . k) exactly
    in exact arithmetic: a plain weighted sum of dot products, no ReLU."""
    rng = np.random.default_rng(12)
    q = rng.standard_normal((6, 8))
    w = rng.standard_normal(6)
    keys = rng.standard_normal((10, 8))
    diff = oracle.indexer_score(q, w, keys) - oracle.indexer_score(-q, w, keys)
    lin = [sum(w[h] * sum(q[h, d] * k[d] for d in range(8)) for h in range(6)) for k in keys]
    np.testing.assert_allclose(diff, lin, rtol=1e-12, atol=1e-12)


def test_indexer_one_hot_weights_select_head():
    """w = e_h reduces the score to max(0, q_h . k): pairs weights with heads."""
    rng = np.random.default_rng(13)
    q = rng.standard_normal((4, 5))
    keys = rng.standard_normal((7, 5))
    for h in range(4):
        w = np.zeros(4)
        w[h] = 1.0
        s = oracle.indexer_score(q, w, keys)
        expect = [max(0.0, sum(q[h, d] * k[d] for d in range(5))) for k in keys]
        np.testing.assert_allclose(s, expect, rtol=1e-13, atol=1e-14)


def test_indexer_nonfinite_becomes_minus_inf():
    q = np.ones((2, 3))
    w = np.ones(2)
    keys = np.array([[1.0, 1.0, 1.0], [np.nan, 0, 0], [np.inf, 0, 0], [1e38, 1e38, 1e38]])
    s = oracle.indexer_score(q, w, keys)
    assert s[0] == 6.0
    assert s[1] == -np.inf and s[2] == -np.inf
    assert s[3] == -np.inf          # 6e38 overflows fp32


def test_indexer_causal_mask():
    rng = np.random.default_rng(14)
    q, w, keys = rng.standard_normal((3, 4)), rng.standard_normal(3), rng.standard_normal((10, 4))
    s = oracle.indexer_score_causal(q, w, keys, start_pos=22, ratio=4)   # valid = 23 // 4 = 5
    assert np.all(s[5:] == -np.inf)
    np.testing.assert_array_equal(s[:5], oracle.indexer_score(q, w, keys)[:5])


# ---------------------------------------------------------------------------
# Top-k
# ---------------------------------------------------------------------------

def test_topk_golden():
    g = _golden("indexer_tiny.json")
    for width, expect in g["topk"].items():
        assert oracle.topk(np.array(g["scores"]), int(width)).tolist() == expect


def _topk_bruteforce(s, width):
    """Rank every finite entry by counting the entries that beat it."""
    n = len(s)
    finite = [math.isfinite(x) for x in s]
    out = [-1] * width
    for j in range(n):
        if not finite[j]:
            continue
        rank = sum(1 for i in range(n) if finite[i] and (s[i] > s[j] or (s[i] == s[j] and i < j)))
        if rank < width:
            out[rank] = j
    return out


@pytest.mark.parametrize("seed", range(6))
def test_topk_bruteforce_with_ties_and_nonfinite(seed):
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(1, 60))
    s = rng.integers(-4, 5, size=n).astype(float) * 0.5
    s[rng.random(n) < 0.15] = np.nan
    s[rng.random(n) < 0.05] = np.inf
    s[rng.random(n) < 0.05] = -np.inf
    s[rng.random(n) < 0.2] = -0.0
    for width in (1, 3, n, n + 4):
        assert oracle.topk(s, width).tolist() == _topk_bruteforce(s.tolist(), width)


def test_topk_matches_stable_argsort():
    s = workloads.random_scores(7, [3000], ties=True)[0].astype(float)
    ref = np.argsort(-s, kind="stable")[:512]
    assert oracle.topk(s, 512).tolist() == ref.tolist()


def test_topk_signed_zero_ties():
    s = np.array([-0.0, 0.0, -0.0, -1.0, 0.0])
    assert oracle.topk(s, 5).tolist() == [0, 1, 2, 4, 3]


def test_topk_causal_offset_and_fill():
    s = np.arange(10, dtype=float)                  # best is the highest index
    out = oracle.topk_causal(s, start_pos=15, offset=100, ratio=4, width=6)  # valid = 4
    assert out.tolist() == [103, 102, 101, 100, -1, -1]


def _queries_bruteforce(q, w, keys, start_pos, offset, width):
    """Per query: exact integer scores (Fractions), the causal count from the
    query's own position, and ranks counted pairwise."""
    out = []
    for j in range(len(q)):
        valid = min(len(keys), (start_pos + j + 1) // 4)
        s = []
        for k in keys[:valid]:
            s.append(sum(Fraction(w[j][h]) * max(0, sum(Fraction(a) * b for a, b in zip(q[j][h], k)))
                          for h in range(len(w[j]))))
        row = [-1] * width
        for a in range(valid):
            rank = sum(1 for b in range(valid) if s[b] > s[a] or (s[b] == s[a] and b < a))
            if rank < width:
                row[rank] = a + offset
        out.append(row)
    return out


def test_indexer_queries_bruteforce():
    rng = np.random.default_rng(31)
    nq, heads, dim, L = 6, 3, 4, 24
    q = rng.integers(-2, 3, size=(nq, heads, dim))
    w = rng.integers(-2, 3, size=(nq, heads))
    keys = rng.integers(-2, 3, size=(L, dim))
    # start_pos 73: counts 18, 18, 18, 19, 19, 19 (the count steps inside the run)
    for start_pos, offset, width in [(73, 0, 30), (73, 5, 7), (90, 2, 10)]:
        s, idx = oracle.indexer_topk_queries(q, w, keys, start_pos, offset=offset, width=width)
        assert idx.tolist() == _queries_bruteforce(q.tolist(), w.tolist(), keys.tolist(), start_pos, offset, width)
        for j in range(nq):
            valid = min(L, (start_pos + j + 1) // 4)
            assert np.all(s[j, valid:] == -np.inf)


def test_indexer_queries_one_query_is_the_positioned_indexer():
    rng = np.random.default_rng(32)
    q, w, keys = rng.standard_normal((1, 4, 8)), rng.standard_normal((1, 4)), rng.standard_normal((50, 8))
    s, idx = oracle.indexer_topk_queries(q, w, keys, 130, offset=3, width=16)
    ref = oracle.indexer_score_causal(q[0], w[0], keys, 130)
    np.testing.assert_array_equal(s[0], ref)
    assert idx[0].tolist() == oracle.topk_causal(ref, 130, offset=3, width=16).tolist()


# ---------------------------------------------------------------------------
# Sparse attention
# ---------------------------------------------------------------------------

def test_attention_golden():
    g = _golden("attention_tiny.json")
    out, inv = oracle.sparse_attention(np.array(g["q"], float), np.array(g["kv"], float),
                                       np.array(g["indices"]), np.array(g["sinks"]), g["scale"])
    np.testing.assert_allclose(out, g["out"], rtol=1e-15, atol=1e-15)
    assert not inv.any()
    k1 = g["kv_len_1"]
    out, inv = oracle.sparse_attention(np.array(k1["q"], float), np.array(k1["kv"], float),
                                       np.array(k1["indices"]), np.array(k1["sinks"]), k1["scale"])
    np.testing.assert_allclose(out, k1["out"], rtol=1e-15)


def test_attention_dense_closed_form():
    """width = kv_len, every row selected and a sink whose exp is 0 in fp32:
    dense softmax attention softmax(scale q K^T) K."""
    rng = np.random.default_rng(21)
    H, F, L = 4, 16, 9
    q, kv = rng.standard_normal((H, F)), rng.standard_normal((L, F))
    scale = 1 / math.sqrt(F)
    out, inv = oracle.sparse_attention(q, kv, np.arange(L), np.full(H, -3.0e38), scale)
    dense = scipy.special.softmax(scale * np.einsum("hf,lf->hl", q, kv), axis=1) @ kv
    np.testing.assert_allclose(out, dense, rtol=1e-12, atol=1e-14)
    assert not inv.any()


def test_attention_sink_identity():
    """O(sink) = O(no sink) * S / (S + e^sink), S = sum_t e^{l_t} per head."""
    rng = np.random.default_rng(22)
    H, F, L = 5, 12, 20
    q, kv = rng.standard_normal((H, F)), rng.standard_normal((L, F))
    idx = rng.permutation(L)[:11]
    scale = 0.3
    sinks = rng.standard_normal(H) * 2
    with_sink, _ = oracle.sparse_attention(q, kv, idx, sinks, scale)
    no_sink, _ = oracle.sparse_attention(q, kv, idx, np.full(H, -3.0e38), scale)
    for h in range(H):
        S = sum(math.exp(scale * float(np.dot(q[h], kv[j]))) for j in idx)
        np.testing.assert_allclose(with_sink[h], no_sink[h] * S / (S + math.exp(sinks[h])),
                                   rtol=1e-12, atol=1e-15)


def test_attention_slot_order_and_sentinels():
    """A set function of the selected rows: slot order and -1 sentinels do not matter."""
    rng = np.random.default_rng(23)
    H, F, L = 3, 8, 30
    q, kv, sinks = rng.standard_normal((H, F)), rng.standard_normal((L, F)), rng.standard_normal(H)
    idx = rng.permutation(L)[:10]
    a, _ = oracle.sparse_attention(q, kv, idx, sinks, 0.5)
    mixed = np.insert(idx[::-1], [2, 5, 5], -1)
    b, _ = oracle.sparse_attention(q, kv, mixed, sinks, 0.5)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-15)


def test_attention_all_sentinels_is_zero():
    q, kv = np.ones((2, 4)), np.ones((3, 4))
    out, inv = oracle.sparse_attention(q, kv, np.array([-1, -1]), np.zeros(2), 1.0)
    assert np.all(out == 0) and not inv.any()


def test_attention_fail_closed():
    rng = np.random.default_rng(24)
    H, F, L = 4, 8, 12
    q, kv, sinks = rng.standard_normal((H, F)), rng.standard_normal((L, F)), rng.standard_normal(H)
    idx = np.array([3, 7, 1, -1])
    base, inv = oracle.sparse_attention(q, kv, idx, sinks, 0.5)
    assert not inv.any() and np.all(base != 0)
    # non-finite q in head 2 -> head 2 zero only
    q2 = q.copy(); q2[2, 5] = np.nan
    out, inv = oracle.sparse_attention(q2, kv, idx, sinks, 0.5)
    assert inv.tolist() == [False, False, True, False] and np.all(out[2] == 0)
    np.testing.assert_array_equal(out[[0, 1, 3]], base[[0, 1, 3]])
    # non-finite KV on a selected row -> every head zero
    kv2 = kv.copy(); kv2[7, 0] = np.inf
    out, inv = oracle.sparse_attention(q, kv2, idx, sinks, 0.5)
    assert inv.all() and np.all(out == 0)
    # ... but not on an unselected row
    kv3 = kv.copy(); kv3[0, 0] = np.nan
    out, inv = oracle.sparse_attention(q, kv3, idx, sinks, 0.5)
    np.testing.assert_array_equal(out, base)
    # out-of-range index -> every head zero
    for bad in (L, -2):
        out, inv = oracle.sparse_attention(q, kv, np.array([3, bad, 1]), sinks, 0.5)
        assert inv.all() and np.all(out == 0)
    # non-finite sink -> that head zero
    s2 = sinks.copy(); s2[1] = np.inf
    out, inv = oracle.sparse_attention(q, kv, idx, s2, 0.5)
    assert inv.tolist() == [False, True, False, False]


def test_attention_lazy_rows_equal_dense():
    """`sparse_attention_rows` (widens only selected rows) equals `sparse_attention`."""
    rng = np.random.default_rng(25)
    L = 40
    bits = workloads.bf16_bits(rng.standard_normal((L, 16)).astype(np.float32))
    q = rng.standard_normal((3, 16))
    sinks = rng.standard_normal(3)
    for idx in (np.array([5, 5, -1, 39, 0]), np.array([2, L, 1]), np.array([-1, -1])):
        a = oracle.sparse_attention(q, oracle.bf16_to_f64(bits), idx, sinks, 0.25)
        b = oracle.sparse_attention_rows(q, oracle._LazyRows(bits, L), idx, sinks, 0.25)
        np.testing.assert_array_equal(a[0], b[0])
        np.testing.assert_array_equal(a[1], b[1])


def test_round_bf16_against_bit_rounding():
    """fp32-representable values: the log/rint rounding equals the integer
    round-half-even on the fp32 bit pattern (an independent method)."""
    rng = np.random.default_rng(26)
    x = rng.standard_normal(20000).astype(np.float32) * np.float32(3.0)
    x[:8] = [1.00390625, 1.01171875, -1.00390625, 0.0, 2.0 ** -130, 3.0, -7.5, 1e-3]
    via_bits = workloads.bits_to_f32(workloads.bf16_bits(x)).astype(np.float64)
    np.testing.assert_array_equal(oracle.round_bf16(x.astype(np.float64)), via_bits)


def test_bf16_decode_exact():
    vals = np.array([1.0, -2.5, 3.140625, 0.0078125], np.float32)
    bits = (vals.view(np.uint32) >> 16).astype(np.uint16)
    np.testing.assert_array_equal(oracle.bf16_to_f64(bits), vals.astype(np.float64))


# ---------------------------------------------------------------------------
# Learned KV compressor (one token per row)
# ---------------------------------------------------------------------------

def _comp_inputs(seed, ratio, head_dim, pos):
    rng = np.random.default_rng(seed)
    coff = 2 if ratio == 4 else 1
    P = coff * head_dim
    f32 = lambda *sh: rng.standard_normal(sh).astype(np.float32)
    return dict(kv=f32(P), score=f32(P), ape=f32(ratio, P), norm=(1.0 + 0.1 * f32(head_dim)).astype(np.float32),
                kv_state=f32(coff * ratio, P), score_state=f32(coff * ratio, P), start_pos=pos, ratio=ratio,
                head_dim=head_dim, eps=1e-6)


def _bf16_ulp(x):
    x = np.abs(np.asarray(x, np.float64))
    return np.exp2(np.floor(np.log2(np.maximum(x, 1e-30))) - 7.0)


@pytest.mark.parametrize("ratio,head_dim", [(4, 128), (4, 512), (128, 512)])
def test_compressor_uniform_scores_give_the_window_mean(ratio, head_dim):
    a = _comp_inputs(1, ratio, head_dim, pos=ratio * 3 - 1)  # completes a block
    coff = 2 if ratio == 4 else 1
    a["score_state"][:] = 0.5
    a["score"][:] = 0.25
    a["ape"][:] = 0.25  # the token's score + ape is 0.5 too: all equal
    out, kv_new, _ = oracle.compress_kv(**a)
    # The softmax of equal scores is uniform: the pooled value is the mean of
    # the window's values (feature f, and head_dim + f for the current block).
    # The window before the shift: the previous block (untouched by the token's
    # write) and the current block (after it; the shift leaves those rows).
    V = kv_new.astype(np.float64)
    if coff == 2:
        prev = np.asarray(a["kv_state"], np.float64)[:ratio, :head_dim]
        win = np.concatenate([prev, V[ratio:, head_dim:]], 0)
    else:
        win = V[:, :head_dim]
    c = oracle.round_bf16(win.mean(0))
    y = c * np.asarray(a["norm"], np.float64) / np.sqrt(np.mean(c * c) + a["eps"])
    np.testing.assert_allclose(out, oracle.round_bf16(y), rtol=0, atol=0)


def test_compressor_dominant_score_selects_its_value():
    a = _comp_inputs(2, 128, 512, pos=127)
    a["score_state"][:] = 0.0
    a["score_state"][37] = 80.0       # row 37 outweighs the others by e^80
    out, kv_new, _ = oracle.compress_kv(**a)
    c = oracle.round_bf16(kv_new[37].astype(np.float64))
    y = c * np.asarray(a["norm"], np.float64) / np.sqrt(np.mean(c * c) + 1e-6)
    np.testing.assert_allclose(out, oracle.round_bf16(y), rtol=0, atol=0)


@pytest.mark.parametrize("ratio,head_dim", [(4, 128), (128, 512)])
def test_compressor_token_write_and_no_output_mid_block(ratio, head_dim):
    pos = ratio * 5 + 1                    # mid block: (pos + 1) % ratio != 0
    a = _comp_inputs(3, ratio, head_dim, pos)
    out, kv_new, sc_new = oracle.compress_kv(**a)
    assert not out.any()
    slot = (ratio if ratio == 4 else 0) + pos % ratio
    changed = np.nonzero((kv_new != a["kv_state"]).any(1) | (sc_new != a["score_state"]).any(1))[0]
    assert list(changed) == [slot]
    np.testing.assert_array_equal(kv_new[slot], a["kv"])
    # score + ape is an fp32 add (the state is fp32), of the token's ape row.
    np.testing.assert_array_equal(sc_new[slot], np.float32(a["score"]) + np.float32(a["ape"][pos % ratio]))


def test_compressor_first_half_of_the_token_waits_for_the_next_block():
    # A NaN in the first half of the completing token is not read by this block.
    a = _comp_inputs(10, 4, 128, pos=7)
    a["kv"][5] = np.nan
    out, kv_new, sc_new = oracle.compress_kv(**a)
    assert out.any()
    assert kv_new[0 + 3, 5] == 0.0 and np.isnan(sc_new[0 + 3, 5])  # shifted into the previous block


def test_compressor_overlap_reads_each_half_from_its_block():
    # ratio 4: window rows 0..3 (previous block) read features [0, D), rows 4..7
    # (current block) read [D, 2D). Garbage in the other halves changes nothing.
    a = _comp_inputs(4, 4, 128, pos=11)
    out, _, _ = oracle.compress_kv(**a)
    b = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in a.items()}
    b["kv_state"][:4, 128:] = 1e6
    b["score_state"][:4, 128:] = 50.0
    b["kv_state"][4:, :128] = -1e6
    b["score_state"][4:, :128] = 50.0
    b["kv"][:128] = 7e5                     # the token's first half lands in row 4+3, unread
    out2, _, _ = oracle.compress_kv(**b)
    np.testing.assert_array_equal(out, out2)


def test_compressor_overlap_shift_after_a_block():
    a = _comp_inputs(5, 4, 512, pos=3)
    out, kv_new, sc_new = oracle.compress_kv(**a)
    assert out.any()
    np.testing.assert_array_equal(kv_new[:4], kv_new[4:])
    np.testing.assert_array_equal(sc_new[:4], sc_new[4:])
    b = _comp_inputs(5, 4, 512, pos=2)      # mid block: no shift
    _, kv2, _ = oracle.compress_kv(**b)
    np.testing.assert_array_equal(kv2[:4], b["kv_state"][:4])


def test_compressor_unit_norm_gives_unit_rms():
    a = _comp_inputs(6, 4, 512, pos=7)
    a["norm"][:] = 1.0
    out, _, _ = oracle.compress_kv(**a)
    rms = np.sqrt(np.mean(out ** 2))
    assert abs(rms - 1.0) < 4e-3  # bf16 rounding of c and of the output; eps 1e-6


@pytest.mark.parametrize("what", ["kv_nan", "norm_inf", "state_score_inf", "state_kv_nan"])
def test_compressor_fail_closed_zeroes_the_row(what):
    a = _comp_inputs(7, 4, 128, pos=7)
    if what == "kv_nan":
        # The token's second half is read by this block (the first half only
        # after the shift): its score becomes NaN and its value 0.
        a["kv"][128 + 5] = np.nan
    elif what == "norm_inf":
        a["norm"][9] = np.inf
    elif what == "state_score_inf":
        a["score_state"][1, 3] = np.inf
    else:
        a["kv_state"][2, 4] = np.nan
    out, kv_new, _ = oracle.compress_kv(**a)
    assert not out.any()
    np.testing.assert_array_equal(kv_new[:4], kv_new[4:])  # the window still shifts
    if what == "kv_nan":
        assert kv_new[4 + 3, 128 + 5] == 0.0


def test_compressor_window_order_does_not_matter():
    a = _comp_inputs(8, 128, 512, pos=127)
    out, kv_new, sc_new = oracle.compress_kv(**a)
    perm = np.random.default_rng(9).permutation(128)
    b = dict(a)
    b["kv_state"] = kv_new[perm]
    b["score_state"] = sc_new[perm]
    slot = int(np.nonzero(perm == 127)[0][0])   # the token's row moves to `slot`
    b["kv"], b["score"] = kv_new[127].copy(), sc_new[127].copy()
    b["ape"] = np.zeros_like(a["ape"])
    b["start_pos"] = 128 * 9 + slot - 128 if slot == 127 else None
    # Recompute with the permuted window and the token written to its new row.
    if b["start_pos"] is None:
        b["start_pos"] = 128 * 9 + 127
        b["kv_state"][slot], b["kv_state"][127] = b["kv_state"][127].copy(), b["kv_state"][slot].copy()
        b["score_state"][slot], b["score_state"][127] = b["score_state"][127].copy(), b["score_state"][slot].copy()
    out2, _, _ = oracle.compress_kv(**b)
    assert np.all(np.abs(out2 - out) <= _bf16_ulp(out) + 1e-12)


# ---------------------------------------------------------------------------
# Decode composition on a small workload
# ---------------------------------------------------------------------------

def test_decode_integer_workload_exact_scores():
    """Config-1-style integer inputs: every score is an exact integer, and the
    selected set's minimum beats every unselected score (ties: lower index)."""
    wl = workloads.make_workload("t", 5, [40, 600], integer=True, per_row_sinks=False)
    res = oracle.decode(wl)
    for e, r in enumerate(wl.rows):
        q = oracle.bf16_to_f64(wl.q_index[r.q_row]).astype(int).tolist()
        w = wl.w_index[r.q_row].astype(int).tolist()
        keys = oracle.bf16_to_f64(wl.keys[e]).astype(int).tolist()
        assert [Fraction(x) for x in res[e]["scores"]] == _indexer_exact(q, w, keys)
        assert res[e]["indices"].tolist() == _topk_bruteforce(res[e]["scores"].tolist(), r.width)


# ---------------------------------------------------------------------------
# Planted mistakes: each must be caught by one of the pins above
# ---------------------------------------------------------------------------

def _no_relu(q, w, keys):
    return (np.asarray(keys) @ np.asarray(q).T) @ np.asarray(w)


def _transposed_weights(q, w, keys):
    d = np.asarray(keys) @ np.asarray(q).T
    return np.maximum(d, 0) @ np.asarray(w)[::-1]


def _topk_high_index_ties(scores, width):
    s = np.asarray(scores, float)
    cand = np.nonzero(np.isfinite(s))[0]
    order = cand[np.lexsort((-cand, -s[cand]))]
    out = np.full(width, -1, np.int32)
    out[: min(width, len(order))] = order[:width]
    return out


_REAL_QUERIES = oracle.indexer_topk_queries


def _queries_one_position(q, w, keys, start_pos, offset=0, ratio=4, width=512):
    # mistake: every query takes the first query's causal count
    s, _ = _REAL_QUERIES(q, w, keys, start_pos, offset, ratio, width)
    idx = np.stack([oracle.topk_causal(np.asarray(oracle.indexer_score_causal(q[j], w[j], keys, start_pos, ratio)),
                                       start_pos, offset, ratio, width) for j in range(len(q))])
    return s, idx


def _queries_first_weights(q, w, keys, start_pos, offset=0, ratio=4, width=512):
    # mistake: every query uses the first query's head weights
    w = np.broadcast_to(np.asarray(w)[:1], np.asarray(w).shape)
    return _REAL_QUERIES(q, w, keys, start_pos, offset, ratio, width)


_REAL_ATTENTION = oracle.sparse_attention
_REAL_COMPRESS = oracle.compress_kv


def _compress_without_ape(**a):
    # mistake: the position bias is not added to the token's score
    return _REAL_COMPRESS(**{**a, "ape": np.zeros_like(np.asarray(a["ape"]))})


def _compress_current_block_only(**a):
    # mistake: an overlapping window pools only its current block
    if a["ratio"] != 4:
        return _REAL_COMPRESS(**a)
    sc = np.array(a["score_state"], np.float32)
    sc[:4] = -np.inf
    out, kv, s = _REAL_COMPRESS(**{**a, "score_state": sc})
    return out, kv, s


def _attention_sink_with_value(q, kv, idx, sinks, scale):
    out, inv = _REAL_ATTENTION(q, kv, idx, sinks, scale)
    # mistake: the sink's mass goes to a value row (the first selected one)
    return out * 0.9 + 0.1 * np.asarray(kv)[max(int(idx[0]), 0)], inv


def test_planted_mistakes_are_caught(monkeypatch):
    caught = []
    for name, fake in [("indexer_score", _no_relu), ("indexer_score", _transposed_weights),
                       ("topk", _topk_high_index_ties),
                       ("indexer_topk_queries", _queries_one_position),
                       ("indexer_topk_queries", _queries_first_weights),
                       ("sparse_attention", _attention_sink_with_value),
                       ("compress_kv", _compress_without_ape), ("compress_kv", _compress_current_block_only)]:
        monkeypatch.setattr(oracle, name, fake)
        tests = {
            "indexer_score": [test_indexer_golden, test_indexer_relu_identity,
                              test_indexer_one_hot_weights_select_head],
            "topk": [test_topk_golden, test_topk_signed_zero_ties],
            "indexer_topk_queries": [test_indexer_queries_bruteforce],
            "sparse_attention": [test_attention_golden, test_attention_dense_closed_form],
            "compress_kv": [lambda: test_compressor_uniform_scores_give_the_window_mean(4, 128),
                            lambda: test_compressor_token_write_and_no_output_mid_block(4, 128)],
        }[name]
        failed = 0
        for t in tests:
            try:
                t()
            except AssertionError:
                failed += 1
        caught.append(failed > 0)
        monkeypatch.undo()
    assert all(caught), caught
