"""The seeded input recipe shared by the oracle and the GPU path (CPU).

The recipe is fixed: one numpy default_rng(seed) per workload, values drawn in
fp32 and rounded to bf16 (nearest, ties to even), per row the order qI, KI,
wI, qA, KV, then the sinks. These tests restate the draws independently and
check the configs' stated properties.
"""

import numpy as np
import pytest

import workloads


def rne_bf16(x):
    """fp32 -> bf16 bits, round to nearest even, by exhaustive comparison of
    the two neighbouring bf16 values (not the bit trick the module uses)."""
    x = np.asarray(x, np.float32).ravel()
    lo = (x.view(np.uint32) >> np.uint32(16)).astype(np.uint32)  # truncation toward zero in magnitude
    hi = lo + np.uint32(1)
    f = lambda b: (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    xd = x.astype(np.float64)
    dlo, dhi = np.abs(xd - f(lo)), np.abs(xd - f(hi))
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (lo % 2 == 1))
    return np.where(pick_hi, hi, lo).astype(np.uint16)


def test_bf16_rounding_matches_an_exhaustive_nearest_even():
    rng = np.random.default_rng(11)
    x = rng.standard_normal(200_000, dtype=np.float32) * np.float32(100.0)
    # exact halfway cases: a bf16 value plus half an ulp
    base = workloads.bits_to_f32(rng.integers(0x3F00, 0x4300, size=1000).astype(np.uint16))
    half = (base.view(np.uint32) + np.uint32(0x8000)).view(np.float32)
    for v in (x, half):
        np.testing.assert_array_equal(workloads.bf16_bits(v), rne_bf16(v))


def test_config0_is_the_stated_draw_sequence():
    wl = workloads.config(0)
    rng = np.random.default_rng(0)
    qI = rne_bf16(rng.standard_normal(size=(64, 128), dtype=np.float32)).reshape(64, 128)
    KI = rne_bf16(rng.standard_normal(size=(2048, 128), dtype=np.float32)).reshape(2048, 128)
    wI = rng.standard_normal(size=64, dtype=np.float32) / np.float32(8.0)
    qA = rne_bf16(rng.standard_normal(size=(64, 512), dtype=np.float32)).reshape(64, 512)
    KV = rne_bf16(rng.standard_normal(size=(2048, 512), dtype=np.float32)).reshape(2048, 512)
    sinks = rng.standard_normal(size=64, dtype=np.float32)
    np.testing.assert_array_equal(wl.q_index[0], qI)
    np.testing.assert_array_equal(wl.keys[0], KI)
    np.testing.assert_array_equal(wl.w_index[0], wI)
    np.testing.assert_array_equal(wl.q_attn[0], qA)
    np.testing.assert_array_equal(wl.kv[0], KV)
    np.testing.assert_array_equal(wl.sinks, sinks)
    assert wl.sinks_row_stride == 0 and wl.scale == pytest.approx(512 ** -0.5)


def test_config1_integers_in_range_and_table():
    wl = workloads.config(1)
    assert [r.kv_len for r in wl.rows] == [300, 512, 1000, 4096]
    assert [r.width for r in wl.rows] == [300, 512, 512, 512]
    assert [r.index_offset for r in wl.rows] == [0, 512, 1024, 1536]
    arrays = [workloads.bits_to_f32(wl.q_index), workloads.bits_to_f32(wl.q_attn), wl.w_index]
    arrays += [workloads.bits_to_f32(k) for k in wl.keys] + [workloads.bits_to_f32(k) for k in wl.kv]
    for a in arrays:
        assert np.all(a == np.round(a)) and a.min() >= -3 and a.max() <= 3
    assert wl.integer_valued and wl.sinks.ndim == 1


def test_config2_row_lengths():
    lens = workloads.config_kv_lens(2)
    assert lens == [55557, 20169, 10811, 22435, 29521, 54122, 31822, 9743]
    assert all(4096 <= L <= 65536 for L in lens)


def test_config4_edges_sinks_and_prototype_keys():
    wl = workloads.config(4)
    assert [r.kv_len for r in wl.rows] == [1, 17, 511, 512, 513, 32768, 65536, 262144]
    assert np.all(wl.sinks[2] == 20.0) and np.all(wl.sinks[5] == -20.0)
    assert wl.sinks_row_stride == 64
    # Replay the first two rows: 64 prototypes are drawn first; each key is a
    # prototype plus N(0, 1e-3) noise, rounded to bf16.
    rng = np.random.default_rng(4)
    protos = rne_bf16(rng.standard_normal(size=(64, 128), dtype=np.float32)).reshape(64, 128)
    same = []
    for e, L in enumerate([1, 17]):
        rng.standard_normal(size=(64, 128), dtype=np.float32)                  # qI
        pick = rng.integers(0, 64, size=L)
        noise = rng.standard_normal(size=(L, 128), dtype=np.float32) * np.float32(1e-3)
        keys = rne_bf16(workloads.bits_to_f32(protos)[pick] + noise).reshape(L, 128)
        np.testing.assert_array_equal(wl.keys[e], keys)
        same.append(np.mean(keys == protos[pick]))
        rng.standard_normal(size=64, dtype=np.float32)                         # wI
        rng.standard_normal(size=(64, 512), dtype=np.float32)                  # qA
        rng.standard_normal(size=(L, 512), dtype=np.float32)                   # KV
    # most elements keep their prototype's value: keys of one prototype score as near-ties
    assert min(same) > 0.5


def test_draws_are_deterministic_and_query_sets_differ():
    a, b = workloads.config(0), workloads.config(0)
    np.testing.assert_array_equal(a.keys[0], b.keys[0])
    q1 = workloads.draw_queries(a, 1001)
    q2 = workloads.draw_queries(a, 1002)
    assert q1[0].shape == a.q_index.shape and q1[2].shape == a.q_attn.shape
    assert not np.array_equal(q1[0], q2[0])
    np.testing.assert_array_equal(q1[0], workloads.draw_queries(a, 1001)[0])


def test_algorithmic_bytes_of_the_bench_workload():
    # 256 L + 1024 W + 16384 + 65536 + 65536 per row, at 8 x 131072
    rows = [workloads.Row(131072, 512, 512 * e, e) for e in range(8)]
    wl = workloads.Workload("t", 0, rows, None, None, [], None, [], np.zeros(64, np.float32), 1.0)
    assert wl.algorithmic_bytes() == 273_809_408
