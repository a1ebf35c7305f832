"""Host-side checks of the C-ABI library: it builds, loads, exports every
declared symbol and rejects bad arguments before enqueueing anything.

No GPU is needed: every call here fails validation on the host, so no CUDA
call is reached (the one exception is guarded to run only without a GPU).
"""

import ctypes
import os
import re

import pytest
import torch

import deepseek_sparse_attention_ragged_gb300 as ds

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsrows.h")


@pytest.fixture(scope="module")
def lib():
    ds.build()
    return ds.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(ds_rows_[a-z_0-9]+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("ds_rows_indexer_score", "ds_rows_topk", "ds_rows_sparse_attn", "ds_rows_decode",
              "ds_rows_workspace_bytes", "ds_rows_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_version(lib):
    assert "sm_103a" in ds.ds_rows_version()


# ---------------------------------------------------------------------------
# raw C-ABI validation (fake, aligned pointers: validation fails first)
# ---------------------------------------------------------------------------

FAKE = 0x7F0000000000  # 256-aligned, never dereferenced


def _set(rows, keys=True, kv=True, n=None):
    tab, cnt = ds._table(rows)
    n = cnt if n is None else n
    ptrs = (ctypes.c_void_p * max(1, cnt))(*[FAKE + 4096 * i for i in range(cnt)])
    rs = ds._RowSet(n, ctypes.cast(tab, ctypes.POINTER(ds.Row)),
                    ctypes.cast(ptrs, ctypes.POINTER(ctypes.c_void_p)) if keys else None,
                    ctypes.cast(ptrs, ctypes.POINTER(ctypes.c_void_p)) if kv else None)
    return rs, (tab, ptrs)


def _err(lib):
    return lib.ds_rows_last_error().decode()


def _attn(lib, rows, scale=0.04, stride=0, ws_bytes=1 << 30, q=FAKE, kv=True, ws=FAKE):
    rs, keep = _set(rows, kv=kv)
    return lib.ds_rows_sparse_attn(ctypes.byref(rs), q, FAKE, stride, FAKE, ctypes.c_float(scale), FAKE, None,
                                   ws, ws_bytes, None)


def test_rows_count(lib):
    assert lib.ds_rows_workspace_bytes(0, None) == 0
    rows9 = [(10, 10, 16 * i, i) for i in range(9)]
    tab, n = ds._table(rows9)
    assert lib.ds_rows_workspace_bytes(9, tab) == 0
    assert "rows must be 1..=8" in _err(lib)
    assert _attn(lib, rows9) == -1


@pytest.mark.parametrize("row,msg", [
    ((0, 1, 0, 0), "nonzero"), ((5, 0, 0, 0), "nonzero"), ((600, 513, 0, 0), "exceeds 512"),
    ((5, 5, 0xFFFFFFFE, 0), "exceeds u32"),
])
def test_bad_row(lib, row, msg):
    assert _attn(lib, [row]) in (-1, -2)
    assert msg in _err(lib)


def test_scale(lib):
    for s in (0.0, -1.0, float("inf"), float("nan")):
        assert _attn(lib, [(8, 8, 0, 0)], scale=s) == -1
        assert "scale" in _err(lib)


def test_duplicate_q_row(lib):
    assert _attn(lib, [(8, 8, 0, 3), (9, 9, 8, 3)]) == -1
    assert "used twice" in _err(lib)


def test_sinks_stride(lib):
    assert _attn(lib, [(8, 8, 0, 0)], stride=7) == -1
    assert "sinks_row_stride" in _err(lib)


def test_workspace_checks(lib):
    rows = [(100, 100, 0, 0)]
    need = ds.ds_rows_workspace_bytes(rows)
    assert _attn(lib, rows, ws_bytes=need - 1) == -2
    assert "workspace holds" in _err(lib)
    assert _attn(lib, rows, ws=FAKE + 16) == -3
    assert _attn(lib, rows, ws=0) == -1


def test_alignment(lib):
    assert _attn(lib, [(8, 8, 0, 0)], q=FAKE + 2) == -3
    assert "16-B aligned" in _err(lib)


def test_missing_cache(lib):
    assert _attn(lib, [(8, 8, 0, 0)], kv=False) == -1
    assert "kv cache is NULL" in _err(lib)


def test_topk_overlapping_outputs(lib):
    rs, keep = _set([(600, 512, 0, 0), (600, 512, 100, 1)])
    rc = lib.ds_rows_topk(ctypes.byref(rs), FAKE, 600, FAKE, FAKE, 1 << 30, None)
    assert rc == -1 and "overlap" in _err(lib)


def test_width_contract(lib):
    """Every call: width <= kv_len (no more slots than keys). The top-k and the
    decode select exactly min(512, kv_len); the attention takes any width up to
    that (a caller's shorter index list)."""
    assert _attn(lib, [(5, 6, 0, 0)]) == -1 and "exceeds kv_len" in _err(lib)
    assert lib.ds_rows_workspace_bytes(1, ds._table([(5, 6, 0, 0)])[0]) == 0
    for row in ((600, 100, 0, 0), (300, 299, 0, 0)):
        rs, keep = _set([row])
        rc = lib.ds_rows_topk(ctypes.byref(rs), FAKE, 600, FAKE, FAKE, 1 << 30, None)
        assert rc == -1 and "must be min(512, kv_len)" in _err(lib)
        rc = lib.ds_rows_topk_static(ctypes.byref(rs), FAKE, 600, FAKE, None)
        assert rc == -1 and "must be min(512, kv_len)" in _err(lib)
        rc = lib.ds_rows_decode(ctypes.byref(rs), FAKE, FAKE, FAKE, FAKE, 0, ctypes.c_float(0.04), FAKE, None,
                                None, FAKE, 1 << 30, None)
        assert rc == -1 and "must be min(512, kv_len)" in _err(lib)
    assert lib.ds_rows_workspace_bytes(1, ds._table([(600, 100, 0, 0)])[0]) > 0  # a valid attention table


def test_topk_static_status_checks(lib):
    assert lib.ds_rows_topk_static_status(None, None) == -1 and "status is NULL" in _err(lib)
    assert lib.ds_rows_topk_static_status(FAKE + 2, None) == -3 and "4-byte aligned" in _err(lib)


def test_score_stride(lib):
    rs, keep = _set([(600, 512, 0, 0)])
    rc = lib.ds_rows_indexer_score(ctypes.byref(rs), FAKE, FAKE, FAKE, 599, None)
    assert rc == -1 and "score_stride" in _err(lib)


def test_decode_checks_everything(lib):
    rs, keep = _set([(600, 512, 0, 0)], keys=False)
    rc = lib.ds_rows_decode(ctypes.byref(rs), FAKE, FAKE, FAKE, FAKE, 0, ctypes.c_float(0.04), FAKE, None, None,
                            FAKE, 1 << 30, None)
    assert rc == -1 and "indexer keys are NULL" in _err(lib)


def test_workspace_bytes_grows_with_rows(lib):
    a = ds.ds_rows_workspace_bytes([(131072, 512, 0, 0)])
    b = ds.ds_rows_workspace_bytes([(131072, 512, 512 * i, i) for i in range(8)])
    assert 0 < a < b
    assert b % 256 == 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="launch-failure path is checked without a device only")
def test_cuda_failure_is_reported_without_device(lib):
    """With no CUDA device, a call that passes validation fails at its first
    CUDA call and reports DS_ECUDA (the launch-error path)."""
    rows = [(64, 64, 0, 0)]
    assert _attn(lib, rows, ws_bytes=ds.ds_rows_workspace_bytes(rows)) == -4
    assert "failed" in _err(lib)


def test_python_binding_checks_tensors():
    with pytest.raises(TypeError):
        ds._require(torch.zeros(4, dtype=torch.float32), "x", torch.bfloat16, 4)
    with pytest.raises(ValueError):
        ds._require(torch.zeros(4, dtype=torch.bfloat16), "x", torch.bfloat16, 4)  # not CUDA


# ---------------------------------------------------------------------------
# positioned indexer rows (dispatch_deepseek_indexer_rows checks)
# ---------------------------------------------------------------------------

def _indexer_topk(lib, rows, ws_bytes=1 << 30, ws=FAKE, keys=True, q=FAKE):
    tab, n = ds._indexer_table(rows)
    ptrs = (ctypes.c_void_p * max(1, n))(*[FAKE + 4096 * i for i in range(n)])
    return lib.ds_rows_indexer_topk(n, tab, ptrs if keys else None, q, FAKE, FAKE, ws, ws_bytes, None)


@pytest.mark.parametrize("row,msg", [
    ((0, 1, 0, 0, 0), "kv_len must be nonzero"),
    ((10, 100, 0, 0, 0), "shorter than 25 causal compressed entries"),
    ((10, 3, -1, 0, 0), "offset must be nonnegative"),
    ((10, 0xFFFFFFFF, 0, 0, 0), "position overflows"),
    ((10, 39, 2**31 - 5, 0, 0), "offset plus compressed index exceeds i32"),
    ((10, 3, 0, 0, 0xFFFFFF00), "output range exceeds u32"),
])
def test_indexer_row_checks(lib, row, msg):
    assert _indexer_topk(lib, [row]) in (-1, -2)
    assert msg in _err(lib)
    tab, n = ds._indexer_table([row])
    assert lib.ds_rows_indexer_topk_workspace_bytes(n, tab) == 0


def test_indexer_rows_edges_accepted(lib):
    # valid_count = (start_pos + 1) / 4 may be 0 (no valid key) or equal kv_len.
    for row in [(10, 2, 0, 0, 0), (10, 39, 0, 0, 0), (10, 39, 2**31 - 10, 0, 0)]:
        tab, n = ds._indexer_table([row])
        assert lib.ds_rows_indexer_topk_workspace_bytes(n, tab) > 0, _err(lib)


def test_indexer_rows_outputs_disjoint_and_counts(lib):
    assert _indexer_topk(lib, [(600, 2399, 0, 0, 0), (600, 2399, 0, 1, 511)]) == -1
    assert "overlap" in _err(lib)
    rows9 = [(10, 39, 0, 0, 512 * i) for i in range(9)]
    assert _indexer_topk(lib, rows9) == -1 and "rows must be 1..=8" in _err(lib)


def test_indexer_rows_pointers_and_workspace(lib):
    rows = [(600, 2399, 0, 0, 0)]
    assert _indexer_topk(lib, rows, keys=False) == -1 and "index_keys is NULL" in _err(lib)
    assert _indexer_topk(lib, rows, q=FAKE + 2) == -3
    need = ds.ds_rows_indexer_topk_workspace_bytes(rows)
    assert _indexer_topk(lib, rows, ws_bytes=need - 1) == -2 and "workspace holds" in _err(lib)
    assert _indexer_topk(lib, rows, ws=FAKE + 16) == -3


def test_decode_host_checks(lib):
    rows = [(600, 512, 0, 0), (300, 300, 512, 1)]
    tab, n = ds._table(rows)
    rs, keep = _set(rows)
    call = lambda *a, ws_bytes=1 << 30: lib.ds_rows_decode_host(ctypes.byref(rs), *a, 0, ctypes.c_float(0.05),
                                                                  FAKE, None, None, FAKE, ws_bytes, None)
    assert call(None, FAKE, FAKE, FAKE) == -1 and "host q_index" in _err(lib)
    assert call(FAKE, FAKE, FAKE, None) == -1 and "host q_index" in _err(lib)
    need = lib.ds_rows_decode_host_workspace_bytes(n, tab, 0)
    assert need > lib.ds_rows_workspace_bytes(n, tab)
    assert call(FAKE, FAKE, FAKE, FAKE, ws_bytes=need - 1) == -2 and "workspace holds" in _err(lib)
    assert lib.ds_rows_decode_host_workspace_bytes(n, tab, 32) == 0  # stride below 64
    # Per-row sinks make the staging larger.
    assert lib.ds_rows_decode_host_workspace_bytes(n, tab, 64) > need


def _queries(lib, rows, query_len, ws_bytes=1 << 30, ws=FAKE):
    tab, n = ds._indexer_table(rows)
    ptrs = (ctypes.c_void_p * max(1, n))(*[FAKE + 4096 * i for i in range(n)])
    return lib.ds_rows_indexer_topk_queries(n, tab, query_len, ptrs, FAKE, FAKE, FAKE, ws, ws_bytes, None)


def test_indexer_queries_checks(lib):
    # The last query's count decides: start_pos 35, 4 queries -> (35 + 4) / 4 = 9.
    assert _queries(lib, [(8, 35, 0, 0, 0)], 4) == -1 and "shorter than 9 causal" in _err(lib)
    tab, n = ds._indexer_table([(9, 35, 0, 0, 0)])
    assert lib.ds_rows_indexer_topk_queries_workspace_bytes(n, tab, 4) > 0, _err(lib)
    # Output ranges span 512 x query_len.
    assert _queries(lib, [(600, 2399, 0, 0, 0), (600, 2399, 0, 1, 1024)], 3) == -1 and "overlap" in _err(lib)
    tab, n = ds._indexer_table([(600, 2399, 0, 0, 0), (600, 2399, 0, 3, 1536)])
    assert lib.ds_rows_indexer_topk_queries_workspace_bytes(n, tab, 3) > 0, _err(lib)
    # rows x query_len is bounded; query_len 0 is rejected.
    assert _queries(lib, [(600, 2399, 0, 0, 0)] * 2, 33) == -1 and "rows x query_len" in _err(lib)
    assert _queries(lib, [(600, 2399, 0, 0, 0)], 0) == -1 and "rows x query_len" in _err(lib)
    assert _queries(lib, [(600, 0xFFFFFFFF - 2, 0, 0, 0)], 4) == -1 and "position overflows" in _err(lib)
    # One query is the positioned indexer: the same workspace.
    rows = [(700, 2399, 0, 0, 0), (70000, 9999, 5, 8, 4096)]
    tab, n = ds._indexer_table(rows)
    assert lib.ds_rows_indexer_topk_queries_workspace_bytes(n, tab, 1) == lib.ds_rows_indexer_topk_workspace_bytes(n, tab)
    assert (lib.ds_rows_indexer_topk_queries_workspace_bytes(n, tab, 8)
            > lib.ds_rows_indexer_topk_workspace_bytes(n, tab))
    need = ds.ds_rows_indexer_topk_queries_workspace_bytes([(600, 2399, 0, 0, 0)], 4)
    assert _queries(lib, [(600, 2399, 0, 0, 0)], 4, ws_bytes=need - 1) == -2 and "workspace holds" in _err(lib)


# ---------------------------------------------------------------------------
# KV compressor rows (dispatch_deepseek_compressor_rows checks)
# ---------------------------------------------------------------------------

def _compress(lib, rows, ratio=4, head_dim=128, eps=1e-6, ptr=FAKE):
    tab = (ds.CompressorRow * max(1, len(rows)))(*[ds.CompressorRow(*r) for r in rows])
    return lib.ds_rows_compress_kv(len(rows), tab, ptr, ptr, ptr, ptr, ratio, head_dim, ctypes.c_float(eps), ptr,
                                   None)


STATE = 2 * 4 * 2 * 128 * 4  # bytes of one (4, 128) state


@pytest.mark.parametrize("ratio,head_dim", [(4, 256), (128, 128), (8, 512), (0, 512)])
def test_compressor_shape_checks(lib, ratio, head_dim):
    assert _compress(lib, [(FAKE, FAKE + STATE, 3)], ratio, head_dim) == -1
    assert "(4,128), (4,512) or (128,512)" in _err(lib)


def test_compressor_argument_checks(lib):
    ok_row = (FAKE, FAKE + STATE, 3)
    for eps in (0.0, -1.0, float("inf"), float("nan")):
        assert _compress(lib, [ok_row], eps=eps) == -1 and "epsilon" in _err(lib)
    for pos in (0, 0xFFFFFFFF):
        assert _compress(lib, [(FAKE, FAKE + STATE, pos)]) == -1 and "position" in _err(lib)
    assert _compress(lib, [ok_row], ptr=FAKE + 4) == -3
    assert _compress(lib, [(FAKE, FAKE + STATE - 16, 3)]) == -1 and "overlap" in _err(lib)
    assert _compress(lib, [ok_row, (FAKE + STATE, FAKE + 2 * STATE, 3)]) == -1 and "overlap" in _err(lib)
    assert _compress(lib, [ok_row, (FAKE + 2 * STATE, FAKE + 3 * STATE, 3)]) != -1 or "overlap" not in _err(lib)
    assert _compress(lib, [(FAKE, FAKE + STATE, 3)] * 9) == -1 and "rows must be 1..=8" in _err(lib)


def test_selftest_bounded_wait_validation(lib):
    # Rejected on the host: nothing is launched.
    assert lib.ds_rows_selftest_bounded_wait(None, FAKE, 1_000_000, None) == -1
    assert "non-NULL" in _err(lib)
    assert lib.ds_rows_selftest_bounded_wait(FAKE, None, 1_000_000, None) == -1
    assert lib.ds_rows_selftest_bounded_wait(FAKE, FAKE, 999, None) == -1
    assert "budget_ns" in _err(lib)
    assert lib.ds_rows_selftest_bounded_wait(FAKE, FAKE, 10_000_000_001, None) == -1


def test_status_bits_match_the_binding():
    text = open(HEADER).read()
    assert re.search(r"#define DS_STATUS_WAIT_TIMEOUT 1u", text)
    assert re.search(r"#define DS_STATUS_OVERFLOW 2u", text)
    assert ds.STATUS_WAIT_TIMEOUT == 1 and ds.STATUS_OVERFLOW == 2
