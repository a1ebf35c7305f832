"""Python binding of libdsrows: ragged DeepSeek sparse-attention decode on GB300.

Thin ctypes marshalling over the C-ABI declared in ``include/dsrows.h``. Every
step of the computation runs in the library's CUDA kernels; this module only
checks tensor types and sizes (as the mlx-native dispatch functions of
``src/ops/deepseek_rows.rs`` do with their ``require`` checks), gathers raw
pointers and calls the entry point of the same name. PyTorch provides device
memory and streams.

The library must be built first (``build()``); without it every call raises.
"""

from __future__ import annotations

import ctypes
import os
from typing import Iterable, List, Optional, Sequence

import torch

from . import build as _build

__all__ = [
    "DsRowsError", "Row", "load", "build", "library_path",
    "ds_rows_workspace_bytes", "workspace", "ds_rows_indexer_score", "ds_rows_topk", "ds_rows_topk_static",
    "topk_static_status",
    "ds_rows_sparse_attn", "ds_rows_decode", "ds_rows_version",
    "ds_rows_decode_host_workspace_bytes", "host_workspace", "ds_rows_decode_host",
    "IndexerRow", "ds_rows_indexer_topk_workspace_bytes", "indexer_topk_workspace", "ds_rows_indexer_topk",
    "ds_rows_indexer_topk_queries_workspace_bytes", "ds_rows_indexer_topk_queries",
    "CompressorRow", "ds_rows_compress_kv",
    "STATUS_WAIT_TIMEOUT", "STATUS_OVERFLOW", "workspace_status", "ds_rows_selftest_bounded_wait",
    "ROWS_MAX", "INDEX_HEADS", "INDEX_DIM", "TOP_K", "HEADS", "DIM",
]

ROWS_MAX = 8
INDEX_HEADS = 64
INDEX_DIM = 128
TOP_K = 512
HEADS = 64
DIM = 512

DS_OK = 0
STATUS_WAIT_TIMEOUT = 1  # DS_STATUS_WAIT_TIMEOUT: a bounded device wait gave up
STATUS_OVERFLOW = 2      # DS_STATUS_OVERFLOW: an internal selection check failed


class DsRowsError(RuntimeError):
    """A call rejected by the library (bad argument, size, alignment, CUDA error)."""

    def __init__(self, code: int, message: str):
        super().__init__(f"[{code}] {message}")
        self.code = code


class Row(ctypes.Structure):
    """One entry of the row table: ds_row_t {kv_len, width, index_offset, q_row}."""

    _fields_ = [("kv_len", ctypes.c_uint32), ("width", ctypes.c_uint32),
                ("index_offset", ctypes.c_uint32), ("q_row", ctypes.c_uint32)]


class IndexerRow(ctypes.Structure):
    """One positioned indexer row: ds_indexer_row_t {kv_len, start_pos, offset, q_row, output_offset}."""

    _fields_ = [("kv_len", ctypes.c_uint32), ("start_pos", ctypes.c_uint32), ("offset", ctypes.c_int32),
                ("q_row", ctypes.c_uint32), ("output_offset", ctypes.c_uint32)]


class CompressorRow(ctypes.Structure):
    """One compressor row: ds_compressor_row_t {kv_state, score_state, start_pos} (device pointers)."""

    _fields_ = [("kv_state", ctypes.c_void_p), ("score_state", ctypes.c_void_p), ("start_pos", ctypes.c_uint32)]


class _RowSet(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int), ("table", ctypes.POINTER(Row)),
                ("index_keys", ctypes.POINTER(ctypes.c_void_p)), ("kv", ctypes.POINTER(ctypes.c_void_p))]


_LIB = None


def library_path() -> str:
    return _build.LIB


def build(force: bool = False) -> str:
    """Compile libdsrows.so in-tree (nvcc, sm_103a)."""
    return _build.build(force=force)


def load():
    """Load libdsrows.so; raises if it has not been built."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libdsrows is not built ({path} missing); call "
                           "deepseek_sparse_attention_ragged_gb300.build()")
    lib = ctypes.CDLL(path)
    vp, sz, i32, u32p = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p
    rs = ctypes.POINTER(_RowSet)
    lib.ds_rows_workspace_bytes.argtypes = [i32, ctypes.POINTER(Row)]
    lib.ds_rows_workspace_bytes.restype = sz
    lib.ds_rows_indexer_score.argtypes = [rs, vp, vp, vp, sz, vp]
    lib.ds_rows_indexer_score.restype = i32
    lib.ds_rows_topk.argtypes = [rs, vp, sz, vp, vp, sz, vp]
    lib.ds_rows_topk.restype = i32
    lib.ds_rows_topk_static.argtypes = [rs, vp, sz, vp, vp]
    lib.ds_rows_topk_static.restype = i32
    lib.ds_rows_topk_static_status.argtypes = [vp, vp]
    lib.ds_rows_topk_static_status.restype = i32
    lib.ds_rows_sparse_attn.argtypes = [rs, vp, vp, sz, vp, ctypes.c_float, vp, u32p, vp, sz, vp]
    lib.ds_rows_sparse_attn.restype = i32
    lib.ds_rows_decode.argtypes = [rs, vp, vp, vp, vp, sz, ctypes.c_float, vp, vp, u32p, vp, sz, vp]
    lib.ds_rows_decode.restype = i32
    lib.ds_rows_decode_host_workspace_bytes.argtypes = [i32, ctypes.POINTER(Row), sz]
    lib.ds_rows_decode_host_workspace_bytes.restype = sz
    lib.ds_rows_decode_host.argtypes = [rs, vp, vp, vp, vp, sz, ctypes.c_float, vp, vp, u32p, vp, sz, vp]
    lib.ds_rows_decode_host.restype = i32
    lib.ds_rows_indexer_topk_workspace_bytes.argtypes = [i32, ctypes.POINTER(IndexerRow)]
    lib.ds_rows_indexer_topk_workspace_bytes.restype = sz
    lib.ds_rows_indexer_topk.argtypes = [i32, ctypes.POINTER(IndexerRow), ctypes.POINTER(vp), vp, vp, vp, vp, sz, vp]
    lib.ds_rows_indexer_topk.restype = i32
    lib.ds_rows_indexer_topk_queries_workspace_bytes.argtypes = [i32, ctypes.POINTER(IndexerRow), ctypes.c_uint32]
    lib.ds_rows_indexer_topk_queries_workspace_bytes.restype = sz
    lib.ds_rows_indexer_topk_queries.argtypes = [i32, ctypes.POINTER(IndexerRow), ctypes.c_uint32,
                                                 ctypes.POINTER(vp), vp, vp, vp, vp, sz, vp]
    lib.ds_rows_indexer_topk_queries.restype = i32
    lib.ds_rows_compress_kv.argtypes = [i32, ctypes.POINTER(CompressorRow), vp, vp, vp, vp, ctypes.c_uint32,
                                         ctypes.c_uint32, ctypes.c_float, vp, vp]
    lib.ds_rows_compress_kv.restype = i32
    lib.ds_rows_selftest_bounded_wait.argtypes = [vp, vp, ctypes.c_uint64, vp]
    lib.ds_rows_selftest_bounded_wait.restype = i32
    lib.ds_rows_last_error.argtypes = []
    lib.ds_rows_last_error.restype = ctypes.c_char_p
    lib.ds_rows_version.argtypes = []
    lib.ds_rows_version.restype = ctypes.c_char_p
    _LIB = lib
    return lib


def ds_rows_version() -> str:
    return load().ds_rows_version().decode()


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------

def _table(rows) -> "ctypes.Array":
    rows = list(rows)
    arr = (Row * max(1, len(rows)))()
    for i, r in enumerate(rows):
        if isinstance(r, Row):
            arr[i] = r
        elif hasattr(r, "kv_len"):
            arr[i] = Row(r.kv_len, r.width, r.index_offset, r.q_row)
        else:
            arr[i] = Row(*r)
    return arr, len(rows)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _check(lib, rc: int):
    if rc != DS_OK:
        raise DsRowsError(rc, lib.ds_rows_last_error().decode())


def _require(t: Optional[torch.Tensor], name: str, dtype, numel: int, *, optional=False):
    """`t` must be a contiguous CUDA tensor of `dtype` holding >= numel elements."""
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() < numel:
        raise ValueError(f"{name} holds {t.numel()} elements, needs {numel}")


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _rowset(tab, n, keys=None, kv=None, rows=None):
    ks = kvs = None
    if keys is not None:
        ks = (ctypes.c_void_p * n)(*[k.data_ptr() for k in keys])
    if kv is not None:
        kvs = (ctypes.c_void_p * n)(*[k.data_ptr() for k in kv])
    rs = _RowSet(n, ctypes.cast(tab, ctypes.POINTER(Row)),
                 ctypes.cast(ks, ctypes.POINTER(ctypes.c_void_p)) if ks is not None else None,
                 ctypes.cast(kvs, ctypes.POINTER(ctypes.c_void_p)) if kvs is not None else None)
    return rs, (ks, kvs)


def _rows_list(rows) -> List:
    out = []
    for r in rows:
        if isinstance(r, Row) or hasattr(r, "kv_len"):
            out.append((int(r.kv_len), int(r.width), int(r.index_offset), int(r.q_row)))
        else:
            out.append(tuple(int(x) for x in r))
    return out


def _check_caches(caches: Sequence[torch.Tensor], rows, dim: int, name: str):
    if len(caches) != len(rows):
        raise ValueError(f"{name}: {len(caches)} caches for {len(rows)} rows")
    for e, (c, r) in enumerate(zip(caches, rows)):
        _require(c, f"{name}[{e}]", torch.bfloat16, r[0] * dim)


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------

def ds_rows_workspace_bytes(rows) -> int:
    lib = load()
    tab, n = _table(rows)
    b = lib.ds_rows_workspace_bytes(n, tab)
    if b == 0:
        raise DsRowsError(-1, lib.ds_rows_last_error().decode())
    return int(b)


def workspace(rows, device=None) -> torch.Tensor:
    """A workspace tensor (uint8, 256-byte aligned by the caching allocator)."""
    return torch.empty(ds_rows_workspace_bytes(rows), dtype=torch.uint8,
                       device=device if device is not None else "cuda")


def workspace_status(workspace_t: torch.Tensor) -> int:
    """The device status word at the head of a workspace (the STATUS_* bits of
    the last call that used it). Reads 4 bytes back to the host, so it waits
    for the work queued on the workspace's device."""
    if workspace_t.dtype != torch.uint8 or workspace_t.numel() < 4:
        raise DsRowsError(-1, "workspace_status: a uint8 workspace tensor is required")
    return int(workspace_t[:4].view(torch.int32).item()) & 0xFFFFFFFF


def ds_rows_selftest_bounded_wait(budget_ns: int = 1_000_000, device=None, stream=None):
    """Run the library's bounded mbarrier wait on a phase that completes and on
    one that nothing completes (giving up after budget_ns); returns
    (status, completed_wait_ok, abandoned_wait_gave_up)."""
    lib = load()
    dev = torch.device(device if device is not None else "cuda")
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    result = torch.full((2,), 7, dtype=torch.int32, device=dev)
    _check(lib, lib.ds_rows_selftest_bounded_wait(status.data_ptr(), result.data_ptr(), int(budget_ns),
                                                  _stream(stream)))
    r = result.cpu().tolist()
    return int(status.item()) & 0xFFFFFFFF, r[0] == 1, r[1] == 1


def ds_rows_indexer_score(rows, q_index, w_index, index_keys, scores, score_stride=None, stream=None):
    """Indexer scores of every row into `scores` (fp32, row e at e*score_stride)."""
    lib = load()
    rl = _rows_list(rows)
    q_rows = max(r[3] for r in rl) + 1
    _require(q_index, "q_index", torch.bfloat16, q_rows * INDEX_HEADS * INDEX_DIM)
    _require(w_index, "w_index", torch.float32, q_rows * INDEX_HEADS)
    _check_caches(index_keys, rl, INDEX_DIM, "index_keys")
    if score_stride is None:
        score_stride = scores.shape[-1] if scores.dim() > 1 else max(r[0] for r in rl)
    _require(scores, "scores", torch.float32, (len(rl) - 1) * score_stride + max(r[0] for r in rl))
    tab, n = _table(rl)
    rs, keep = _rowset(tab, n, keys=index_keys)
    _check(lib, lib.ds_rows_indexer_score(ctypes.byref(rs), _ptr(q_index), _ptr(w_index), _ptr(scores),
                                          int(score_stride), _stream(stream)))


def ds_rows_topk(rows, scores, score_stride, indices, workspace_t, stream=None):
    """Top-`width` indices of each row's scores into `indices` at index_offset."""
    lib = load()
    rl = _rows_list(rows)
    _require(scores, "scores", torch.float32, (len(rl) - 1) * score_stride + max(r[0] for r in rl))
    _require(indices, "indices", torch.int32, max(r[2] + r[1] for r in rl))
    _require(workspace_t, "workspace", torch.uint8, 0)
    tab, n = _table(rl)
    rs, keep = _rowset(tab, n)
    _check(lib, lib.ds_rows_topk(ctypes.byref(rs), _ptr(scores), int(score_stride), _ptr(indices),
                                 _ptr(workspace_t), workspace_t.numel(), _stream(stream)))


def ds_rows_topk_static(rows, scores, score_stride, indices, stream=None):
    """ds_rows_topk without a workspace: for callers that cannot allocate device
    memory when they run this stage. The library keeps the scratch in one fixed
    array per device, shared by every call on that device: calls that overlap
    on the GPU race on it, so order them (one stream, or events)."""
    lib = load()
    rl = _rows_list(rows)
    _require(scores, "scores", torch.float32, (len(rl) - 1) * score_stride + max(r[0] for r in rl))
    _require(indices, "indices", torch.int32, max(r[2] + r[1] for r in rl))
    tab, n = _table(rl)
    rs, keep = _rowset(tab, n)
    _check(lib, lib.ds_rows_topk_static(ctypes.byref(rs), _ptr(scores), int(score_stride), _ptr(indices),
                                        _stream(stream)))


def topk_static_status(device=None, stream=None) -> int:
    """The status word of ds_rows_topk_static on `device` (the STATUS_* bits of
    the last call there). Reads 4 bytes back to the host, so it waits for the
    work queued on `stream`."""
    lib = load()
    dev = torch.device(device if device is not None else "cuda")
    word = torch.full((1,), -1, dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        _check(lib, lib.ds_rows_topk_static_status(word.data_ptr(), _stream(stream)))
        return int(word.item()) & 0xFFFFFFFF


def _attn_checks(rl, q_attn, sinks, sinks_row_stride, out, kv, invalid):
    q_rows = max(r[3] for r in rl) + 1
    _require(q_attn, "q_attn", torch.bfloat16, q_rows * HEADS * DIM)
    _require(out, "out", torch.bfloat16, q_rows * HEADS * DIM)
    _require(sinks, "sinks", torch.float32, HEADS if sinks_row_stride == 0 else q_rows * sinks_row_stride)
    _require(invalid, "invalid", torch.int32, q_rows * HEADS, optional=True)
    _check_caches(kv, rl, DIM, "kv")


def ds_rows_sparse_attn(rows, q_attn, sinks, sinks_row_stride, indices, scale, out, kv,
                        invalid=None, workspace_t=None, stream=None):
    """Gather + sink-softmax attention of each row over its selected indices."""
    lib = load()
    rl = _rows_list(rows)
    _attn_checks(rl, q_attn, sinks, sinks_row_stride, out, kv, invalid)
    _require(indices, "indices", torch.int32, max(r[2] + r[1] for r in rl))
    if workspace_t is None:
        workspace_t = workspace(rl, q_attn.device)
    tab, n = _table(rl)
    rs, keep = _rowset(tab, n, kv=kv)
    _check(lib, lib.ds_rows_sparse_attn(ctypes.byref(rs), _ptr(q_attn), _ptr(sinks), int(sinks_row_stride),
                                        _ptr(indices), float(scale), _ptr(out), _ptr(invalid),
                                        _ptr(workspace_t), workspace_t.numel(), _stream(stream)))


def ds_rows_decode(rows, q_index, w_index, index_keys, q_attn, kv, sinks, sinks_row_stride, scale, out,
                   indices=None, invalid=None, workspace_t=None, stream=None):
    """The whole decode step: indexer score -> top-k -> gather + sink attention."""
    lib = load()
    rl = _rows_list(rows)
    q_rows = max(r[3] for r in rl) + 1
    _require(q_index, "q_index", torch.bfloat16, q_rows * INDEX_HEADS * INDEX_DIM)
    _require(w_index, "w_index", torch.float32, q_rows * INDEX_HEADS)
    _check_caches(index_keys, rl, INDEX_DIM, "index_keys")
    _attn_checks(rl, q_attn, sinks, sinks_row_stride, out, kv, invalid)
    _require(indices, "indices", torch.int32, max(r[2] + r[1] for r in rl), optional=True)
    if workspace_t is None:
        workspace_t = workspace(rl, q_attn.device)
    tab, n = _table(rl)
    rs, keep = _rowset(tab, n, keys=index_keys, kv=kv)
    _check(lib, lib.ds_rows_decode(ctypes.byref(rs), _ptr(q_index), _ptr(w_index), _ptr(q_attn), _ptr(sinks),
                                   int(sinks_row_stride), float(scale), _ptr(out), _ptr(indices), _ptr(invalid),
                                   _ptr(workspace_t), workspace_t.numel(), _stream(stream)))


def _require_host(t: Optional[torch.Tensor], name: str, dtype, numel: int, *, optional=False):
    """`t` must be a contiguous CPU tensor of `dtype` holding >= numel elements
    (pinned, for the library's copies to be asynchronous)."""
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() < numel:
        raise ValueError(f"{name} holds {t.numel()} elements, needs {numel}")


def ds_rows_decode_host_workspace_bytes(rows, sinks_row_stride=0) -> int:
    lib = load()
    tab, n = _table(_rows_list(rows))
    b = lib.ds_rows_decode_host_workspace_bytes(n, tab, int(sinks_row_stride))
    if b == 0:
        raise DsRowsError(-1, lib.ds_rows_last_error().decode() or "invalid row table")
    return int(b)


def host_workspace(rows, sinks_row_stride=0, device=None) -> torch.Tensor:
    """A workspace tensor for ds_rows_decode_host (uint8, 256-byte aligned)."""
    return torch.empty(ds_rows_decode_host_workspace_bytes(rows, sinks_row_stride), dtype=torch.uint8,
                       device=device if device is not None else "cuda")


def ds_rows_decode_host(rows, q_index, w_index, index_keys, q_attn, kv, sinks, sinks_row_stride, scale, out,
                        indices=None, invalid=None, workspace_t=None, stream=None):
    """ds_rows_decode with the step's inputs and outputs in host memory (pinned
    CPU tensors); the caches stay on the device. Asynchronous on `stream`:
    synchronise it before reading `out`."""
    lib = load()
    rl = _rows_list(rows)
    q_rows = max(r[3] for r in rl) + 1
    _require_host(q_index, "q_index", torch.bfloat16, q_rows * INDEX_HEADS * INDEX_DIM)
    _require_host(w_index, "w_index", torch.float32, q_rows * INDEX_HEADS)
    _require_host(q_attn, "q_attn", torch.bfloat16, q_rows * HEADS * DIM)
    _require_host(sinks, "sinks", torch.float32, HEADS if sinks_row_stride == 0 else
                  (q_rows - 1) * sinks_row_stride + HEADS)
    _require_host(out, "out", torch.bfloat16, q_rows * HEADS * DIM)
    _require_host(indices, "indices", torch.int32, max(r[2] + r[1] for r in rl), optional=True)
    _require_host(invalid, "invalid", torch.int32, q_rows * HEADS, optional=True)
    _check_caches(index_keys, rl, INDEX_DIM, "index_keys")
    _check_caches(kv, rl, DIM, "kv")
    if workspace_t is None:
        workspace_t = host_workspace(rl, sinks_row_stride, kv[0].device)
    tab, n = _table(rl)
    rs, keep = _rowset(tab, n, keys=index_keys, kv=kv)
    _check(lib, lib.ds_rows_decode_host(ctypes.byref(rs), _ptr(q_index), _ptr(w_index), _ptr(q_attn), _ptr(sinks),
                                        int(sinks_row_stride), float(scale), _ptr(out), _ptr(indices),
                                        _ptr(invalid), _ptr(workspace_t), workspace_t.numel(), _stream(stream)))


# ---------------------------------------------------------------------------
# positioned indexer + causal top-512
# ---------------------------------------------------------------------------

def _indexer_table(rows):
    rows = list(rows)
    arr = (IndexerRow * max(1, len(rows)))()
    for i, r in enumerate(rows):
        if isinstance(r, IndexerRow):
            arr[i] = r
        elif hasattr(r, "start_pos"):
            arr[i] = IndexerRow(r.kv_len, r.start_pos, r.offset, r.q_row, r.output_offset)
        else:
            arr[i] = IndexerRow(*r)
    return arr, len(rows)


def ds_rows_indexer_topk_queries_workspace_bytes(rows, query_len=1) -> int:
    lib = load()
    tab, n = _indexer_table(rows)
    b = lib.ds_rows_indexer_topk_queries_workspace_bytes(n, tab, int(query_len))
    if b == 0:
        raise DsRowsError(-1, lib.ds_rows_last_error().decode())
    return int(b)


def ds_rows_indexer_topk_workspace_bytes(rows) -> int:
    lib = load()
    tab, n = _indexer_table(rows)
    b = lib.ds_rows_indexer_topk_workspace_bytes(n, tab)
    if b == 0:
        raise DsRowsError(-1, lib.ds_rows_last_error().decode())
    return int(b)


def indexer_topk_workspace(rows, device=None, query_len=1) -> torch.Tensor:
    """A workspace tensor for ds_rows_indexer_topk(_queries) (uint8, 256-byte aligned)."""
    return torch.empty(ds_rows_indexer_topk_queries_workspace_bytes(rows, query_len), dtype=torch.uint8,
                       device=device if device is not None else "cuda")


def _indexer_call(fn, rows, query_len, q_index, w_index, index_keys, indices, workspace_t, stream):
    lib = load()
    tab, n = _indexer_table(rows)
    q_rows = max(tab[e].q_row for e in range(n)) + query_len
    _require(q_index, "q_index", torch.bfloat16, q_rows * INDEX_HEADS * INDEX_DIM)
    _require(w_index, "w_index", torch.float32, q_rows * INDEX_HEADS)
    if len(index_keys) != n:
        raise ValueError(f"index_keys: {len(index_keys)} caches for {n} rows")
    for e in range(n):
        _require(index_keys[e], f"index_keys[{e}]", torch.bfloat16, tab[e].kv_len * INDEX_DIM)
    _require(indices, "indices", torch.int32, max(tab[e].output_offset for e in range(n)) + TOP_K * query_len)
    if workspace_t is None:
        workspace_t = indexer_topk_workspace(list(tab)[:n], q_index.device, query_len)
    ks = (ctypes.c_void_p * n)(*[k.data_ptr() for k in index_keys])
    args = (_ptr(q_index), _ptr(w_index), _ptr(indices), _ptr(workspace_t), workspace_t.numel(), _stream(stream))
    if fn == "single":
        _check(lib, lib.ds_rows_indexer_topk(n, tab, ks, *args))
    else:
        _check(lib, lib.ds_rows_indexer_topk_queries(n, tab, int(query_len), ks, *args))


def ds_rows_indexer_topk(rows, q_index, w_index, index_keys, indices, workspace_t=None, stream=None):
    """Positioned indexer score and causal top-512 of each row (IndexerRow entries):
    512 indices (+ offset, -1 fill) per row at output_offset."""
    _indexer_call("single", rows, 1, q_index, w_index, index_keys, indices, workspace_t, stream)


def ds_rows_indexer_topk_queries(rows, query_len, q_index, w_index, index_keys, indices, workspace_t=None,
                                 stream=None):
    """ds_rows_indexer_topk for query_len consecutive queries per row: query j of a
    row uses query row q_row + j, position start_pos + j, and writes its 512
    indices at output_offset + 512 j."""
    _indexer_call("queries", rows, query_len, q_index, w_index, index_keys, indices, workspace_t, stream)


# ---------------------------------------------------------------------------
# learned KV compressor, one decode token per row
# ---------------------------------------------------------------------------

def ds_rows_compress_kv(kv_states, score_states, start_pos, kv, score, ape, norm, ratio, head_dim, epsilon, out,
                        stream=None):
    """One token of the learned KV compressor per row. kv_states / score_states:
    per-row fp32 [coff*ratio, coff*head_dim] CUDA tensors, updated in place;
    start_pos: per-row positions; kv, score fp32 [rows, coff*head_dim]; ape
    fp32 [ratio, coff*head_dim]; norm fp32 [head_dim]; out bf16 [rows, head_dim]."""
    lib = load()
    n = len(start_pos)
    if len(kv_states) != n or len(score_states) != n:
        raise ValueError("one kv_state, score_state and start_pos per row")
    coff = 2 if ratio == 4 else 1
    proj = coff * head_dim
    for e in range(n):
        _require(kv_states[e], f"kv_states[{e}]", torch.float32, coff * ratio * proj)
        _require(score_states[e], f"score_states[{e}]", torch.float32, coff * ratio * proj)
    _require(kv, "kv", torch.float32, n * proj)
    _require(score, "score", torch.float32, n * proj)
    _require(ape, "ape", torch.float32, ratio * proj)
    _require(norm, "norm", torch.float32, head_dim)
    _require(out, "out", torch.bfloat16, n * head_dim)
    tab = (CompressorRow * max(1, n))()
    for e in range(n):
        tab[e] = CompressorRow(kv_states[e].data_ptr(), score_states[e].data_ptr(), int(start_pos[e]))
    _check(lib, lib.ds_rows_compress_kv(n, tab, _ptr(kv), _ptr(score), _ptr(ape), _ptr(norm), int(ratio),
                                        int(head_dim), float(epsilon), _ptr(out), _stream(stream)))
