"""The host-buffer decode (ds_rows_decode_host) against the device-buffer
decode (ds_rows_decode), through the C-ABI: the same step with the inputs in
pinned host memory and the outputs copied back must be bitwise the same, for
dense query rows (whole-array copies) and sparse ones (per-row copies)."""

import functools

import numpy as np
import pytest
import torch

import deepseek_sparse_attention_ragged_gb300 as ds
import workloads
from workloads.device import to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    ds.build()
    ds.load()


@functools.lru_cache(maxsize=None)
def cfg_dev(i):
    return to_device(workloads.config(i), "cuda")


def device_decode(dev, rows, keys, kv):
    nq = max(r.q_row for r in rows) + 1
    out = torch.full((nq, 64, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    n_idx = max(r.index_offset + r.width for r in rows)
    idx = torch.full((n_idx,), -7, dtype=torch.int32, device="cuda")
    inv = torch.full((nq, 64), 7, dtype=torch.int32, device="cuda")
    ws = ds.workspace(rows)
    ds.ds_rows_decode(rows, dev.q_index, dev.w_index, keys, dev.q_attn, kv, dev.sinks, dev.sinks_row_stride,
                      dev.scale, out, indices=idx, invalid=inv, workspace_t=ws)
    torch.cuda.synchronize()
    assert ds.workspace_status(ws) == 0
    return out.cpu(), idx.cpu(), inv.cpu()


def host_decode(dev, rows, keys, kv, stream=None, pinned=True):
    nq = max(r.q_row for r in rows) + 1
    pin = (lambda t: t.pin_memory()) if pinned else (lambda t: t)
    h_qI, h_wI, h_qA, h_sk = (pin(t.cpu()) for t in (dev.q_index, dev.w_index, dev.q_attn, dev.sinks))
    out = pin(torch.full((nq, 64, 512), float("nan"), dtype=torch.bfloat16))
    n_idx = max(r.index_offset + r.width for r in rows)
    idx = pin(torch.full((n_idx,), -7, dtype=torch.int32))
    inv = pin(torch.full((nq, 64), 7, dtype=torch.int32))
    ws = ds.host_workspace(rows, dev.sinks_row_stride)
    ds.ds_rows_decode_host(rows, h_qI, h_wI, keys, h_qA, kv, h_sk, dev.sinks_row_stride, dev.scale, out,
                           indices=idx, invalid=inv, workspace_t=ws, stream=stream)
    (stream or torch.cuda.current_stream()).synchronize()
    assert ds.workspace_status(ws) == 0
    return out, idx, inv


@pytest.mark.parametrize("i,pinned", [(1, True), (2, True), (4, True), (2, False), (4, False)])
def test_host_decode_equals_device_decode(i, pinned):
    """Pinned host arrays are read and written in place by the kernels;
    pageable ones go through device staging and copies."""
    dev = cfg_dev(i)
    a = device_decode(dev, dev.rows, dev.keys, dev.kv)
    b = host_decode(dev, dev.rows, dev.keys, dev.kv, pinned=pinned)
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1], b[1])
    assert torch.equal(a[2], b[2])


@pytest.mark.parametrize("pinned", [True, False])
def test_host_decode_sparse_query_rows_on_another_stream(pinned):
    # Entries 1 and 3 only: query rows 1 and 3 of 4, so each copy is per entry
    # and rows 0 and 2 of the host outputs stay untouched.
    dev = cfg_dev(2)
    rows = [dev.rows[1], dev.rows[3]]
    keys, kv = [dev.keys[1], dev.keys[3]], [dev.kv[1], dev.kv[3]]
    a = device_decode(dev, rows, keys, kv)
    s = torch.cuda.Stream()
    b = host_decode(dev, rows, keys, kv, stream=s, pinned=pinned)
    for r in rows:
        assert torch.equal(a[0][r.q_row].view(torch.int16), b[0][r.q_row].view(torch.int16))
        assert torch.equal(a[2][r.q_row], b[2][r.q_row])
        sl = slice(r.index_offset, r.index_offset + r.width)
        assert torch.equal(a[1][sl], b[1][sl])
    for q in (0, 2):
        assert torch.isnan(b[0][q].float()).all()
        assert (b[2][q] == 7).all()


def test_host_decode_repeated_calls_on_one_workspace():
    """Back-to-back calls on one stream and one workspace, each with other
    queries: every call's outputs are its own."""
    dev = cfg_dev(2)
    wl = workloads.config(2)
    ws = ds.host_workspace(dev.rows, dev.sinks_row_stride, "cuda")
    outs = []
    s = torch.cuda.Stream()
    pinned = []
    for k in range(3):
        qI, wI, qA = workloads.draw_queries(wl, 2000 + k)
        from workloads.device import bf16_tensor
        h = (bf16_tensor(qI, "cpu").pin_memory(), torch.from_numpy(wI).pin_memory(),
             bf16_tensor(qA, "cpu").pin_memory(), dev.sinks.cpu().pin_memory())
        out = torch.empty((8, 64, 512), dtype=torch.bfloat16).pin_memory()
        pinned.append((h, out))
        ds.ds_rows_decode_host(dev.rows, h[0], h[1], dev.keys, h[2], dev.kv, h[3], dev.sinks_row_stride,
                               dev.scale, out, workspace_t=ws, stream=s)
    s.synchronize()
    assert ds.workspace_status(ws) == 0
    for k, (h, out) in enumerate(pinned):
        ref = torch.empty((8, 64, 512), dtype=torch.bfloat16, device="cuda")
        ds.ds_rows_decode(dev.rows, h[0].cuda(), h[1].cuda(), dev.keys, h[2].cuda(), dev.kv, h[3].cuda(),
                          dev.sinks_row_stride, dev.scale, ref)
        torch.cuda.synchronize()
        assert torch.equal(ref.cpu().view(torch.int16), out.view(torch.int16)), f"call {k}"


def test_host_decode_in_a_cuda_graph():
    """The call can be captured; a replay with new host inputs gives the decode
    of those inputs."""
    from workloads.device import bf16_tensor
    dev = cfg_dev(2)
    wl = workloads.config(2)
    s = torch.cuda.Stream()
    ws = ds.host_workspace(dev.rows, dev.sinks_row_stride, "cuda")
    h_qI, h_wI, h_qA = (dev.q_index.cpu().pin_memory(), dev.w_index.cpu().pin_memory(),
                        dev.q_attn.cpu().pin_memory())
    h_sk = dev.sinks.cpu().pin_memory()
    out = torch.empty((8, 64, 512), dtype=torch.bfloat16).pin_memory()
    call = lambda: ds.ds_rows_decode_host(dev.rows, h_qI, h_wI, dev.keys, h_qA, dev.kv, h_sk, dev.sinks_row_stride,
                                          dev.scale, out, workspace_t=ws, stream=s)
    with torch.cuda.stream(s):
        call()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    qI, wI, qA = workloads.draw_queries(wl, 3000)
    h_qI.copy_(bf16_tensor(qI, "cpu"))
    h_wI.copy_(torch.from_numpy(wI))
    h_qA.copy_(bf16_tensor(qA, "cpu"))
    with torch.cuda.stream(s):
        g.replay()
    s.synchronize()
    assert ds.workspace_status(ws) == 0
    ref = torch.empty((8, 64, 512), dtype=torch.bfloat16, device="cuda")
    ds.ds_rows_decode(dev.rows, h_qI.cuda(), h_wI.cuda(), dev.keys, h_qA.cuda(), dev.kv, dev.sinks,
                      dev.sinks_row_stride, dev.scale, ref)
    torch.cuda.synchronize()
    assert torch.equal(ref.cpu().view(torch.int16), out.view(torch.int16))
