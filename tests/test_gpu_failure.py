"""Device-side failure detection without a fault: the library's bounded wait
gives up on a phase that nothing completes, records the timeout in the status
word, and the device stays usable; a normal call leaves the status clear."""

import time

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


@pytest.mark.parametrize("budget_ns", [100_000, 5_000_000])
def test_bounded_wait_gives_up_and_reports(budget_ns):
    t0 = time.perf_counter()
    status, completed_ok, gave_up = ds.ds_rows_selftest_bounded_wait(budget_ns)
    elapsed = time.perf_counter() - t0
    assert completed_ok, "a wait on a completed phase must succeed"
    assert gave_up, "a wait on a phase nothing completes must give up"
    assert status == ds.STATUS_WAIT_TIMEOUT
    assert elapsed < 5.0


def test_device_usable_after_timeout_and_status_clear_after_decode():
    ds.ds_rows_selftest_bounded_wait(1_000_000)
    dev = to_device(workloads.config(0), "cuda")
    ws = ds.workspace(dev.rows)
    ws.fill_(0xFF)  # a stale status word must not survive the call
    out = torch.empty((1, 64, 512), dtype=torch.bfloat16, device="cuda")
    ds.ds_rows_decode(dev.rows, dev.q_index, dev.w_index, dev.keys, dev.q_attn, dev.kv, dev.sinks,
                      dev.sinks_row_stride, dev.scale, out, workspace_t=ws)
    torch.cuda.synchronize()
    assert ds.workspace_status(ws) == 0
    assert torch.isfinite(out.float()).all()
