"""The N-GPU path is N independent replicas: the only cross-rank steps are
the barrier and the maximum of the ranks' times. Checked with world_size 2
over gloo on the CPU (no GPU needed)."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from deepseek_sparse_attention_ragged_gb300.replicas import job_rate, max_over_ranks


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        # The slower replica (rank 1: 7.5 ms) bounds the job.
        total_ms = 5.0 if rank == 0 else 7.5
        worst = max_over_ranks(total_ms)
        rate = job_rate(world, 8, 100, worst)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{worst} {rate}\n")
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    for r in range(world):
        worst, rate = map(float, (tmp_path / f"rank{r}.txt").read_text().split())
        assert worst == 7.5
        # 2 replicas x 8 rows x 100 steps in 7.5 ms
        assert rate == pytest.approx(2 * 8 * 100 / 7.5e-3)


def test_single_process_needs_no_group():
    assert not dist.is_initialized()
    assert max_over_ranks(3.25) == 3.25
    assert job_rate(1, 8, 10, 2.0) == pytest.approx(8 * 10 / 2e-3)
    with pytest.raises(ValueError):
        job_rate(1, 8, 10, 0.0)
