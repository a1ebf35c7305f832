"""Upload a `workloads.Workload` to a CUDA device as torch tensors (no arithmetic)."""

from __future__ import annotations

import dataclasses
from typing import List

import numpy as np
import torch


def bf16_tensor(bits: np.ndarray, device) -> torch.Tensor:
    """uint16 bf16 bit patterns -> torch.bfloat16 tensor on `device` (same bits)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).to(device)


@dataclasses.dataclass
class DeviceWorkload:
    rows: list
    q_index: torch.Tensor
    w_index: torch.Tensor
    keys: List[torch.Tensor]
    q_attn: torch.Tensor
    kv: List[torch.Tensor]
    sinks: torch.Tensor
    sinks_row_stride: int
    scale: float


def to_device(wl, device="cuda") -> DeviceWorkload:
    return DeviceWorkload(
        rows=list(wl.rows),
        q_index=bf16_tensor(wl.q_index, device),
        w_index=torch.from_numpy(np.ascontiguousarray(wl.w_index)).to(device),
        keys=[bf16_tensor(k, device) for k in wl.keys],
        q_attn=bf16_tensor(wl.q_attn, device),
        kv=[bf16_tensor(k, device) for k in wl.kv],
        sinks=torch.from_numpy(np.ascontiguousarray(wl.sinks)).to(device),
        sinks_row_stride=wl.sinks_row_stride,
        scale=float(wl.scale),
    )
