"""Host-side marshalling shared by the benchmark and the tests: bf16 bit
arrays (numpy uint16) as torch bfloat16 device tensors, and an index-key cache
filled with a workload's keys through idx_store_keys."""
from __future__ import annotations

import numpy as np
import torch

from . import dsaidx
from . import workloads as wl


def bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    """uint16 bf16 bit patterns -> a bfloat16 tensor on `device` (bits kept)."""
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).view(
        torch.bfloat16).to(device)


def build_cache(W: wl.Workload, mode: int, fill: int = 0xA5, device="cuda", rotate: bool = False,
                fp4: bool = False):
    """A pool of W.num_blocks blocks in key format `mode` (unused bytes set to
    `fill`) holding every key of W at the slots of its block table (stored
    with the Walsh-Hadamard rotation and / or the fp4 round trip when asked)."""
    cache = dsaidx.IndexCache.allocate(W.num_blocks, W.bs, mode, device=device, fill=fill)
    if sum(W.seq_lens):
        k = bf16_tensor(W.all_keys(), device)
        slots = torch.from_numpy(W.all_slots()).to(device)
        dsaidx.store_keys(cache, k, slots, rotate=rotate, fp4=fp4)
    return cache


def hadamard_rotate_bf16(x: torch.Tensor) -> torch.Tensor:
    """Caller-side rotation of bf16 query rows [..., 128] (the score calls take
    queries already rotated): y = H x with the orthonormal Sylvester-order
    Walsh-Hadamard matrix, in fp64 on the device, rounded to bf16."""
    d = x.shape[-1]
    H = torch.ones((1, 1), dtype=torch.float64, device=x.device)
    while H.shape[0] < d:
        H = torch.cat([torch.cat([H, H], 1), torch.cat([H, -H], 1)], 0)
    y = x.to(torch.float64) @ (H / d ** 0.5).T
    return y.to(torch.float32).to(torch.bfloat16)
