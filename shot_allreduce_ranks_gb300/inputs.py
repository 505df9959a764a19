"""Seeded synthetic inputs for the virtual-rank allreduce.

This module only draws numbers; it holds none of the reduction's arithmetic,
so both the CUDA path's tests and the oracle can be fed from it.

Recipe (the pages use no dataset; their workloads are bf16 tensors of the
shapes in the aiter write-mode table and the helion one-shot size sweep):
  * ``normal``: rank r of seed s draws ``torch.randn(N)`` in fp32 from a CPU
    generator seeded with ``s * 1_000_003 + r`` and casts it to bf16.
  * ``ints``: same seeding, ``torch.randint(-8, 9, (N,))`` (uniform integers in
    [-8, 8], exact in bf16), cast to bf16.  Any rank-order sum of up to 8 of
    them is an integer of magnitude <= 64, exactly representable, so the
    result is independent of summation order.
  * ``position``: a position- and rank-dependent integer fill
    ``((7 * i + 13 * r) % 17) - 8`` so that a permutation of blocks, offsets or
    ranks cannot produce the right answer.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

SEED_STRIDE = 1_000_003


@dataclass(frozen=True)
class Workload:
    name: str
    R: int
    count: int
    fill: str = "normal"
    shape: tuple = ()

    @property
    def bytes_per_rank(self) -> int:
        return 2 * self.count


def _shape_workloads():
    out = {}
    out["r8_4096"] = Workload("r8_4096", 8, 4096, "normal", (4096,))
    for rows, cols in [(440, 5120), (512, 5120), (512, 7168), (512, 8192),
                       (632, 5120), (680, 5120)]:
        name = "r8_%dx%d" % (rows, cols)
        out[name] = Workload(name, 8, rows * cols, "normal", (rows, cols))
    for k in range(9):
        n = 4096 << k
        label = "%dk" % (n // 1024) if n < (1 << 20) else "1m"
        for fill in ("ints", "normal"):
            name = "r8_%s_%s" % (label, fill)
            out[name] = Workload(name, 8, n, fill, (n,))
    for R in (4, 8):
        name = "r%d_64mib" % R
        out[name] = Workload(name, R, 33_554_432, "normal", (33_554_432,))
    return out


#: Every workload named by the five benchmark configurations.
WORKLOADS = _shape_workloads()


def generator(seed: int, rank: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed * SEED_STRIDE + rank)
    return g


def rank_input(count: int, rank: int, seed: int = 0, fill: str = "normal",
               dtype=torch.bfloat16) -> torch.Tensor:
    """One rank's input as a CPU tensor of ``count`` elements of ``dtype``
    (bf16 by default; fp16 and fp32 draw the same fp32 numbers)."""
    if fill == "normal":
        x = torch.randn(count, dtype=torch.float32, generator=generator(seed, rank))
        return x.to(dtype)
    if fill == "ints":
        x = torch.randint(-8, 9, (count,), dtype=torch.int32, generator=generator(seed, rank))
        return x.to(dtype)
    if fill == "position":
        i = torch.arange(count, dtype=torch.int64)
        return (((7 * i + 13 * rank) % 17) - 8).to(dtype)
    if fill == "ones":
        return torch.ones(count, dtype=dtype)
    raise ValueError("unknown fill %r" % fill)


def make_inputs(R: int, count: int, seed: int = 0, fill: str = "normal", dtype=torch.bfloat16):
    """All R ranks' inputs as CPU tensors."""
    return [rank_input(count, r, seed, fill, dtype) for r in range(R)]


def bits(t: torch.Tensor) -> np.ndarray:
    """The bit patterns of a CPU tensor (uint16 for bf16/fp16, uint32 for
    fp32; no copy)."""
    if t.device.type != "cpu":
        raise TypeError("expected a CPU tensor")
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.contiguous().view(torch.int32).numpy().view(np.uint32)
    raise TypeError("expected a bf16, fp16 or fp32 tensor")


def from_bits(a: np.ndarray) -> torch.Tensor:
    """A CPU bf16 tensor sharing memory with uint16 bit patterns."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
