"""Seeded synthetic inputs for the quantized all-reduce workloads.

This module only draws random numbers and lays them out; it holds none of the
codec's arithmetic, and both the CUDA-path tests / benchmark and the CPU
oracle's callers take their inputs from here.  Values travel as raw uint16 bit
patterns of fp16 or bf16.

Workloads (tensor-parallel activations, the message an all-reduce sums):
  c1  R=2, 4096 fp16 values per rank (2 tiles), N(0,1), plus crafted blocks
      in tile 1: all-zero, a single +-1e3 outlier, all-equal values.
  c2  R=4, decode-step activation 16 tokens x 8192 hidden, bf16, N(0,1) with
      1% of the channels (the same ones on every rank) scaled x20.
  c3  R=8, prefill activation 1024 tokens x 5120 hidden, bf16, Student-t with
      3 degrees of freedom, 8 channels scaled x50.
  c4  R=4, batch 32 x seq 1024 x hidden 4096 fp16, N(0, sd 0.5).
  sweep  R in {2,4,8}, fp16 or bf16, any N, N(0,1) viewed as rows of 4096
      channels with 8 seeded outlier channels x20.
Rank r of a workload with base seed b draws from PCG64(b + 1000*r).
"""
from __future__ import annotations

import numpy as np

FP16 = 0
BF16 = 1

C1 = dict(name="c1", R=2, N=4096, dtype=FP16, bits=(4, 3))
C2 = dict(name="c2", R=4, N=16 * 8192, dtype=BF16, bits=(8, 6, 4, 3))
C3 = dict(name="c3", R=8, N=1024 * 5120, dtype=BF16, bits=(4, 3))
C4 = dict(name="c4", R=4, N=32 * 1024 * 4096, dtype=FP16, bits=(8, 4))

FP16_MAX = 65504.0


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def to_bits(vals: np.ndarray, dtype: int) -> np.ndarray:
    """float32 values -> uint16 patterns of the storage type.

    fp16 uses numpy's own conversion (values clipped to the finite range
    first); bf16 keeps the top half of the float32 pattern.  Any finite value
    of the storage type is a valid input, so how the draw is rounded does not
    matter, only that it is seeded.
    """
    vals = np.asarray(vals, dtype=np.float32)
    if dtype == FP16:
        return np.clip(vals, -FP16_MAX, FP16_MAX).astype(np.float16).view(np.uint16)
    return (vals.view(np.uint32) >> 16).astype(np.uint16)


def c1_rank(r: int) -> np.ndarray:
    x = _rng(1 + 1000 * r).standard_normal(C1["N"], dtype=np.float32)
    blk = lambda g: slice(32 * g, 32 * g + 32)  # noqa: E731  (blocks 64.. are tile 1)
    x[blk(64)] = 0.0
    x[32 * 65 + 7] = 1000.0 if r == 0 else -1000.0
    x[32 * 66 + 7] = 1000.0
    x[blk(67)] = 0.7
    x[blk(68)] = -0.75
    x[blk(69)] = 1.0
    return to_bits(x, FP16)


def c2_rank(r: int) -> np.ndarray:
    x = _rng(2 + 1000 * r).standard_normal((16, 8192), dtype=np.float32)
    ch = _rng(2).choice(8192, size=82, replace=False)
    x[:, ch] *= 20.0
    return to_bits(x.reshape(-1), BF16)


def c3_rank(r: int) -> np.ndarray:
    x = _rng(3 + 1000 * r).standard_t(3.0, size=(1024, 5120)).astype(np.float32)
    ch = _rng(3).choice(5120, size=8, replace=False)
    x[:, ch] *= 50.0
    return to_bits(x.reshape(-1), BF16)


def c4_rank(r: int) -> np.ndarray:
    x = _rng(4 + 1000 * r).normal(0.0, 0.5, size=C4["N"]).astype(np.float32)
    return to_bits(x, FP16)


def sweep_rank(r: int, n: int, dtype: int, seed: int = 5) -> np.ndarray:
    x = _rng(seed + 1000 * r).standard_normal(n, dtype=np.float32)
    ch = _rng(seed).choice(4096, size=8, replace=False)
    full = (n // 4096) * 4096  # rows of 4096 channels; channel = value index mod 4096
    x[:full].reshape(-1, 4096)[:, ch] *= 20.0
    tail = x[full:]
    tail[np.isin(np.arange(tail.size), ch)] *= 20.0
    return to_bits(x, dtype)


def fuzz_case(seed: int) -> dict:
    """A random case for the fuzz tests: rank count, size, width, storage
    type and R seeded messages mixing plain Gaussian blocks at a random
    scale, heavy-tailed values, all-zero and constant blocks and lone
    outliers."""
    rng = _rng(7000 + seed)
    R = int(rng.integers(1, 9))
    kind = rng.integers(0, 10)
    if kind < 5:
        n = int(rng.integers(1, 6000))
    elif kind < 9:
        n = int(rng.integers(6000, 80000))
    else:
        n = int(rng.integers(1 << 20, (1 << 20) + 5000))
    dtype = int(rng.integers(0, 2))
    scale = float(10.0 ** rng.uniform(-3, 3))
    xs = []
    for _ in range(R):
        if rng.random() < 0.3:
            x = rng.standard_t(3.0, size=n).astype(np.float32) * scale
        else:
            x = rng.standard_normal(n, dtype=np.float32) * scale
        blocks = (n + 31) // 32
        for _ in range(int(rng.integers(0, 4))):
            g = int(rng.integers(0, blocks))
            x[32 * g: 32 * g + 32] = 0.0
        for _ in range(int(rng.integers(0, 4))):
            g = int(rng.integers(0, blocks))
            x[32 * g: 32 * g + 32] = np.float32(rng.standard_normal() * scale)
        for _ in range(int(rng.integers(0, 4))):
            x[int(rng.integers(0, n))] = np.float32(rng.choice([-1, 1]) * scale * 10.0 ** rng.uniform(1, 3))
        xs.append(to_bits(x, dtype))
    return dict(R=R, n=n, dtype=dtype, bits=int(rng.choice([8, 6, 4, 3])),
                fc=((4, 4), (4, 8), (8, 8))[int(rng.integers(0, 3))], xs=xs)


def ranks(cfg: dict) -> list[np.ndarray]:
    gen = {"c1": c1_rank, "c2": c2_rank, "c3": c3_rank, "c4": c4_rank}[cfg["name"]]
    return [gen(r) for r in range(cfg["R"])]


def device_sweep(R: int, n: int, dtype: int, seed: int, device):
    """The sweep workload drawn on the device with torch's seeded generator
    (for messages too large to draw on the host in reasonable time).
    Returns a list of R int16 CUDA tensors holding the uint16 patterns."""
    import torch

    tdt = torch.float16 if dtype == FP16 else torch.bfloat16
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    ch = torch.randperm(4096, generator=g, device=device)[:8]
    out = []
    for r in range(R):
        g.manual_seed(seed + 1000 * r)
        x = torch.randn(n, generator=g, device=device, dtype=torch.float32)
        col = torch.arange(n, device=device) % 4096
        x = torch.where(torch.isin(col, ch), x * 20.0, x)
        out.append(x.to(tdt).view(torch.int16))
        del x, col
    return out
