"""Helpers shared by the GPU parity tests: moving seeded inputs to the device,
running the CUDA path through the C ABI binding, running the oracle on whole
messages or on sampled tiles, and the comparison rules.

Comparison rules:
  - wires (codes and scales) are integer/byte data: bit-exact;
  - fp16 / bf16 outputs: the stated tolerance is fp16 within 1 ulp, bf16
    within 1 ulp or |diff| <= 1e-3 * max|x| over all ranks' inputs; every
    step of the method is deterministic, so the outputs are also expected to
    be bit-identical, and that is asserted separately.
"""
from __future__ import annotations

import numpy as np
import torch

import bit_quantized_all_gb300 as qr
import oracle

TORCH_DT = {0: torch.float16, 1: torch.bfloat16}


def to_dev(x: np.ndarray, dtype: int, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(device)
    return t.view(TORCH_DT[dtype])


def to_host_u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_host_u8(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().numpy()


def _ordered(u16: np.ndarray) -> np.ndarray:
    """Map fp16/bf16 bit patterns to integers whose order is the value order
    (for ulp distances); +0 and -0 both map to 0."""
    u = u16.astype(np.int64)
    mag = u & 0x7FFF
    return np.where(u & 0x8000, -mag, mag)


def assert_outputs_match(y_gpu: np.ndarray, y_ref: np.ndarray, dtype: int, xmax: float, what: str = ""):
    assert y_gpu.shape == y_ref.shape, (what, y_gpu.shape, y_ref.shape)
    ulps = np.abs(_ordered(y_gpu) - _ordered(y_ref))
    if dtype == 0:
        within = ulps <= 1
    else:
        diff = np.abs(oracle.widen(1, y_gpu).astype(np.float64) - oracle.widen(1, y_ref).astype(np.float64))
        within = (ulps <= 1) | (diff <= 1e-3 * xmax)
    bad = np.flatnonzero(~within)
    assert bad.size == 0, f"{what}: {bad.size} outputs outside tolerance, first at {bad[:5]}"
    diff_idx = np.flatnonzero(y_gpu != y_ref)
    assert diff_idx.size == 0, (f"{what}: {diff_idx.size} outputs within tolerance but not bit-identical, "
                                f"first at {diff_idx[:5]}")


def assert_wire_equal(w_gpu: np.ndarray, w_ref: np.ndarray, bits: int, what: str = ""):
    assert w_gpu.shape == w_ref.shape, (what, w_gpu.shape, w_ref.shape)
    if not np.array_equal(w_gpu, w_ref):
        tb = qr.qr_tile_bytes(bits)
        d = np.flatnonzero(w_gpu != w_ref)
        raise AssertionError(f"{what}: {d.size} wire bytes differ; first at byte {d[0]} "
                             f"(tile {d[0] // tb}, offset {d[0] % tb})")


def xmax_of(xs, dtype) -> float:
    return float(max(np.max(np.abs(oracle.widen(dtype, x))) for x in xs))


# ---------------------------------------------------------------------------
# the CUDA path, through the binding (which calls the C ABI)
# ---------------------------------------------------------------------------
def gpu_unfused(bits: int, xs_dev):
    n = xs_dev[0].numel()
    wires = [qr.qr_encode(bits, x) for x in xs_dev]
    red = qr.qr_segment_reduce(bits, wires, n)
    y = qr.qr_decode(bits, red, n, dtype=xs_dev[0].dtype)
    return wires, red, y


def gpu_fused(bits: int, xs_dev, ctas: int = 0):
    return qr.qr_allreduce(bits, xs_dev, ctas=ctas)


# ---------------------------------------------------------------------------
# sampled tiles for messages too large for the oracle in seconds
# ---------------------------------------------------------------------------
def sample_tiles(T: int, k: int, seed: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    pick = rng.choice(T, size=min(k, T), replace=False) if T > 2 else np.arange(T)
    return np.unique(np.concatenate([pick, [0, T - 1]]))


def gather_tiles_u16(t: torch.Tensor, tiles: np.ndarray, n: int) -> list[np.ndarray]:
    """The fp16/bf16 values of each sampled tile (the last may be short)."""
    flat = t.reshape(-1)
    idx = torch.as_tensor(tiles, device=flat.device)
    full = idx[idx * 2048 + 2048 <= n]
    out = {}
    if full.numel():
        rows = (full[:, None] * 2048 + torch.arange(2048, device=flat.device)[None, :]).reshape(-1)
        vals = to_host_u16(flat[rows]).reshape(-1, 2048)
        for i, ti in enumerate(full.tolist()):
            out[ti] = vals[i]
    for ti in tiles.tolist():
        if ti not in out:
            out[ti] = to_host_u16(flat[ti * 2048: min(n, ti * 2048 + 2048)])
    return [out[ti] for ti in tiles.tolist()]


def gather_wire_tiles(w: torch.Tensor, tiles: np.ndarray, bits: int) -> np.ndarray:
    tb = qr.qr_tile_bytes(bits)
    idx = torch.as_tensor(tiles, device=w.device)
    rows = (idx[:, None] * tb + torch.arange(tb, device=w.device)[None, :]).reshape(-1)
    return to_host_u8(w[rows])
