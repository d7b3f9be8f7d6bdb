"""Pins of the oracle's own fp16 / bf16 conversions against a library routine.

The oracle writes its IEEE-754 binary16 and bfloat16 conversions from the
format definitions; here they are checked against torch's CPU conversions
(``Tensor.half()`` / ``Tensor.bfloat16()``, round-half-to-even) over every
16-bit pattern, every rounding tie between neighbouring values, and 10^7
random float32 patterns spread over all exponents.
"""
import numpy as np
import pytest
import torch


def _same_f32(a: np.ndarray, b: np.ndarray) -> bool:
    nan = np.isnan(a) & np.isnan(b)
    return bool(np.all(nan | (a.view(np.uint32) == b.view(np.uint32))))


def _same_16(a: np.ndarray, b: np.ndarray, is_nan: np.ndarray) -> bool:
    return bool(np.all(is_nan | (a == b)))


def _torch_half(f: np.ndarray) -> np.ndarray:
    return torch.from_numpy(f).half().view(torch.int16).numpy().view(np.uint16)


def _torch_bf16(f: np.ndarray) -> np.ndarray:
    return torch.from_numpy(f).bfloat16().view(torch.int16).numpy().view(np.uint16)


ALL16 = np.arange(65536, dtype=np.uint32).astype(np.uint16)


def test_f16_widen_every_pattern(orc):
    ref = torch.from_numpy(ALL16.view(np.int16)).view(torch.float16).float().numpy()
    assert _same_f32(orc.f16_to_f32(ALL16), ref)


def test_bf16_widen_every_pattern(orc):
    ref = torch.from_numpy(ALL16.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert _same_f32(orc.bf16_to_f32(ALL16), ref)


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_narrow_roundtrips_every_value(orc, fmt):
    widen = orc.f16_to_f32 if fmt == "f16" else orc.bf16_to_f32
    narrow = orc.f32_to_f16 if fmt == "f16" else orc.f32_to_bf16
    f = widen(ALL16)
    back = narrow(f)
    assert _same_16(back, ALL16, np.isnan(f))


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_narrow_ties_and_neighbours(orc, fmt):
    """Every midpoint between two adjacent finite values (a tie), and the
    float32 values just above and below it, against torch."""
    widen = orc.f16_to_f32 if fmt == "f16" else orc.bf16_to_f32
    narrow = orc.f32_to_f16 if fmt == "f16" else orc.f32_to_bf16
    ref = _torch_half if fmt == "f16" else _torch_bf16
    pos = np.arange(0, 0x7C00 if fmt == "f16" else 0x7F80, dtype=np.uint32).astype(np.uint16)
    lo = widen(pos[:-1]).astype(np.float64)
    hi = widen(pos[1:]).astype(np.float64)
    mid = ((lo + hi) / 2).astype(np.float32)  # exact: a dyadic with few bits
    assert np.all(mid.astype(np.float64) == (lo + hi) / 2)
    cases = [mid, np.nextafter(mid, np.float32(np.inf)), np.nextafter(mid, np.float32(0))]
    for c in cases:
        for v in (c, -c):
            v = np.ascontiguousarray(v, dtype=np.float32)
            assert np.array_equal(narrow(v), ref(v))


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_narrow_random_patterns(orc, fmt):
    narrow = orc.f32_to_f16 if fmt == "f16" else orc.f32_to_bf16
    ref = _torch_half if fmt == "f16" else _torch_bf16
    rng = np.random.Generator(np.random.PCG64(12345))
    bits = rng.integers(0, 2**32, size=10_000_000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = np.ascontiguousarray(f[~np.isnan(f)])
    assert np.array_equal(narrow(f), ref(f))
    # values concentrated around the fp16 range, including subnormals and overflow
    g = (rng.standard_normal(2_000_000) * np.exp2(rng.integers(-30, 18, 2_000_000))).astype(np.float32)
    assert np.array_equal(narrow(g), ref(g))


def test_f16_overflow_and_underflow_edges(orc):
    # 65504 is the largest finite; 65520 is the tie that rounds to infinity
    f = np.array([65504, 65519.996, 65520, 1e9, 2.0**-25, 2.0**-25 * 1.0000001, 2.0**-24], np.float32)
    assert [hex(v) for v in orc.f32_to_f16(f)] == [hex(v) for v in _torch_half(f)]
    assert list(orc.f32_to_f16(f)) == [0x7BFF, 0x7BFF, 0x7C00, 0x7C00, 0x0000, 0x0001, 0x0001]
