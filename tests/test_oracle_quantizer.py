"""Pins of the oracle's block quantizer (send path) and dequantizer (receive
path), from "QuickReduce INT3 quantization and benchmarking on MI355",
Design Highlights and Quantization and Dequantization Paths.

- the fp16 scale equals torch's fp16 rounding of absmax/|qmin| (saturated);
- every code whose exact value x/s is not within 2^-14 of a rounding boundary
  equals the nearest integer of x/s (computed in float64), clipped;
- error bound |x - D(E(x))| <= s*(1/2 + 2^-15) for in-range values, and the
  clipped positives decode to qmax*s;
- zero blocks, closed-form blocks, fp16 saturation / underflow of the scale,
  zero padding of tails.
"""
import numpy as np
import pytest
import torch

BITS = [3, 4, 6, 8]


def _blocks(n_blocks, seed, scale_spread=True):
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((n_blocks, 32)).astype(np.float32)
    if scale_spread:
        x *= np.exp2(rng.integers(-12, 12, size=(n_blocks, 1))).astype(np.float32)
    # a few single-outlier blocks
    x[::7, 5] *= 40.0
    return x


def _f16_bits_torch(v: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(v, np.float32)).half().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("bits", BITS)
def test_scale_is_fp16_rounding_of_absmax_over_qmin(orc, bits):
    bias = 1 << (bits - 1)
    x = _blocks(4000, bits)
    for blk in x:
        u, sh = orc.quantize_block(bits, blk)
        d = np.float32(np.max(np.abs(blk)) / np.float32(bias))
        exp = int(_f16_bits_torch(np.array([d]))[0])
        if exp == 0x7C00:
            exp = 0x7BFF
        assert sh == exp


@pytest.mark.parametrize("bits", BITS)
def test_codes_are_nearest_integers_clipped(orc, bits):
    bias = 1 << (bits - 1)
    qmin, qmax = -bias, bias - 1
    x = _blocks(6000, 10 + bits)
    checked = 0
    for blk in x:
        u, sh = orc.quantize_block(bits, blk)
        s = float(orc.f16_to_f32(np.array([sh], np.uint16))[0])
        assert u.min() >= 0 and u.max() <= 2 * bias - 1
        q = u.astype(np.int64) - bias
        if s == 0.0:
            assert np.all(q == 0)
            continue
        v = blk.astype(np.float64) / s  # exact ratio, up to float64 rounding
        near_tie = np.abs(v - np.floor(v) - 0.5) < 2.0**-14
        expect = np.clip(np.floor(v + 0.5), qmin, qmax)
        ok = near_tie | (expect == q)
        assert np.all(ok), (blk, q, expect)
        checked += int(np.sum(~near_tie))
    assert checked > 6000 * 30


@pytest.mark.parametrize("bits", BITS)
def test_error_bound(orc, bits):
    bias = 1 << (bits - 1)
    qmax = bias - 1
    x = _blocks(3000, 20 + bits).reshape(-1)
    wire = orc.encode_f32(bits, x)
    y = orc.decode_f32(bits, wire, x.size).astype(np.float64)
    tiles = wire.reshape(-1, orc.tile_bytes(bits))
    sc = tiles[:, orc.scale_offset(bits):].copy().view(np.uint16).reshape(-1)
    s = np.repeat(orc.f16_to_f32(sc).astype(np.float64), 32)[: x.size]
    xd = x.astype(np.float64)
    ratio = xd / np.where(s > 0, s, 1)
    clipped = ratio > qmax + 0.5
    # below qmin - 1/2 only when s rounded far below absmax/|qmin| (subnormal fp16)
    clipped_lo = ratio < -bias - 0.5
    inside = ~(clipped | clipped_lo)
    err = np.abs(xd - y)
    assert np.all(err[inside] <= s[inside] * (0.5 + 2.0**-15))
    assert np.all(y[clipped] == qmax * s[clipped])
    assert np.all(y[clipped_lo] == -bias * s[clipped_lo])
    assert np.all(s[clipped_lo] < 2.0**-14)
    assert np.all(err[clipped_lo] <= bias * 2.0**-25)
    # fp32 inputs: s = fp16(absmax/|qmin|) is within half an fp16 spacing h of
    # the exact ratio (h = 2^-25 for subnormal scales, s*2^-11 at most for
    # normal ones), so a clipped value misses by at most
    # absmax - qmax*s <= |qmin|*(s + h) - qmax*s = s + |qmin|*h
    sc_ = s[clipped]
    h = np.where(sc_ < 2.0**-14, 2.0**-25, np.exp2(np.floor(np.log2(sc_)) - 11))
    assert np.all(err[clipped] <= sc_ + bias * h)


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("dtype", [0, 1])
def test_zero_block(orc, bits, dtype):
    bias = 1 << (bits - 1)
    x = np.zeros(2048 + 37, np.uint16)
    wire = orc.encode(bits, dtype, x)
    tiles = wire.reshape(2, -1)
    assert np.all(tiles[:, orc.scale_offset(bits):] == 0)  # scale +0
    assert np.all(orc.unpack_codes(bits, wire) == bias)   # every code is the bias
    y = orc.decode(bits, dtype, wire, x.size)
    assert np.all(y == 0)  # +0, not -0
    # negative zeros are a zero block too
    xneg = np.full(64, 0x8000, np.uint16)
    w2 = orc.encode(bits, dtype, xneg)
    assert np.all(orc.decode(bits, dtype, w2, 64) == 0)


@pytest.mark.parametrize("bits", BITS)
def test_closed_form_all_equal_blocks(orc, bits):
    bias = 1 << (bits - 1)
    qmax = bias - 1
    for v in [0.75, 1.0, 3.0, 0.0078125, 96.0, 1234.0]:
        # all-equal negative: code qmin, decodes back to v exactly when v/|qmin| is an fp16 value
        u, sh = orc.quantize_block(bits, np.full(32, -v, np.float32))
        assert np.all(u == 0)
        s = float(orc.f16_to_f32(np.array([sh], np.uint16))[0])
        assert s == v / bias
        assert -bias * s == -v
        # all-equal positive: clipped to qmax, decodes to qmax * s
        u, sh = orc.quantize_block(bits, np.full(32, v, np.float32))
        assert np.all(u == 2 * bias - 1)
        assert float(orc.f16_to_f32(np.array([sh], np.uint16))[0]) * qmax == v * qmax / bias


def test_int3_example_values(orc):
    """INT3, block of all +0.7 (fp16) and all -0.75: the scale is absmax/4."""
    x = np.zeros(2048, np.float32)
    x[:32] = 0.7
    x[32:64] = -0.75
    xin = orc.narrow(0, x)
    a = float(orc.widen(0, xin)[0])  # fp16(0.7) = 0.7001953125
    wire = orc.encode(3, 0, xin)
    sc = wire[768:768 + 4].view(np.uint16)
    assert float(orc.f16_to_f32(sc[:1])[0]) == a / 4
    assert float(orc.f16_to_f32(sc[1:2])[0]) == 0.1875
    yf = orc.decode_f32(3, wire, 64)
    assert np.all(yf[:32] == np.float32(3 * a / 4))  # clipped at +3, exact in fp32
    assert np.all(yf[32:] == np.float32(-0.75))      # exact at -4
    # the fp16 output rounds 3*a/4 = 4302/8192 (13 significant bits) to 0.525390625
    y = orc.widen(0, orc.decode(3, 0, wire, 64))
    assert np.all(y[:32] == np.float32(0.525390625)) and np.all(y[32:] == -0.75)


@pytest.mark.parametrize("bits", BITS)
def test_scale_saturates_and_underflows_bf16(orc, bits):
    bias = 1 << (bits - 1)
    big = np.float32(65504.0 * bias * 4)  # absmax/|qmin| far above 65504
    x = np.zeros(64, np.float32)
    x[:32] = np.linspace(-1, 1, 32) * big
    x[32:] = np.linspace(-1, 1, 32) * np.float32(1e-12)  # below the fp16 range
    xin = orc.narrow(1, x)
    wire = orc.encode(bits, 1, xin)
    sc = wire[orc.scale_offset(bits): orc.scale_offset(bits) + 4].view(np.uint16)
    assert sc[0] == 0x7BFF  # saturated at 65504
    assert sc[1] == 0x0000  # underflow -> zero scale
    y = orc.decode_f32(bits, wire, 64)
    xw = orc.widen(1, xin)
    assert y[0] == -bias * 65504.0 and y[31] == (bias - 1) * 65504.0
    assert np.all(y[32:] == 0.0)
    # every decoded value of the saturated block stays within the clip range
    assert np.all(np.abs(y[:32]) <= bias * 65504.0) and np.all(np.sign(y[:32]) * np.sign(xw[:32]) >= 0)


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("dtype", [0, 1])
def test_tail_is_zero_padded(orc, bits, dtype):
    rng = np.random.Generator(np.random.PCG64(7))
    n = 2048 * 3 + 37
    x = orc.narrow(dtype, rng.standard_normal(n).astype(np.float32))
    padded = np.zeros(2048 * 4, np.uint16)
    padded[:n] = x
    w1 = orc.encode(bits, dtype, x)
    w2 = orc.encode(bits, dtype, padded)
    assert np.array_equal(w1, w2)
    y = orc.decode(bits, dtype, w1, n)
    assert y.size == n
    assert np.array_equal(y, orc.decode(bits, dtype, w2, 2048 * 4)[:n])


def test_non_finite_input_is_rejected(orc):
    x = np.zeros(32, np.float32)
    x[3] = np.inf
    with pytest.raises(ValueError):
        orc.quantize_block(4, x)
    with pytest.raises(ValueError):
        orc.quantize_block(9, np.zeros(32, np.float32))
