"""Pins of the oracle's two-shot reduction.

Phase-1B decodes the R rank copies of a tile, sums them and re-quantizes
("QuickReduce INT3 quantization and benchmarking on MI355", Quantization and
Dequantization Paths; "Flash Communication" review record, key machinery:
sum locally, re-quantize the partial sums); Phase-2 dequantizes the result.

- R identical inputs whose blocks all hold their qmin: the output is exactly
  R * D(E(x)) (R*s is the new scale, every code is unchanged);
- R=2: swapping the ranks changes nothing;
- R=1: segment_reduce(w) = E(D(w)); allreduce = D(E(D(E(x)))), which equals
  a plain quantize-dequantize D(E(x)) on every block holding its qmin;
- rank order: a hand-worked R=3 case where fp32 addition in rank order
  0,1,2 gives a different answer from any other order;
- the all-reduce stays within the sum of the quantization error bounds of
  the exact sum of the inputs.
"""
import numpy as np
import pytest

import workloads

BITS = [3, 4, 6, 8]


def _qmin_blocks(n, seed, dtype, orc):
    """Random values where every block's largest magnitude is negative."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((n // 32, 32)).astype(np.float32)
    x *= np.exp2(rng.integers(-6, 6, size=(n // 32, 1))).astype(np.float32)
    i = np.argmax(np.abs(x), axis=1)
    rows = np.arange(x.shape[0])
    x[rows, i] = -np.abs(x[rows, i])
    xin = orc.narrow(dtype, x.reshape(-1))
    # re-check after rounding to the storage type: the negative one is still the max
    xw = orc.widen(dtype, xin).reshape(-1, 32)
    assert np.all(np.max(np.abs(xw), axis=1) == -np.min(xw, axis=1))
    return xin


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("R", [2, 4, 8])
@pytest.mark.parametrize("dtype", [0, 1])
def test_identical_ranks_scale_by_R(orc, bits, R, dtype):
    x = _qmin_blocks(2048 * 2, 31 * bits + R, dtype, orc)
    y = orc.allreduce(bits, dtype, [x] * R)
    qdq = orc.decode_f32(bits, orc.encode(bits, dtype, x), x.size)
    expect = orc.narrow(dtype, (qdq * np.float32(R)).astype(np.float32))
    assert np.array_equal(y, expect)


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("dtype", [0, 1])
def test_two_ranks_commute(orc, bits, dtype):
    rng = np.random.Generator(np.random.PCG64(bits))
    a = orc.narrow(dtype, rng.standard_normal(4096 + 100).astype(np.float32))
    b = orc.narrow(dtype, (3 * rng.standard_normal(4096 + 100)).astype(np.float32))
    assert np.array_equal(orc.allreduce(bits, dtype, [a, b]), orc.allreduce(bits, dtype, [b, a]))


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("dtype", [0, 1])
def test_one_rank_identities(orc, bits, dtype):
    rng = np.random.Generator(np.random.PCG64(50 + bits))
    x = orc.narrow(dtype, rng.standard_normal(2048 * 3 + 5).astype(np.float32))
    n = x.size
    w = orc.encode(bits, dtype, x)
    # Phase-1B with one rank: the "sum" is the decoded copy, re-quantized
    assert np.array_equal(orc.segment_reduce(bits, [w], n),
                          orc.encode_f32(bits, orc.decode_f32(bits, w, n)))
    # the whole pipeline is two quantize-dequantize round trips
    twice = orc.decode(bits, dtype, orc.encode_f32(bits, orc.decode_f32(bits, w, n)), n)
    assert np.array_equal(orc.allreduce(bits, dtype, [x]), twice)
    # ... which equals one round trip on blocks that hold their qmin
    xq = _qmin_blocks(2048 * 2, 60 + bits, dtype, orc)
    assert np.array_equal(orc.allreduce(bits, dtype, [xq]),
                          orc.decode(bits, dtype, orc.encode(bits, dtype, xq), xq.size))


@pytest.mark.parametrize("dtype", [0, 1])
def test_sum_runs_in_rank_order(orc, dtype):
    """INT8, R=3, value 0 of block 0 (all other values zero):
    rank 0 decodes to -1016 exactly (scale 1016/128 = 7.9375, code qmin),
    rank 1 decodes to -2^-16 exactly (scale 2^-23, a subnormal fp16, code qmin),
    rank 2 holds +1024: scale 8, x/s = 128 clips to 127, decodes to +1016.
    In rank order, -1016 + -2^-16 rounds back to -1016 (2^-16 is a quarter of
    the fp32 spacing 2^-14 at 1016), then + 1016 = 0: an all-zero block.
    Adding rank 0 and rank 2 first would leave -2^-16."""
    x = np.zeros((3, 2048), np.float32)
    x[0, 0] = -1016.0
    x[1, 0] = -(2.0**-16)
    x[2, 0] = 1024.0
    xs = [orc.narrow(dtype, r) for r in x]
    for r in range(3):
        assert orc.widen(dtype, xs[r])[0] == x[r, 0]
    dec = [orc.decode_f32(8, orc.encode(8, dtype, r), 2048)[0] for r in xs]
    assert dec == [-1016.0, -(2.0**-16), 1016.0]
    y = orc.allreduce(8, dtype, xs)
    assert np.all(y == 0)
    # the other order gives the tiny value
    y2 = orc.allreduce(8, dtype, [xs[0], xs[2], xs[1]])
    assert orc.widen(dtype, y2)[0] == -(2.0**-16)


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("R", [2, 3, 8])
def test_error_bound_against_exact_sum(orc, bits, R):
    bias = 1 << (bits - 1)
    rng = np.random.Generator(np.random.PCG64(70 + bits + R))
    n = 2048 * 2 + 301
    xs = [orc.narrow(1, (rng.standard_normal(n) * (1 + r)).astype(np.float32)) for r in range(R)]
    exact = np.sum([orc.widen(1, x).astype(np.float64) for x in xs], axis=0)
    y = orc.widen(1, orc.allreduce(bits, 1, xs)).astype(np.float64)

    def block_scales(wire):
        t = wire.reshape(-1, orc.tile_bytes(bits))
        sc = t[:, orc.scale_offset(bits):].copy().view(np.uint16).reshape(-1)
        return np.repeat(orc.f16_to_f32(sc).astype(np.float64), 32)[:n]

    # per-rank error <= s_r (clipping included), reduced error <= s_red, plus
    # the fp32 adds and the final bf16 rounding
    bound = np.zeros(n)
    wires = [orc.encode(bits, 1, x) for x in xs]
    for w in wires:
        bound += block_scales(w) * (1 + 2.0**-9)
    red = orc.segment_reduce(bits, wires, n)
    bound += block_scales(red) * (1 + 2.0**-9) * (1 + 2.0**-8)
    bound += np.abs(exact) * 2.0**-8 + 1e-30
    assert np.all(np.abs(y - exact) <= bound)
    # and the decoded reduced wire is the quantized sum of the decoded ranks
    acc = np.zeros(n, np.float32)
    for w in wires:
        acc = (acc + orc.decode_f32(bits, w, n)).astype(np.float32)
    assert np.array_equal(red, orc.encode_f32(bits, acc))
    assert bias > 0


def test_workload_c1_crafted_blocks(orc):
    """c1 at INT4: the crafted blocks of tile 1 reduce as worked out by hand."""
    xs = workloads.ranks(workloads.C1)
    y = orc.widen(0, orc.allreduce(4, 0, xs))
    # block 64 all-zero on both ranks -> +0
    assert np.all(y[64 * 32: 65 * 32] == 0)
    # block 67 all +0.7 on both ranks: each rank decodes 7/8 * fp16(0.7);
    # the sum 2*0.7*7/8 re-quantizes onto its own qmax again
    a = float(orc.widen(0, orc.narrow(0, np.array([0.7], np.float32)))[0])
    r_dec = np.float32(7 * (a / 8))
    s2 = float(orc.f16_to_f32(orc.f32_to_f16(np.array([2 * r_dec / 8], np.float32)))[0])
    out67 = orc.widen(0, orc.narrow(0, np.array([7 * s2], np.float32)))[0]  # fp16 output rounding
    assert np.all(y[67 * 32: 68 * 32] == out67)
    # block 68 all -0.75: exact on each rank and after the sum
    assert np.all(y[68 * 32: 69 * 32] == -1.5)
    # block 66: value 7 is +1000 on both ranks: scale 125 each, clipped to 875;
    # the sum 1750 sets the new scale 1750/8 = 218.75 and clips to 7 * 218.75
    # = 1531.25, which the fp16 output rounds to 1531 (spacing 1 in [1024, 2048))
    assert y[66 * 32 + 7] == 1531.0
    # block 65: value 7 is +1000 on rank 0 (clipped to 875) and -1000 on rank 1
    # (exact at qmin): the sum -125 is exact at the new qmin, scale 15.625
    assert y[65 * 32 + 7] == -125.0
    assert np.all(np.delete(y[65 * 32: 66 * 32], 7) == 0)
