"""Pins of the oracle's Flash Communication codec (asymmetric quantization in
groups of 128; "Flash Communication" review record, arXiv 2412.04964: key
machinery, pith summary, minor comments on "INT6" and Algorithm 1).

- hand-built known-answer tiles (tests/golden/fc_known_answer_tiles.json);
- constant groups decode exactly; the group minimum decodes exactly;
- every code whose exact (x - z)/s is not within 2^-14 of a rounding boundary
  equals the float64 nearest integer, capped at 2^b - 1;
- error bound |x - decode| <= s/2 (plus the final fp32 rounding);
- Phase-1B: one rank re-quantizes its own decode; identical ranks on exact
  grids scale by R exactly; two ranks commute; the rank order is the order
  of the fp32 adds; the mixed INT4 -> INT8 ("INT6") pipeline uses INT4 wires
  for the reduce-scatter and INT8 for the all-gather; error bound against the
  exact sum.
"""
import json
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fc_known_answer_tiles.json")


def _cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


def _group0_values(case):
    i = np.arange(128)
    if case["bits"] == 4:
        u = i % 16
    else:
        u = 2 * i
        u[127] = 255
    return (case["lo"] + u * case["d"]).astype(np.float32), u


def test_tile_sizes(orc):
    assert orc.fc_tile_bytes(4) == 1024 + 128
    assert orc.fc_tile_bytes(8) == 2048 + 128
    for b in (3, 5, 6, 2, 16):
        assert orc.fc_tile_bytes(b) == 0
    assert orc.fc_wire_bytes(4, 2049) == 2 * 1152


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
@pytest.mark.parametrize("dtype", [0, 1], ids=["fp16", "bf16"])
def test_known_answer_tiles(orc, case, dtype):
    bits = case["bits"]
    x = np.zeros(2048, np.float32)
    g0, u = _group0_values(case)
    x[:128] = g0
    xin = orc.narrow(dtype, x)
    assert np.array_equal(orc.widen(dtype, xin), x)
    w = orc.fc_encode(bits, dtype, xin)
    assert w.size == orc.fc_tile_bytes(bits)
    for off, hexstr in case["expect_hex"].items():
        off = int(off)
        got = w[off: off + len(hexstr) // 2].tobytes().hex()
        assert got == hexstr, (case["name"], off, got, hexstr)
    assert np.array_equal(orc.fc_decode_f32(bits, w, 2048), x)


@pytest.mark.parametrize("bits", [4, 8])
def test_constant_groups_are_exact(orc, bits):
    for c in (0.0, -0.0, 1.0, -3.25, 1e-3, 12345.0):
        u, s, z = orc.fc_quantize_group(bits, np.full(128, c, np.float32))
        assert s == 0.0 and z == np.float32(c) and np.all(u == 0)
    x = np.repeat(np.linspace(-5, 5, 16).astype(np.float32), 128)
    assert np.array_equal(orc.fc_decode_f32(bits, orc.fc_encode_f32(bits, x), x.size), x)


def _groups(n, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((n, 128)).astype(np.float32)
    x *= np.exp2(rng.integers(-10, 10, size=(n, 1))).astype(np.float32)
    x += rng.standard_normal((n, 1)).astype(np.float32) * np.float32(3)  # offsets: asymmetric ranges
    x[::5, 7] *= 25.0
    return x


@pytest.mark.parametrize("bits", [4, 8])
def test_min_decodes_exactly_and_codes_span_the_range(orc, bits):
    x = _groups(500, bits)
    for g in x:
        u, s, z = orc.fc_quantize_group(bits, g)
        assert z == g.min()
        assert u[np.argmin(g)] == 0
        if s > 0:
            assert u[np.argmax(g)] == (1 << bits) - 1
    w = orc.fc_encode_f32(bits, x.reshape(-1))
    y = orc.fc_decode_f32(bits, w, x.size).reshape(-1, 128)
    rows = np.arange(x.shape[0])
    assert np.array_equal(y[rows, np.argmin(x, axis=1)], x.min(axis=1))


@pytest.mark.parametrize("bits", [4, 8])
def test_codes_are_nearest_integers(orc, bits):
    umax = (1 << bits) - 1
    x = _groups(2000, 10 + bits)
    checked = 0
    for g in x:
        u, s, z = orc.fc_quantize_group(bits, g)
        assert s == np.float32(np.float32(g.max() - g.min()) / np.float32(umax))
        if s == 0:
            continue
        v = (g.astype(np.float64) - float(z)) / float(s)
        near = np.abs(v - np.floor(v) - 0.5) < 2.0**-14
        expect = np.minimum(np.floor(v + 0.5), umax)
        assert np.all(near | (u == expect))
        checked += int(np.sum(~near))
    assert checked > 2000 * 120


@pytest.mark.parametrize("bits", [4, 8])
def test_error_bound(orc, bits):
    x = _groups(1500, 20 + bits).reshape(-1)
    w = orc.fc_encode_f32(bits, x)
    y = orc.fc_decode_f32(bits, w, x.size).astype(np.float64)
    t = w.reshape(-1, orc.fc_tile_bytes(bits))
    meta = 256 * bits
    s = np.repeat(t[:, meta:meta + 64].copy().view(np.float32).reshape(-1).astype(np.float64), 128)[:x.size]
    xd = x.astype(np.float64)
    # half a step, plus the relative error of r = RN(1/s) over at most 2^b steps,
    # plus the final rounding of u*s + z
    bound = s * (0.5 + 2.0**-15) + np.abs(y) * 2.0**-23
    assert np.all(np.abs(xd - y) <= bound)


def test_zero_minimum_is_stored_as_plus_zero(orc):
    """-0 and +0 are the same value: a group whose minimum is zero stores the
    zero point +0 whichever sign its zeros carry, and its code-0 values
    decode to +0."""
    for first in (-0.0, 0.0):
        g = np.zeros(128, np.float32)
        g[0], g[1], g[5] = first, -0.0, 2.5
        u, s, z = orc.fc_quantize_group(4, g)
        assert np.float32(z).view(np.uint32) == 0
        x = np.zeros(2048, np.float32)
        x[:128] = g
        y = orc.fc_decode(4, 1, orc.fc_encode_f32(4, x), 2048)
        assert y[0] == 0 and y[1] == 0  # +0 bit patterns


def test_decode_is_one_fused_rounding(orc):
    """INT4 group with minimum -1 and maximum 4: s = RN(5/15) = RN(1/3) =
    0.3333333432674408, r = RN(1/s) = 3, and the value 0 gets code 3.  With one
    rounding, 3*s - 1 = 2^-25 exactly (3*s = 1 + 2^-25); rounding the product
    first would give 1 - 1 = 0."""
    g = np.zeros(128, np.float32)
    g[0], g[1] = -1.0, 4.0
    u, s, z = orc.fc_quantize_group(4, g)
    assert s == np.float32(1.0 / 3.0) and z == -1.0 and u[2] == 3
    x = np.zeros(2048, np.float32)
    x[:128] = g
    y = orc.fc_decode_f32(4, orc.fc_encode_f32(4, x), 2048)
    assert y[2] == 2.0**-25


def test_code_is_nearest_integer_of_exact_product(orc):
    """The code is the nearest integer to the exact product (x - z) * r, one
    rounding.  Group with minimum -4.0053387 (0xc0802bbc) and maximum 2.8191404
    (0x40346ccc): s = 0.45496526 (0x3ee8f135), r = 2.19797 (0x400cab8a); for
    x = -0.593099 (0xbf17d556), d = x - z = 3.4122396 (0x405a6222) and the exact
    product d*r = 7.49999987... gives code 7, while rounding the product to fp32
    first (7.5, a tie) would give 8."""
    bits = np.array([0xc0802bbc, 0x40346ccc, 0xbf17d556], np.uint32).view(np.float32)
    g = np.full(128, bits[2], np.float32)
    g[0], g[1] = bits[0], bits[1]
    u, s, z = orc.fc_quantize_group(4, g)
    assert np.float32(s).view(np.uint32) == 0x3ee8f135
    assert u[0] == 0 and u[1] == 15 and np.all(u[2:] == 7)


def test_non_finite_or_overflowing_range_is_rejected(orc):
    g = np.zeros(128, np.float32)
    g[0] = np.inf
    with pytest.raises(ValueError):
        orc.fc_quantize_group(4, g)
    g[0], g[1] = 3e38, -3e38
    with pytest.raises(ValueError):
        orc.fc_quantize_group(8, g)
    with pytest.raises(ValueError):
        orc.fc_quantize_group(6, np.zeros(128, np.float32))


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("dtype", [0, 1])
def test_one_rank_and_mixed_widths(orc, bits, dtype):
    rng = np.random.Generator(np.random.PCG64(bits + dtype))
    x = orc.narrow(dtype, (rng.standard_normal(2048 * 3 + 5) + 0.5).astype(np.float32))
    n = x.size
    w = orc.fc_encode(bits, dtype, x)
    for bo in (4, 8):
        red = orc.fc_segment_reduce(bits, bo, [w], n)
        assert red.size == orc.fc_wire_bytes(bo, n)
        assert np.array_equal(red, orc.fc_encode_f32(bo, orc.fc_decode_f32(bits, w, n)))
        y = orc.fc_allreduce(bits, bo, dtype, [x])
        assert np.array_equal(y, orc.fc_decode(bo, dtype, red, n))


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("R", [2, 4, 8])
def test_identical_ranks_on_exact_grids(orc, bits, R):
    """Values lo + u*d on every rank: the sum is R times each value exactly,
    its range R times the range, so the scale is R*d and every code repeats."""
    umax = (1 << bits) - 1
    rng = np.random.Generator(np.random.PCG64(R * bits))
    u = rng.integers(0, umax + 1, size=(16, 128))
    u[:, 0], u[:, 1] = 0, umax
    lo = -np.exp2(rng.integers(-3, 3, size=(16, 1))).astype(np.float64)
    d = np.exp2(rng.integers(-6, -2, size=(16, 1))).astype(np.float64)
    x = (lo + u * d).astype(np.float32).reshape(-1)
    for dtype in (0, 1):
        xin = orc.narrow(dtype, x)
        if not np.array_equal(orc.widen(dtype, xin), x):
            continue  # not exact in this storage type
        y = orc.fc_allreduce(bits, bits, dtype, [xin] * R)
        assert np.array_equal(orc.widen(dtype, y), (x * np.float32(R)).astype(np.float32))


def test_two_ranks_commute_and_rank_order(orc):
    rng = np.random.Generator(np.random.PCG64(99))
    a = orc.narrow(1, rng.standard_normal(4096).astype(np.float32))
    b = orc.narrow(1, (3 + rng.standard_normal(4096)).astype(np.float32))
    for bits in (4, 8):
        assert np.array_equal(orc.fc_allreduce(bits, 8, 1, [a, b]), orc.fc_allreduce(bits, 8, 1, [b, a]))
    # Rank order: INT8 groups that decode exactly (constant groups): value 0
    # is -1024 on rank 0, -2^-16 on rank 1, +1024 on rank 2 (each rank's group
    # is constant, so each decodes exactly).  -1024 + -2^-16 rounds back to
    # -1024 in fp32 (2^-16 is below half the spacing 2^-13 at 1024), then
    # + 1024 = 0; adding ranks 0 and 2 first would leave -2^-16.
    xs = [np.full(128, v, np.float32) for v in (-1024.0, -(2.0**-16), 1024.0)]
    xs = [orc.narrow(1, np.concatenate([v, np.zeros(2048 - 128, np.float32)])) for v in xs]
    y = orc.widen(1, orc.fc_allreduce(8, 8, 1, xs))
    assert np.all(y == 0)
    y2 = orc.widen(1, orc.fc_allreduce(8, 8, 1, [xs[0], xs[2], xs[1]]))
    assert np.all(y2[:128] == -(2.0**-16))


@pytest.mark.parametrize("bits_rs,bits_ag", [(4, 4), (4, 8), (8, 8)])
@pytest.mark.parametrize("R", [2, 3, 8])
def test_error_bound_against_exact_sum(orc, bits_rs, bits_ag, R):
    rng = np.random.Generator(np.random.PCG64(70 + bits_rs + bits_ag + R))
    n = 2048 * 2 + 301
    xs = [orc.narrow(1, (rng.standard_normal(n) * (1 + r) + r).astype(np.float32)) for r in range(R)]
    exact = np.sum([orc.widen(1, x).astype(np.float64) for x in xs], axis=0)
    y = orc.widen(1, orc.fc_allreduce(bits_rs, bits_ag, 1, xs)).astype(np.float64)

    def steps(wire, bits):
        t = wire.reshape(-1, orc.fc_tile_bytes(bits))
        meta = 256 * bits
        return np.repeat(t[:, meta:meta + 64].copy().view(np.float32).reshape(-1).astype(np.float64), 128)[:n]

    wires = [orc.fc_encode(bits_rs, 1, x) for x in xs]
    bound = np.zeros(n)
    for w in wires:
        bound += steps(w, bits_rs) * (0.5 + 2.0**-14)
    red = orc.fc_segment_reduce(bits_rs, bits_ag, wires, n)
    bound += steps(red, bits_ag) * (0.5 + 2.0**-14)
    bound += np.abs(exact) * 2.0**-7 + 1e-30  # fp32 adds and the bf16 output rounding
    assert np.all(np.abs(y - exact) <= bound)
    acc = np.zeros(n, np.float32)
    for w in wires:
        acc = (acc + orc.fc_decode_f32(bits_rs, w, n)).astype(np.float32)
    assert np.array_equal(red, orc.fc_encode_f32(bits_ag, acc))
