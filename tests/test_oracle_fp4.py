"""Pins of the oracle's FP4 codec (QuickReduce INT3 blog, introduction: an FP4
quantization path "essentially interchangeable" with INT4; the pages give no
format, so the oracle reads it as the INT4 block framework with E2M1
elements, one fp16 scale per 32 values, scale = fp16(absmax / 6)).

- the E2M1 element: all 16 codes' values and the rounding of fp32 values
  onto the grid (nearest, ties to the even code, saturation at 6, signed
  zero) against ml_dtypes' float4_e2m1fn conversion, an independent
  implementation, over every fp32 pattern of a dense range and random
  patterns of every magnitude;
- the block scale against torch's fp32 division and fp16 rounding;
- a hand-built known-answer tile (codes, nibble order, scale position);
- zero blocks, the error bound, the tile size shared with INT4;
- Phase-1B: one rank, identical ranks on exact grids scale by R exactly,
  the rank order of the fp32 adds.
"""
import numpy as np
import pytest
import torch

GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _e2m1():
    ml = pytest.importorskip("ml_dtypes")
    return ml.float4_e2m1fn


def test_tile_is_the_int4_tile(orc):
    assert orc.fp4_tile_bytes() == orc.tile_bytes(4) == 1152
    assert orc.fp4_wire_bytes(2049) == 2 * 1152


def test_code_values_against_an_independent_decoder(orc):
    e2m1 = _e2m1()
    ref = np.arange(16, dtype=np.uint8).view(e2m1).astype(np.float32)
    got = np.array([orc.fp4_value(c) for c in range(16)], np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))  # signed zeros too
    assert list(got[:8]) == GRID


def test_rounding_every_pattern_of_a_dense_range(orc):
    """Every fp32 pattern from 0 to 8 (and the negatives) and every pattern
    within 64 ulps of each tie and each grid value."""
    e2m1 = _e2m1()
    lo, hi = np.float32(0).view(np.uint32), np.float32(8.0).view(np.uint32)
    t = np.arange(lo, hi + 1, 97, dtype=np.uint64).astype(np.uint32).view(np.float32)
    pts = np.array(GRID + [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.5, 7.0], np.float32).view(np.uint32)
    near = (pts[:, None].astype(np.int64) + np.arange(-64, 65)[None, :]).clip(0).astype(np.uint32).view(np.float32)
    t = np.concatenate([t, near.reshape(-1)])
    t = np.concatenate([t, -t])
    got = orc.fp4_round_n(t)
    ref = t.astype(e2m1).view(np.uint8)
    bad = np.flatnonzero(got != ref)
    assert bad.size == 0, (t[bad[:5]], got[bad[:5]], ref[bad[:5]])


def test_rounding_random_patterns_of_every_magnitude(orc):
    e2m1 = _e2m1()
    rng = np.random.Generator(np.random.PCG64(41))
    t = rng.integers(0, 2**32, size=2_000_000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    t = t[np.isfinite(t)]
    got = orc.fp4_round_n(t)
    ref = t.astype(e2m1).view(np.uint8)
    bad = np.flatnonzero(got != ref)
    assert bad.size == 0, (t[bad[:5]], got[bad[:5]], ref[bad[:5]])


def test_ties_go_to_the_even_code(orc):
    for t, code in ((0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6)):
        assert orc.fp4_round(t) == code
        assert orc.fp4_round(-t) == code | 8
    assert orc.fp4_round(6.0) == 7 and orc.fp4_round(1e30) == 7 and orc.fp4_round(-1e30) == 15
    assert orc.fp4_round(-0.0) == 8 and orc.fp4_round(-1e-30) == 8 and orc.fp4_round(0.0) == 0


def test_block_scale_against_torch(orc):
    rng = np.random.Generator(np.random.PCG64(42))
    for _ in range(3000):
        x = (rng.standard_normal(32) * 10.0 ** rng.uniform(-8, 6)).astype(np.float32)
        _, sh = orc.fp4_quantize_block(x)
        A = torch.tensor(np.abs(x).max(), dtype=torch.float32)
        d = A / torch.tensor(6.0, dtype=torch.float32)  # IEEE fp32 division
        s = d.to(torch.float16)
        if torch.isinf(s):
            s = torch.tensor(65504.0, dtype=torch.float16)
        assert sh == int(s.view(torch.int16).item()) & 0xFFFF


def test_known_answer_block_and_layout(orc):
    """Block 0 holds the 16 code values exactly at scale 1 (absmax 6, so
    d = 1 and r = 1), twice; the rest of the tile is zero.  Codes by hand:
    lane j of slot k at bits 4j of the u32 at 4k; scale 1.0 = 0x3C00 at 1024."""
    x = np.zeros(2048, np.float32)
    vals = np.array(GRID + [-v for v in GRID], np.float32)  # codes 0..7, 8..15 (-0 at 8)
    x[:16] = vals
    x[16:32] = vals[::-1]
    w = orc.fp4_encode_f32(x)
    assert w.size == 1152
    words = w[:16].view(np.uint32)
    assert words[0] == 0x76543210
    assert words[1] == 0xFEDCBA98
    assert words[2] == 0x89ABCDEF
    assert words[3] == 0x01234567
    assert w[16:1024].max() == 0
    assert int(w[1024]) | (int(w[1025]) << 8) == 0x3C00
    assert w[1026:].max() == 0  # zero blocks: scale +0
    y = orc.fp4_decode_f32(w, 2048)
    assert np.array_equal(y[:32].view(np.uint32), x[:32].view(np.uint32))


def test_zero_block(orc):
    c, sh = orc.fp4_quantize_block(np.zeros(32, np.float32))
    assert sh == 0 and not c.any()
    c, sh = orc.fp4_quantize_block(np.full(32, 1e-30, np.float32))  # below the fp16 range
    assert sh == 0 and not c.any()


def test_error_bound(orc):
    """|x - decode| <= s * (half the grid spacing at |x|/s), plus the
    rounding of x*r; beyond 6*s (a scale rounded down) at most A - 6*s."""
    rng = np.random.Generator(np.random.PCG64(43))
    for _ in range(2000):
        x = (rng.standard_t(3, 32) * 10.0 ** rng.uniform(-3, 3)).astype(np.float32)
        c, sh = orc.fp4_quantize_block(x)
        s = float(np.array([sh], np.uint16).view(np.float16)[0])
        dec = np.array([orc.fp4_value(int(k)) for k in c], np.float64) * s
        a = np.abs(x.astype(np.float64)) / s
        half = np.where(a <= 2, 0.25, np.where(a <= 4, 0.5, 1.0))
        bound = s * half * (1 + 2**-20) + np.maximum(0.0, np.abs(x) - 6 * s)
        assert np.all(np.abs(x - dec) <= bound + 1e-30)


def test_one_rank_reduces_to_its_own_requantization(orc):
    rng = np.random.Generator(np.random.PCG64(44))
    x = (rng.standard_normal(5000) * 3).astype(np.float32)
    w = orc.fp4_encode_f32(x)
    assert np.array_equal(orc.fp4_segment_reduce([w], 5000), orc.fp4_encode_f32(orc.fp4_decode_f32(w, 5000)))


@pytest.mark.parametrize("R", [2, 4, 8])
def test_identical_ranks_on_exact_grids_scale_by_R(orc, R):
    """Every block holds a +-6 code, so for a power-of-two R the fp32 sums are
    R times the decoded values, the new scale is R*s and every code survives:
    the all-reduce of R identical ranks is exactly R * D(E(x))."""
    rng = np.random.Generator(np.random.PCG64(45 + R))
    n = 4096
    x = (rng.standard_normal(n) * 2).astype(np.float32)
    x[::32] = 9.0  # each block's absmax: 9 / 6 = 1.5, an fp16 value, so the block holds code 7
    xin = orc.narrow(1, x)
    once = orc.fp4_decode_f32(orc.fp4_encode(1, xin), n)
    y = orc.widen(1, orc.fp4_allreduce(1, [xin] * R))
    assert np.array_equal(y, (once * R).astype(np.float32))


def test_rank_order_is_the_order_of_the_fp32_adds(orc):
    """Four ranks whose lane-0 values decode to 1, 0.25, 2^-24 and 2^-24 (lane
    1 holds 6 on rank 0, so the reduced block's scale is 1).  In rank order
    1.25 + 2^-24 ties back to 1.25 twice, which re-quantizes to the even code
    (1.0); in reverse order 2^-24 + 2^-24 + 0.25 + 1 = 1.25 + 2^-23 is above
    the tie and goes to 1.5."""
    n = 32

    def wire(lane0, lane, big):
        x = np.zeros(n, np.float32)
        x[0], x[lane] = lane0, big
        return orc.fp4_encode_f32(x)

    w0 = wire(1.0, 1, 6.0)                      # scale 1
    w1 = wire(0.25, 2, 3.0)                     # scale 1/2, 0.25 = code 1
    w2 = wire(2.0**-24, 3, 6.0 * 2.0**-23)      # scale 2^-23 (fp16 subnormal), 2^-24 = code 1
    for w, v in ((w0, 1.0), (w1, 0.25), (w2, 2.0**-24)):
        assert orc.fp4_decode_f32(w, n)[0] == v
    in_order = orc.fp4_decode_f32(orc.fp4_segment_reduce([w0, w1, w2, w2], n), n)
    reverse = orc.fp4_decode_f32(orc.fp4_segment_reduce([w2, w2, w1, w0], n), n)
    assert in_order[0] == 1.0 and reverse[0] == 1.5
    assert in_order[1] == reverse[1] == 6.0
