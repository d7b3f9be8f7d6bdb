"""The argument behind Phase-1B's exact integer sum, checked on the host.

Phase-1B ("QuickReduce INT3 quantization and benchmarking on MI355",
Quantization and Dequantization Paths) decodes each rank's block, q_r * s_r,
and adds the R copies in rank order in fp32.  The symmetric codec's kernels
take a shortcut for most blocks: with unit = 2^(floor(log2 smin) - 10) (smin
the smallest nonzero fp16 scale of the block over the ranks), every scale is an
integer multiple M_r of unit; when every M_r < 2^16 (and, for INT6 with at
most four ranks, sum_r M_r < 2^17) the kernels add sum_r M_r * u_r in 32-bit
integers, starting from the bit pattern of the float 1.5*2^23 - bias * sum_r M_r
(INT6 from five ranks: from the integer -bias * sum_r M_r), and turn the result
into fp32 with one fused multiply-add by unit (or an int-to-float conversion
and a multiply by unit).

This test restates that arithmetic in numpy -- independently of the CUDA
code -- on blocks built to sit on both sides of the condition, and checks that
wherever the condition holds it yields exactly the fp32 rank-order sum (a zero
may differ in sign only), so that the kernels' shortcut cannot change a byte.
"""
import numpy as np
import pytest

MAGIC = np.float32(1.5 * 2.0**23)


def _scales(rng, R, nb):
    """fp16 scales (as float64) of nb blocks for R ranks, a mix of spreads."""
    kind = rng.integers(0, 7, nb)
    u = rng.uniform(size=(R, nb))
    s = np.exp2(rng.uniform(-20.0, 15.0, (R, nb)))                     # log-uniform
    s = np.where(kind == 0, 1.0 + u, s)                                # one binade
    s = np.where(kind == 1, 1.0 + 62.96875 * u, s)                     # up to M ~ 2^16
    s = np.where(kind == 2, np.where(u < 0.4, 0.0, 0.5 + 3.5 * u), s)  # zeros in some ranks
    s = np.where(kind == 3, 2.0**-24 + (2.0**-14 - 2.0**-24) * u, s)   # subnormal
    s = np.where(kind == 4, 16384.0 + (65504.0 - 16384.0) * u, s)      # near the fp16 maximum
    s = np.where(kind == 5, (1.0 + 15.0 * u) * 2.0**-8, s)             # a few binades
    s = s.astype(np.float16).astype(np.float64)
    # near the INT6 sum limit: sum M = 2^17 - 1 and 2^17 from three ranks
    if R >= 3:
        j = rng.integers(0, R, nb)
        col = np.arange(nb)
        for k, m in ((6, (2047, 63520, 65504)),):
            sel = kind == k
            s[:, sel] = 0.0
            for d in range(3):
                s[(j[sel] + d) % R, col[sel]] = m[d] / 1024.0
            half = sel & (rng.random(nb) < 0.5)  # the other side of the limit
            s[(j[half] + 0) % R, col[half]] = 2016 / 1024.0
            s[(j[half] + 1) % R, col[half]] = 63552 / 1024.0
    return s


def _condition(s, bits, R):
    """The kernels' test, from the scales of each block: (holds, unit, M)."""
    nz = np.where(s > 0, s, np.inf)
    smin = nz.min(axis=0)
    some = np.isfinite(smin)
    e = np.floor(np.log2(np.where(some, smin, 1.0)))
    unit = np.exp2(e - 10.0)
    M = s / unit
    assert np.all(M[:, some] == np.round(M[:, some])), "every scale is a multiple of unit"
    holds = some & (M.max(axis=0) < 2**16)
    if bits == 6 and R <= 4:
        holds &= M.sum(axis=0) < 2**17
    return holds, unit, M.astype(np.int64)


def _integer_path(u, M, unit, bits, R):
    """The kernels' integer arithmetic for each block and value: u[r, b, i]
    codes 0 .. 2^bits - 1, M[r, b], unit[b]; returns the fp32 results."""
    bias = 1 << (bits - 1)
    msum = M.sum(axis=0)
    dot = np.einsum("rb,rbi->bi", M, u)  # sum_r M_r * u_r, exact in int64
    if bits != 6 or R <= 4:  # the pattern of 1.5*2^23 - bias * sum M, plus the products
        base = int(MAGIC.view(np.uint32)) - bias * msum
        pat = base[:, None] + dot
        assert np.all((pat >= 0x4B000000) & (pat < 0x4B800000)), "the accumulator stays in [2^23, 2^24)"
        F = pat.astype(np.uint32).view(np.float32).astype(np.float64)
        acc = F * unit[:, None] - float(MAGIC) * unit[:, None]  # one fma: exact, S * unit
    else:  # -bias * sum M plus the products, as a 32-bit integer S
        S = dot - bias * msum[:, None]
        assert np.all(np.abs(S) < 2**24)
        acc = S.astype(np.float32).astype(np.float64) * unit[:, None]
    out = acc.astype(np.float32)
    assert np.all(out.astype(np.float64) == acc), "the result is exact in fp32"
    return out


def _rank_order_sum(u, s, bits):
    """Phase-1B's definition: fp32 acc += q_r * s_r in rank order (q * s is
    exact in fp32)."""
    q = (u - (1 << (bits - 1))).astype(np.float64)
    acc = np.zeros(u.shape[1:], dtype=np.float32)
    for r in range(u.shape[0]):
        acc = acc + (q[r] * s[r][:, None]).astype(np.float32)
    return acc


@pytest.mark.parametrize("R", [2, 3, 4, 5, 8])
@pytest.mark.parametrize("bits", [3, 4, 6])
def test_integer_sum_equals_the_rank_order_sum_where_the_condition_holds(bits, R):
    rng = np.random.Generator(np.random.PCG64(100 * bits + R))
    nb = 4000
    s = _scales(rng, R, nb)
    u = rng.integers(0, 1 << bits, (R, nb, 32))
    # extreme codes in some blocks: every rank at 0, or at the top code
    u[:, :200] = 0
    u[:, 200:400] = (1 << bits) - 1
    holds, unit, M = _condition(s, bits, R)
    assert holds.mean() > 0.4, "the mix exercises the shortcut"
    assert (~holds).sum() > 0, "and the fallback"
    got = _integer_path(u[:, holds], M[:, holds], unit[holds], bits, R)
    ref = _rank_order_sum(u[:, holds], s[:, holds], bits)
    assert np.array_equal(got, ref)  # == treats -0 and +0 as equal


def test_the_int6_sum_limit_is_needed_for_the_pattern():
    """At INT6 with sum M past 2^17 the pattern would leave [2^23, 2^24):
    the limit is what keeps the shortcut's accumulator a float of unit
    spacing."""
    bias = 32
    msum = (1 << 17) + 32
    assert int(MAGIC.view(np.uint32)) - bias * msum < 0x4B000000
