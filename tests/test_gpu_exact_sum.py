"""Phase-1B's exact integer sum and its fallback, on wires built to sit on
both sides of the condition that selects it.

The symmetric codec's Phase-1B sums a block's R decoded copies with integer
dot products when the ranks' nonzero scales are all integer multiples M_r of
the smallest one's unit (2^(floor(log2 smin) - 10)) below 2^16, and at INT6
also sum_r M_r < 2^17; then no partial sum of the rank order rounds, and the
integer sum equals the oracle's fp32 sum.  Every other block takes the float
path.  These wires mix, within every warp, blocks of each kind: scales in one
binade; spread to just inside the limit (M = 65504) and just past it
(M = 65536); zero scales in some ranks; every rank zero; subnormal scales;
scales near the fp16 maximum; a negative zero and a negative scale; a spread
of 10^6; log-uniform random scales; and, from three ranks, sum_r M_r just
below 2^17 (131071) and at it (131072).  The codes are random bytes.  Every reduced wire equals the oracle's
Phase-1B output byte for byte, through the default kernel choice and the
staged kernel, at rank counts that pair every rank and that leave one alone,
and at the sizes where the one-block-ahead and staged kernels run.
"""
import numpy as np
import pytest
import torch

import bit_quantized_all_gb300 as qr
import oracle
from qr_testlib import assert_wire_equal, to_host_u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from bit_quantized_all_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available()


def _f16(v):
    return np.array(v, dtype=np.float16).view(np.uint16)


def _block_scales(rng, kind, R):
    """fp16 scale bit patterns of one block for R ranks."""
    top = 63.96875  # the largest scale with M below the limit 2^16 when smin = 1
    past = 64.0     # the smallest with M at the limit
    if kind == 0:    # one binade
        s = _f16(rng.uniform(1.0, 2.0, R))
    elif kind == 1:  # spread to just inside the limit
        s = _f16(rng.uniform(1.0, top, R))
        s[rng.integers(R)] = _f16(1.0)
        s[rng.integers(R)] = _f16(top)
    elif kind == 2:  # just past it
        s = _f16(rng.uniform(1.0, top, R))
        j = rng.permutation(R)
        s[j[0]] = _f16(1.0)
        s[j[1 % R]] = _f16(past)
    elif kind == 3:  # zero scales in some ranks
        s = _f16(rng.uniform(0.5, 4.0, R))
        s[rng.random(R) < 0.4] = 0
    elif kind == 4:  # every rank zero
        s = np.zeros(R, dtype=np.uint16)
    elif kind == 5:  # subnormal scales (and a normal one near them)
        s = _f16(rng.uniform(2.0**-24, 2.0**-14, R))
    elif kind == 6:  # near the fp16 maximum
        s = _f16(rng.uniform(16384.0, 65504.0, R))
    elif kind == 7:  # a negative zero in one rank
        s = _f16(rng.uniform(1.0, 3.0, R))
        s[rng.integers(R)] = 0x8000
    elif kind == 8:  # a negative scale in one rank
        s = _f16(rng.uniform(1.0, 3.0, R))
        s[rng.integers(R)] = _f16(-1.5)
    elif kind == 9:  # a spread of 10^6
        s = _f16(rng.uniform(1.0, 2.0, R) * 1e-3)
        s[rng.integers(R)] = _f16(1000.0)
    elif kind in (11, 12) and R >= 3:  # sum M = 2047 + 63520 + 65504 = 2^17 - 1, or 2016 + 63552 + 65504 = 2^17
        s = np.zeros(R, dtype=np.uint16)
        j = rng.permutation(R)
        s[j[0]] = _f16(2047 / 1024 if kind == 11 else 2016 / 1024)
        s[j[1]] = _f16(63520 / 1024 if kind == 11 else 63552 / 1024)
        s[j[2]] = _f16(63.96875)
    else:            # log-uniform over most of the fp16 range
        s = _f16(np.exp2(rng.uniform(-20.0, 15.0, R)))
    return s.astype(np.uint16)


def _wires(bits, R, T, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    tb = qr.qr_tile_bytes(bits)
    code_bytes = 256 * bits
    wires = [np.empty(T * tb, dtype=np.uint8) for _ in range(R)]
    for t in range(T):
        for r in range(R):
            wires[r][t * tb: t * tb + code_bytes] = rng.integers(0, 256, code_bytes, dtype=np.uint8)
        for g in range(64):
            kind = int(rng.integers(0, 13)) if rng.random() < 0.5 else (g % 13)
            s = _block_scales(rng, kind, R)
            for r in range(R):
                off = t * tb + code_bytes + 2 * g
                wires[r][off: off + 2] = np.array([s[r]], dtype=np.uint16).view(np.uint8)
    return wires


def _wires_fast(bits, R, T, seed):
    """_wires' mix of block kinds for many tiles at once (vectorized): each
    block takes one of the kinds above, its scales drawn per rank."""
    rng = np.random.Generator(np.random.PCG64(seed))
    tb = qr.qr_tile_bytes(bits)
    code_bytes = 256 * bits
    nb = 64 * T
    kind = rng.integers(0, 13, nb)
    u = rng.uniform(size=(R, nb))
    s = np.exp2(rng.uniform(-20.0, 15.0, (R, nb)))                        # log-uniform
    s = np.where(kind == 0, 1.0 + u, s)                                   # one binade
    s = np.where(kind == 1, 1.0 + 62.96875 * u, s)                        # to the limit
    s = np.where(kind == 3, np.where(u < 0.4, 0.0, 0.5 + 3.5 * u), s)     # zeros in some ranks
    s = np.where(kind == 4, 0.0, s)                                       # every rank zero
    s = np.where(kind == 5, 2.0**-24 + (2.0**-14 - 2.0**-24) * u, s)      # subnormal
    s = np.where(kind == 6, 16384.0 + (65504.0 - 16384.0) * u, s)         # near the maximum
    s = np.where(kind == 9, (1.0 + u) * 1e-3, s)                          # spread of 10^6
    bits16 = s.astype(np.float16).view(np.uint16).copy()
    j = rng.integers(0, R, nb)
    col = np.arange(nb)
    bits16[j, col] = np.where(kind == 1, _f16(63.96875), bits16[j, col])  # M = 65504
    bits16[j, col] = np.where(kind == 2, _f16(64.0), bits16[j, col])      # M = 65536 ...
    bits16[(j + 1) % R, col] = np.where(kind == 2, _f16(1.0), bits16[(j + 1) % R, col])  # ... with smin = 1
    bits16[j, col] = np.where(kind == 7, 0x8000, bits16[j, col])          # a negative zero
    bits16[j, col] = np.where(kind == 8, _f16(-1.5), bits16[j, col])      # a negative scale
    bits16[j, col] = np.where(kind == 9, _f16(1000.0), bits16[j, col])
    if R >= 3:  # sum M just below 2^17 (kind 11) and at it (kind 12)
        for k, m in ((11, (2047, 63520, 65504)), (12, (2016, 63552, 65504))):
            sel = kind == k
            bits16[:, sel] = 0
            for d in range(3):
                bits16[(j[sel] + d) % R, col[sel]] = _f16(m[d] / 1024)
    wires = []
    for r in range(R):
        w = np.empty((T, tb), dtype=np.uint8)
        w[:, :code_bytes] = rng.integers(0, 256, (T, code_bytes), dtype=np.uint8)
        w[:, code_bytes:] = bits16[r].reshape(T, 64).view(np.uint8)
        wires.append(w.reshape(-1))
    return wires


@pytest.mark.parametrize("R", [2, 8])
@pytest.mark.parametrize("bits", [3, 4, 6])
def test_long_message_kernels_on_both_sides_of_the_condition(bits, R):
    """At 48 tiles per SM and more, where Phase-1B runs the one-block-ahead
    or the staged kernel (a ragged tail included)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    T = 48 * sms + 3
    n = T * 2048 - 777
    wires = _wires_fast(bits, R, T, 77 * bits + R)
    ref = oracle.segment_reduce(bits, wires, n)
    dev = [torch.from_numpy(w).cuda() for w in wires]
    got = to_host_u8(qr.qr_segment_reduce(bits, dev, n))
    assert_wire_equal(got, ref, bits, f"INT{bits} R={R} n={n} long message")
    assert qr.qr_wait_timeouts() == 0


@pytest.mark.parametrize("R", [2, 3, 5, 8])
@pytest.mark.parametrize("bits", [3, 4, 6])
def test_reduced_wire_equals_the_oracle_on_both_sides_of_the_condition(bits, R):
    T = 40
    for n in (T * 2048, T * 2048 - 1000):
        wires = _wires(bits, R, T, 1000 * bits + 10 * R + (n & 1))
        ref = oracle.segment_reduce(bits, wires, n)
        dev = [torch.from_numpy(w).cuda() for w in wires]
        got = to_host_u8(qr.qr_segment_reduce(bits, dev, n))
        assert_wire_equal(got, ref, bits, f"INT{bits} R={R} n={n} default kernel")
        if bits != 3:
            got = to_host_u8(qr.qr_segment_reduce(bits, dev, n, staged=True))
            assert_wire_equal(got, ref, bits, f"INT{bits} R={R} n={n} staged kernel")
    assert qr.qr_wait_timeouts() == 0
