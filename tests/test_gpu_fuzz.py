"""Seeded random cases against the oracle, bit for bit: rank counts 1..8,
sizes from one value to past 2^20 with ragged tails, every width, fp16 and
bf16, and messages that mix Gaussian and heavy-tailed values at scales from
1e-3 to 1e3 with all-zero blocks, constant blocks and lone outliers
(workloads.fuzz_case).  Every path: the fused kernel as the library picks
it and forced onto the staged kernel, encode / Phase-1B / decode with their
wires, the three-launch and the flag-joined two-shot, the per-rank two-shot
calls issued for every rank from one process, random grid sizes,
16-byte-aligned buffers, the wire-emitting variant, the asymmetric codec's
paths and the FP4 codec's."""
import os

import numpy as np
import pytest
import torch

import bit_quantized_all_gb300 as qr
import oracle
import workloads
from bit_quantized_all_gb300.peer import twoshot_peer_local
from qr_testlib import assert_outputs_match, assert_wire_equal, to_dev, to_host_u16, to_host_u8, xmax_of

pytestmark = pytest.mark.gpu

# seeds a:b from QR_FUZZ_SEEDS (default 0:150)
CASES = range(*(int(v) for v in os.environ.get("QR_FUZZ_SEEDS", "0:150").split(":")))


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


@pytest.mark.parametrize("seed", CASES)
def test_symmetric_codec_every_path(seed):
    c = workloads.fuzz_case(seed)
    R, n, dt, bits, xs = c["R"], c["n"], c["dtype"], c["bits"], c["xs"]
    what = f"seed {seed}: R={R} n={n} dtype={dt} bits={bits}"
    xmax = xmax_of(xs, dt)
    y_ref = oracle.allreduce(bits, dt, xs)
    w_ref = [oracle.encode(bits, dt, x) for x in xs]
    red_ref = oracle.segment_reduce(bits, w_ref, n)
    xs_dev = [to_dev(x, dt) for x in xs]

    assert_outputs_match(to_host_u16(qr.qr_allreduce(bits, xs_dev)), y_ref, dt, xmax, what + " fused")
    assert_outputs_match(to_host_u16(qr.qr_allreduce_staged(bits, xs_dev)), y_ref, dt, xmax, what + " staged")

    wires = [qr.qr_encode(bits, x) for x in xs_dev]
    for r in range(R):
        assert_wire_equal(to_host_u8(wires[r]), w_ref[r], bits, f"{what} wire {r}")
    red = qr.qr_segment_reduce(bits, wires, n)
    assert_wire_equal(to_host_u8(red), red_ref, bits, what + " reduced wire")
    if bits != 3:
        assert_wire_equal(to_host_u8(qr.qr_segment_reduce(bits, wires, n, staged=True)), red_ref, bits,
                          what + " reduced wire (staged)")
    y_u = qr.qr_decode(bits, red, n, dtype=xs_dev[0].dtype)
    assert_outputs_match(to_host_u16(y_u), y_ref, dt, xmax, what + " unfused")

    for flags in (False, True):
        ys, _ = qr.qr_allreduce_twoshot(bits, xs_dev, flags=flags)
        for j, y in enumerate(ys):
            assert_outputs_match(to_host_u16(y), y_ref, dt, xmax, f"{what} two-shot flags={flags} rank {j}")
    ys, _ = twoshot_peer_local(bits, xs_dev)
    for j, y in enumerate(ys):
        assert_outputs_match(to_host_u16(y), y_ref, dt, xmax, f"{what} per-rank two-shot rank {j}")
    assert qr.qr_wait_timeouts() == 0


@pytest.mark.parametrize("seed", CASES)
def test_asymmetric_codec_every_path(seed):
    c = workloads.fuzz_case(seed)
    R, n, dt, xs = c["R"], c["n"], c["dtype"], c["xs"]
    brs, bag = c["fc"]
    what = f"seed {seed}: R={R} n={n} dtype={dt} widths {brs}->{bag}"
    rng = np.random.Generator(np.random.PCG64(11000 + seed))
    xmax = xmax_of(xs, dt)
    y_ref = oracle.fc_allreduce(brs, bag, dt, xs)
    w_ref = [oracle.fc_encode(brs, dt, x) for x in xs]
    red_ref = oracle.fc_segment_reduce(brs, bag, w_ref, n)
    xs_dev = [to_dev(x, dt) for x in xs]

    assert_outputs_match(to_host_u16(qr.qr_fc_allreduce(brs, bag, xs_dev)), y_ref, dt, xmax, what + " fused")
    ctas = int(rng.integers(1, 2000))
    assert_outputs_match(to_host_u16(qr.qr_fc_allreduce(brs, bag, xs_dev, ctas=ctas)), y_ref, dt, xmax,
                         f"{what} register-fed, {ctas} CTAs")
    ctas = int(rng.integers(0, 200))
    assert_outputs_match(to_host_u16(qr.qr_fc_allreduce_staged(brs, bag, xs_dev, ctas=ctas)), y_ref, dt, xmax,
                         f"{what} staged, {ctas} CTAs")

    wires = [qr.qr_fc_encode(brs, x) for x in xs_dev]
    for r in range(R):
        assert np.array_equal(to_host_u8(wires[r]), w_ref[r]), f"{what} wire {r}"
    red = qr.qr_fc_segment_reduce(brs, bag, wires, n)
    assert np.array_equal(to_host_u8(red), red_ref), what + " reduced wire"
    red_st = qr.qr_fc_segment_reduce(brs, bag, wires, n, staged=True)
    assert np.array_equal(to_host_u8(red_st), red_ref), what + " reduced wire (staged)"
    y_u = qr.qr_fc_decode(bag, red, n, dtype=xs_dev[0].dtype)
    assert_outputs_match(to_host_u16(y_u), y_ref, dt, xmax, what + " unfused")
    ys, _ = qr.qr_fc_allreduce_twoshot(brs, bag, xs_dev)
    for j, y in enumerate(ys):
        assert_outputs_match(to_host_u16(y), y_ref, dt, xmax, f"{what} two-shot rank {j}")
    ys, _ = twoshot_peer_local(("fc", brs, bag), xs_dev)
    for j, y in enumerate(ys):
        assert_outputs_match(to_host_u16(y), y_ref, dt, xmax, f"{what} per-rank two-shot rank {j}")
    assert qr.qr_wait_timeouts() == 0


def _offset_by_16_bytes(x: torch.Tensor) -> torch.Tensor:
    """x's values in a buffer that starts 16 bytes past a 32-byte boundary."""
    buf = torch.empty(x.numel() + 16, dtype=x.dtype, device=x.device)
    v = buf[8: 8 + x.numel()]
    assert v.data_ptr() % 32 == 16
    v.copy_(x)
    return v


@pytest.mark.parametrize("seed", CASES)
def test_symmetric_codec_launch_shapes_alignment_and_emission(seed):
    """The same cases on random grid sizes, on 16-byte (not 32-byte) aligned
    buffers, and through the variant that also writes the Phase-1 and
    reduced wires."""
    c = workloads.fuzz_case(seed)
    R, n, dt, bits, xs = c["R"], c["n"], c["dtype"], c["bits"], c["xs"]
    what = f"seed {seed}: R={R} n={n} dtype={dt} bits={bits}"
    rng = np.random.Generator(np.random.PCG64(9000 + seed))
    xmax = xmax_of(xs, dt)
    y_ref = oracle.allreduce(bits, dt, xs)
    xs_dev = [to_dev(x, dt) for x in xs]

    ctas = int(rng.integers(1, 2000))
    assert_outputs_match(to_host_u16(qr.qr_allreduce(bits, xs_dev, ctas=ctas)), y_ref, dt, xmax,
                         f"{what} register-fed, {ctas} CTAs")
    ctas = int(rng.integers(1, 200))
    assert_outputs_match(to_host_u16(qr.qr_allreduce_staged(bits, xs_dev, ctas=ctas)), y_ref, dt, xmax,
                         f"{what} staged, {ctas} CTAs")

    xs16 = [_offset_by_16_bytes(x) for x in xs_dev]
    y16 = _offset_by_16_bytes(torch.zeros_like(xs_dev[0]))
    qr.qr_allreduce(bits, xs16, y=y16)
    assert_outputs_match(to_host_u16(y16), y_ref, dt, xmax, what + " 16-byte aligned")

    y, wires, red = qr.qr_allreduce_emit(bits, xs_dev)
    assert_outputs_match(to_host_u16(y), y_ref, dt, xmax, what + " emit")
    w_ref = [oracle.encode(bits, dt, x) for x in xs]
    for r in range(R):
        assert_wire_equal(to_host_u8(wires[r]), w_ref[r], bits, f"{what} emitted wire {r}")
    assert_wire_equal(to_host_u8(red), oracle.segment_reduce(bits, w_ref, n), bits, what + " emitted reduced wire")
    assert qr.qr_wait_timeouts() == 0


@pytest.mark.parametrize("seed", CASES)
def test_fp4_codec_every_path(seed):
    c = workloads.fuzz_case(seed)
    R, n, dt, xs = c["R"], c["n"], c["dtype"], c["xs"]
    what = f"seed {seed}: R={R} n={n} dtype={dt} FP4"
    rng = np.random.Generator(np.random.PCG64(13000 + seed))
    xmax = xmax_of(xs, dt)
    y_ref = oracle.fp4_allreduce(dt, xs)
    w_ref = [oracle.fp4_encode(dt, x) for x in xs]
    xs_dev = [to_dev(x, dt) for x in xs]
    ctas = int(rng.integers(0, 200))
    assert_outputs_match(to_host_u16(qr.qr_fp4_allreduce(xs_dev, ctas=ctas)), y_ref, dt, xmax,
                         f"{what} fused, {ctas} CTAs")
    wires = [qr.qr_fp4_encode(x) for x in xs_dev]
    for r in range(R):
        assert np.array_equal(to_host_u8(wires[r]), w_ref[r]), f"{what} wire {r}"
    red = qr.qr_fp4_segment_reduce(wires, n, ctas=int(rng.integers(0, 200)))
    assert np.array_equal(to_host_u8(red), oracle.fp4_segment_reduce(w_ref, n)), what + " reduced wire"
    y_u = qr.qr_fp4_decode(red, n, dtype=xs_dev[0].dtype)
    assert_outputs_match(to_host_u16(y_u), y_ref, dt, xmax, what + " unfused")
    ys, _ = qr.qr_fp4_allreduce_twoshot(xs_dev)
    for j, y in enumerate(ys):
        assert_outputs_match(to_host_u16(y), y_ref, dt, xmax, f"{what} two-shot rank {j}")
    ys, _ = twoshot_peer_local("fp4", xs_dev)
    for j, y in enumerate(ys):
        assert_outputs_match(to_host_u16(y), y_ref, dt, xmax, f"{what} per-rank two-shot rank {j}")
    assert qr.qr_wait_timeouts() == 0
