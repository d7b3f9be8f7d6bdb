"""Seeded random cases against the oracle, bit for bit: rank counts 1..8,
sizes from one value to past 2^20 with ragged tails, every width, fp16 and
bf16, and messages that mix Gaussian and heavy-tailed values at scales from
1e-3 to 1e3 with all-zero blocks, constant blocks and lone outliers
(workloads.fuzz_case).  Every path: the fused kernel as the library picks
it and forced onto the staged kernel, encode / Phase-1B / decode with their
wires, the three-launch and the flag-joined two-shot, and the asymmetric
codec's fused path."""
import numpy as np
import pytest
import torch

import bit_quantized_all_gb300 as qr
import oracle
import workloads
from qr_testlib import assert_outputs_match, assert_wire_equal, to_dev, to_host_u16, to_host_u8, xmax_of

pytestmark = pytest.mark.gpu

CASES = range(150)


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
    assert qr.qr_wait_timeouts() == 0


@pytest.mark.parametrize("seed", CASES)
def test_asymmetric_codec_fused(seed):
    c = workloads.fuzz_case(seed)
    R, n, dt, xs = c["R"], c["n"], c["dtype"], c["xs"]
    brs, bag = c["fc"]
    what = f"seed {seed}: R={R} n={n} dtype={dt} widths {brs}->{bag}"
    y_ref = oracle.fc_allreduce(brs, bag, dt, xs)
    xs_dev = [to_dev(x, dt) for x in xs]
    y = to_host_u16(qr.qr_fc_allreduce(brs, bag, xs_dev))
    assert_outputs_match(y, y_ref, dt, xmax_of(xs, dt), what)
    assert qr.qr_wait_timeouts() == 0
