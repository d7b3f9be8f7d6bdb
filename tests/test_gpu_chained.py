"""Back-to-back dependent calls on one stream.  The library launches its
kernels with programmatic stream serialization (a kernel may start while its
predecessor on the stream finishes, and waits for the predecessor's
completion before it touches global memory), so each call here reads what
the call before it wrote, with no synchronization in between: twelve rounds
of y <- allreduce(y, x_1, ..., x_{R-1}) per path, compared bit for bit with
the oracle iterated the same way.  A kernel that read its input before its
predecessor finished would see a stale or half-written y."""
import numpy as np
import pytest
import torch

import bit_quantized_all_gb300 as qr
import oracle
from qr_testlib import to_dev, to_host_u16

pytestmark = pytest.mark.gpu

ROUNDS = 12


@pytest.fixture(scope="module", autouse=True)
def lib():
    from bit_quantized_all_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available()
    qr.lib()


def _ranks(R, n, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    return [oracle.narrow(1, (rng.standard_normal(n) * (1 + r)).astype(np.float32)) for r in range(R)]


def _gpu_step(path, bits, xs):
    if path == "fused":
        return qr.qr_allreduce(bits, xs)
    if path == "staged":
        return qr.qr_allreduce_staged(bits, xs)
    if path == "unfused":
        n = xs[0].numel()
        red = qr.qr_segment_reduce(bits, [qr.qr_encode(bits, x) for x in xs], n)
        return qr.qr_decode(bits, red, n, dtype=xs[0].dtype)
    if path == "twoshot":
        return qr.qr_allreduce_twoshot(bits, xs)[0][-1]  # (outputs, workspace): the last rank's output
    if path == "fc":
        return qr.qr_fc_allreduce(4, 8, xs)
    if path == "fp4":
        return qr.qr_fp4_allreduce(xs)
    raise ValueError(path)


def _oracle_step(path, bits, xs):
    if path == "fc":
        return oracle.fc_allreduce(4, 8, 1, xs)
    if path == "fp4":
        return oracle.fp4_allreduce(1, xs)
    return oracle.allreduce(bits, 1, xs)


@pytest.mark.parametrize("path,bits", [("fused", 4), ("fused", 3), ("staged", 4), ("staged", 3), ("unfused", 4),
                                       ("unfused", 6), ("twoshot", 3), ("fc", 0), ("fp4", 0)])
def test_each_call_reads_its_predecessors_output(path, bits):
    R, n = 4, 2048 * 300 + 17
    xs = _ranks(R, n, 31 + bits)
    dev = [to_dev(x, 1) for x in xs]
    y = dev[0]
    for _ in range(ROUNDS):  # no synchronization between the calls
        y = _gpu_step(path, bits, [y] + dev[1:])
    got = to_host_u16(y)
    ref = xs[0]
    for _ in range(ROUNDS):
        ref = _oracle_step(path, bits, [ref] + xs[1:])
    assert np.array_equal(got, ref), f"{path} INT{bits}: first difference at {np.flatnonzero(got != ref)[:5]}"
    assert qr.qr_wait_timeouts() == 0
