"""qr_allreduce_twoshot_static: the two-shot all-reduce for callers that
cannot allocate device memory (for example code that runs inside another
component's memory budget or caching allocator, or a plain C caller with no
allocator of its own).  It takes its workspace from a buffer the library
keeps in device memory instead of from the caller.

Called through the C ABI, its R outputs must equal those of the entry point
that takes a caller-provided workspace (qr_allreduce_twoshot) and the
oracle's all-reduce, within the tolerance the other parity tests use (and in
fact bit for bit), on two calls in a row with different data -- the second
call runs over whatever the first left in the shared buffer.  A call makes
no device allocation (free device memory and the caching allocator's count
are unchanged across it).  A message whose exchange does not fit the buffer
is refused before anything runs, and the largest one that fits is served.

This file is collected last, so a run that stops at the first failure has
already run every other test.
"""
import numpy as np
import pytest
import torch

import bit_quantized_all_gb300 as qr
import oracle
from bit_quantized_all_gb300 import capi
from qr_testlib import assert_outputs_match, sample_tiles, to_dev, to_host_u16, xmax_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from bit_quantized_all_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    qr.lib()


def _ranks(R, n, dtype, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    out = []
    for r in range(R):
        v = rng.standard_normal(n).astype(np.float32) * np.float32(1 + r)
        v[rng.integers(0, n, size=max(1, n // 200))] *= 30.0
        out.append(oracle.narrow(dtype, v))
    return out


def _static_call(bits, dtype, xs_dev, ys):
    st = torch.cuda.current_stream().cuda_stream
    return capi.qr_allreduce_twoshot_static(bits, dtype, len(xs_dev), [x.data_ptr() for x in xs_dev],
                                            xs_dev[0].numel(), [y.data_ptr() for y in ys], st)


@pytest.mark.parametrize("bits,R,n,dtype", [(4, 8, 2048 * 100 + 37, 1), (3, 4, 16 * 8192, 1),
                                            (8, 2, 2048 * 7 + 1, 0), (6, 3, 4096, 0)])
def test_matches_the_workspace_entry_point_and_the_oracle_twice(bits, R, n, dtype):
    assert qr.qr_twoshot_workspace_bytes(bits, R, n) <= qr.TWOSHOT_STATIC_WORKSPACE_BYTES
    for call, seed in enumerate((1, 2)):  # two calls in a row, different data
        xs = _ranks(R, n, dtype, 100 * bits + 10 * R + seed)
        xs_dev = [to_dev(x, dtype) for x in xs]
        ref, _ = qr.qr_allreduce_twoshot(bits, xs_dev)
        ys = [torch.full_like(xs_dev[0], float("nan")) for _ in range(R)]
        status = _static_call(bits, dtype, xs_dev, ys)
        assert status == qr.QR_OK, qr.status_string(status)
        torch.cuda.synchronize()
        xmax = xmax_of(xs, dtype)
        y_orc = oracle.allreduce(bits, dtype, xs)
        for j in range(R):
            got = to_host_u16(ys[j])
            assert_outputs_match(got, to_host_u16(ref[j]), dtype, xmax, f"call {call} rank {j} INT{bits} R={R}")
            assert_outputs_match(got, y_orc, dtype, xmax, f"call {call} rank {j} INT{bits} R={R} vs oracle")


def test_allocates_nothing():
    """After a first call (which loads the library's module and looks up the
    buffer's address), further calls leave the device's free memory and the
    caching allocator's count where they were."""
    bits, R, n, dtype = 4, 8, 2048 * 64 + 5, 1
    xs = _ranks(R, n, dtype, 77)
    xs_dev = [to_dev(x, dtype) for x in xs]
    ys = [torch.empty_like(xs_dev[0]) for _ in range(R)]
    assert _static_call(bits, dtype, xs_dev, ys) == qr.QR_OK
    torch.cuda.synchronize()
    free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    for _ in range(3):
        assert _static_call(bits, dtype, xs_dev, ys) == qr.QR_OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_allocated() == alloc0
    y_orc = oracle.allreduce(bits, dtype, xs)
    for j in range(R):
        assert_outputs_match(to_host_u16(ys[j]), y_orc, dtype, xmax_of(xs, dtype), f"rank {j}")


def test_small_call_after_a_large_one():
    """A large R=8 INT4 exchange fills most of the buffer; a small R=3 INT6
    call with a different layout then runs over its leftovers."""
    big = _ranks(8, 2048 * 3000 + 3, 1, 5)
    big_dev = [to_dev(x, 1) for x in big]
    yb = [torch.empty_like(big_dev[0]) for _ in range(8)]
    assert qr.qr_twoshot_workspace_bytes(4, 8, big[0].size) > qr.TWOSHOT_STATIC_WORKSPACE_BYTES // 2
    assert _static_call(4, 1, big_dev, yb) == qr.QR_OK
    small = _ranks(3, 2048 * 9 + 100, 0, 6)
    small_dev = [to_dev(x, 0) for x in small]
    ys = [torch.empty_like(small_dev[0]) for _ in range(3)]
    assert _static_call(6, 0, small_dev, ys) == qr.QR_OK
    torch.cuda.synchronize()
    y_orc = oracle.allreduce(6, 0, small)
    for j in range(3):
        assert_outputs_match(to_host_u16(ys[j]), y_orc, 0, xmax_of(small, 0), f"small call rank {j}")


def test_refuses_messages_beyond_the_buffer_and_serves_the_largest_that_fits():
    """R=8 at INT8: 1712 tiles per rank need 72 * 214 tiles of 2176 bytes,
    just under 32 MiB, and run; one value more needs a 1713th tile, whose
    exchange does not fit, and is refused without touching the outputs."""
    R, bits, dtype = 8, 8, 1
    n_fit = 1712 * 2048
    assert qr.qr_twoshot_workspace_bytes(bits, R, n_fit) <= qr.TWOSHOT_STATIC_WORKSPACE_BYTES
    assert qr.qr_twoshot_workspace_bytes(bits, R, n_fit + 1) > qr.TWOSHOT_STATIC_WORKSPACE_BYTES
    # one value too many: refused, outputs untouched
    xs = [torch.zeros(n_fit + 1, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    ys = [torch.full((n_fit + 1,), 7.0, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    assert _static_call(bits, dtype, xs, ys) == qr.QR_ERR_SIZE
    torch.cuda.synchronize()
    for y in ys:
        assert bool(torch.all(y == 7.0))
    # far beyond the buffer: refused too
    n_big = 1 << 22
    assert qr.qr_twoshot_workspace_bytes(bits, R, n_big) > qr.TWOSHOT_STATIC_WORKSPACE_BYTES
    xb = [torch.zeros(n_big, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    yb = [torch.zeros(n_big, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    assert _static_call(bits, dtype, xb, yb) == qr.QR_ERR_SIZE
    del xs, ys, xb, yb
    # exactly at the limit: served, equal to the workspace entry point and,
    # on sampled tiles, to the oracle
    xh = _ranks(R, n_fit, dtype, 31)
    xd = [to_dev(x, dtype) for x in xh]
    yd = [torch.empty_like(xd[0]) for _ in range(R)]
    assert _static_call(bits, dtype, xd, yd) == qr.QR_OK
    ref, _ = qr.qr_allreduce_twoshot(bits, xd)
    torch.cuda.synchronize()
    for j in range(R):
        assert torch.equal(yd[j].view(torch.int16), ref[j].view(torch.int16)), j
    xmax = xmax_of(xh, dtype)
    for t in sample_tiles(n_fit // 2048, 24, seed=4).tolist():
        y_t = oracle.allreduce(bits, dtype, [x[t * 2048:(t + 1) * 2048] for x in xh])
        for j in (0, R - 1):
            assert_outputs_match(to_host_u16(yd[j][t * 2048:(t + 1) * 2048]), y_t, dtype, xmax, f"tile {t} rank {j}")
