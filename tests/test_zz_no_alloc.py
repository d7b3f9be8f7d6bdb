"""qr_allreduce_twoshot_static: the two-shot all-reduce for callers that
cannot allocate device memory (for example code that runs inside another
component's memory budget or caching allocator, or a plain C caller with no
allocator of its own).  It takes its workspace from a buffer the library
keeps in device memory instead of from the caller.

Called through the C ABI, its R outputs must equal those of the entry point
that takes a caller-provided workspace (qr_allreduce_twoshot), within the
tolerance the other parity tests use (and in fact bit for bit), on two calls
in a row with different data -- the second call runs over whatever the first
left in the shared buffer.  A message whose exchange does not fit the buffer
is refused before anything runs.

This file is collected last, so a run that stops at the first failure has
already run every other test.
"""
import numpy as np
import pytest
import torch

import bit_quantized_all_gb300 as qr
import oracle
from bit_quantized_all_gb300 import capi
from qr_testlib import assert_outputs_match, to_dev, to_host_u16, xmax_of

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


@pytest.mark.parametrize("bits,R,n,dtype", [(4, 8, 2048 * 100 + 37, 1), (3, 4, 16 * 8192, 1),
                                            (8, 2, 2048 * 7 + 1, 0), (6, 3, 4096, 0)])
def test_matches_the_workspace_entry_point_twice(bits, R, n, dtype):
    assert qr.qr_twoshot_workspace_bytes(bits, R, n) <= qr.TWOSHOT_STATIC_WORKSPACE_BYTES
    st = torch.cuda.current_stream().cuda_stream
    for call, seed in enumerate((1, 2)):  # two calls in a row, different data
        xs = _ranks(R, n, dtype, 100 * bits + 10 * R + seed)
        xs_dev = [to_dev(x, dtype) for x in xs]
        ref, _ = qr.qr_allreduce_twoshot(bits, xs_dev)
        ys = [torch.full_like(xs_dev[0], float("nan")) for _ in range(R)]
        status = capi.qr_allreduce_twoshot_static(bits, dtype, R, [x.data_ptr() for x in xs_dev], n,
                                                  [y.data_ptr() for y in ys], st)
        assert status == qr.QR_OK, qr.status_string(status)
        torch.cuda.synchronize()
        xmax = xmax_of(xs, dtype)
        for j in range(R):
            assert_outputs_match(to_host_u16(ys[j]), to_host_u16(ref[j]), dtype, xmax,
                                 f"call {call} rank {j} INT{bits} R={R}")


def test_refuses_messages_beyond_the_buffer():
    R, bits = 8, 8
    n = 1 << 22  # 4 M values per rank at INT8, R=8: needs more than the buffer
    assert qr.qr_twoshot_workspace_bytes(bits, R, n) > qr.TWOSHOT_STATIC_WORKSPACE_BYTES
    xs = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    ys = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    status = capi.qr_allreduce_twoshot_static(bits, 1, R, [x.data_ptr() for x in xs], n,
                                              [y.data_ptr() for y in ys], torch.cuda.current_stream().cuda_stream)
    assert status == qr.QR_ERR_SIZE
