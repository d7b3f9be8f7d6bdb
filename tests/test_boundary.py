"""The C ABI boundary, without a GPU.

- libqr.so loads and exports every function include/qr.h declares;
- the size functions follow their closed forms (1152 B INT4 and 896 B INT3
  tiles, printed in "QuickReduce INT3 quantization and benchmarking on
  MI355", Design Highlights);
- each validation error is returned for invalid arguments.  Every call here
  fails validation, which the library does on the host before any CUDA call,
  so nothing is launched and no pointer is dereferenced (the pointers are
  made-up addresses);
- the binding fails loudly when the library is missing, and the product
  package never touches the oracle.
"""
import os
import re

import pytest

import bit_quantized_all_gb300 as qr
from bit_quantized_all_gb300 import capi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qr.h")

A = 0x7F0000000000  # made-up, 16-byte aligned "device" addresses: never dereferenced
B = 0x7F1000000000
Y = 0x7F2000000000


# The validation tests pass made-up addresses.  Where a GPU can be reached, a
# validation bug would launch a kernel on them, so they run only where none can.
no_gpu_only = pytest.mark.skipif(
    __import__("torch").cuda.is_available(),
    reason="made-up device addresses are only passed where no GPU can be reached")


@pytest.fixture(scope="module", autouse=True)
def built():
    from bit_quantized_all_gb300 import build
    build.build()
    qr.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qr_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = _declared()
    assert "qr_allreduce" in names and "qr_encode" in names
    L = qr.lib()
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(qr.EXPORTS)


def test_sizes():
    assert qr.qr_tile_values() == 2048
    assert qr.qr_tile_bytes(4) == 1152 and qr.qr_tile_bytes(3) == 896
    assert qr.qr_tile_bytes(8) == 2176 and qr.qr_tile_bytes(6) == 1664
    for b in (0, 1, 2, 5, 7, 9, 16, -4):
        assert qr.qr_tile_bytes(b) == 0
        assert qr.qr_wire_bytes(b, 100) == 0
    for b in (3, 4, 6, 8):
        tb = qr.qr_tile_bytes(b)
        assert qr.qr_wire_bytes(b, 0) == 0
        assert qr.qr_wire_bytes(b, 1) == tb
        assert qr.qr_wire_bytes(b, 2048) == tb
        assert qr.qr_wire_bytes(b, 2049) == 2 * tb
        assert qr.qr_wire_bytes(b, 2048 * 65536) == 65536 * tb
        for n in (2**64 - 1, 2**62 + 5, 2**60):
            tiles = -(-n // 2048)
            exact = tiles * tb
            assert qr.qr_wire_bytes(b, n) == (exact if exact < 2**64 else 0)  # 0 on size_t overflow


def test_status_strings():
    for code, stem in [(0, "QR_OK"), (1, "QR_ERR_INVALID_ARG"), (2, "QR_ERR_UNSUPPORTED"),
                       (3, "QR_ERR_MISALIGNED"), (4, "QR_ERR_SIZE"), (5, "QR_ERR_CUDA")]:
        assert qr.status_string(code).startswith(stem)
    assert qr.status_string(99).startswith("QR_ERR_UNKNOWN")


@no_gpu_only
def test_encode_decode_validation():
    n = 4096
    assert capi.qr_encode(4, 0, A, 0, B) == qr.QR_ERR_INVALID_ARG          # n == 0
    assert capi.qr_encode(4, 0, None, n, B) == qr.QR_ERR_INVALID_ARG       # null x
    assert capi.qr_encode(4, 0, A, n, None) == qr.QR_ERR_INVALID_ARG       # null wire
    assert capi.qr_encode(5, 0, A, n, B) == qr.QR_ERR_UNSUPPORTED          # bits
    assert capi.qr_encode(4, 2, A, n, B) == qr.QR_ERR_UNSUPPORTED          # dtype
    assert capi.qr_encode(4, 0, A, 2**63, B) == qr.QR_ERR_SIZE             # 2n overflows
    assert capi.qr_encode(4, 0, A + 8, n, B) == qr.QR_ERR_MISALIGNED
    assert capi.qr_encode(4, 0, A, n, B + 2) == qr.QR_ERR_MISALIGNED
    assert capi.qr_encode(4, 0, A, n, A + 1024) == qr.QR_ERR_INVALID_ARG   # wire overlaps x
    assert capi.qr_encode(4, 0, A, n, A) == qr.QR_ERR_INVALID_ARG          # even exactly
    assert capi.qr_decode(3, 1, A, 0, Y) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_decode(3, 1, None, n, Y) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_decode(2, 1, A, n, Y) == qr.QR_ERR_UNSUPPORTED
    assert capi.qr_decode(3, -1, A, n, Y) == qr.QR_ERR_UNSUPPORTED
    assert capi.qr_decode(3, 1, A + 4, n, Y) == qr.QR_ERR_MISALIGNED
    assert capi.qr_decode(3, 1, A, n, A + 16) == qr.QR_ERR_INVALID_ARG    # y overlaps wire


@no_gpu_only
def test_reduce_validation():
    n = 2048 * 3
    W = qr.qr_wire_bytes(4, n)
    assert capi.qr_segment_reduce(4, 0, [A], n, Y) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_segment_reduce(4, 2, [A, None], n, Y) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_segment_reduce(4, 2, [A, B], n, None) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_segment_reduce(4, 2, None, n, Y) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_segment_reduce(4, 9, [A + 16 * i for i in range(9)], n, Y) == qr.QR_ERR_UNSUPPORTED
    assert capi.qr_segment_reduce(7, 2, [A, B], n, Y) == qr.QR_ERR_UNSUPPORTED
    assert capi.qr_segment_reduce(4, 2, [A, B + 8], n, Y) == qr.QR_ERR_MISALIGNED
    assert capi.qr_segment_reduce(4, 2, [A, B], n, A + W - 16) == qr.QR_ERR_INVALID_ARG  # partial overlap
    assert capi.qr_segment_reduce(4, 2, [A, B], 2**62 * 3, Y) == qr.QR_ERR_SIZE
    assert capi.qr_segment_reduce_staged(4, 2, [A, B], n, Y, -1) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_fc_segment_reduce_staged(4, 8, 2, [A, B], n, Y, -1) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_fc_segment_reduce_staged(8, 4, 2, [A, B], n, Y, 0) == qr.QR_ERR_UNSUPPORTED
    assert capi.qr_segment_reduce_staged(4, 2, [A, B + 8], n, Y, 0) == qr.QR_ERR_MISALIGNED
    assert capi.qr_segment_reduce_staged(7, 2, [A, B], n, Y, 0) == qr.QR_ERR_UNSUPPORTED
    assert capi.qr_segment_reduce_staged(4, 2, [A, B], n, A + W - 16, 0) == qr.QR_ERR_INVALID_ARG


@no_gpu_only
def test_allreduce_validation():
    n = 2048 * 2 + 37
    V = 2 * n
    W = qr.qr_wire_bytes(3, n)
    xs = [A, B]
    assert capi.qr_allreduce(3, 0, 2, xs, 0, Y) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_allreduce(3, 0, 0, xs, n, Y) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_allreduce(3, 0, 2, [A, None], n, Y) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_allreduce(3, 0, 2, xs, n, None) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_allreduce(3, 0, 9, [A + 4096 * i for i in range(9)], n, Y) == qr.QR_ERR_UNSUPPORTED
    assert capi.qr_allreduce(1, 0, 2, xs, n, Y) == qr.QR_ERR_UNSUPPORTED
    assert capi.qr_allreduce(3, 5, 2, xs, n, Y) == qr.QR_ERR_UNSUPPORTED
    assert capi.qr_allreduce(3, 0, 2, [A, B + 2], n, Y) == qr.QR_ERR_MISALIGNED
    assert capi.qr_allreduce(3, 0, 2, xs, n, Y + 8) == qr.QR_ERR_MISALIGNED
    assert capi.qr_allreduce(3, 0, 2, xs, n, A + 16) == qr.QR_ERR_INVALID_ARG   # y partially overlaps x[0]
    assert capi.qr_allreduce(3, 0, 2, xs, n, B - 4096) == qr.QR_ERR_INVALID_ARG  # y's end overlaps x[1]
    assert capi.qr_allreduce(3, 0, 2, xs, 2**63, Y) == qr.QR_ERR_SIZE
    assert capi.qr_allreduce_ctas(3, 0, 2, xs, n, Y, -1) == qr.QR_ERR_INVALID_ARG
    # the staged kernel: the same checks, ctas >= 0, and 32-byte alignment
    assert capi.qr_allreduce_staged(3, 0, 2, xs, n, Y, -1) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_allreduce_staged(3, 0, 2, xs, 0, Y, 0) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_allreduce_staged(1, 0, 2, xs, n, Y, 0) == qr.QR_ERR_UNSUPPORTED
    assert capi.qr_allreduce_staged(3, 0, 2, [A, B + 16], n, Y, 0) == qr.QR_ERR_MISALIGNED
    assert capi.qr_allreduce_staged(3, 0, 2, xs, n, Y + 16, 0) == qr.QR_ERR_MISALIGNED
    assert capi.qr_allreduce_staged(3, 0, 2, xs, n, A + 32, 0) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_allreduce_staged(3, 0, 2, xs, 2**63, Y, 0) == qr.QR_ERR_SIZE
    assert capi.qr_fc_allreduce_staged(4, 8, 0, 2, xs, n, Y, -1) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_fc_allreduce_ctas(4, 8, 0, 2, xs, n, Y, -1) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_fc_allreduce_staged(4, 4, 0, 2, [A, B + 16], n, Y, 0) == qr.QR_ERR_MISALIGNED
    assert capi.qr_fc_allreduce_staged(3, 8, 0, 2, xs, n, Y, 0) == qr.QR_ERR_UNSUPPORTED
    # the timeout counter's reader rejects a null destination without touching the device
    assert qr.lib().qr_wait_timeouts(None) == qr.QR_ERR_INVALID_ARG
    # emit: every output disjoint from every other buffer
    wo = [Y + 2**20, Y + 2**21]
    assert capi.qr_allreduce_emit(3, 0, 2, xs, n, Y, [wo[0], None], None) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_allreduce_emit(3, 0, 2, xs, n, Y, [wo[0], A], None) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_allreduce_emit(3, 0, 2, xs, n, Y, [wo[0], wo[0] + W - 16], None) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_allreduce_emit(3, 0, 2, xs, n, Y, wo, wo[1]) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_allreduce_emit(3, 0, 2, xs, n, Y, wo, Y) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_allreduce_emit(3, 0, 2, xs, n, Y, wo, Y + 2**22 + 8) == qr.QR_ERR_MISALIGNED
    assert capi.qr_allreduce_emit(3, 0, 2, xs, n, Y, [wo[0], wo[1] + 4], None) == qr.QR_ERR_MISALIGNED


def test_fc_sizes():
    assert qr.qr_fc_tile_bytes(4) == 1152 and qr.qr_fc_tile_bytes(8) == 2176
    for b in (3, 6, 0, 16):
        assert qr.qr_fc_tile_bytes(b) == 0 and qr.qr_fc_wire_bytes(b, 10) == 0
    assert qr.qr_fc_wire_bytes(4, 2049) == 2 * 1152


@no_gpu_only
def test_fc_validation():
    n = 2048 + 5
    assert capi.qr_fc_encode(4, 0, A, 0, B) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_fc_encode(3, 0, A, n, B) == qr.QR_ERR_UNSUPPORTED    # FC is INT4 / INT8 only
    assert capi.qr_fc_encode(6, 1, A, n, B) == qr.QR_ERR_UNSUPPORTED
    assert capi.qr_fc_encode(4, 0, A + 2, n, B) == qr.QR_ERR_MISALIGNED
    assert capi.qr_fc_encode(8, 0, A, n, A + 32) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_fc_decode(8, 1, None, n, Y) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_fc_decode(5, 1, A, n, Y) == qr.QR_ERR_UNSUPPORTED
    assert capi.qr_fc_decode(4, 1, A, n, A + 16) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_fc_segment_reduce(8, 4, 2, [A, B], n, Y) == qr.QR_ERR_UNSUPPORTED  # (8,4) is not a scheme
    assert capi.qr_fc_segment_reduce(4, 8, 0, [A], n, Y) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_fc_segment_reduce(4, 8, 9, [A + 4096 * i for i in range(9)], n, Y) == qr.QR_ERR_UNSUPPORTED
    assert capi.qr_fc_segment_reduce(4, 8, 2, [A, B], n, A) == qr.QR_ERR_INVALID_ARG  # widths differ: no in-place
    assert capi.qr_fc_segment_reduce(4, 4, 2, [A, B], n, A + 16) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_fc_allreduce(8, 4, 0, 2, [A, B], n, Y) == qr.QR_ERR_UNSUPPORTED
    assert capi.qr_fc_allreduce(4, 8, 2, 2, [A, B], n, Y) == qr.QR_ERR_UNSUPPORTED     # dtype
    assert capi.qr_fc_allreduce(4, 8, 0, 2, [A, None], n, Y) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_fc_allreduce(4, 8, 0, 2, [A, B], n, A + 16) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_fc_allreduce(4, 8, 0, 2, [A, B + 8], n, Y) == qr.QR_ERR_MISALIGNED
    assert capi.qr_fc_allreduce(4, 8, 0, 2, [A, B], 2**63, Y) == qr.QR_ERR_SIZE


def test_fp4_sizes():
    assert qr.qr_fp4_tile_bytes() == qr.qr_tile_bytes(4) == 1152
    assert qr.qr_fp4_wire_bytes(2049) == 2 * 1152 and qr.qr_fp4_wire_bytes(1) == 1152


@no_gpu_only
def test_fp4_validation():
    n = 2048 + 5
    assert capi.qr_fp4_encode(0, A, 0, B) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_fp4_encode(0, None, n, B) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_fp4_encode(2, A, n, B) == qr.QR_ERR_UNSUPPORTED       # dtype
    assert capi.qr_fp4_encode(0, A + 2, n, B) == qr.QR_ERR_MISALIGNED
    assert capi.qr_fp4_encode(1, A, n, A + 32) == qr.QR_ERR_INVALID_ARG   # wire overlaps x
    assert capi.qr_fp4_decode(1, None, n, Y) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_fp4_decode(3, A, n, Y) == qr.QR_ERR_UNSUPPORTED
    assert capi.qr_fp4_decode(1, A, n, A + 16) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_fp4_decode(1, A, n, Y + 8) == qr.QR_ERR_MISALIGNED
    assert capi.qr_fp4_segment_reduce(0, [A], n, Y, 0) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_fp4_segment_reduce(2, [A, None], n, Y, 0) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_fp4_segment_reduce(2, [A, B], n, Y, -1) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_fp4_segment_reduce(9, [A + 4096 * i for i in range(9)], n, Y, 0) == qr.QR_ERR_UNSUPPORTED
    assert capi.qr_fp4_segment_reduce(2, [A, B + 8], n, Y, 0) == qr.QR_ERR_MISALIGNED
    assert capi.qr_fp4_segment_reduce(2, [A, B], n, A + 16, 0) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_fp4_segment_reduce(2, [A, B], 2**63, Y, 0) == qr.QR_ERR_SIZE
    assert capi.qr_fp4_allreduce(0, 2, [A, None], n, Y, 0) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_fp4_allreduce(0, 2, [A, B], n, Y, -1) == qr.QR_ERR_INVALID_ARG
    assert capi.qr_fp4_allreduce(2, 2, [A, B], n, Y, 0) == qr.QR_ERR_UNSUPPORTED    # dtype
    assert capi.qr_fp4_allreduce(0, 9, [A + 4096 * i for i in range(9)], n, Y, 0) == qr.QR_ERR_UNSUPPORTED
    assert capi.qr_fp4_allreduce(0, 2, [A, B + 16], n, Y, 0) == qr.QR_ERR_MISALIGNED  # 32-byte alignment
    assert capi.qr_fp4_allreduce(0, 2, [A, B], n, Y + 16, 0) == qr.QR_ERR_MISALIGNED
    assert capi.qr_fp4_allreduce(0, 2, [A, B], n, A + 32, 0) == qr.QR_ERR_INVALID_ARG  # partial overlap
    assert capi.qr_fp4_allreduce(0, 2, [A, B], 2**63, Y, 0) == qr.QR_ERR_SIZE


def test_twoshot_workspace_bytes():
    for bits in (3, 4, 6, 8):
        tb = qr.qr_tile_bytes(bits)
        for R in (1, 2, 3, 8):
            for n in (1, 2048, 2049, 2048 * 17 + 5, 2**27):
                T = -(-n // 2048)
                seg = -(-T // R)
                assert qr.qr_twoshot_workspace_bytes(bits, R, n) == R * (R + 1) * seg * tb
    assert qr.qr_twoshot_workspace_bytes(5, 2, 100) == 0
    assert qr.qr_twoshot_workspace_bytes(4, 0, 100) == 0
    assert qr.qr_twoshot_workspace_bytes(4, 9, 100) == 0
    assert qr.qr_twoshot_workspace_bytes(8, 8, 2**64 - 1) == 0


def test_fc_twoshot_workspace_bytes():
    for brs, bag in ((4, 4), (4, 8), (8, 8)):
        ti, to = 256 * brs + 128, 256 * bag + 128
        for R in (1, 2, 3, 8):
            for n in (1, 2048, 2049, 2048 * 17 + 5, 2**27):
                T = -(-n // 2048)
                seg = -(-T // R)
                assert qr.qr_fc_twoshot_workspace_bytes(brs, bag, R, n) == R * R * seg * ti + T * to
    assert qr.qr_fc_twoshot_workspace_bytes(8, 4, 2, 100) == 0
    assert qr.qr_fc_twoshot_workspace_bytes(4, 6, 2, 100) == 0
    assert qr.qr_fc_twoshot_workspace_bytes(4, 4, 0, 100) == 0
    assert qr.qr_fc_twoshot_workspace_bytes(4, 4, 9, 100) == 0
    assert qr.qr_fc_twoshot_workspace_bytes(8, 8, 8, 2**64 - 1) == 0


def test_fp4_twoshot_workspace_bytes():
    for R in (1, 2, 3, 8):
        for n in (1, 2048, 2049, 2048 * 17 + 5, 2**27):
            assert qr.qr_fp4_twoshot_workspace_bytes(R, n) == qr.qr_twoshot_workspace_bytes(4, R, n)
    assert qr.qr_fp4_twoshot_workspace_bytes(0, 100) == 0
    assert qr.qr_fp4_twoshot_workspace_bytes(9, 100) == 0


@no_gpu_only
def test_fp4_twoshot_validation():
    n = 2048 * 5 + 3
    need = qr.qr_fp4_twoshot_workspace_bytes(2, n)
    WS = 0x7F3000000000
    xs, ys = [A, B], [Y, Y + 2**24]
    call = capi.qr_fp4_allreduce_twoshot
    assert call(0, 2, xs, n, ys, None, need) == qr.QR_ERR_INVALID_ARG
    assert call(0, 2, xs, n, [Y, None], WS, need) == qr.QR_ERR_INVALID_ARG
    assert call(0, 2, xs, 0, ys, WS, need) == qr.QR_ERR_INVALID_ARG
    assert call(2, 2, xs, n, ys, WS, need) == qr.QR_ERR_UNSUPPORTED              # dtype
    assert call(0, 9, [A + 4096 * i for i in range(9)], n, [Y + 2**22 * i for i in range(9)], WS,
                need) == qr.QR_ERR_UNSUPPORTED
    assert call(0, 2, xs, n, ys, WS, need - 1) == qr.QR_ERR_SIZE
    assert call(0, 2, xs, n, ys, WS + 8, need) == qr.QR_ERR_MISALIGNED
    assert call(0, 2, xs, n, [Y, Y + 4096], WS, need) == qr.QR_ERR_INVALID_ARG      # outputs overlap
    assert call(0, 2, xs, n, [A + 16, Y], WS, need) == qr.QR_ERR_INVALID_ARG         # partial in-place
    assert call(0, 2, xs, n, ys, A, need) == qr.QR_ERR_INVALID_ARG                 # workspace over an input


@no_gpu_only
def test_fc_twoshot_validation():
    n = 2048 * 5 + 3
    need = qr.qr_fc_twoshot_workspace_bytes(4, 8, 2, n)
    WS = 0x7F3000000000
    xs, ys = [A, B], [Y, Y + 2**24]
    call = capi.qr_fc_allreduce_twoshot
    assert call(4, 8, 0, 2, xs, n, ys, None, need) == qr.QR_ERR_INVALID_ARG
    assert call(4, 8, 0, 2, xs, n, [Y, None], WS, need) == qr.QR_ERR_INVALID_ARG
    assert call(4, 8, 0, 2, xs, 0, ys, WS, need) == qr.QR_ERR_INVALID_ARG
    assert call(8, 4, 0, 2, xs, n, ys, WS, need) == qr.QR_ERR_UNSUPPORTED       # no 8 -> 4 pair
    assert call(4, 8, 2, 2, xs, n, ys, WS, need) == qr.QR_ERR_UNSUPPORTED       # dtype
    assert call(4, 8, 0, 9, [A + 4096 * i for i in range(9)], n, [Y + 2**22 * i for i in range(9)], WS,
                need) == qr.QR_ERR_UNSUPPORTED
    assert call(4, 8, 0, 2, xs, n, ys, WS, need - 1) == qr.QR_ERR_SIZE
    assert call(4, 8, 0, 2, xs, n, ys, WS + 8, need) == qr.QR_ERR_MISALIGNED
    assert call(4, 8, 0, 2, [A + 8, B], n, ys, WS, need) == qr.QR_ERR_MISALIGNED
    assert call(4, 8, 0, 2, xs, n, [Y, Y + 4096], WS, need) == qr.QR_ERR_INVALID_ARG   # outputs overlap
    assert call(4, 8, 0, 2, xs, n, [A + 16, Y], WS, need) == qr.QR_ERR_INVALID_ARG      # partial in-place
    assert call(4, 8, 0, 2, xs, n, ys, A, need) == qr.QR_ERR_INVALID_ARG              # workspace over an input
    assert call(4, 8, 0, 2, xs, 2**63, ys, WS, need) == qr.QR_ERR_SIZE


@no_gpu_only
def test_twoshot_validation():
    n = 2048 * 5 + 3
    need = qr.qr_twoshot_workspace_bytes(4, 2, n)
    WS = 0x7F3000000000
    V = 2 * n
    xs, ys = [A, B], [Y, Y + 2**24]
    call = capi.qr_allreduce_twoshot
    assert call(4, 0, 2, xs, n, ys, None, need) == qr.QR_ERR_INVALID_ARG
    assert call(4, 0, 2, xs, n, [Y, None], WS, need) == qr.QR_ERR_INVALID_ARG
    assert call(4, 0, 2, xs, 0, ys, WS, need) == qr.QR_ERR_INVALID_ARG
    assert call(5, 0, 2, xs, n, ys, WS, need) == qr.QR_ERR_UNSUPPORTED
    assert call(4, 0, 9, [A + 4096 * i for i in range(9)], n, [Y + 2**22 * i for i in range(9)], WS,
                need) == qr.QR_ERR_UNSUPPORTED
    assert call(4, 0, 2, xs, n, ys, WS, need - 1) == qr.QR_ERR_SIZE            # workspace too small
    assert call(4, 0, 2, xs, n, ys, WS + 8, need) == qr.QR_ERR_MISALIGNED
    assert call(4, 0, 2, xs, n, [Y, Y + 4096], WS, need) == qr.QR_ERR_INVALID_ARG   # outputs overlap
    assert call(4, 0, 2, xs, n, [Y, Y], WS, need) == qr.QR_ERR_INVALID_ARG
    assert call(4, 0, 2, xs, n, [A + 16, Y], WS, need) == qr.QR_ERR_INVALID_ARG      # partial in-place
    assert call(4, 0, 2, xs, n, ys, A, need) == qr.QR_ERR_INVALID_ARG              # workspace over an input
    # the one-launch version: the same checks against its larger workspace
    T = -(-n // 2048)
    fneed = qr.lib().qr_twoshot_flags_workspace_bytes(4, 2, n)
    assert fneed == -(-need // 16) * 16 + 4 * (2 * T + 1)
    fcall = capi.qr_allreduce_twoshot_flags
    assert fcall(4, 0, 2, xs, n, ys, WS, fneed - 1) == qr.QR_ERR_SIZE
    assert fcall(4, 0, 2, xs, n, ys, WS, need) == qr.QR_ERR_SIZE
    assert fcall(4, 0, 2, xs, n, ys, WS + 8, fneed) == qr.QR_ERR_MISALIGNED
    assert fcall(4, 0, 2, xs, n, [A + 16, Y], WS, fneed) == qr.QR_ERR_INVALID_ARG
    assert fcall(5, 0, 2, xs, n, ys, WS, fneed) == qr.QR_ERR_UNSUPPORTED
    assert fcall(4, 0, 2, xs, n, ys, None, fneed) == qr.QR_ERR_INVALID_ARG
    assert qr.lib().qr_twoshot_flags_workspace_bytes(4, 9, n) == 0
    # the failure-path self-test: the same checks, and the dropped sender must be a rank
    dcall = capi.qr_selftest_twoshot_flags_drop
    for drop in (-1, 2, 8):
        assert dcall(4, 0, 2, xs, n, ys, WS, fneed, drop) == qr.QR_ERR_INVALID_ARG
    assert dcall(4, 0, 2, xs, n, ys, WS, fneed - 1, 0) == qr.QR_ERR_SIZE
    assert dcall(4, 0, 2, xs, n, ys, WS + 8, fneed, 1) == qr.QR_ERR_MISALIGNED


def test_peer_workspace_bytes():
    from bit_quantized_all_gb300 import peer
    L = peer._lib()
    for bits in (3, 4, 6, 8):
        tb = qr.qr_tile_bytes(bits)
        for R in (1, 2, 3, 8):
            for n in (1, 2048, 2049, 2048 * 17 + 5, 2**27):
                T = -(-n // 2048)
                seg = -(-T // R)
                assert L.qr_twoshot_peer_workspace_bytes(bits, R, n) == 2 * R * seg * tb
    assert L.qr_twoshot_peer_workspace_bytes(5, 2, 100) == 0
    assert L.qr_twoshot_peer_workspace_bytes(4, 0, 100) == 0
    assert L.qr_twoshot_peer_workspace_bytes(4, 9, 100) == 0
    assert L.qr_twoshot_peer_workspace_bytes(4, 2, 0) == 0
    assert L.qr_twoshot_peer_workspace_bytes(8, 8, 2**64 - 1) == 0
    assert L.qr_ipc_handle_bytes() == peer.QR_IPC_HANDLE_BYTES == 72


@no_gpu_only
def test_peer_validation():
    from bit_quantized_all_gb300 import peer
    L = peer._lib()
    n = 2048 * 5 + 3
    need = L.qr_twoshot_peer_workspace_bytes(4, 2, n)
    W0, W1 = 0x7F3000000000, 0x7F4000000000
    ws = peer._ptrs([W0, W1])
    send, red, dec = L.qr_twoshot_peer_send, L.qr_twoshot_peer_reduce, L.qr_twoshot_peer_decode
    assert send(4, 0, 2, 0, None, n, ws, None) == qr.QR_ERR_INVALID_ARG           # no input
    assert send(4, 0, 2, 0, A, n, None, None) == qr.QR_ERR_INVALID_ARG            # no workspaces
    assert send(4, 0, 2, 0, A, n, peer._ptrs([W0, None]), None) == qr.QR_ERR_INVALID_ARG
    assert send(4, 0, 2, 2, A, n, ws, None) == qr.QR_ERR_INVALID_ARG              # rank out of range
    assert send(4, 0, 2, -1, A, n, ws, None) == qr.QR_ERR_INVALID_ARG
    assert send(4, 0, 2, 0, A, 0, ws, None) == qr.QR_ERR_INVALID_ARG
    assert send(5, 0, 2, 0, A, n, ws, None) == qr.QR_ERR_UNSUPPORTED
    assert send(4, 2, 2, 0, A, n, ws, None) == qr.QR_ERR_UNSUPPORTED              # dtype
    assert send(4, 0, 9, 0, A, n, peer._ptrs([W0 + 2**30 * i for i in range(9)]), None) == qr.QR_ERR_UNSUPPORTED
    assert send(4, 0, 2, 0, A + 8, n, ws, None) == qr.QR_ERR_MISALIGNED
    assert send(4, 0, 2, 0, A, n, peer._ptrs([W0, W1 + 8]), None) == qr.QR_ERR_MISALIGNED
    assert send(4, 0, 2, 0, A, n, peer._ptrs([W0, W0 + 64]), None) == qr.QR_ERR_INVALID_ARG   # overlapping
    assert send(4, 0, 2, 0, W0 + 16, n, ws, None) == qr.QR_ERR_INVALID_ARG                   # input in a workspace
    assert red(4, 2, 2, n, ws, None) == qr.QR_ERR_INVALID_ARG
    assert red(4, 2, 0, n, None, None) == qr.QR_ERR_INVALID_ARG
    assert red(4, 2, 0, n, peer._ptrs([W0, W0 + need - 16]), None) == qr.QR_ERR_INVALID_ARG
    assert red(7, 2, 0, n, ws, None) == qr.QR_ERR_UNSUPPORTED
    assert dec(4, 0, 2, n, None, Y, None) == qr.QR_ERR_INVALID_ARG
    assert dec(4, 0, 2, n, W0, None, None) == qr.QR_ERR_INVALID_ARG
    assert dec(4, 0, 2, n, W0 + 8, Y, None) == qr.QR_ERR_MISALIGNED
    assert dec(4, 0, 2, n, W0, W0 + 32, None) == qr.QR_ERR_INVALID_ARG              # output in the workspace
    assert dec(4, 3, 2, n, W0, Y, None) == qr.QR_ERR_UNSUPPORTED
    assert L.qr_ipc_get_handle(None, None) == qr.QR_ERR_INVALID_ARG
    assert L.qr_ipc_open_handle(None, None) == qr.QR_ERR_INVALID_ARG
    assert L.qr_ipc_close_handle(None) == qr.QR_ERR_INVALID_ARG
    assert L.qr_ipc_close_handle(W0) == qr.QR_ERR_INVALID_ARG                       # never opened


def test_codec_peer_workspace_bytes():
    """recv at the reduce-scatter width, then the gathered wire at the
    all-gather width: R*seg tiles of each."""
    from bit_quantized_all_gb300 import peer
    L = peer._lib()
    for rs, ag in qr.FC_PAIRS:
        ti, to = qr.qr_fc_tile_bytes(rs), qr.qr_fc_tile_bytes(ag)
        for R in (1, 2, 3, 8):
            for n in (1, 2048, 2049, 2048 * 17 + 5, 2**27):
                seg = -(-(-(-n // 2048)) // R)
                assert L.qr_fc_twoshot_peer_workspace_bytes(rs, ag, R, n) == R * seg * (ti + to)
    for R in (1, 2, 5, 8):
        for n in (1, 2049, 2**26 + 3):
            assert L.qr_fp4_twoshot_peer_workspace_bytes(R, n) == L.qr_twoshot_peer_workspace_bytes(4, R, n)
    assert L.qr_fc_twoshot_peer_workspace_bytes(8, 4, 2, 100) == 0      # not a width pair
    assert L.qr_fc_twoshot_peer_workspace_bytes(4, 6, 2, 100) == 0
    assert L.qr_fc_twoshot_peer_workspace_bytes(4, 8, 9, 100) == 0
    assert L.qr_fc_twoshot_peer_workspace_bytes(4, 8, 2, 0) == 0
    assert L.qr_fc_twoshot_peer_workspace_bytes(8, 8, 8, 2**64 - 1) == 0
    assert L.qr_fp4_twoshot_peer_workspace_bytes(0, 100) == 0
    assert L.qr_fp4_twoshot_peer_workspace_bytes(9, 100) == 0
    assert L.qr_fp4_twoshot_peer_workspace_bytes(8, 2**64 - 1) == 0


@no_gpu_only
@pytest.mark.parametrize("codec", ["fc", "fp4"])
def test_codec_peer_validation(codec):
    """The asymmetric and FP4 per-rank calls check their arguments as the
    symmetric ones do, in the same order, before any CUDA call."""
    from bit_quantized_all_gb300 import peer
    L = peer._lib()
    n = 2048 * 5 + 3
    W0, W1 = 0x7F3000000000, 0x7F4000000000
    ws = peer._ptrs([W0, W1])
    if codec == "fc":
        need = L.qr_fc_twoshot_peer_workspace_bytes(4, 8, 2, n)

        def send(dt, R, rank, x, n_, w, rs=4, ag=8):
            return L.qr_fc_twoshot_peer_send(rs, ag, dt, R, rank, x, n_, w, None)

        def red(R, rank, n_, w, rs=4, ag=8):
            return L.qr_fc_twoshot_peer_reduce(rs, ag, R, rank, n_, w, None)

        def dec(dt, R, n_, w, y, rs=4, ag=8):
            return L.qr_fc_twoshot_peer_decode(rs, ag, dt, R, n_, w, y, None)

        assert send(0, 2, 0, A, n, ws, rs=8, ag=4) == qr.QR_ERR_UNSUPPORTED
        assert red(2, 0, n, ws, rs=6) == qr.QR_ERR_UNSUPPORTED
        assert dec(0, 2, n, W0, Y, ag=3) == qr.QR_ERR_UNSUPPORTED
    else:
        need = L.qr_fp4_twoshot_peer_workspace_bytes(2, n)

        def send(dt, R, rank, x, n_, w):
            return L.qr_fp4_twoshot_peer_send(dt, R, rank, x, n_, w, None)

        def red(R, rank, n_, w):
            return L.qr_fp4_twoshot_peer_reduce(R, rank, n_, w, None)

        def dec(dt, R, n_, w, y):
            return L.qr_fp4_twoshot_peer_decode(dt, R, n_, w, y, None)
    assert need > 0
    assert send(0, 2, 0, None, n, ws) == qr.QR_ERR_INVALID_ARG           # no input
    assert send(0, 2, 0, A, n, None) == qr.QR_ERR_INVALID_ARG            # no workspaces
    assert send(0, 2, 0, A, n, peer._ptrs([W0, None])) == qr.QR_ERR_INVALID_ARG
    assert send(0, 2, 2, A, n, ws) == qr.QR_ERR_INVALID_ARG              # rank out of range
    assert send(0, 2, -1, A, n, ws) == qr.QR_ERR_INVALID_ARG
    assert send(0, 2, 0, A, 0, ws) == qr.QR_ERR_INVALID_ARG
    assert send(0, 0, 0, A, n, ws) == qr.QR_ERR_INVALID_ARG              # R < 1
    assert send(2, 2, 0, A, n, ws) == qr.QR_ERR_UNSUPPORTED              # dtype
    assert send(0, 9, 0, A, n, peer._ptrs([W0 + 2**30 * i for i in range(9)])) == qr.QR_ERR_UNSUPPORTED
    assert send(0, 2, 0, A, 2**62, ws) == qr.QR_ERR_SIZE
    assert send(0, 2, 0, A + 8, n, ws) == qr.QR_ERR_MISALIGNED
    assert send(0, 2, 0, A, n, peer._ptrs([W0, W1 + 8])) == qr.QR_ERR_MISALIGNED
    assert send(0, 2, 0, A, n, peer._ptrs([W0, W0 + 64])) == qr.QR_ERR_INVALID_ARG   # overlapping
    assert send(0, 2, 0, A, n, peer._ptrs([W0, W0 + need - 16])) == qr.QR_ERR_INVALID_ARG
    assert send(0, 2, 0, W0 + 16, n, ws) == qr.QR_ERR_INVALID_ARG        # input in a workspace
    assert red(2, 2, n, ws) == qr.QR_ERR_INVALID_ARG
    assert red(2, 0, n, None) == qr.QR_ERR_INVALID_ARG
    assert red(2, 0, 0, ws) == qr.QR_ERR_INVALID_ARG
    assert red(9, 0, n, peer._ptrs([W0 + 2**30 * i for i in range(9)])) == qr.QR_ERR_UNSUPPORTED
    assert red(2, 0, n, peer._ptrs([W0, W0 + need - 16])) == qr.QR_ERR_INVALID_ARG
    assert red(2, 0, n, peer._ptrs([W0, W1 + 4])) == qr.QR_ERR_MISALIGNED
    assert red(2, 0, 2**62, ws) == qr.QR_ERR_SIZE
    assert dec(0, 2, n, None, Y) == qr.QR_ERR_INVALID_ARG
    assert dec(0, 2, n, W0, None) == qr.QR_ERR_INVALID_ARG
    assert dec(0, 2, 0, W0, Y) == qr.QR_ERR_INVALID_ARG
    assert dec(0, 2, n, W0 + 8, Y) == qr.QR_ERR_MISALIGNED
    assert dec(0, 2, n, W0, Y + 2) == qr.QR_ERR_MISALIGNED
    assert dec(0, 2, n, W0, W0 + 32) == qr.QR_ERR_INVALID_ARG            # output in the workspace
    assert dec(3, 2, n, W0, Y) == qr.QR_ERR_UNSUPPORTED
    assert dec(0, 9, n, W0, Y) == qr.QR_ERR_UNSUPPORTED
    assert dec(0, 2, 2**62, W0, Y) == qr.QR_ERR_SIZE


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(qr, "LIB_PATH", str(tmp_path / "missing" / "libqr.so"))
    monkeypatch.setattr(qr, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        qr.qr_tile_bytes(4)


def test_product_package_does_not_touch_the_oracle():
    pkg = os.path.join(ROOT, "bit_quantized_all_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"\boracle\b|qr_oracle|liboracle|orc_", text), f


def test_concurrent_builds_take_turns(monkeypatch):
    """Two builds at once (as the ranks of one job may start them) never
    compile at the same time: the second waits for the lock, then finds the
    library up to date and compiles nothing."""
    import threading
    import time

    from bit_quantized_all_gb300 import build as b
    state = {"active": 0, "overlap": False, "compiles": 0, "stale": True}

    def fake_build(verbose, ptxas_info):
        state["active"] += 1
        state["overlap"] |= state["active"] > 1
        state["compiles"] += 1
        time.sleep(0.3)
        state["stale"] = False
        state["active"] -= 1
        return b.LIB_PATH

    monkeypatch.setattr(b, "_build_locked", fake_build)
    monkeypatch.setattr(b, "_stale", lambda: state["stale"])
    threads = [threading.Thread(target=b.build) for _ in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=30)
    assert not state["overlap"]
    assert state["compiles"] == 1
