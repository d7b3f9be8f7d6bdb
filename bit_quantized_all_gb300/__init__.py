"""Block-quantized two-shot all-reduce codec (QuickReduce / Flash
Communication) for one GB300 GPU: Python binding of ``libqr.so``.

The functions carry the names of the C ABI in ``include/qr.h``.  They only
marshal arguments: check tensor dtypes, sizes, devices and contiguity, pick the
caller's current stream, and call the library through ``ctypes``.  Every step
of the codec runs in the library's CUDA kernels; there is no CPU path.  If
``libqr.so`` has not been built, every call raises.

Tensors: fp16 / bf16 messages are ``torch.float16`` / ``torch.bfloat16`` CUDA
tensors (any shape, contiguous; n = numel); wires are ``torch.uint8`` CUDA
tensors of at least ``qr_wire_bytes(bits, n)`` bytes.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqr.so")

QR_OK = 0
QR_ERR_INVALID_ARG = 1
QR_ERR_UNSUPPORTED = 2
QR_ERR_MISALIGNED = 3
QR_ERR_SIZE = 4
QR_ERR_CUDA = 5

QR_FP16 = 0
QR_BF16 = 1
QR_MAX_RANKS = 8
BITS = (3, 4, 6, 8)

EXPORTS = ("qr_tile_values", "qr_tile_bytes", "qr_wire_bytes", "qr_encode", "qr_segment_reduce",
           "qr_decode", "qr_allreduce", "qr_allreduce_emit", "qr_allreduce_ctas", "qr_status_string",
           "qr_fc_tile_bytes", "qr_fc_wire_bytes", "qr_fc_encode", "qr_fc_segment_reduce", "qr_fc_decode",
           "qr_fc_allreduce", "qr_twoshot_workspace_bytes", "qr_allreduce_twoshot",
           "qr_allreduce_twoshot_static", "qr_wait_timeouts", "qr_selftest_bounded_wait",
           "qr_allreduce_staged", "qr_fc_allreduce_staged", "qr_fc_allreduce_ctas",
           "qr_segment_reduce_staged", "qr_fc_segment_reduce_staged", "qr_twoshot_flags_workspace_bytes",
           "qr_allreduce_twoshot_flags", "qr_fp4_tile_bytes", "qr_fp4_wire_bytes", "qr_fp4_encode",
           "qr_fp4_decode", "qr_fp4_segment_reduce", "qr_fp4_allreduce", "qr_selftest_twoshot_flags_drop",
           "qr_twoshot_peer_workspace_bytes", "qr_twoshot_peer_send", "qr_twoshot_peer_reduce",
           "qr_twoshot_peer_decode", "qr_ipc_handle_bytes", "qr_ipc_get_handle", "qr_ipc_open_handle",
           "qr_ipc_close_handle", "qr_fc_twoshot_workspace_bytes", "qr_fc_allreduce_twoshot",
           "qr_fp4_twoshot_workspace_bytes", "qr_fp4_allreduce_twoshot", "qr_fc_twoshot_peer_workspace_bytes",
           "qr_fc_twoshot_peer_send", "qr_fc_twoshot_peer_reduce", "qr_fc_twoshot_peer_decode",
           "qr_fp4_twoshot_peer_workspace_bytes", "qr_fp4_twoshot_peer_send", "qr_fp4_twoshot_peer_reduce",
           "qr_fp4_twoshot_peer_decode")
TWOSHOT_STATIC_WORKSPACE_BYTES = 32 << 20  # QR_TWOSHOT_STATIC_WORKSPACE_BYTES
FC_BITS = (4, 8)
FC_PAIRS = ((4, 4), (4, 8), (8, 8))  # (reduce-scatter, all-gather) widths; (4, 8) is the mixed "INT6"

_lock = threading.Lock()
_lib = None


class QRError(RuntimeError):
    """A qr_* call returned a status other than QR_OK."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def lib() -> ctypes.CDLL:
    """The loaded libqr.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is not built; run bit_quantized_all_gb300.build.build() "
                    "(needs nvcc). There is no CPU fallback.")
            L = ctypes.CDLL(LIB_PATH)
            vp = ctypes.c_void_p
            sz = ctypes.c_size_t
            i32 = ctypes.c_int
            vpp = ctypes.POINTER(ctypes.c_void_p)
            sig = {
                "qr_tile_values": (sz, []),
                "qr_tile_bytes": (sz, [i32]),
                "qr_wire_bytes": (sz, [i32, sz]),
                "qr_encode": (i32, [i32, i32, vp, sz, vp, vp]),
                "qr_segment_reduce": (i32, [i32, i32, vpp, sz, vp, vp]),
                "qr_decode": (i32, [i32, i32, vp, sz, vp, vp]),
                "qr_allreduce": (i32, [i32, i32, i32, vpp, sz, vp, vp]),
                "qr_allreduce_emit": (i32, [i32, i32, i32, vpp, sz, vp, vpp, vp, vp]),
                "qr_allreduce_ctas": (i32, [i32, i32, i32, vpp, sz, vp, i32, vp]),
                "qr_status_string": (ctypes.c_char_p, [i32]),
                "qr_fc_tile_bytes": (sz, [i32]),
                "qr_fc_wire_bytes": (sz, [i32, sz]),
                "qr_fc_encode": (i32, [i32, i32, vp, sz, vp, vp]),
                "qr_fc_segment_reduce": (i32, [i32, i32, i32, vpp, sz, vp, vp]),
                "qr_fc_decode": (i32, [i32, i32, vp, sz, vp, vp]),
                "qr_fc_allreduce": (i32, [i32, i32, i32, i32, vpp, sz, vp, vp]),
                "qr_twoshot_workspace_bytes": (sz, [i32, i32, sz]),
                "qr_allreduce_twoshot": (i32, [i32, i32, i32, vpp, sz, vpp, vp, sz, vp]),
                "qr_twoshot_flags_workspace_bytes": (sz, [i32, i32, sz]),
                "qr_allreduce_twoshot_flags": (i32, [i32, i32, i32, vpp, sz, vpp, vp, sz, vp]),
                "qr_allreduce_twoshot_static": (i32, [i32, i32, i32, vpp, sz, vpp, vp]),
                "qr_selftest_twoshot_flags_drop": (i32, [i32, i32, i32, vpp, sz, vpp, vp, sz, i32, vp]),
                "qr_wait_timeouts": (i32, [ctypes.POINTER(ctypes.c_uint)]),
                "qr_allreduce_staged": (i32, [i32, i32, i32, vpp, sz, vp, i32, vp]),
                "qr_fc_allreduce_staged": (i32, [i32, i32, i32, i32, vpp, sz, vp, i32, vp]),
                "qr_fc_twoshot_workspace_bytes": (sz, [i32, i32, i32, sz]),
                "qr_fc_allreduce_twoshot": (i32, [i32, i32, i32, i32, vpp, sz, vpp, vp, sz, vp]),
                "qr_fp4_twoshot_workspace_bytes": (sz, [i32, sz]),
                "qr_fp4_allreduce_twoshot": (i32, [i32, i32, vpp, sz, vpp, vp, sz, vp]),
                "qr_fc_allreduce_ctas": (i32, [i32, i32, i32, i32, vpp, sz, vp, i32, vp]),
                "qr_segment_reduce_staged": (i32, [i32, i32, vpp, sz, vp, i32, vp]),
                "qr_fc_segment_reduce_staged": (i32, [i32, i32, i32, vpp, sz, vp, i32, vp]),
                "qr_selftest_bounded_wait": (i32, [vp]),
                "qr_fp4_tile_bytes": (sz, []),
                "qr_fp4_wire_bytes": (sz, [sz]),
                "qr_fp4_encode": (i32, [i32, vp, sz, vp, vp]),
                "qr_fp4_decode": (i32, [i32, vp, sz, vp, vp]),
                "qr_fp4_segment_reduce": (i32, [i32, vpp, sz, vp, i32, vp]),
                "qr_fp4_allreduce": (i32, [i32, i32, vpp, sz, vp, i32, vp]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().qr_status_string(status).decode()


def _ptr_array(ptrs):
    """A host array of device pointers (ints or None) for the C ABI."""
    if ptrs is None:
        return None
    return (ctypes.c_void_p * len(ptrs))(*ptrs)


def _check(status: int, where: str) -> None:
    if status != QR_OK:
        raise QRError(status, where)


# ---------------------------------------------------------------------------
# raw C ABI: integer device pointers, integer stream handle, status returned
# ---------------------------------------------------------------------------
class capi:
    """Direct calls of the C ABI with raw pointers; each returns the status."""

    @staticmethod
    def qr_encode(bits, dtype, x, n, wire, stream=None):
        return lib().qr_encode(bits, dtype, x, n, wire, stream)

    @staticmethod
    def qr_decode(bits, dtype, wire, n, y, stream=None):
        return lib().qr_decode(bits, dtype, wire, n, y, stream)

    @staticmethod
    def qr_segment_reduce(bits, R, wires, n, out, stream=None):
        return lib().qr_segment_reduce(bits, R, _ptr_array(wires), n, out, stream)

    @staticmethod
    def qr_segment_reduce_staged(bits, R, wires, n, out, ctas, stream=None):
        return lib().qr_segment_reduce_staged(bits, R, _ptr_array(wires), n, out, ctas, stream)

    @staticmethod
    def qr_allreduce(bits, dtype, R, xs, n, y, stream=None):
        return lib().qr_allreduce(bits, dtype, R, _ptr_array(xs), n, y, stream)

    @staticmethod
    def qr_allreduce_emit(bits, dtype, R, xs, n, y, wire_out, red_out, stream=None):
        return lib().qr_allreduce_emit(bits, dtype, R, _ptr_array(xs), n, y, _ptr_array(wire_out),
                                       red_out, stream)

    @staticmethod
    def qr_allreduce_ctas(bits, dtype, R, xs, n, y, ctas, stream=None):
        return lib().qr_allreduce_ctas(bits, dtype, R, _ptr_array(xs), n, y, ctas, stream)

    @staticmethod
    def qr_allreduce_staged(bits, dtype, R, xs, n, y, ctas, stream=None):
        return lib().qr_allreduce_staged(bits, dtype, R, _ptr_array(xs), n, y, ctas, stream)

    @staticmethod
    def qr_fp4_allreduce_twoshot(dtype, R, xs, n, ys, workspace, workspace_bytes, stream=None):
        return lib().qr_fp4_allreduce_twoshot(dtype, R, _ptr_array(xs), n, _ptr_array(ys), workspace,
                                              workspace_bytes, stream)

    @staticmethod
    def qr_fc_allreduce_twoshot(bits_rs, bits_ag, dtype, R, xs, n, ys, workspace, workspace_bytes, stream=None):
        return lib().qr_fc_allreduce_twoshot(bits_rs, bits_ag, dtype, R, _ptr_array(xs), n, _ptr_array(ys),
                                             workspace, workspace_bytes, stream)

    @staticmethod
    def qr_allreduce_twoshot(bits, dtype, R, xs, n, ys, workspace, workspace_bytes, stream=None):
        return lib().qr_allreduce_twoshot(bits, dtype, R, _ptr_array(xs), n, _ptr_array(ys), workspace,
                                          workspace_bytes, stream)

    @staticmethod
    def qr_allreduce_twoshot_flags(bits, dtype, R, xs, n, ys, workspace, workspace_bytes, stream=None):
        return lib().qr_allreduce_twoshot_flags(bits, dtype, R, _ptr_array(xs), n, _ptr_array(ys), workspace,
                                                workspace_bytes, stream)

    @staticmethod
    def qr_allreduce_twoshot_static(bits, dtype, R, xs, n, ys, stream=None):
        return lib().qr_allreduce_twoshot_static(bits, dtype, R, _ptr_array(xs), n, _ptr_array(ys), stream)

    @staticmethod
    def qr_selftest_twoshot_flags_drop(bits, dtype, R, xs, n, ys, workspace, workspace_bytes, drop_sender,
                                       stream=None):
        return lib().qr_selftest_twoshot_flags_drop(bits, dtype, R, _ptr_array(xs), n, _ptr_array(ys), workspace,
                                                    workspace_bytes, drop_sender, stream)

    @staticmethod
    def qr_wait_timeouts():
        """(status, count) -- reads and clears the device's wait-timeout counter."""
        c = ctypes.c_uint(0)
        st = lib().qr_wait_timeouts(ctypes.byref(c))
        return st, c.value

    @staticmethod
    def qr_selftest_bounded_wait(stream=None):
        return lib().qr_selftest_bounded_wait(stream)

    @staticmethod
    def qr_fc_encode(bits, dtype, x, n, wire, stream=None):
        return lib().qr_fc_encode(bits, dtype, x, n, wire, stream)

    @staticmethod
    def qr_fp4_encode(dtype, x, n, wire, stream=None):
        return lib().qr_fp4_encode(dtype, x, n, wire, stream)

    @staticmethod
    def qr_fp4_decode(dtype, wire, n, y, stream=None):
        return lib().qr_fp4_decode(dtype, wire, n, y, stream)

    @staticmethod
    def qr_fp4_segment_reduce(R, wires, n, out, ctas, stream=None):
        return lib().qr_fp4_segment_reduce(R, _ptr_array(wires), n, out, ctas, stream)

    @staticmethod
    def qr_fp4_allreduce(dtype, R, xs, n, y, ctas, stream=None):
        return lib().qr_fp4_allreduce(dtype, R, _ptr_array(xs), n, y, ctas, stream)

    @staticmethod
    def qr_fc_decode(bits, dtype, wire, n, y, stream=None):
        return lib().qr_fc_decode(bits, dtype, wire, n, y, stream)

    @staticmethod
    def qr_fc_segment_reduce(bits_in, bits_out, R, wires, n, out, stream=None):
        return lib().qr_fc_segment_reduce(bits_in, bits_out, R, _ptr_array(wires), n, out, stream)

    @staticmethod
    def qr_fc_segment_reduce_staged(bits_in, bits_out, R, wires, n, out, ctas, stream=None):
        return lib().qr_fc_segment_reduce_staged(bits_in, bits_out, R, _ptr_array(wires), n, out, ctas, stream)

    @staticmethod
    def qr_fc_allreduce_ctas(bits_rs, bits_ag, dtype, R, xs, n, y, ctas, stream=None):
        return lib().qr_fc_allreduce_ctas(bits_rs, bits_ag, dtype, R, _ptr_array(xs), n, y, ctas, stream)

    @staticmethod
    def qr_fc_allreduce_staged(bits_rs, bits_ag, dtype, R, xs, n, y, ctas, stream=None):
        return lib().qr_fc_allreduce_staged(bits_rs, bits_ag, dtype, R, _ptr_array(xs), n, y, ctas, stream)

    @staticmethod
    def qr_fc_allreduce(bits_rs, bits_ag, dtype, R, xs, n, y, stream=None):
        return lib().qr_fc_allreduce(bits_rs, bits_ag, dtype, R, _ptr_array(xs), n, y, stream)


# ---------------------------------------------------------------------------
# sizes
# ---------------------------------------------------------------------------
def qr_tile_values() -> int:
    return int(lib().qr_tile_values())


def qr_tile_bytes(bits: int) -> int:
    return int(lib().qr_tile_bytes(bits))


def qr_wire_bytes(bits: int, n: int) -> int:
    return int(lib().qr_wire_bytes(bits, n))


# ---------------------------------------------------------------------------
# torch-tensor front end
# ---------------------------------------------------------------------------
_DTYPES = {torch.float16: QR_FP16, torch.bfloat16: QR_BF16}
_TORCH = {QR_FP16: torch.float16, QR_BF16: torch.bfloat16}


def _dtype_code(t: torch.Tensor, what: str) -> int:
    if t.dtype not in _DTYPES:
        raise TypeError(f"{what} must be torch.float16 or torch.bfloat16, got {t.dtype}")
    return _DTYPES[t.dtype]


def _cuda_contig(t: torch.Tensor, what: str) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{what} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor (there is no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")


def _wire_tensor(t: torch.Tensor, bits: int, n: int, what: str) -> None:
    _cuda_contig(t, what)
    if t.dtype != torch.uint8:
        raise TypeError(f"{what} must be torch.uint8 (a packed wire), got {t.dtype}")
    need = qr_wire_bytes(bits, n)
    if t.numel() < need:
        raise ValueError(f"{what} holds {t.numel()} bytes; {need} are needed for {n} values at INT{bits}")


def _stream(device: torch.device, stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _same_device(ts, what):
    dev = ts[0].device
    for t in ts:
        if t.device != dev:
            raise ValueError(f"{what}: every tensor must be on {dev}")
    return dev


def new_wire(bits: int, n: int, device) -> torch.Tensor:
    """An uninitialised wire buffer for an n-value message."""
    return torch.empty(qr_wire_bytes(bits, n), dtype=torch.uint8, device=device)


def qr_encode(bits: int, x: torch.Tensor, wire: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Send path: quantize x into a packed wire (returned)."""
    _cuda_contig(x, "x")
    dt = _dtype_code(x, "x")
    n = x.numel()
    if wire is None:
        wire = new_wire(bits, n, x.device)
    _wire_tensor(wire, bits, n, "wire")
    _same_device([x, wire], "qr_encode")
    _check(capi.qr_encode(bits, dt, x.data_ptr(), n, wire.data_ptr(), _stream(x.device, stream)), "qr_encode")
    return wire


def qr_decode(bits: int, wire: torch.Tensor, n: int, dtype: torch.dtype = torch.bfloat16,
              y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Receive path: decode the first n values of a wire into fp16/bf16."""
    _wire_tensor(wire, bits, n, "wire")
    if y is None:
        if dtype not in _DTYPES:
            raise TypeError(f"dtype must be torch.float16 or torch.bfloat16, got {dtype}")
        y = torch.empty(n, dtype=dtype, device=wire.device)
    _cuda_contig(y, "y")
    dt = _dtype_code(y, "y")
    if y.numel() != n:
        raise ValueError(f"y holds {y.numel()} values, expected {n}")
    _same_device([wire, y], "qr_decode")
    _check(capi.qr_decode(bits, dt, wire.data_ptr(), n, y.data_ptr(), _stream(y.device, stream)), "qr_decode")
    return y


def qr_segment_reduce(bits: int, wires, n: int, out: torch.Tensor | None = None, stream=None,
                      staged: bool = False, ctas: int = 0) -> torch.Tensor:
    """Phase-1B: decode the R wires, sum in fp32 in rank order, re-quantize.
    `staged` runs the staged kernel (qr_segment_reduce_staged) at any size."""
    wires = list(wires)
    if not 1 <= len(wires) <= QR_MAX_RANKS:
        raise ValueError(f"1 to {QR_MAX_RANKS} wires are supported, got {len(wires)}")
    for i, w in enumerate(wires):
        _wire_tensor(w, bits, n, f"wires[{i}]")
    if out is None:
        out = new_wire(bits, n, wires[0].device)
    _wire_tensor(out, bits, n, "out")
    dev = _same_device(wires + [out], "qr_segment_reduce")
    ptrs = [w.data_ptr() for w in wires]
    if staged:
        status = capi.qr_segment_reduce_staged(bits, len(wires), ptrs, n, out.data_ptr(), ctas, _stream(dev, stream))
    else:
        status = capi.qr_segment_reduce(bits, len(wires), ptrs, n, out.data_ptr(), _stream(dev, stream))
    _check(status, "qr_segment_reduce")
    return out


def _check_inputs(xs):
    xs = list(xs)
    if not 1 <= len(xs) <= QR_MAX_RANKS:
        raise ValueError(f"1 to {QR_MAX_RANKS} ranks are supported, got {len(xs)}")
    for i, x in enumerate(xs):
        _cuda_contig(x, f"xs[{i}]")
    dt = _dtype_code(xs[0], "xs[0]")
    for i, x in enumerate(xs):
        if x.dtype != xs[0].dtype:
            raise TypeError(f"xs[{i}] is {x.dtype}; every rank must be {xs[0].dtype}")
        if x.numel() != xs[0].numel():
            raise ValueError(f"xs[{i}] holds {x.numel()} values; every rank must hold {xs[0].numel()}")
    return xs, dt, xs[0].numel()


def qr_allreduce(bits: int, xs, y: torch.Tensor | None = None, stream=None, ctas: int = 0) -> torch.Tensor:
    """The fused two-shot all-reduce of R rank tensors (one kernel)."""
    xs, dt, n = _check_inputs(xs)
    if y is None:
        y = torch.empty_like(xs[0])
    _cuda_contig(y, "y")
    if y.dtype != xs[0].dtype or y.numel() != n:
        raise ValueError("y must match the inputs' dtype and size")
    dev = _same_device(xs + [y], "qr_allreduce")
    ptrs = [x.data_ptr() for x in xs]
    st = _stream(dev, stream)
    if ctas:
        status = capi.qr_allreduce_ctas(bits, dt, len(xs), ptrs, n, y.data_ptr(), ctas, st)
    else:
        status = capi.qr_allreduce(bits, dt, len(xs), ptrs, n, y.data_ptr(), st)
    _check(status, "qr_allreduce")
    return y


def qr_allreduce_staged(bits: int, xs, y: torch.Tensor | None = None, stream=None, ctas: int = 0) -> torch.Tensor:
    """qr_allreduce on the staged kernel (bulk copies into shared memory, one
    persistent CTA per SM) at any size; every tensor 32-byte aligned."""
    xs, dt, n = _check_inputs(xs)
    if y is None:
        y = torch.empty_like(xs[0])
    _cuda_contig(y, "y")
    if y.dtype != xs[0].dtype or y.numel() != n:
        raise ValueError("y must match the inputs' dtype and size")
    dev = _same_device(xs + [y], "qr_allreduce_staged")
    status = capi.qr_allreduce_staged(bits, dt, len(xs), [x.data_ptr() for x in xs], n, y.data_ptr(), ctas,
                                      _stream(dev, stream))
    _check(status, "qr_allreduce_staged")
    return y


def qr_allreduce_emit(bits: int, xs, y: torch.Tensor | None = None, wire_out=None,
                      red_out: torch.Tensor | None = None, stream=None):
    """qr_allreduce that also returns the R Phase-1 wires and the reduced wire."""
    xs, dt, n = _check_inputs(xs)
    dev = _same_device(xs, "qr_allreduce_emit")
    if y is None:
        y = torch.empty_like(xs[0])
    if wire_out is None:
        wire_out = [new_wire(bits, n, dev) for _ in xs]
    if red_out is None:
        red_out = new_wire(bits, n, dev)
    _cuda_contig(y, "y")
    if y.dtype != xs[0].dtype or y.numel() != n:
        raise ValueError("y must match the inputs' dtype and size")
    if len(wire_out) != len(xs):
        raise ValueError("wire_out needs one wire per rank")
    for i, w in enumerate(wire_out):
        _wire_tensor(w, bits, n, f"wire_out[{i}]")
    _wire_tensor(red_out, bits, n, "red_out")
    _same_device(xs + [y, red_out] + list(wire_out), "qr_allreduce_emit")
    _check(capi.qr_allreduce_emit(bits, dt, len(xs), [x.data_ptr() for x in xs], n, y.data_ptr(),
                                  [w.data_ptr() for w in wire_out], red_out.data_ptr(),
                                  _stream(dev, stream)), "qr_allreduce_emit")
    return y, wire_out, red_out


def qr_wait_timeouts() -> int:
    """Device-side waits that ran out on the current device since the last
    call (0 in a correct run); reads and resets the count in one atomic step
    after waiting for all work enqueued on the device."""
    st, count = capi.qr_wait_timeouts()
    _check(st, "qr_wait_timeouts")
    return count


def qr_twoshot_workspace_bytes(bits: int, R: int, n: int) -> int:
    return int(lib().qr_twoshot_workspace_bytes(bits, R, n))


def qr_allreduce_twoshot(bits: int, xs, ys=None, workspace: torch.Tensor | None = None, stream=None,
                         flags: bool = False):
    """The two-shot all-reduce with its exchange laid out per rank and per
    owner in `workspace`: returns (the R outputs, the workspace).  With
    `flags`, the one-launch version whose phases are joined by ready flags,
    one pair per two-tile chunk (qr_allreduce_twoshot_flags; its workspace
    also holds the 2T + 1 flag words)."""
    xs, dt, n = _check_inputs(xs)
    R = len(xs)
    dev = _same_device(xs, "qr_allreduce_twoshot")
    if ys is None:
        ys = [torch.empty_like(xs[0]) for _ in range(R)]
    ys = list(ys)
    if len(ys) != R:
        raise ValueError("one output per rank is needed")
    for i, y in enumerate(ys):
        _cuda_contig(y, f"ys[{i}]")
        if y.dtype != xs[0].dtype or y.numel() != n:
            raise ValueError(f"ys[{i}] must match the inputs' dtype and size")
    need = (lib().qr_twoshot_flags_workspace_bytes if flags else lib().qr_twoshot_workspace_bytes)(bits, R, n)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    _cuda_contig(workspace, "workspace")
    if workspace.dtype != torch.uint8:
        raise TypeError(f"workspace must be torch.uint8, got {workspace.dtype}")
    _same_device(xs + ys + [workspace], "qr_allreduce_twoshot")
    call = capi.qr_allreduce_twoshot_flags if flags else capi.qr_allreduce_twoshot
    _check(call(bits, dt, R, [x.data_ptr() for x in xs], n, [y.data_ptr() for y in ys], workspace.data_ptr(),
                workspace.numel(), _stream(dev, stream)), "qr_allreduce_twoshot")
    return ys, workspace


# ---------------------------------------------------------------------------
# the Flash Communication codec (asymmetric groups of 128)
# ---------------------------------------------------------------------------
def qr_fc_tile_bytes(bits: int) -> int:
    return int(lib().qr_fc_tile_bytes(bits))


def qr_fc_wire_bytes(bits: int, n: int) -> int:
    return int(lib().qr_fc_wire_bytes(bits, n))


def _fc_wire_tensor(t: torch.Tensor, bits: int, n: int, what: str) -> None:
    _cuda_contig(t, what)
    if t.dtype != torch.uint8:
        raise TypeError(f"{what} must be torch.uint8 (a packed wire), got {t.dtype}")
    need = qr_fc_wire_bytes(bits, n)
    if t.numel() < need:
        raise ValueError(f"{what} holds {t.numel()} bytes; {need} are needed for {n} values at INT{bits}")


def qr_fc_encode(bits: int, x: torch.Tensor, wire: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Send path of the asymmetric group-128 codec."""
    _cuda_contig(x, "x")
    dt = _dtype_code(x, "x")
    n = x.numel()
    if wire is None:
        wire = torch.empty(qr_fc_wire_bytes(bits, n), dtype=torch.uint8, device=x.device)
    _fc_wire_tensor(wire, bits, n, "wire")
    _same_device([x, wire], "qr_fc_encode")
    _check(capi.qr_fc_encode(bits, dt, x.data_ptr(), n, wire.data_ptr(), _stream(x.device, stream)), "qr_fc_encode")
    return wire


def qr_fc_decode(bits: int, wire: torch.Tensor, n: int, dtype: torch.dtype = torch.bfloat16,
                 y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    _fc_wire_tensor(wire, bits, n, "wire")
    if y is None:
        if dtype not in _DTYPES:
            raise TypeError(f"dtype must be torch.float16 or torch.bfloat16, got {dtype}")
        y = torch.empty(n, dtype=dtype, device=wire.device)
    _cuda_contig(y, "y")
    dt = _dtype_code(y, "y")
    if y.numel() != n:
        raise ValueError(f"y holds {y.numel()} values, expected {n}")
    _same_device([wire, y], "qr_fc_decode")
    _check(capi.qr_fc_decode(bits, dt, wire.data_ptr(), n, y.data_ptr(), _stream(y.device, stream)), "qr_fc_decode")
    return y


def qr_fc_segment_reduce(bits_in: int, bits_out: int, wires, n: int, out: torch.Tensor | None = None,
                         stream=None, staged: bool = False, ctas: int = 0) -> torch.Tensor:
    wires = list(wires)
    if not 1 <= len(wires) <= QR_MAX_RANKS:
        raise ValueError(f"1 to {QR_MAX_RANKS} wires are supported, got {len(wires)}")
    for i, w in enumerate(wires):
        _fc_wire_tensor(w, bits_in, n, f"wires[{i}]")
    if out is None:
        out = torch.empty(qr_fc_wire_bytes(bits_out, n), dtype=torch.uint8, device=wires[0].device)
    _fc_wire_tensor(out, bits_out, n, "out")
    dev = _same_device(wires + [out], "qr_fc_segment_reduce")
    ptrs = [w.data_ptr() for w in wires]
    if staged:
        status = capi.qr_fc_segment_reduce_staged(bits_in, bits_out, len(wires), ptrs, n, out.data_ptr(), ctas,
                                                  _stream(dev, stream))
    else:
        status = capi.qr_fc_segment_reduce(bits_in, bits_out, len(wires), ptrs, n, out.data_ptr(),
                                           _stream(dev, stream))
    _check(status, "qr_fc_segment_reduce")
    return out


def qr_fc_allreduce(bits_rs: int, bits_ag: int, xs, y: torch.Tensor | None = None, stream=None,
                    ctas: int = 0) -> torch.Tensor:
    """The fused two-shot all-reduce with the asymmetric group-128 codec:
    reduce-scatter at bits_rs, all-gather at bits_ag ((4, 8) is "INT6")."""
    xs, dt, n = _check_inputs(xs)
    if y is None:
        y = torch.empty_like(xs[0])
    _cuda_contig(y, "y")
    if y.dtype != xs[0].dtype or y.numel() != n:
        raise ValueError("y must match the inputs' dtype and size")
    dev = _same_device(xs + [y], "qr_fc_allreduce")
    ptrs = [x.data_ptr() for x in xs]
    if ctas:
        status = capi.qr_fc_allreduce_ctas(bits_rs, bits_ag, dt, len(xs), ptrs, n, y.data_ptr(), ctas,
                                           _stream(dev, stream))
    else:
        status = capi.qr_fc_allreduce(bits_rs, bits_ag, dt, len(xs), ptrs, n, y.data_ptr(), _stream(dev, stream))
    _check(status, "qr_fc_allreduce")
    return y


def qr_fc_allreduce_staged(bits_rs: int, bits_ag: int, xs, y: torch.Tensor | None = None, stream=None,
                           ctas: int = 0) -> torch.Tensor:
    """qr_fc_allreduce on the staged kernel (bulk copies into shared memory,
    one persistent CTA per SM) at any size; every tensor 32-byte aligned."""
    xs, dt, n = _check_inputs(xs)
    if y is None:
        y = torch.empty_like(xs[0])
    _cuda_contig(y, "y")
    if y.dtype != xs[0].dtype or y.numel() != n:
        raise ValueError("y must match the inputs' dtype and size")
    dev = _same_device(xs + [y], "qr_fc_allreduce_staged")
    _check(capi.qr_fc_allreduce_staged(bits_rs, bits_ag, dt, len(xs), [x.data_ptr() for x in xs], n, y.data_ptr(),
                                       ctas, _stream(dev, stream)), "qr_fc_allreduce_staged")
    return y


def qr_fc_twoshot_workspace_bytes(bits_rs: int, bits_ag: int, R: int, n: int) -> int:
    return int(lib().qr_fc_twoshot_workspace_bytes(bits_rs, bits_ag, R, n))


def qr_fc_allreduce_twoshot(bits_rs: int, bits_ag: int, xs, ys=None, workspace: torch.Tensor | None = None,
                            stream=None):
    """The asymmetric codec's two-shot all-reduce with its exchange laid out
    per rank and per owner in `workspace` (quantize at bits_rs, all-to-all,
    owners' reduction re-quantized at bits_ag, all-gather, decode): returns
    (the R outputs, the workspace)."""
    xs, dt, n = _check_inputs(xs)
    R = len(xs)
    dev = _same_device(xs, "qr_fc_allreduce_twoshot")
    if ys is None:
        ys = [torch.empty_like(xs[0]) for _ in range(R)]
    ys = list(ys)
    if len(ys) != R:
        raise ValueError("one output per rank is needed")
    for i, y in enumerate(ys):
        _cuda_contig(y, f"ys[{i}]")
        if y.dtype != xs[0].dtype or y.numel() != n:
            raise ValueError(f"ys[{i}] must match the inputs' dtype and size")
    need = qr_fc_twoshot_workspace_bytes(bits_rs, bits_ag, R, n)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    _cuda_contig(workspace, "workspace")
    if workspace.dtype != torch.uint8:
        raise TypeError(f"workspace must be torch.uint8, got {workspace.dtype}")
    _same_device(xs + ys + [workspace], "qr_fc_allreduce_twoshot")
    _check(capi.qr_fc_allreduce_twoshot(bits_rs, bits_ag, dt, R, [x.data_ptr() for x in xs], n,
                                        [y.data_ptr() for y in ys], workspace.data_ptr(), workspace.numel(),
                                        _stream(dev, stream)), "qr_fc_allreduce_twoshot")
    return ys, workspace


# ---------------------------------------------------------------------------
# the FP4 codec (the INT4 block framework with E2M1 elements)
# ---------------------------------------------------------------------------
def qr_fp4_twoshot_workspace_bytes(R: int, n: int) -> int:
    return int(lib().qr_fp4_twoshot_workspace_bytes(R, n))


def qr_fp4_allreduce_twoshot(xs, ys=None, workspace: torch.Tensor | None = None, stream=None):
    """The FP4 codec's two-shot all-reduce with its exchange laid out per rank
    and per owner in `workspace`: returns (the R outputs, the workspace)."""
    xs, dt, n = _check_inputs(xs)
    R = len(xs)
    dev = _same_device(xs, "qr_fp4_allreduce_twoshot")
    if ys is None:
        ys = [torch.empty_like(xs[0]) for _ in range(R)]
    ys = list(ys)
    if len(ys) != R:
        raise ValueError("one output per rank is needed")
    for i, y in enumerate(ys):
        _cuda_contig(y, f"ys[{i}]")
        if y.dtype != xs[0].dtype or y.numel() != n:
            raise ValueError(f"ys[{i}] must match the inputs' dtype and size")
    need = qr_fp4_twoshot_workspace_bytes(R, n)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    _cuda_contig(workspace, "workspace")
    if workspace.dtype != torch.uint8:
        raise TypeError(f"workspace must be torch.uint8, got {workspace.dtype}")
    _same_device(xs + ys + [workspace], "qr_fp4_allreduce_twoshot")
    _check(capi.qr_fp4_allreduce_twoshot(dt, R, [x.data_ptr() for x in xs], n, [y.data_ptr() for y in ys],
                                         workspace.data_ptr(), workspace.numel(), _stream(dev, stream)),
           "qr_fp4_allreduce_twoshot")
    return ys, workspace


def qr_fp4_tile_bytes() -> int:
    return int(lib().qr_fp4_tile_bytes())


def qr_fp4_wire_bytes(n: int) -> int:
    return int(lib().qr_fp4_wire_bytes(n))


def _fp4_wire_tensor(t: torch.Tensor, n: int, what: str) -> None:
    _cuda_contig(t, what)
    if t.dtype != torch.uint8:
        raise TypeError(f"{what} must be torch.uint8 (a packed wire), got {t.dtype}")
    need = qr_fp4_wire_bytes(n)
    if t.numel() < need:
        raise ValueError(f"{what} holds {t.numel()} bytes; {need} are needed for {n} values at FP4")


def qr_fp4_encode(x: torch.Tensor, wire: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Send path of the FP4 codec."""
    _cuda_contig(x, "x")
    dt = _dtype_code(x, "x")
    n = x.numel()
    if wire is None:
        wire = torch.empty(qr_fp4_wire_bytes(n), dtype=torch.uint8, device=x.device)
    _fp4_wire_tensor(wire, n, "wire")
    _same_device([x, wire], "qr_fp4_encode")
    _check(capi.qr_fp4_encode(dt, x.data_ptr(), n, wire.data_ptr(), _stream(x.device, stream)), "qr_fp4_encode")
    return wire


def qr_fp4_decode(wire: torch.Tensor, n: int, dtype: torch.dtype = torch.bfloat16,
                  y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Receive path of the FP4 codec: the first n values of a wire."""
    _fp4_wire_tensor(wire, n, "wire")
    if y is None:
        if dtype not in _DTYPES:
            raise TypeError(f"dtype must be torch.float16 or torch.bfloat16, got {dtype}")
        y = torch.empty(n, dtype=dtype, device=wire.device)
    _cuda_contig(y, "y")
    dt = _dtype_code(y, "y")
    if y.numel() != n:
        raise ValueError(f"y holds {y.numel()} values, expected {n}")
    _same_device([wire, y], "qr_fp4_decode")
    _check(capi.qr_fp4_decode(dt, wire.data_ptr(), n, y.data_ptr(), _stream(y.device, stream)), "qr_fp4_decode")
    return y


def qr_fp4_segment_reduce(wires, n: int, out: torch.Tensor | None = None, stream=None,
                          ctas: int = 0) -> torch.Tensor:
    """Phase-1B of the FP4 codec (the staged kernel with `ctas` persistent CTAs;
    with ctas = 0 the library may take a register-fed kernel on long messages)."""
    wires = list(wires)
    if not 1 <= len(wires) <= QR_MAX_RANKS:
        raise ValueError(f"1 to {QR_MAX_RANKS} wires are supported, got {len(wires)}")
    for i, w in enumerate(wires):
        _fp4_wire_tensor(w, n, f"wires[{i}]")
    if out is None:
        out = torch.empty(qr_fp4_wire_bytes(n), dtype=torch.uint8, device=wires[0].device)
    _fp4_wire_tensor(out, n, "out")
    dev = _same_device(wires + [out], "qr_fp4_segment_reduce")
    _check(capi.qr_fp4_segment_reduce(len(wires), [w.data_ptr() for w in wires], n, out.data_ptr(), ctas,
                                      _stream(dev, stream)), "qr_fp4_segment_reduce")
    return out


def qr_fp4_allreduce(xs, y: torch.Tensor | None = None, stream=None, ctas: int = 0) -> torch.Tensor:
    """The fused FP4 all-reduce (the staged kernel; every tensor 32-byte aligned)."""
    xs, dt, n = _check_inputs(xs)
    if y is None:
        y = torch.empty_like(xs[0])
    _cuda_contig(y, "y")
    if y.dtype != xs[0].dtype or y.numel() != n:
        raise ValueError("y must match the inputs' dtype and size")
    dev = _same_device(xs + [y], "qr_fp4_allreduce")
    _check(capi.qr_fp4_allreduce(dt, len(xs), [x.data_ptr() for x in xs], n, y.data_ptr(), ctas,
                                 _stream(dev, stream)), "qr_fp4_allreduce")
    return y
