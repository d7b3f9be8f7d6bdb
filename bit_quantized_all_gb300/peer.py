"""The two-shot all-reduce run by R separate processes, one per rank: the
per-rank calls of ``libqr.so`` (``qr_twoshot_peer_send / _reduce / _decode``,
and their ``qr_fc_`` / ``qr_fp4_`` counterparts for the other two codecs)
with the peers' workspaces mapped through CUDA IPC and the three phases
joined by host barriers.

The codec is named by ``bits``: 3, 4, 6 or 8 for the symmetric block codec,
``("fc", bits_rs, bits_ag)`` for the asymmetric group-128 codec (width pairs
(4, 4), (4, 8), (8, 8)), ``"fp4"`` for the FP4 codec.

Each rank allocates one workspace in its own device memory, shares a handle
to it with the other ranks (``torch.distributed.all_gather_object``) and maps
theirs.  A step is, on every rank::

    send   -- quantize this rank's message, store segment k into rank k's workspace
    join   -- every rank's send has finished on its GPU
    reduce -- this rank, as owner, sums its segment's R copies and stores the
              re-quantized tiles into every rank's gathered wire
    join   -- every rank's reduce has finished
    decode -- decode this rank's gathered wire into its output

A join is the rank's stream synchronized, then a barrier of the process group
(gloo: it runs on the host).  No kernel waits on another rank, so a rank that
stops is noticed on the host: the next join of the others fails with
``PeerError`` (the group's timeout bounds the wait) before they launch
anything that would read what the missing rank should have written.

The compute runs in the library's kernels; this module only moves handles,
pointers and barriers.  ``ops`` is the seam between the two: ``CudaPeerOps``
(the default) calls the library; a test can pass an object with the same
methods to exercise the host protocol without a GPU.
"""
from __future__ import annotations

import ctypes
import datetime
import numbers

import torch

from . import _check, _stream, lib

QR_IPC_HANDLE_BYTES = 72


class PeerError(RuntimeError):
    """A peer did not reach a join (it stopped, or the group timed out)."""


def _lib():
    L = lib()
    if not getattr(L, "_peer_sigs", False):
        vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        vpp = ctypes.POINTER(ctypes.c_void_p)
        sigs = {
            "qr_twoshot_peer_workspace_bytes": (sz, [i32, i32, sz]),
            "qr_twoshot_peer_send": (i32, [i32, i32, i32, i32, vp, sz, vpp, vp]),
            "qr_twoshot_peer_reduce": (i32, [i32, i32, i32, sz, vpp, vp]),
            "qr_twoshot_peer_decode": (i32, [i32, i32, i32, sz, vp, vp, vp]),
            "qr_fc_twoshot_peer_workspace_bytes": (sz, [i32, i32, i32, sz]),
            "qr_fc_twoshot_peer_send": (i32, [i32, i32, i32, i32, i32, vp, sz, vpp, vp]),
            "qr_fc_twoshot_peer_reduce": (i32, [i32, i32, i32, i32, sz, vpp, vp]),
            "qr_fc_twoshot_peer_decode": (i32, [i32, i32, i32, i32, sz, vp, vp, vp]),
            "qr_fp4_twoshot_peer_workspace_bytes": (sz, [i32, sz]),
            "qr_fp4_twoshot_peer_send": (i32, [i32, i32, i32, vp, sz, vpp, vp]),
            "qr_fp4_twoshot_peer_reduce": (i32, [i32, i32, sz, vpp, vp]),
            "qr_fp4_twoshot_peer_decode": (i32, [i32, i32, sz, vp, vp, vp]),
            "qr_ipc_handle_bytes": (sz, []),
            "qr_ipc_get_handle": (i32, [vp, vp]),
            "qr_ipc_open_handle": (i32, [vp, ctypes.POINTER(ctypes.c_void_p)]),
            "qr_ipc_close_handle": (i32, [vp]),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        L._peer_sigs = True
    return L


def _ptrs(ptrs):
    return (ctypes.c_void_p * len(ptrs))(*ptrs)


def codec_of(bits):
    """("qr", bits), ("fc", bits_rs, bits_ag) or ("fp4",) for a codec named
    as this module's ``bits`` arguments name it."""
    if isinstance(bits, str) and bits == "fp4":
        return ("fp4",)
    if isinstance(bits, tuple) and len(bits) == 3 and bits[0] == "fc":
        return ("fc", int(bits[1]), int(bits[2]))
    if isinstance(bits, numbers.Integral) and not isinstance(bits, bool):
        return ("qr", int(bits))
    raise ValueError(f"unknown two-shot codec {bits!r}: 3/4/6/8, ('fc', bits_rs, bits_ag) or 'fp4'")


class CudaPeerOps:
    """The library's per-rank calls and CUDA IPC, on one device."""

    def __init__(self, device=None):
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)

    def workspace_bytes(self, bits, R: int, n: int) -> int:
        c, L = codec_of(bits), _lib()
        if c[0] == "fc":
            return int(L.qr_fc_twoshot_peer_workspace_bytes(c[1], c[2], R, n))
        if c[0] == "fp4":
            return int(L.qr_fp4_twoshot_peer_workspace_bytes(R, n))
        return int(L.qr_twoshot_peer_workspace_bytes(c[1], R, n))

    def alloc(self, nbytes: int):
        buf = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        return buf, buf.data_ptr()

    def get_handle(self, ptr: int) -> bytes:
        h = ctypes.create_string_buffer(QR_IPC_HANDLE_BYTES)
        _check(_lib().qr_ipc_get_handle(ptr, h), "qr_ipc_get_handle")
        return h.raw

    def open_handle(self, handle: bytes) -> int:
        out = ctypes.c_void_p()
        buf = ctypes.create_string_buffer(handle, QR_IPC_HANDLE_BYTES)
        _check(_lib().qr_ipc_open_handle(buf, ctypes.byref(out)), "qr_ipc_open_handle")
        return int(out.value)

    def close_handle(self, ptr: int) -> None:
        _check(_lib().qr_ipc_close_handle(ptr), "qr_ipc_close_handle")

    def send(self, bits, dtype, R, rank, x_ptr, n, peers, stream):
        c, L, P = codec_of(bits), _lib(), _ptrs(peers)
        if c[0] == "fc":
            _check(L.qr_fc_twoshot_peer_send(c[1], c[2], dtype, R, rank, x_ptr, n, P, stream),
                   "qr_fc_twoshot_peer_send")
        elif c[0] == "fp4":
            _check(L.qr_fp4_twoshot_peer_send(dtype, R, rank, x_ptr, n, P, stream), "qr_fp4_twoshot_peer_send")
        else:
            _check(L.qr_twoshot_peer_send(c[1], dtype, R, rank, x_ptr, n, P, stream), "qr_twoshot_peer_send")

    def reduce(self, bits, R, rank, n, peers, stream):
        c, L, P = codec_of(bits), _lib(), _ptrs(peers)
        if c[0] == "fc":
            _check(L.qr_fc_twoshot_peer_reduce(c[1], c[2], R, rank, n, P, stream), "qr_fc_twoshot_peer_reduce")
        elif c[0] == "fp4":
            _check(L.qr_fp4_twoshot_peer_reduce(R, rank, n, P, stream), "qr_fp4_twoshot_peer_reduce")
        else:
            _check(L.qr_twoshot_peer_reduce(c[1], R, rank, n, P, stream), "qr_twoshot_peer_reduce")

    def decode(self, bits, dtype, R, n, ws_ptr, y_ptr, stream):
        c, L = codec_of(bits), _lib()
        if c[0] == "fc":
            _check(L.qr_fc_twoshot_peer_decode(c[1], c[2], dtype, R, n, ws_ptr, y_ptr, stream),
                   "qr_fc_twoshot_peer_decode")
        elif c[0] == "fp4":
            _check(L.qr_fp4_twoshot_peer_decode(dtype, R, n, ws_ptr, y_ptr, stream), "qr_fp4_twoshot_peer_decode")
        else:
            _check(L.qr_twoshot_peer_decode(c[1], dtype, R, n, ws_ptr, y_ptr, stream), "qr_twoshot_peer_decode")

    def stream(self, stream=None):
        return _stream(self.device, stream)

    def synchronize(self, stream) -> None:
        torch.cuda.synchronize(self.device)


class PeerTwoShot:
    """One rank of the per-rank two-shot all-reduce over a process group.

    ``bits``: the codec (3, 4, 6 or 8; ``("fc", bits_rs, bits_ag)``;
    ``"fp4"``); ``n``: values per rank; ``dtype``: 0 (fp16) or 1 (bf16).  Construct it on every rank of ``group`` (collective: handles are
    exchanged); ``allreduce(x_ptr, y_ptr)`` is collective too.  ``x_ptr`` /
    ``y_ptr`` are device pointers of n 16-bit values in this rank's memory
    (the tensor helpers take tensors)."""

    def __init__(self, bits, n: int, dtype: int, group=None, ops=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.R = dist.get_world_size(group)
        self.bits, self.n, self.dtype = bits, n, dtype
        self.ops = CudaPeerOps() if ops is None else ops
        need = self.ops.workspace_bytes(bits, self.R, n)
        # every rank must agree on the shape: a peer's kernels store into this
        # rank's workspace at offsets computed from their own (bits, n)
        shapes = [None] * self.R
        dist.all_gather_object(shapes, (bits, n, dtype, need), group=group)
        if any(sh != shapes[0] for sh in shapes):
            raise ValueError(f"rank {self.rank}: the ranks disagree on (bits, n, dtype, workspace bytes): {shapes}")
        if need == 0:
            raise ValueError(f"unsupported two-shot shape: bits={bits} R={self.R} n={n}")
        self.workspace, self.ws_ptr = self.ops.alloc(need)
        handles = [None] * self.R
        dist.all_gather_object(handles, self.ops.get_handle(self.ws_ptr), group=group)
        self.peers = []
        self._opened = []
        for j, h in enumerate(handles):
            if j == self.rank:
                self.peers.append(self.ws_ptr)
            else:
                p = self.ops.open_handle(h)
                self._opened.append(p)
                self.peers.append(p)
        self.steps = 0
        self._join("setup")

    def _join(self, where: str, stream=None) -> None:
        self.ops.synchronize(stream)
        try:
            self.dist.barrier(group=self.group)
        except Exception as e:  # noqa: BLE001  (gloo raises RuntimeError or DistBackendError)
            raise PeerError(f"rank {self.rank}: a peer did not reach the join after {where} "
                            f"(step {self.steps}): {e}") from e

    def allreduce(self, x_ptr: int, y_ptr: int, stream=None) -> None:
        s = self.ops.stream(stream)
        self.ops.send(self.bits, self.dtype, self.R, self.rank, x_ptr, self.n, self.peers, s)
        self._join("send", stream)
        self.ops.reduce(self.bits, self.R, self.rank, self.n, self.peers, s)
        self._join("reduce", stream)
        self.ops.decode(self.bits, self.dtype, self.R, self.n, self.ws_ptr, y_ptr, s)
        self.steps += 1

    def allreduce_tensor(self, x: torch.Tensor, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        if x.dtype not in (torch.float16, torch.bfloat16) or not x.is_contiguous() or x.numel() != self.n:
            raise ValueError("x must be a contiguous fp16/bf16 tensor of n values")
        if (x.dtype == torch.bfloat16) != (self.dtype == 1):
            raise TypeError("x's dtype does not match the dtype this rank was set up with")
        y = torch.empty_like(x) if y is None else y
        if y.dtype != x.dtype or y.numel() != self.n or not y.is_contiguous():
            raise ValueError("y must match x")
        self.allreduce(x.data_ptr(), y.data_ptr(), stream)
        return y

    def close(self) -> None:
        """Collective: every rank stops using the peers' workspaces, then unmaps them."""
        self._join("close")
        for p in self._opened:
            self.ops.close_handle(p)
        self._opened = []


def twoshot_peer_local(bits, xs, ys=None, workspaces=None, stream=None):
    """All R ranks' per-rank calls from one process, on one device and one
    stream: R workspaces in this process, every rank's send, then every
    owner's reduce, then every rank's decode (the stream order is the join).
    Returns (the R outputs, the R workspaces).  Each output equals the
    codec's fused all-reduce (qr_allreduce, qr_fc_allreduce or
    qr_fp4_allreduce).  `bits` names the codec as for PeerTwoShot;
    `workspaces` (R uint8 tensors of the codec's peer workspace bytes each)
    and `ys` may be passed in to reuse them."""
    from . import _check_inputs, _same_device
    xs, dt, n = _check_inputs(xs)
    R = len(xs)
    dev = _same_device(xs, "twoshot_peer_local")
    ops = CudaPeerOps(dev)
    need = ops.workspace_bytes(bits, R, n)
    if need == 0:
        raise ValueError(f"unsupported two-shot shape: bits={bits} R={R} n={n}")
    if workspaces is None:
        ws = [torch.empty(need, dtype=torch.uint8, device=dev) for _ in range(R)]
    else:
        ws = list(workspaces)
        if len(ws) != R or any(w.dtype != torch.uint8 or w.numel() < need or not w.is_contiguous()
                               or w.device != dev for w in ws):
            raise ValueError(f"workspaces must be {R} contiguous uint8 tensors of at least {need} bytes on {dev}")
    ys = [torch.empty_like(xs[0]) for _ in range(R)] if ys is None else list(ys)
    for y in ys:
        if y.dtype != xs[0].dtype or y.numel() != n or not y.is_contiguous() or y.device != dev:
            raise ValueError("every output must match the inputs")
    peers = [w.data_ptr() for w in ws]
    s = ops.stream(stream)
    for j in range(R):
        ops.send(bits, dt, R, j, xs[j].data_ptr(), n, peers, s)
    for j in range(R):
        ops.reduce(bits, R, j, n, peers, s)
    for j in range(R):
        ops.decode(bits, dt, R, n, peers[j], ys[j].data_ptr(), s)
    return ys, ws


def init_group(rank: int, world: int, port: int, timeout_s: float = 60.0):
    """A gloo process group on 127.0.0.1 for the host joins."""
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=timeout_s))
    return dist.group.WORLD


__all__ = ["PeerTwoShot", "PeerError", "CudaPeerOps", "codec_of", "twoshot_peer_local", "init_group",
           "QR_IPC_HANDLE_BYTES"]
