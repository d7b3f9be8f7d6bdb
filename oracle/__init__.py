"""CPU oracle for the block-quantized two-shot all-reduce codec.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the benchmark's CPU-baseline / reference arm may import this package.  The
product library (``bit_quantized_all_gb300``) never imports, loads or calls it,
and it shares no code with the CUDA path: the arithmetic lives in the plain C
file ``qr_oracle.c`` next to this one, compiled with gcc (``-O2
-ffp-contract=off``, no fast-math).  This module is argument marshalling only.

What the oracle computes, and the passages it follows, is described in
``qr_oracle.h``.  Every array here is numpy; fp16 / bf16 values travel as their
raw ``uint16`` bit patterns.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qr_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

FP16 = 0
BF16 = 1
BITS = (3, 4, 6, 8)

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``qr_oracle.c`` into ``liboracle.so`` beside it (gcc)."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC),
                                                  os.path.getmtime(os.path.join(_HERE, "qr_oracle.h"))))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
               "-Wall", "-Wextra", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path: str) -> ctypes.CDLL:
    L = ctypes.CDLL(path)
    u8p = ctypes.POINTER(ctypes.c_uint8)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f32p = ctypes.POINTER(ctypes.c_float)
    sz = ctypes.c_size_t
    i32 = ctypes.c_int
    sig = {
        "orc_f32_to_f16": (ctypes.c_uint16, [ctypes.c_float]),
        "orc_f16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
        "orc_f32_to_bf16": (ctypes.c_uint16, [ctypes.c_float]),
        "orc_bf16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
        "orc_f32_to_f16_n": (None, [f32p, sz, u16p]),
        "orc_f16_to_f32_n": (None, [u16p, sz, f32p]),
        "orc_f32_to_bf16_n": (None, [f32p, sz, u16p]),
        "orc_bf16_to_f32_n": (None, [u16p, sz, f32p]),
        "orc_tile_values": (sz, []),
        "orc_tile_bytes": (sz, [i32]),
        "orc_wire_bytes": (sz, [i32, sz]),
        "orc_pack_codes": (i32, [i32, u8p, sz, u8p]),
        "orc_unpack_codes": (i32, [i32, u8p, sz, u8p]),
        "orc_quantize_block": (i32, [i32, f32p, u8p, u16p]),
        "orc_encode_f32": (i32, [i32, f32p, sz, u8p]),
        "orc_encode": (i32, [i32, i32, u16p, sz, u8p]),
        "orc_decode_f32": (i32, [i32, u8p, sz, f32p]),
        "orc_decode": (i32, [i32, i32, u8p, sz, u16p]),
        "orc_segment_reduce": (i32, [i32, i32, ctypes.POINTER(u8p), sz, u8p]),
        "orc_allreduce": (i32, [i32, i32, i32, ctypes.POINTER(u16p), sz, u16p]),
        "orc_fc_tile_bytes": (sz, [i32]),
        "orc_fc_wire_bytes": (sz, [i32, sz]),
        "orc_fc_quantize_group": (i32, [i32, f32p, u8p, f32p, f32p]),
        "orc_fc_encode_f32": (i32, [i32, f32p, sz, u8p]),
        "orc_fc_encode": (i32, [i32, i32, u16p, sz, u8p]),
        "orc_fc_decode_f32": (i32, [i32, u8p, sz, f32p]),
        "orc_fc_decode": (i32, [i32, i32, u8p, sz, u16p]),
        "orc_fc_segment_reduce": (i32, [i32, i32, i32, ctypes.POINTER(u8p), sz, u8p]),
        "orc_fc_allreduce": (i32, [i32, i32, i32, i32, ctypes.POINTER(u16p), sz, u16p]),
        "orc_fp4_value": (ctypes.c_float, [ctypes.c_uint8]),
        "orc_fp4_round": (ctypes.c_uint8, [ctypes.c_float]),
        "orc_fp4_round_n": (None, [f32p, sz, u8p]),
        "orc_fp4_tile_bytes": (sz, []),
        "orc_fp4_wire_bytes": (sz, [sz]),
        "orc_fp4_quantize_block": (i32, [f32p, u8p, u16p]),
        "orc_fp4_encode_f32": (i32, [f32p, sz, u8p]),
        "orc_fp4_encode": (i32, [i32, u16p, sz, u8p]),
        "orc_fp4_decode_f32": (i32, [u8p, sz, f32p]),
        "orc_fp4_decode": (i32, [i32, u8p, sz, u16p]),
        "orc_fp4_segment_reduce": (i32, [i32, ctypes.POINTER(u8p), sz, u8p]),
        "orc_fp4_allreduce": (i32, [i32, i32, ctypes.POINTER(u16p), sz, u16p]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(_LIB_PATH)
    return _lib


@contextlib.contextmanager
def using_library(path: str):
    """Temporarily route every function of this module through another build
    of the oracle (the mutation tests use this to run the pins against copies
    with planted mistakes)."""
    global _lib
    lib()
    with _lock:
        saved, _lib = _lib, _bind(path)
    try:
        yield
    finally:
        with _lock:
            _lib = saved


def _p(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")


# ---- formats -------------------------------------------------------------

def f32_to_f16(f) -> np.ndarray:
    f = np.ascontiguousarray(f, dtype=np.float32)
    h = np.empty(f.shape, np.uint16)
    lib().orc_f32_to_f16_n(_p(f, ctypes.c_float), f.size, _p(h, ctypes.c_uint16))
    return h


def f16_to_f32(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    f = np.empty(h.shape, np.float32)
    lib().orc_f16_to_f32_n(_p(h, ctypes.c_uint16), h.size, _p(f, ctypes.c_float))
    return f


def f32_to_bf16(f) -> np.ndarray:
    f = np.ascontiguousarray(f, dtype=np.float32)
    h = np.empty(f.shape, np.uint16)
    lib().orc_f32_to_bf16_n(_p(f, ctypes.c_float), f.size, _p(h, ctypes.c_uint16))
    return h


def bf16_to_f32(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    f = np.empty(h.shape, np.float32)
    lib().orc_bf16_to_f32_n(_p(h, ctypes.c_uint16), h.size, _p(f, ctypes.c_float))
    return f


def widen(dtype: int, h) -> np.ndarray:
    return f16_to_f32(h) if dtype == FP16 else bf16_to_f32(h)


def narrow(dtype: int, f) -> np.ndarray:
    return f32_to_f16(f) if dtype == FP16 else f32_to_bf16(f)


# ---- sizes ---------------------------------------------------------------

def tile_values() -> int:
    return int(lib().orc_tile_values())


def tile_bytes(bits: int) -> int:
    return int(lib().orc_tile_bytes(bits))


def wire_bytes(bits: int, n: int) -> int:
    return int(lib().orc_wire_bytes(bits, n))


def scale_offset(bits: int) -> int:
    """Byte offset of the 64 fp16 scales inside a tile (after the codes)."""
    return tile_bytes(bits) - 128


# ---- packing and the block quantizer -------------------------------------

def pack_codes(bits: int, u) -> np.ndarray:
    """u: uint8 codes, a whole number of 2048-value tiles -> wire (scales 0)."""
    u = np.ascontiguousarray(u, dtype=np.uint8).reshape(-1)
    assert u.size % 2048 == 0
    nt = u.size // 2048
    w = np.zeros(nt * tile_bytes(bits), np.uint8)
    _check(lib().orc_pack_codes(bits, _p(u, ctypes.c_uint8), nt, _p(w, ctypes.c_uint8)), "pack")
    return w


def unpack_codes(bits: int, wire) -> np.ndarray:
    wire = np.ascontiguousarray(wire, dtype=np.uint8).reshape(-1)
    tb = tile_bytes(bits)
    assert wire.size % tb == 0
    nt = wire.size // tb
    u = np.empty(nt * 2048, np.uint8)
    _check(lib().orc_unpack_codes(bits, _p(wire, ctypes.c_uint8), nt, _p(u, ctypes.c_uint8)), "unpack")
    return u


def quantize_block(bits: int, x):
    """x: 32 fp32 values -> (codes uint8[32], fp16 scale bits)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.size == 32
    u = np.empty(32, np.uint8)
    s = np.zeros(1, np.uint16)
    _check(lib().orc_quantize_block(bits, _p(x, ctypes.c_float), _p(u, ctypes.c_uint8),
                                    _p(s, ctypes.c_uint16)), "quantize_block")
    return u, int(s[0])


# ---- the codec -----------------------------------------------------------

def encode_f32(bits: int, x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    w = np.empty(wire_bytes(bits, x.size), np.uint8)
    _check(lib().orc_encode_f32(bits, _p(x, ctypes.c_float), x.size, _p(w, ctypes.c_uint8)), "encode_f32")
    return w


def encode(bits: int, dtype: int, x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.uint16).reshape(-1)
    w = np.empty(wire_bytes(bits, x.size), np.uint8)
    _check(lib().orc_encode(bits, dtype, _p(x, ctypes.c_uint16), x.size, _p(w, ctypes.c_uint8)), "encode")
    return w


def decode_f32(bits: int, wire, n: int) -> np.ndarray:
    wire = np.ascontiguousarray(wire, dtype=np.uint8)
    assert wire.size >= wire_bytes(bits, n)
    out = np.empty(n, np.float32)
    _check(lib().orc_decode_f32(bits, _p(wire, ctypes.c_uint8), n, _p(out, ctypes.c_float)), "decode_f32")
    return out


def decode(bits: int, dtype: int, wire, n: int) -> np.ndarray:
    wire = np.ascontiguousarray(wire, dtype=np.uint8)
    assert wire.size >= wire_bytes(bits, n)
    y = np.empty(n, np.uint16)
    _check(lib().orc_decode(bits, dtype, _p(wire, ctypes.c_uint8), n, _p(y, ctypes.c_uint16)), "decode")
    return y


def segment_reduce(bits: int, wires, n: int) -> np.ndarray:
    ws = [np.ascontiguousarray(w, dtype=np.uint8) for w in wires]
    for w in ws:
        assert w.size >= wire_bytes(bits, n)
    arr = (ctypes.POINTER(ctypes.c_uint8) * len(ws))(*[_p(w, ctypes.c_uint8) for w in ws])
    out = np.empty(wire_bytes(bits, n), np.uint8)
    _check(lib().orc_segment_reduce(bits, len(ws), arr, n, _p(out, ctypes.c_uint8)), "segment_reduce")
    return out


def allreduce(bits: int, dtype: int, xs) -> np.ndarray:
    xs = [np.ascontiguousarray(x, dtype=np.uint16).reshape(-1) for x in xs]
    n = xs[0].size
    assert all(x.size == n for x in xs)
    arr = (ctypes.POINTER(ctypes.c_uint16) * len(xs))(*[_p(x, ctypes.c_uint16) for x in xs])
    y = np.empty(n, np.uint16)
    _check(lib().orc_allreduce(bits, dtype, len(xs), arr, n, _p(y, ctypes.c_uint16)), "allreduce")
    return y


# ---- the Flash Communication codec (asymmetric, groups of 128) -------------

FC_BITS = (4, 8)


def fc_tile_bytes(bits: int) -> int:
    return int(lib().orc_fc_tile_bytes(bits))


def fc_wire_bytes(bits: int, n: int) -> int:
    return int(lib().orc_fc_wire_bytes(bits, n))


def fc_quantize_group(bits: int, x):
    """x: 128 fp32 values -> (codes uint8[128], scale, zero point)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.size == 128
    u = np.empty(128, np.uint8)
    s = np.zeros(1, np.float32)
    z = np.zeros(1, np.float32)
    _check(lib().orc_fc_quantize_group(bits, _p(x, ctypes.c_float), _p(u, ctypes.c_uint8),
                                       _p(s, ctypes.c_float), _p(z, ctypes.c_float)), "fc_quantize_group")
    return u, float(s[0]), float(z[0])


def fc_encode_f32(bits: int, x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    w = np.empty(fc_wire_bytes(bits, x.size), np.uint8)
    _check(lib().orc_fc_encode_f32(bits, _p(x, ctypes.c_float), x.size, _p(w, ctypes.c_uint8)), "fc_encode_f32")
    return w


def fc_encode(bits: int, dtype: int, x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.uint16).reshape(-1)
    w = np.empty(fc_wire_bytes(bits, x.size), np.uint8)
    _check(lib().orc_fc_encode(bits, dtype, _p(x, ctypes.c_uint16), x.size, _p(w, ctypes.c_uint8)), "fc_encode")
    return w


def fc_decode_f32(bits: int, wire, n: int) -> np.ndarray:
    wire = np.ascontiguousarray(wire, dtype=np.uint8)
    assert wire.size >= fc_wire_bytes(bits, n)
    out = np.empty(n, np.float32)
    _check(lib().orc_fc_decode_f32(bits, _p(wire, ctypes.c_uint8), n, _p(out, ctypes.c_float)), "fc_decode_f32")
    return out


def fc_decode(bits: int, dtype: int, wire, n: int) -> np.ndarray:
    wire = np.ascontiguousarray(wire, dtype=np.uint8)
    assert wire.size >= fc_wire_bytes(bits, n)
    y = np.empty(n, np.uint16)
    _check(lib().orc_fc_decode(bits, dtype, _p(wire, ctypes.c_uint8), n, _p(y, ctypes.c_uint16)), "fc_decode")
    return y


def fc_segment_reduce(bits_in: int, bits_out: int, wires, n: int) -> np.ndarray:
    ws = [np.ascontiguousarray(w, dtype=np.uint8) for w in wires]
    for w in ws:
        assert w.size >= fc_wire_bytes(bits_in, n)
    arr = (ctypes.POINTER(ctypes.c_uint8) * len(ws))(*[_p(w, ctypes.c_uint8) for w in ws])
    out = np.empty(fc_wire_bytes(bits_out, n), np.uint8)
    _check(lib().orc_fc_segment_reduce(bits_in, bits_out, len(ws), arr, n, _p(out, ctypes.c_uint8)),
           "fc_segment_reduce")
    return out


def fc_allreduce(bits_rs: int, bits_ag: int, dtype: int, xs) -> np.ndarray:
    xs = [np.ascontiguousarray(x, dtype=np.uint16).reshape(-1) for x in xs]
    n = xs[0].size
    assert all(x.size == n for x in xs)
    arr = (ctypes.POINTER(ctypes.c_uint16) * len(xs))(*[_p(x, ctypes.c_uint16) for x in xs])
    y = np.empty(n, np.uint16)
    _check(lib().orc_fc_allreduce(bits_rs, bits_ag, dtype, len(xs), arr, n, _p(y, ctypes.c_uint16)),
           "fc_allreduce")
    return y


# ---- the FP4 (E2M1) codec: the INT4 block framework with E2M1 elements -----

def fp4_value(code: int) -> float:
    return float(lib().orc_fp4_value(code))


def fp4_round(t: float) -> int:
    return int(lib().orc_fp4_round(float(t)))


def fp4_round_n(t) -> np.ndarray:
    t = np.ascontiguousarray(t, dtype=np.float32).reshape(-1)
    c = np.empty(t.size, np.uint8)
    lib().orc_fp4_round_n(_p(t, ctypes.c_float), t.size, _p(c, ctypes.c_uint8))
    return c


def fp4_tile_bytes() -> int:
    return int(lib().orc_fp4_tile_bytes())


def fp4_wire_bytes(n: int) -> int:
    return int(lib().orc_fp4_wire_bytes(n))


def fp4_quantize_block(x):
    """(codes, fp16 scale bits) of one 32-value block."""
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    assert x.size == 32
    c = np.empty(32, np.uint8)
    sh = np.zeros(1, np.uint16)
    _check(lib().orc_fp4_quantize_block(_p(x, ctypes.c_float), _p(c, ctypes.c_uint8), _p(sh, ctypes.c_uint16)),
           "fp4_quantize_block")
    return c, int(sh[0])


def fp4_encode_f32(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    w = np.empty(fp4_wire_bytes(x.size), np.uint8)
    _check(lib().orc_fp4_encode_f32(_p(x, ctypes.c_float), x.size, _p(w, ctypes.c_uint8)), "fp4_encode_f32")
    return w


def fp4_encode(dtype: int, x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.uint16).reshape(-1)
    w = np.empty(fp4_wire_bytes(x.size), np.uint8)
    _check(lib().orc_fp4_encode(dtype, _p(x, ctypes.c_uint16), x.size, _p(w, ctypes.c_uint8)), "fp4_encode")
    return w


def fp4_decode_f32(wire, n: int) -> np.ndarray:
    wire = np.ascontiguousarray(wire, dtype=np.uint8)
    assert wire.size >= fp4_wire_bytes(n)
    out = np.empty(n, np.float32)
    _check(lib().orc_fp4_decode_f32(_p(wire, ctypes.c_uint8), n, _p(out, ctypes.c_float)), "fp4_decode_f32")
    return out


def fp4_decode(dtype: int, wire, n: int) -> np.ndarray:
    wire = np.ascontiguousarray(wire, dtype=np.uint8)
    assert wire.size >= fp4_wire_bytes(n)
    y = np.empty(n, np.uint16)
    _check(lib().orc_fp4_decode(dtype, _p(wire, ctypes.c_uint8), n, _p(y, ctypes.c_uint16)), "fp4_decode")
    return y


def fp4_segment_reduce(wires, n: int) -> np.ndarray:
    wires = [np.ascontiguousarray(w, dtype=np.uint8) for w in wires]
    arr = (ctypes.POINTER(ctypes.c_uint8) * len(wires))(*[_p(w, ctypes.c_uint8) for w in wires])
    out = np.empty(fp4_wire_bytes(n), np.uint8)
    _check(lib().orc_fp4_segment_reduce(len(wires), arr, n, _p(out, ctypes.c_uint8)), "fp4_segment_reduce")
    return out


def fp4_allreduce(dtype: int, xs) -> np.ndarray:
    xs = [np.ascontiguousarray(x, dtype=np.uint16).reshape(-1) for x in xs]
    n = xs[0].size
    assert all(x.size == n for x in xs)
    arr = (ctypes.POINTER(ctypes.c_uint16) * len(xs))(*[_p(x, ctypes.c_uint16) for x in xs])
    y = np.empty(n, np.uint16)
    _check(lib().orc_fp4_allreduce(dtype, len(xs), arr, n, _p(y, ctypes.c_uint16)), "fp4_allreduce")
    return y
