"""Parity of the CUDA path (through the C ABI) against the oracle on the GPU.

Element by element on whole messages where the oracle finishes in seconds
(workloads c1, c2, c3, ragged and edge sizes, special values), and on seeded
samples of tiles (plus the first and last tile) for the large workloads (c4,
the 2 GiB-per-rank sweep point, the benchmark's own configuration).  Tiles
are independent in every step, so a sampled tile is checked exactly.
Properties that hold at any size (fused == unfused, determinism, grid-size
independence, in-place) are checked on the device over whole messages.
"""
import numpy as np
import pytest
import torch

import bit_quantized_all_gb300 as qr
import oracle
import workloads
from bit_quantized_all_gb300 import capi
from qr_testlib import (assert_outputs_match, assert_wire_equal, gather_tiles_u16, gather_wire_tiles,
                        gpu_fused, gpu_unfused, sample_tiles, to_dev, to_host_u8, to_host_u16, xmax_of)

pytestmark = pytest.mark.gpu

BITS = [3, 4, 6, 8]


@pytest.fixture(scope="module", autouse=True)
def lib():
    from bit_quantized_all_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    qr.lib()


_cache = {}


def _cfg_inputs(cfg):
    if cfg["name"] not in _cache:
        _cache[cfg["name"]] = workloads.ranks(cfg)
    return _cache[cfg["name"]]


def full_check(bits, dtype, xs, what):
    """Every path against the oracle on whole messages."""
    n = xs[0].size
    xs_dev = [to_dev(x, dtype) for x in xs]
    # oracle
    w_ref = [oracle.encode(bits, dtype, x) for x in xs]
    red_ref = oracle.segment_reduce(bits, w_ref, n)
    y_ref = oracle.decode(bits, dtype, red_ref, n)
    xmax = xmax_of(xs, dtype)
    # unfused: encode -> segment_reduce -> decode
    wires, red, y = gpu_unfused(bits, xs_dev)
    for r in range(len(xs)):
        assert_wire_equal(to_host_u8(wires[r]), w_ref[r], bits, f"{what} encode rank {r}")
    assert_wire_equal(to_host_u8(red), red_ref, bits, f"{what} segment_reduce")
    assert_outputs_match(to_host_u16(y), y_ref, dtype, xmax, f"{what} decode")
    # the oracle's own composition equals its all-reduce
    assert np.array_equal(oracle.allreduce(bits, dtype, xs), y_ref)
    # fused
    yf = gpu_fused(bits, xs_dev)
    assert_outputs_match(to_host_u16(yf), y_ref, dtype, xmax, f"{what} fused")
    # fused, emitting the wires
    ye, we, rede = qr.qr_allreduce_emit(bits, xs_dev)
    assert_outputs_match(to_host_u16(ye), y_ref, dtype, xmax, f"{what} emit y")
    for r in range(len(xs)):
        assert_wire_equal(to_host_u8(we[r]), w_ref[r], bits, f"{what} emit wire {r}")
    assert_wire_equal(to_host_u8(rede), red_ref, bits, f"{what} emit reduced wire")


@pytest.mark.parametrize("bits", [4, 3])
def test_c1_small_crafted(bits):
    full_check(bits, 0, _cfg_inputs(workloads.C1), f"c1 INT{bits}")


@pytest.mark.parametrize("bits", BITS)
def test_c2_decode_step(bits):
    full_check(bits, 1, _cfg_inputs(workloads.C2), f"c2 INT{bits}")


@pytest.mark.parametrize("bits", [4, 3])
def test_c3_prefill(bits):
    full_check(bits, 1, _cfg_inputs(workloads.C3), f"c3 INT{bits}")


def _rand_ranks(R, n, dtype, seed, scale=1.0):
    rng = np.random.Generator(np.random.PCG64(seed))
    out = []
    for r in range(R):
        v = rng.standard_normal(n).astype(np.float32) * np.float32(scale * (1 + r))
        v[rng.integers(0, n, size=max(1, n // 500))] *= 30.0
        out.append(oracle.narrow(dtype, v))
    return out


@pytest.mark.parametrize("n", [1, 7, 8, 9, 31, 33, 2047, 2048, 2049, 2048 * 5 + 37])
@pytest.mark.parametrize("R", [1, 2, 3, 8])
def test_ragged_sizes(n, R):
    for bits in BITS:
        for dtype in (0, 1):
            xs = _rand_ranks(R, n, dtype, seed=1000 * R + n + bits + 10 * dtype)
            full_check(bits, dtype, xs, f"n={n} R={R} INT{bits} dt={dtype}")


@pytest.mark.parametrize("R", [1, 2, 3, 4, 5, 6, 7, 8])
def test_every_rank_count(R):
    n = 2048 * 3 + 37
    for bits in BITS:
        for dtype in (0, 1):
            xs = _rand_ranks(R, n, dtype, seed=500 + 10 * R + bits + dtype)
            full_check(bits, dtype, xs, f"R={R} INT{bits} dt={dtype}")


@pytest.mark.parametrize("dtype", [0, 1])
def test_mixed_scale_ranges_in_one_warp(dtype):
    """Neighbouring blocks with subnormal, normal and saturated fp16 scales,
    so that some warps need the clip at qmin and others do not."""
    n = 2048 * 8 + 37
    rng = np.random.Generator(np.random.PCG64(31 + dtype))
    lo, hi = (-27, 14) if dtype == 0 else (-40, 40)
    for R in (1, 2, 5, 8):
        xs = []
        for r in range(R):
            v = rng.standard_normal(n).astype(np.float32)
            v *= np.repeat(np.exp2(rng.integers(lo, hi, size=-(-n // 32))), 32)[:n].astype(np.float32)
            if dtype == 0:
                v = np.clip(v, -60000.0 / R, 60000.0 / R)
            xs.append(oracle.narrow(dtype, v))
        for bits in BITS:
            full_check(bits, dtype, xs, f"mixed scales R={R} INT{bits} dt={dtype}")


@pytest.mark.parametrize("bits", BITS)
def test_fused_with_16_byte_aligned_pointers(bits):
    """Pointers that are 16- but not 32-byte aligned take the general fused
    kernel; the result is the same."""
    R, n, dtype = 3, 2048 * 5 + 37, 1
    xs = _rand_ranks(R, n, dtype, seed=900 + bits)
    bufs = []
    for x in xs:
        b = torch.zeros(2 * n + 64, dtype=torch.uint8, device="cuda")
        b[16:16 + 2 * n] = torch.from_numpy(x.view(np.uint8)).cuda()
        bufs.append(b)
    yb = torch.zeros(2 * n + 64, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    ptrs = [b.data_ptr() + 16 for b in bufs]
    assert all(p % 32 == 16 for p in ptrs)
    assert capi.qr_allreduce(bits, dtype, R, ptrs, n, yb.data_ptr() + 16, st) == qr.QR_OK
    # the unfused kernels on the same 16-byte-aligned pointers
    W = qr.qr_wire_bytes(bits, n)
    wb = [torch.zeros(W + 64, dtype=torch.uint8, device="cuda") for _ in range(R + 1)]
    yu = torch.zeros(2 * n + 64, dtype=torch.uint8, device="cuda")
    wp = [b.data_ptr() + 16 for b in wb]
    for r in range(R):
        assert capi.qr_encode(bits, dtype, ptrs[r], n, wp[r], st) == qr.QR_OK
    assert capi.qr_segment_reduce(bits, R, wp[:R], n, wp[R], st) == qr.QR_OK
    assert capi.qr_decode(bits, dtype, wp[R], n, yu.data_ptr() + 16, st) == qr.QR_OK
    torch.cuda.synchronize()
    w_ref = [oracle.encode(bits, dtype, x) for x in xs]
    for r in range(R):
        assert_wire_equal(to_host_u8(wb[r])[16:16 + W], w_ref[r], bits, f"16B-aligned encode {r}")
    assert_wire_equal(to_host_u8(wb[R])[16:16 + W], oracle.segment_reduce(bits, w_ref, n), bits, "16B reduce")
    y_ref = oracle.allreduce(bits, dtype, xs)
    got = to_host_u8(yb)[16:16 + 2 * n].copy().view(np.uint16)
    assert np.array_equal(got, y_ref)
    assert np.array_equal(to_host_u8(yu)[16:16 + 2 * n].copy().view(np.uint16), y_ref)


GUARD = 4096  # canary bytes before and after every buffer


def _guarded(nbytes, device="cuda"):
    buf = torch.full((GUARD + nbytes + GUARD,), 0xA5, dtype=torch.uint8, device=device)
    return buf, buf.data_ptr() + GUARD


def _canary_ok(buf, nbytes):
    h = to_host_u8(buf)
    return bool(np.all(h[:GUARD] == 0xA5) and np.all(h[GUARD + nbytes:] == 0xA5))


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("n", [37, 2048 * 3 + 37, 2048 * 4])
def test_no_writes_outside_buffers(bits, dtype, n):
    """Guard regions around inputs, wires and outputs keep their canary;
    outputs are written for the first n values only."""
    R = 3
    xs = _rand_ranks(R, n, dtype, seed=77 + n + bits)
    W = qr.qr_wire_bytes(bits, n)
    xbufs = []
    for x in xs:
        b, p = _guarded(2 * n)
        b[GUARD:GUARD + 2 * n] = torch.from_numpy(x.view(np.uint8)).cuda()
        xbufs.append((b, p))
    wbufs = [_guarded(W) for _ in range(R)]
    rbuf = _guarded(W)
    ybuf = _guarded(2 * n)
    yfbuf = _guarded(2 * n)
    st = torch.cuda.current_stream().cuda_stream
    for r in range(R):
        assert capi.qr_encode(bits, dtype, xbufs[r][1], n, wbufs[r][1], st) == qr.QR_OK
    assert capi.qr_segment_reduce(bits, R, [w[1] for w in wbufs], n, rbuf[1], st) == qr.QR_OK
    assert capi.qr_decode(bits, dtype, rbuf[1], n, ybuf[1], st) == qr.QR_OK
    assert capi.qr_allreduce(bits, dtype, R, [x[1] for x in xbufs], n, yfbuf[1], st) == qr.QR_OK
    ewbufs = [_guarded(W) for _ in range(R)]
    erbuf = _guarded(W)
    eybuf = _guarded(2 * n)
    assert capi.qr_allreduce_emit(bits, dtype, R, [x[1] for x in xbufs], n, eybuf[1],
                                  [w[1] for w in ewbufs], erbuf[1], st) == qr.QR_OK
    torch.cuda.synchronize()
    for b, _ in xbufs:
        assert _canary_ok(b, 2 * n)
    for b, _ in wbufs + [rbuf] + ewbufs + [erbuf]:
        assert _canary_ok(b, W)
    for b in (ybuf, yfbuf, eybuf):
        assert _canary_ok(b[0], 2 * n)
    y_ref = oracle.allreduce(bits, dtype, xs)
    for b in (ybuf, yfbuf, eybuf):
        got = to_host_u8(b[0])[GUARD:GUARD + 2 * n].copy().view(np.uint16)
        assert np.array_equal(got, y_ref)


def test_special_values():
    n = 2048 * 2
    for dtype in (0, 1):
        blocks = []
        z = np.zeros(n, np.float32)
        blocks.append(z)                                        # all zero
        e = np.zeros(n, np.float32)
        e[:1024] = 0.7
        e[1024:2048] = -0.75
        e[2048:] = np.repeat(np.linspace(-3, 3, 64), 32)        # all-equal blocks
        blocks.append(e)
        t = np.zeros(n, np.float32)
        t[::2] = 6e-8 if dtype == 0 else 1e-30                  # tiny: scale underflow
        t[1::7] = -3e-8 if dtype == 0 else -2e-31
        blocks.append(t)
        # finite inputs on every rank (x (1 + 0.25 r) <= x 2.75); the fp16 sums
        # overflow to inf in the output, the bf16 scales saturate at 65504
        big = np.full(n, 21000.0 if dtype == 0 else 3e30, np.float32)
        big[1::3] *= -1
        blocks.append(big)
        for bits in BITS:
            for R in (2, 4, 8):
                for v in blocks:
                    xs = [oracle.narrow(dtype, v * np.float32(1 + 0.25 * r)) for r in range(R)]
                    full_check(bits, dtype, xs, f"special INT{bits} R={R} dt={dtype}")


@pytest.mark.parametrize("bits", BITS)
def test_properties_on_device(bits):
    n = 2048 * 257 + 37
    R = 4
    xs_dev = [to_dev(x, 1) for x in _rand_ranks(R, n, 1, seed=bits)]
    y0 = gpu_fused(bits, xs_dev)
    # determinism and grid-size independence
    for ctas in (1, 3, 152, 5000):
        assert torch.equal(gpu_fused(bits, xs_dev, ctas=ctas).view(torch.int16), y0.view(torch.int16))
    assert torch.equal(gpu_fused(bits, xs_dev).view(torch.int16), y0.view(torch.int16))
    # fused == unfused
    _, _, yu = gpu_unfused(bits, xs_dev)
    assert torch.equal(yu.view(torch.int16), y0.view(torch.int16))
    # in place: y aliases rank 0
    xs2 = [x.clone() for x in xs_dev]
    out = qr.qr_allreduce(bits, xs2, y=xs2[0])
    assert out.data_ptr() == xs2[0].data_ptr()
    assert torch.equal(xs2[0].view(torch.int16), y0.view(torch.int16))
    # R=2 rank swap
    a = gpu_fused(bits, xs_dev[:2])
    b = gpu_fused(bits, xs_dev[1::-1])
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def _sampled_check(bits, dtype, xs_dev, k, seed, what, unfused=True):
    """Compare sampled tiles of every path with the oracle run on those tiles."""
    n = xs_dev[0].numel()
    T = -(-n // 2048)
    tiles = sample_tiles(T, k, seed)
    per_rank = [gather_tiles_u16(x, tiles, n) for x in xs_dev]  # [R][tile] -> values
    yf = gpu_fused(bits, xs_dev)
    yf_tiles = gather_tiles_u16(yf, tiles, n)
    if unfused:
        wires, red, yu = gpu_unfused(bits, xs_dev)
        assert torch.equal(yu.view(torch.int16), yf.view(torch.int16)), f"{what}: fused != unfused"
        w_tiles = [gather_wire_tiles(w, tiles, bits) for w in wires]
        red_tiles = gather_wire_tiles(red, tiles, bits)
    tb = qr.qr_tile_bytes(bits)
    xmax = float(max(x.abs().max().float().item() for x in xs_dev))
    for i, t in enumerate(tiles.tolist()):
        xs_t = [per_rank[r][i] for r in range(len(xs_dev))]
        m = xs_t[0].size
        w_ref = [oracle.encode(bits, dtype, x) for x in xs_t]
        red_ref = oracle.segment_reduce(bits, w_ref, m)
        y_ref = oracle.decode(bits, dtype, red_ref, m)
        assert_outputs_match(yf_tiles[i], y_ref, dtype, xmax, f"{what} tile {t}")
        if unfused:
            for r in range(len(xs_dev)):
                assert_wire_equal(w_tiles[r][i * tb:(i + 1) * tb], w_ref[r], bits, f"{what} tile {t} rank {r}")
            assert_wire_equal(red_tiles[i * tb:(i + 1) * tb], red_ref, bits, f"{what} tile {t} reduced")


@pytest.mark.parametrize("bits", [8, 4])
def test_c4_sampled(bits):
    xs = _cfg_inputs(workloads.C4)
    xs_dev = [to_dev(x, 0) for x in xs]
    _sampled_check(bits, 0, xs_dev, 1024, seed=bits, what=f"c4 INT{bits}")


SWEEP = [(1 << 14), (1 << 14) + 37, (1 << 20) + 37, (1 << 24)]


@pytest.mark.parametrize("n", SWEEP)
@pytest.mark.parametrize("R", [2, 4, 8])
@pytest.mark.parametrize("dtype", [0, 1])
def test_sweep_points(n, R, dtype):
    xs = [workloads.sweep_rank(r, n, dtype) for r in range(R)]
    for bits in BITS:
        if n <= (1 << 20) + 37:
            full_check(bits, dtype, xs, f"sweep n={n} R={R} dt={dtype} INT{bits}")
        else:
            xs_dev = [to_dev(x, dtype) for x in xs]
            _sampled_check(bits, dtype, xs_dev, 256, seed=n + R + bits, what=f"sweep n={n} R={R} INT{bits}")


@pytest.mark.parametrize("bits", [4, 3])
def test_bench_configuration_sampled(bits):
    """The benchmark's workload and launch: R=8, 2^27 bf16 values per rank
    (256 MiB per rank), default grid."""
    import bench
    if "bench" not in _cache:
        _cache["bench"] = bench.host_inputs()
    xs_dev = [to_dev(x, 1) for x in _cache["bench"]]
    _sampled_check(bits, 1, xs_dev, 512, seed=bits, what=f"bench INT{bits}")


def test_largest_sweep_point_sampled():
    """The largest message: R=8, 2^30 values (2 GiB) per rank."""
    xs_dev = workloads.device_sweep(8, 1 << 30, 0, seed=9, device="cuda")
    xs_dev = [x.view(torch.float16) for x in xs_dev]
    for bits in (4, 3):
        _sampled_check(bits, 0, xs_dev, 128, seed=bits, what=f"2GiB INT{bits}", unfused=False)
    del xs_dev
    torch.cuda.empty_cache()


def test_binding_rejects_wrong_tensors():
    """Wrong-format tensors are rejected, never misread (dtype checks of the
    binding, in the style of the vLLM W4A16 zero-point regression test)."""
    x = torch.zeros(4096, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(TypeError):
        qr.qr_encode(4, x.float())
    with pytest.raises(TypeError):
        qr.qr_allreduce(4, [x, x.half()])
    with pytest.raises(ValueError):
        qr.qr_allreduce(4, [x, x[:2048]])
    with pytest.raises(ValueError):
        qr.qr_encode(4, x.cpu())
    w = qr.qr_encode(4, x)
    with pytest.raises(TypeError):
        qr.qr_decode(4, w.view(torch.int8), 4096)
    with pytest.raises(ValueError):
        qr.qr_decode(4, w[:100], 4096)
    with pytest.raises(ValueError):
        qr.qr_allreduce(4, [x] * 9)
    with pytest.raises(ValueError):
        qr.qr_allreduce(4, [x, x], y=torch.empty(4095, dtype=torch.bfloat16, device="cuda"))
    # partial overlap of y with an input, on real buffers: rejected by the library
    big = torch.zeros(8192 + 64, dtype=torch.bfloat16, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    assert capi.qr_allreduce(4, 1, 2, [big.data_ptr(), big.data_ptr()], 4096,
                             big.data_ptr() + 64, st) == qr.QR_ERR_INVALID_ARG
