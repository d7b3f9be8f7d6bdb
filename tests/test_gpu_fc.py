"""Parity of the Flash Communication codec's CUDA path (through the C ABI)
against the oracle: the asymmetric group-128 codec at INT4 and INT8 and the
three reduce-scatter / all-gather schemes INT4 (4,4), INT8 (8,8) and the mixed
"INT6" (4,8) of the "Flash Communication" review record.  Wires byte for byte,
outputs bit for bit (and within the stated tolerance)."""
import numpy as np
import pytest
import torch

import bit_quantized_all_gb300 as qr
import oracle
import workloads
from bit_quantized_all_gb300 import capi
from qr_testlib import (assert_outputs_match, assert_wire_equal, gather_tiles_u16, sample_tiles, to_dev, to_host_u8,
                        to_host_u16, xmax_of)

pytestmark = pytest.mark.gpu

PAIRS = [(4, 4), (4, 8), (8, 8)]


@pytest.fixture(scope="module", autouse=True)
def lib():
    from bit_quantized_all_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    qr.lib()


_cache = {}


def _cfg(cfg):
    if cfg["name"] not in _cache:
        _cache[cfg["name"]] = workloads.ranks(cfg)
    return _cache[cfg["name"]]


def fc_full_check(brs, bag, dtype, xs, what):
    n = xs[0].size
    xs_dev = [to_dev(x, dtype) for x in xs]
    w_ref = [oracle.fc_encode(brs, dtype, x) for x in xs]
    red_ref = oracle.fc_segment_reduce(brs, bag, w_ref, n)
    y_ref = oracle.fc_decode(bag, dtype, red_ref, n)
    xmax = xmax_of(xs, dtype)
    wires = [qr.qr_fc_encode(brs, x) for x in xs_dev]
    red = qr.qr_fc_segment_reduce(brs, bag, wires, n)
    y = qr.qr_fc_decode(bag, red, n, dtype=xs_dev[0].dtype)
    for r in range(len(xs)):
        assert_wire_equal(to_host_u8(wires[r]), w_ref[r], brs, f"{what} fc_encode rank {r}")
    assert_wire_equal(to_host_u8(red), red_ref, bag, f"{what} fc_segment_reduce")
    assert_outputs_match(to_host_u16(y), y_ref, dtype, xmax, f"{what} fc_decode")
    assert np.array_equal(oracle.fc_allreduce(brs, bag, dtype, xs), y_ref)
    yf = qr.qr_fc_allreduce(brs, bag, xs_dev)
    assert_outputs_match(to_host_u16(yf), y_ref, dtype, xmax, f"{what} fused")


@pytest.mark.parametrize("pair", PAIRS)
def test_c1(pair):
    fc_full_check(*pair, 0, _cfg(workloads.C1), f"c1 {pair}")


@pytest.mark.parametrize("pair", PAIRS)
def test_c2(pair):
    fc_full_check(*pair, 1, _cfg(workloads.C2), f"c2 {pair}")


@pytest.mark.parametrize("pair", PAIRS)
def test_c3(pair):
    fc_full_check(*pair, 1, _cfg(workloads.C3), f"c3 {pair}")


def _rand_ranks(R, n, dtype, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    out = []
    for r in range(R):
        v = (rng.standard_normal(n) * (1 + r) + 0.3 * r).astype(np.float32)
        v[rng.integers(0, n, size=max(1, n // 400))] *= 25.0
        out.append(oracle.narrow(dtype, v))
    return out


@pytest.mark.parametrize("n", [1, 37, 128, 129, 2047, 2048, 2049, 2048 * 3 + 37])
@pytest.mark.parametrize("R", [1, 2, 3, 8])
def test_ragged_sizes(n, R):
    for pair in PAIRS:
        for dtype in (0, 1):
            fc_full_check(*pair, dtype, _rand_ranks(R, n, dtype, 10 * n + R), f"n={n} R={R} {pair} dt={dtype}")


@pytest.mark.parametrize("R", [1, 2, 3, 4, 5, 6, 7, 8])
def test_every_rank_count(R):
    n = 2048 * 2 + 300
    for pair in PAIRS:
        for dtype in (0, 1):
            fc_full_check(*pair, dtype, _rand_ranks(R, n, dtype, 77 + R), f"R={R} {pair} dt={dtype}")


@pytest.mark.parametrize("pair,R", [((4, 4), 8), ((4, 8), 5), ((4, 4), 4), ((8, 8), 3), ((4, 4), 2), ((4, 8), 3)])
def test_phase1b_many_tiles_per_cta(pair, R):
    """Enough tiles that every CTA of the Phase-1B grid-stride kernels reduces
    several (odd and even counts: both register sets of the one-tile-ahead
    kernel take turns), whole wire against the oracle."""
    n = 2048 * 7001 + 5
    fc_full_check(*pair, 1, _rand_ranks(R, n, 1, 500 + R), f"many tiles R={R} {pair}")


@pytest.mark.parametrize("n", [2048 * 40 + 37, 2048 * 3 + 1, 700])
@pytest.mark.parametrize("R", [1, 2, 3, 5, 8])
def test_twoshot(n, R):
    """The two-shot exchange laid out per rank and per owner: every rank's
    output equals the fused all-reduce and the oracle's, the owners' receive
    buffers hold the oracle's wire segments, the gathered wire is the
    oracle's Phase-1B output; fewer tiles than ranks at the small sizes."""
    T = -(-n // 2048)
    seg = -(-T // R)
    for brs, bag in PAIRS:
        dt = 1 if brs == 4 else 0
        xs = _rand_ranks(R, n, dt, 300 + 7 * R + brs + bag)
        xs_dev = [to_dev(x, dt) for x in xs]
        ys, ws = qr.qr_fc_allreduce_twoshot(brs, bag, xs_dev)
        yf = qr.qr_fc_allreduce(brs, bag, xs_dev)
        torch.cuda.synchronize()
        y_ref = oracle.fc_allreduce(brs, bag, dt, xs)
        for j in range(R):
            assert np.array_equal(to_host_u16(ys[j]), y_ref), (brs, bag, R, n, j)
            assert torch.equal(ys[j].view(torch.int16), yf.view(torch.int16))
        ti, to = qr.qr_fc_tile_bytes(brs), qr.qr_fc_tile_bytes(bag)
        host = to_host_u8(ws)
        w_ref = [oracle.fc_encode(brs, dt, x) for x in xs]
        for k in range(R):
            t0, t1 = k * seg, min(T, (k + 1) * seg)
            for j in range(R):
                got = host[((k * R + j) * seg) * ti:((k * R + j) * seg + max(0, t1 - t0)) * ti]
                assert np.array_equal(got, w_ref[j][t0 * ti:max(t0, t1) * ti]), (brs, bag, R, n, k, j)
        g = R * R * seg * ti
        assert np.array_equal(host[g:g + T * to], oracle.fc_segment_reduce(brs, bag, w_ref, n)), (brs, bag, R, n)
    assert qr.qr_wait_timeouts() == 0


def test_twoshot_in_place():
    n = 2048 * 33 + 5
    xs = _rand_ranks(4, n, 1, 77)
    y_ref = oracle.fc_allreduce(4, 8, 1, xs)
    xs_dev = [to_dev(x, 1) for x in xs]
    ys, _ = qr.qr_fc_allreduce_twoshot(4, 8, xs_dev, ys=xs_dev)   # every output over its own input
    torch.cuda.synchronize()
    for j in range(4):
        assert np.array_equal(to_host_u16(xs_dev[j]), y_ref)


def test_special_groups():
    n = 2048 * 2
    for dtype in (0, 1):
        cases = []
        c = np.repeat(np.linspace(-7, 7, n // 128).astype(np.float32), 128)       # constant groups
        cases.append(c)
        z = np.zeros(n, np.float32)                                               # +-0 groups
        zi = oracle.narrow(dtype, z)
        zi[::3] = 0x8000
        cases.append(oracle.widen(dtype, zi))
        rng = np.random.Generator(np.random.PCG64(5 + dtype))
        m = rng.standard_normal(n).astype(np.float32)                             # mixed ranges
        m *= np.repeat(np.exp2(rng.integers(-20, 12 if dtype == 0 else 60, size=n // 128)), 128).astype(np.float32)
        if dtype == 0:
            m = np.clip(m, -8000, 8000)
        cases.append(m)
        for v in cases:
            for R in (1, 3, 8):
                xs = [oracle.narrow(dtype, v * np.float32(1 + 0.125 * r)) for r in range(R)]
                for pair in PAIRS:
                    fc_full_check(*pair, dtype, xs, f"special R={R} {pair} dt={dtype}")


@pytest.mark.parametrize("pair", PAIRS)
def test_16_byte_aligned_pointers(pair):
    brs, bag = pair
    R, n, dtype = 3, 2048 * 4 + 37, 1
    xs = _rand_ranks(R, n, dtype, 900 + brs + bag)
    st = torch.cuda.current_stream().cuda_stream
    bufs = []
    for x in xs:
        b = torch.zeros(2 * n + 64, dtype=torch.uint8, device="cuda")
        b[16:16 + 2 * n] = torch.from_numpy(x.view(np.uint8)).cuda()
        bufs.append(b)
    ptrs = [b.data_ptr() + 16 for b in bufs]
    yb = torch.zeros(2 * n + 64, dtype=torch.uint8, device="cuda")
    assert capi.qr_fc_allreduce(brs, bag, dtype, R, ptrs, n, yb.data_ptr() + 16, st) == qr.QR_OK
    Wi, Wo = qr.qr_fc_wire_bytes(brs, n), qr.qr_fc_wire_bytes(bag, n)
    wb = [torch.zeros(Wi + 64, dtype=torch.uint8, device="cuda") for _ in range(R)]
    rb = torch.zeros(Wo + 64, dtype=torch.uint8, device="cuda")
    yu = torch.zeros(2 * n + 64, dtype=torch.uint8, device="cuda")
    for r in range(R):
        assert capi.qr_fc_encode(brs, dtype, ptrs[r], n, wb[r].data_ptr() + 16, st) == qr.QR_OK
    assert capi.qr_fc_segment_reduce(brs, bag, R, [w.data_ptr() + 16 for w in wb], n, rb.data_ptr() + 16,
                                     st) == qr.QR_OK
    assert capi.qr_fc_decode(bag, dtype, rb.data_ptr() + 16, n, yu.data_ptr() + 16, st) == qr.QR_OK
    torch.cuda.synchronize()
    y_ref = oracle.fc_allreduce(brs, bag, dtype, xs)
    assert np.array_equal(to_host_u8(yb)[16:16 + 2 * n].copy().view(np.uint16), y_ref)
    assert np.array_equal(to_host_u8(yu)[16:16 + 2 * n].copy().view(np.uint16), y_ref)
    # canaries: bytes around the outputs untouched
    assert np.all(to_host_u8(yb)[:16] == 0) and np.all(to_host_u8(yb)[16 + 2 * n:] == 0)
    assert np.all(to_host_u8(rb)[:16] == 0) and np.all(to_host_u8(rb)[16 + Wo:] == 0)


@pytest.mark.parametrize("pair", PAIRS)
def test_c4_sampled(pair):
    brs, bag = pair
    xs = _cfg(workloads.C4)
    xs_dev = [to_dev(x, 0) for x in xs]
    n = xs[0].size
    yf = qr.qr_fc_allreduce(brs, bag, xs_dev)
    wires = [qr.qr_fc_encode(brs, x) for x in xs_dev]
    red = qr.qr_fc_segment_reduce(brs, bag, wires, n)
    yu = qr.qr_fc_decode(bag, red, n, dtype=torch.float16)
    assert torch.equal(yf.view(torch.int16), yu.view(torch.int16))
    tiles = sample_tiles(-(-n // 2048), 512, seed=brs * 10 + bag)
    yt = gather_tiles_u16(yf, tiles, n)
    per_rank = [gather_tiles_u16(x, tiles, n) for x in xs_dev]
    for i, t in enumerate(tiles.tolist()):
        y_ref = oracle.fc_allreduce(brs, bag, 0, [per_rank[r][i] for r in range(len(xs))])
        assert np.array_equal(yt[i], y_ref), f"c4 {pair} tile {t}"


def test_in_place_and_determinism():
    n = 2048 * 129 + 5
    xs_dev = [to_dev(x, 1) for x in _rand_ranks(4, n, 1, 3)]
    for pair in PAIRS:
        y0 = qr.qr_fc_allreduce(*pair, xs_dev)
        assert torch.equal(qr.qr_fc_allreduce(*pair, xs_dev).view(torch.int16), y0.view(torch.int16))
        xs2 = [x.clone() for x in xs_dev]
        qr.qr_fc_allreduce(*pair, xs2, y=xs2[2])
        assert torch.equal(xs2[2].view(torch.int16), y0.view(torch.int16))
