"""Parity of the two-shot all-reduce whose exchange is laid out as across R
GPUs (qr_allreduce_twoshot) against the oracle.

Every rank's output equals the oracle's all-reduce bit for bit; the
workspace holds, byte for byte, each owner's received copies of every
sender's quantized segment (the oracle's encode of that sender, cut at the
segment) and the gathered reduced wire (the oracle's Phase-1B output).
"""
import numpy as np
import pytest
import torch

import bit_quantized_all_gb300 as qr
import oracle
import workloads
from qr_testlib import assert_outputs_match, assert_wire_equal, to_dev, to_host_u8, to_host_u16, xmax_of

pytestmark = pytest.mark.gpu

BITS = [3, 4, 6, 8]


@pytest.fixture(scope="module", autouse=True)
def lib():
    from bit_quantized_all_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    qr.lib()


def twoshot_check(bits, dtype, xs, what):
    R, n = len(xs), xs[0].size
    xs_dev = [to_dev(x, dtype) for x in xs]
    ys, ws = qr.qr_allreduce_twoshot(bits, xs_dev)
    torch.cuda.synchronize()
    w_ref = [oracle.encode(bits, dtype, x) for x in xs]
    red_ref = oracle.segment_reduce(bits, w_ref, n)
    y_ref = oracle.decode(bits, dtype, red_ref, n)
    xmax = xmax_of(xs, dtype)
    for j, y in enumerate(ys):
        assert_outputs_match(to_host_u16(y), y_ref, dtype, xmax, f"{what} rank {j} output")
    tb = qr.qr_tile_bytes(bits)
    T = -(-n // 2048)
    seg = -(-T // R)
    wsh = to_host_u8(ws)
    for k in range(R):
        t0, t1 = k * seg, min(T, (k + 1) * seg)
        if t0 >= T:
            break
        for j in range(R):
            off = (k * R + j) * seg * tb
            assert_wire_equal(wsh[off: off + (t1 - t0) * tb], w_ref[j][t0 * tb: t1 * tb], bits,
                              f"{what} owner {k} copy from rank {j}")
    red_off = R * R * seg * tb
    assert_wire_equal(wsh[red_off: red_off + T * tb], red_ref, bits, f"{what} gathered wire")
    # the fused kernel gives the same bytes
    yf = qr.qr_allreduce(bits, xs_dev)
    assert torch.equal(yf.view(torch.int16), ys[0].view(torch.int16))


def _rand_ranks(R, n, dtype, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    out = []
    for r in range(R):
        v = rng.standard_normal(n).astype(np.float32) * np.float32(1 + r)
        v[rng.integers(0, n, size=max(1, n // 300))] *= 25.0
        out.append(oracle.narrow(dtype, v))
    return out


@pytest.mark.parametrize("cfg", [workloads.C1, workloads.C2, workloads.C3], ids=lambda c: c["name"])
def test_workloads(cfg):
    xs = workloads.ranks(cfg)
    for bits in cfg["bits"]:
        twoshot_check(bits, cfg["dtype"], xs, f"{cfg['name']} INT{bits}")


@pytest.mark.parametrize("n", [1, 37, 2048, 2049, 2048 * 3, 2048 * 5 + 37, 2048 * 9 + 1])
@pytest.mark.parametrize("R", [1, 2, 3, 8])
def test_segment_shapes(n, R):
    """Fewer tiles than ranks (empty owners), uneven last segments, ragged tails."""
    for bits in BITS:
        for dtype in (0, 1):
            twoshot_check(bits, dtype, _rand_ranks(R, n, dtype, 40 * n + R + bits), f"n={n} R={R} INT{bits}")


@pytest.mark.parametrize("R", [4, 5, 6, 7])
def test_other_rank_counts(R):
    n = 2048 * 11 + 100
    for bits in BITS:
        twoshot_check(bits, 1, _rand_ranks(R, n, 1, 700 + R + bits), f"R={R} INT{bits}")


def test_in_place_and_repeat():
    n = 2048 * 64 + 5
    R = 4
    xs_dev = [to_dev(x, 0) for x in _rand_ranks(R, n, 0, 5)]
    y0 = qr.qr_allreduce(4, xs_dev)
    ys, ws = qr.qr_allreduce_twoshot(4, xs_dev)
    ys2, _ = qr.qr_allreduce_twoshot(4, xs_dev, workspace=ws)  # the same workspace again
    for a, b in zip(ys, ys2):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    xs2 = [x.clone() for x in xs_dev]
    out, _ = qr.qr_allreduce_twoshot(4, xs2, ys=xs2)  # every rank in place
    for y in out:
        assert torch.equal(y.view(torch.int16), y0.view(torch.int16))


def test_large_sampled():
    """The benchmark's size class: R=8, 2^27 values per rank; outputs equal
    the fused kernel's (which is checked against the oracle elsewhere) and a
    sample of gathered tiles equals the oracle's reduction of those tiles."""
    n, R = 1 << 27, 8
    xs_dev = [x.view(torch.bfloat16) for x in workloads.device_sweep(R, n, 1, seed=11, device="cuda")]
    yf = qr.qr_allreduce(4, xs_dev)
    ys, ws = qr.qr_allreduce_twoshot(4, xs_dev)
    for y in ys:
        assert torch.equal(y.view(torch.int16), yf.view(torch.int16))
    T, tb = n // 2048, qr.qr_tile_bytes(4)
    seg = -(-T // R)
    red_off = R * R * seg * tb
    rng = np.random.Generator(np.random.PCG64(3))
    for t in rng.choice(T, size=64, replace=False).tolist() + [0, T - 1]:
        xt = [x[t * 2048:(t + 1) * 2048].contiguous().view(torch.int16).cpu().numpy().view(np.uint16) for x in xs_dev]
        red_t = oracle.segment_reduce(4, [oracle.encode(4, 1, v) for v in xt], 2048)
        got = ws[red_off + t * tb: red_off + (t + 1) * tb].cpu().numpy()
        assert_wire_equal(got, red_t, 4, f"gathered tile {t}")


# ---------------------------------------------------------------------------
# the one-launch version whose phases are joined by per-tile ready flags
# ---------------------------------------------------------------------------
def flags_check(bits, dtype, xs, what):
    R, n = len(xs), xs[0].size
    xs_dev = [to_dev(x, dtype) for x in xs]
    ys, ws = qr.qr_allreduce_twoshot(bits, xs_dev, flags=True)
    torch.cuda.synchronize()
    y_ref = oracle.allreduce(bits, dtype, xs)
    xmax = xmax_of(xs, dtype)
    for j, y in enumerate(ys):
        assert_outputs_match(to_host_u16(y), y_ref, dtype, xmax, f"{what} rank {j} output")
    # the exchange buffers hold what the three-launch version leaves there
    # (the parts either version writes: each owner's received tiles and the
    # T gathered tiles; owners past the last tile own nothing)
    ys3, ws3 = qr.qr_allreduce_twoshot(bits, xs_dev)
    torch.cuda.synchronize()
    base = ws3.numel()
    T = -(-n // 2048)
    tb = qr.qr_tile_bytes(bits)
    seg = -(-T // R)
    a, b = to_host_u8(ws[:base]), to_host_u8(ws3)
    for k in range(R):
        t0, t1 = k * seg, min(T, (k + 1) * seg)
        for j in range(R):
            off = (k * R + j) * seg * tb
            if t0 < T:
                assert_wire_equal(a[off: off + (t1 - t0) * tb], b[off: off + (t1 - t0) * tb], bits,
                                  f"{what} owner {k} copy from rank {j}")
    red_off = R * R * seg * tb
    assert_wire_equal(a[red_off: red_off + T * tb], b[red_off: red_off + T * tb], bits, f"{what} gathered wire")
    # and the protocol ran to completion: the per-chunk flags in use (a
    # prefix of each range) saw R sends and one reduction each, no abort
    off = -(-base // 16) * 16
    words = ws[off: off + 4 * (2 * T + 1)].cpu().numpy().view(np.uint32)
    sent, reduced = words[:T], words[T:2 * T]
    used = int(np.count_nonzero(sent))
    assert used >= 1 and np.all(sent[:used] == R) and np.all(sent[used:] == 0), what
    assert np.all(reduced[:used] == 1) and np.all(reduced[used:] == 0) and words[2 * T] == 0, what
    assert used * 8 >= T, what  # chunks of at most 8 tiles cover every tile
    assert qr.qr_wait_timeouts() == 0


@pytest.mark.parametrize("n", [1, 37, 2048, 2049, 2048 * 9 + 1, 2048 * 64 + 5])
@pytest.mark.parametrize("R", [1, 2, 3, 8])
def test_flags_segment_shapes(n, R):
    for bits in BITS:
        flags_check(bits, 1, _rand_ranks(R, n, 1, 30 * n + R + bits), f"flags n={n} R={R} INT{bits}")


@pytest.mark.parametrize("cfg", [workloads.C1, workloads.C2, workloads.C3], ids=lambda c: c["name"])
def test_flags_workloads(cfg):
    xs = workloads.ranks(cfg)
    for bits in cfg["bits"]:
        flags_check(bits, cfg["dtype"], xs, f"flags {cfg['name']} INT{bits}")


def test_flags_in_place_and_large():
    """Every rank in place; and the benchmark's size class against the fused kernel."""
    n, R = 2048 * 200 + 9, 4
    xs_dev = [to_dev(x, 0) for x in _rand_ranks(R, n, 0, 8)]
    y0 = qr.qr_allreduce(4, xs_dev)
    xs2 = [x.clone() for x in xs_dev]
    out, _ = qr.qr_allreduce_twoshot(4, xs2, ys=xs2, flags=True)
    for y in out:
        assert torch.equal(y.view(torch.int16), y0.view(torch.int16))
    n, R = 1 << 27, 8
    xs_dev = [x.view(torch.bfloat16) for x in workloads.device_sweep(R, n, 1, seed=12, device="cuda")]
    for bits in (4, 3):
        yf = qr.qr_allreduce(bits, xs_dev)
        ys, _ = qr.qr_allreduce_twoshot(bits, xs_dev, flags=True)
        for y in ys:
            assert torch.equal(y.view(torch.int16), yf.view(torch.int16)), bits
    assert qr.qr_wait_timeouts() == 0


@pytest.mark.parametrize("R,drop", [(2, 1), (8, 0), (8, 5)])
def test_flags_wait_runs_out_when_a_sender_never_announces(R, drop):
    """The failure path of the flag-joined protocol: sender `drop` writes its
    tiles into the owners' buffers but never raises their flags (as a peer
    that stopped would).  The owners' waits give up after one second; the
    launch returns, raises the abort word, counts exactly one timeout, and
    leaves the context usable: the next normal call over the same workspace
    matches the oracle bit for bit."""
    n, bits, dtype = 2048 * 40 + 11, 4, 1
    xs = _rand_ranks(R, n, dtype, 900 + 10 * R + drop)
    xs_dev = [to_dev(x, dtype) for x in xs]
    ws = torch.empty(qr.lib().qr_twoshot_flags_workspace_bytes(bits, R, n), dtype=torch.uint8, device="cuda")
    ys = [torch.zeros_like(xs_dev[0]) for _ in range(R)]
    assert qr.qr_wait_timeouts() == 0
    from bit_quantized_all_gb300 import capi
    st = torch.cuda.current_stream().cuda_stream
    status = capi.qr_selftest_twoshot_flags_drop(bits, dtype, R, [x.data_ptr() for x in xs_dev], n,
                                                 [y.data_ptr() for y in ys], ws.data_ptr(), ws.numel(), drop, st)
    assert status == qr.QR_OK  # enqueued; the failure shows only on the device
    torch.cuda.synchronize()
    assert qr.qr_wait_timeouts() == 1
    T = -(-n // 2048)
    off = -(-qr.qr_twoshot_workspace_bytes(bits, R, n) // 16) * 16
    words = ws[off: off + 4 * (2 * T + 1)].cpu().numpy().view(np.uint32)
    assert words[2 * T] == 1  # the abort word
    sent = words[:T]
    assert np.all(sent <= R - 1)  # no chunk ever saw all R announcements
    assert np.all(words[T:2 * T] == 0)  # nothing was reduced
    # a normal call over the same workspace
    ys2, _ = qr.qr_allreduce_twoshot(bits, xs_dev, workspace=ws, flags=True)
    torch.cuda.synchronize()
    y_ref = oracle.allreduce(bits, dtype, xs)
    for j, y in enumerate(ys2):
        assert_outputs_match(to_host_u16(y), y_ref, dtype, xmax_of(xs, dtype), f"after the drop, rank {j}")
    assert qr.qr_wait_timeouts() == 0
