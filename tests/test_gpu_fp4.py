"""The FP4 codec's CUDA path against the oracle, bit for bit: wires (codes and
scales), Phase-1B's reduced wire, decoded outputs and the fused all-reduce,
on the workloads' shapes and on edge cases (ragged and one-value messages,
every rank count, zero / constant / signed-zero / saturating / subnormal-
scale blocks)."""
import numpy as np
import pytest
import torch

import bit_quantized_all_gb300 as qr
import oracle
import workloads
from qr_testlib import assert_outputs_match, to_dev, to_host_u16, to_host_u8, xmax_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


def _check_all(xs, dt, what):
    n = xs[0].size
    xmax = xmax_of(xs, dt)
    w_ref = [oracle.fp4_encode(dt, x) for x in xs]
    red_ref = oracle.fp4_segment_reduce(w_ref, n)
    y_ref = oracle.fp4_allreduce(dt, xs)
    xs_dev = [to_dev(x, dt) for x in xs]
    wires = [qr.qr_fp4_encode(x) for x in xs_dev]
    for r, w in enumerate(wires):
        got = to_host_u8(w)
        assert np.array_equal(got, w_ref[r]), f"{what}: wire {r} differs at bytes {np.flatnonzero(got != w_ref[r])[:5]}"
    red = qr.qr_fp4_segment_reduce(wires, n)
    got = to_host_u8(red)
    assert np.array_equal(got, red_ref), f"{what}: reduced wire differs at bytes {np.flatnonzero(got != red_ref)[:5]}"
    y_u = qr.qr_fp4_decode(red, n, dtype=xs_dev[0].dtype)
    assert_outputs_match(to_host_u16(y_u), y_ref, dt, xmax, what + " unfused")
    y = qr.qr_fp4_allreduce(xs_dev)
    assert_outputs_match(to_host_u16(y), y_ref, dt, xmax, what + " fused")
    assert qr.qr_wait_timeouts() == 0


def _rand(R, n, dt, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    out = []
    for r in range(R):
        v = (rng.standard_normal(n) * (1 + r)).astype(np.float32)
        v[rng.integers(0, n, size=max(1, n // 300))] *= 40.0
        out.append(oracle.narrow(dt, v))
    return out


@pytest.mark.parametrize("n", [2048 * 40 + 37, 2048 * 3 + 1, 700])
@pytest.mark.parametrize("R", [1, 2, 3, 5, 8])
def test_twoshot(n, R):
    """The two-shot exchange laid out per rank and per owner: every rank's
    output equals the fused all-reduce and the oracle's, the owners' receive
    buffers hold the oracle's wire segments, the gathered wire is the
    oracle's Phase-1B output; fewer tiles than ranks at the small sizes."""
    T = -(-n // 2048)
    seg = -(-T // R)
    tb = qr.qr_fp4_tile_bytes()
    for dt in (0, 1):
        xs = _rand(R, n, dt, 600 + 11 * R + dt)
        xs_dev = [to_dev(x, dt) for x in xs]
        ys, ws = qr.qr_fp4_allreduce_twoshot(xs_dev)
        yf = qr.qr_fp4_allreduce(xs_dev)
        torch.cuda.synchronize()
        y_ref = oracle.fp4_allreduce(dt, xs)
        for j in range(R):
            assert np.array_equal(to_host_u16(ys[j]), y_ref), (R, n, dt, j)
            assert torch.equal(ys[j].view(torch.int16), yf.view(torch.int16))
        host = to_host_u8(ws)
        w_ref = [oracle.fp4_encode(dt, x) for x in xs]
        for k in range(R):
            t0, t1 = k * seg, min(T, (k + 1) * seg)
            for j in range(R):
                got = host[((k * R + j) * seg) * tb:((k * R + j) * seg + max(0, t1 - t0)) * tb]
                assert np.array_equal(got, w_ref[j][t0 * tb:max(t0, t1) * tb]), (R, n, dt, k, j)
        g = R * R * seg * tb
        assert np.array_equal(host[g:g + T * tb], oracle.fp4_segment_reduce(w_ref, n)), (R, n, dt)
    assert qr.qr_wait_timeouts() == 0


def test_twoshot_in_place():
    n = 2048 * 33 + 5
    xs = _rand(4, n, 1, 5)
    y_ref = oracle.fp4_allreduce(1, xs)
    xs_dev = [to_dev(x, 1) for x in xs]
    qr.qr_fp4_allreduce_twoshot(xs_dev, ys=xs_dev)
    torch.cuda.synchronize()
    for j in range(4):
        assert np.array_equal(to_host_u16(xs_dev[j]), y_ref)


def test_c1_crafted_blocks():
    _check_all(workloads.ranks(workloads.C1), 0, "c1")


def test_c2_decode_step():
    _check_all(workloads.ranks(workloads.C2), 1, "c2")


def test_c3_prefill():
    _check_all(workloads.ranks(workloads.C3), 1, "c3")


@pytest.mark.parametrize("n", [1, 31, 33, 2047, 2048, 2049, 2048 * 5 + 37])
@pytest.mark.parametrize("R", [1, 2, 3, 8])
def test_ragged_sizes(n, R):
    xs = [workloads.sweep_rank(r, n, 1, seed=60 + R) for r in range(R)]
    _check_all(xs, 1, f"n={n} R={R}")


@pytest.mark.parametrize("R", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("dt", [0, 1])
def test_every_rank_count(R, dt):
    xs = [workloads.sweep_rank(r, 4 * 2048 + 300, dt, seed=70 + R) for r in range(R)]
    _check_all(xs, dt, f"R={R} dtype={dt}")


def test_special_blocks():
    """Zero, constant, signed-zero, tie-heavy, saturating (bf16 beyond the
    fp16 scale range) and subnormal-scale blocks in every rank."""
    n = 2048 * 2
    rng = np.random.Generator(np.random.PCG64(80))
    xs = []
    for r in range(4):
        x = (rng.standard_normal(n) * (r + 1)).astype(np.float32)
        x[0:32] = 0.0
        x[32:64] = -0.0
        x[64:96] = 2.5 * (r + 1)                          # constant
        x[96:128] = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0] * 4, np.float32)  # ties at scale 1
        x[128:160] = 1e30 * (r + 1)                       # bf16 only: scale saturates at 65504
        x[160:192] = 3e-7 * rng.standard_normal(32)       # fp16-subnormal scale
        x[224:256] = 1e-12 * rng.standard_normal(32)      # scale underflows to 0: every code 0
        x[192] = -0.0
        xs.append(workloads.to_bits(x, 1))
    _check_all(xs, 1, "special blocks")


def test_staged_grid_sizes_and_in_place():
    R, n = 4, 300 * 2048 + 7
    xs = [workloads.sweep_rank(r, n, 1, seed=90) for r in range(R)]
    y_ref = oracle.fp4_allreduce(1, xs)
    xs_dev = [to_dev(x, 1) for x in xs]
    for ctas in (1, 7, 152, 1000):
        assert np.array_equal(to_host_u16(qr.qr_fp4_allreduce(xs_dev, ctas=ctas)), y_ref), ctas
    wires = [qr.qr_fp4_encode(x) for x in xs_dev]
    red0 = to_host_u8(qr.qr_fp4_segment_reduce(wires, n))
    for ctas in (1, 5, 1000):
        assert np.array_equal(to_host_u8(qr.qr_fp4_segment_reduce(wires, n, ctas=ctas)), red0), ctas
    qr.qr_fp4_segment_reduce(wires, n, out=wires[1])  # in place over an input
    assert np.array_equal(to_host_u8(wires[1]), red0)
    qr.qr_fp4_allreduce(xs_dev, y=xs_dev[2])
    assert np.array_equal(to_host_u16(xs_dev[2]), y_ref)
    assert qr.qr_wait_timeouts() == 0


def test_large_message_sampled():
    """R=8 at 2^26 bf16 values per rank: whole-message equality of the fused
    and unfused GPU outputs, and the oracle on sampled tiles."""
    R, n = 8, 1 << 26
    dev = torch.device("cuda")
    xs = [x.view(torch.bfloat16) for x in workloads.device_sweep(R, n, 1, 5, dev)]
    y = qr.qr_fp4_allreduce(xs)
    red = qr.qr_fp4_segment_reduce([qr.qr_fp4_encode(x) for x in xs], n)
    y_u = qr.qr_fp4_decode(red, n, dtype=torch.bfloat16)
    assert torch.equal(y.view(torch.int16), y_u.view(torch.int16))
    rng = np.random.Generator(np.random.PCG64(91))
    for t in np.unique(np.concatenate([rng.choice(n // 2048, 64, replace=False), [0, n // 2048 - 1]])):
        sl = slice(int(t) * 2048, int(t) * 2048 + 2048)
        xt = [to_host_u16(x[sl]) for x in xs]
        assert np.array_equal(to_host_u16(y[sl]), oracle.fp4_allreduce(1, xt)), int(t)
    assert qr.qr_wait_timeouts() == 0


def test_binding_rejects_wrong_tensors():
    x = torch.zeros(100, dtype=torch.float32, device="cuda")
    with pytest.raises(TypeError):
        qr.qr_fp4_encode(x)
    w = qr.qr_fp4_encode(torch.zeros(100, dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(ValueError):
        qr.qr_fp4_decode(w, 5000)
