"""The per-rank two-shot all-reduce with the library's kernels, for the
symmetric, the asymmetric (Flash Communication) and the FP4 codec: R
processes on the one GPU, each with its own CUDA context, its own workspace
and its own message, the peers' workspaces mapped through CUDA IPC
(qr_ipc_*), the phases joined by host barriers (no kernel waits on another
process).

Every rank's output equals the oracle's all-reduce of the R messages bit for
bit, and the fused kernel's output in that process; the gathered wire in
every rank's workspace equals the oracle's Phase-1B output byte for byte; two
steps run in a row over the same workspaces with different data; ragged
tails and fewer tiles than ranks are covered.  The same calls on a multi-GPU
node would store across NVLink; that is not measured here."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def lib():
    from bit_quantized_all_gb300 import build
    build.build()
    import oracle
    oracle.build()
    assert torch.cuda.is_available()


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(R, n, dtype, seed):
    import oracle
    rng = np.random.Generator(np.random.PCG64(seed))
    out = []
    for r in range(R):
        v = rng.standard_normal(n).astype(np.float32) * np.float32(1 + r)
        v[rng.integers(0, n, size=max(1, n // 100))] *= 40.0
        out.append(oracle.narrow(dtype, v))
    return out


def _codec_refs(bits, dtype, xs, n, R):
    """The oracle's all-reduce output and gathered (Phase-1B) wire for the
    codec `bits` names (3/4/6/8, ("fc", bits_rs, bits_ag) or "fp4"), with the
    gathered wire's byte offset in a rank's peer workspace and its length."""
    import oracle
    T = -(-n // 2048)
    seg = -(-T // R)
    if bits == "fp4":
        ref = oracle.fp4_allreduce(dtype, xs)
        red = oracle.fp4_segment_reduce([oracle.fp4_encode(dtype, x) for x in xs], n)
        tbi = tbo = oracle.fp4_tile_bytes()
    elif isinstance(bits, tuple):
        _, rs, ag = bits
        ref = oracle.fc_allreduce(rs, ag, dtype, xs)
        red = oracle.fc_segment_reduce(rs, ag, [oracle.fc_encode(rs, dtype, x) for x in xs], n)
        tbi, tbo = oracle.fc_tile_bytes(rs), oracle.fc_tile_bytes(ag)
    else:
        ref = oracle.allreduce(bits, dtype, xs)
        red = oracle.segment_reduce(bits, [oracle.encode(bits, dtype, x) for x in xs], n)
        tbi = tbo = oracle.tile_bytes(bits)
    return ref, red, R * seg * tbi, T * tbo


def _fused(bits, dev):
    """The codec's fused all-reduce of the R device tensors, as host uint16."""
    import bit_quantized_all_gb300 as qr
    if bits == "fp4":
        y = qr.qr_fp4_allreduce(dev)
    elif isinstance(bits, tuple):
        y = qr.qr_fc_allreduce(bits[1], bits[2], dev)
    else:
        y = qr.qr_allreduce(bits, dev)
    return y.view(torch.int16).cpu().numpy().view(np.uint16)


def _worker(rank, world, port, cases, q):
    sys.path.insert(0, ROOT)
    os.environ["PYTORCH_CUDA_ALLOC_CONF"] = "expandable_segments:False"  # IPC needs plain allocations
    import torch
    import torch.distributed as dist
    torch.cuda.set_device(0)
    import bit_quantized_all_gb300 as qr
    from bit_quantized_all_gb300.peer import PeerTwoShot, init_group
    tdt = {0: torch.float16, 1: torch.bfloat16}
    group = init_group(rank, world, port, timeout_s=120.0)
    try:
        for ci, (bits, n, dtype) in enumerate(cases):
            peer = PeerTwoShot(bits, n, dtype, group=group)
            for step in range(2):
                xs = _inputs(world, n, dtype, 1000 * ci + 10 * step + 3)
                dev = [torch.from_numpy(x.view(np.int16)).cuda().view(tdt[dtype]) for x in xs]
                y = peer.allreduce_tensor(dev[rank])
                torch.cuda.synchronize()
                got = y.view(torch.int16).cpu().numpy().view(np.uint16)
                ref, red_ref, g, glen = _codec_refs(bits, dtype, xs, n, world)
                fused = _fused(bits, dev)
                red = peer.workspace[g: g + glen].cpu().numpy()
                status = []
                if not np.array_equal(got, ref):
                    status.append(f"output differs from the oracle at {np.flatnonzero(got != ref)[:5]}")
                if not np.array_equal(got, fused):
                    status.append("output differs from the fused kernel")
                if not np.array_equal(red, red_ref):
                    status.append(f"gathered wire differs at byte {np.flatnonzero(red != red_ref)[:3]}")
                q.put((rank, ci, step, "ok" if not status else "; ".join(status)))
            peer.close()
        q.put((rank, -1, -1, f"timeouts={qr.qr_wait_timeouts()}"))
    except Exception as e:  # noqa: BLE001  (reported to the parent)
        q.put((rank, -2, -2, f"exception: {type(e).__name__}: {e}"))
    finally:
        try:
            dist.destroy_process_group()
        except Exception:  # noqa: BLE001
            pass


def _run(world, cases):
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, cases, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=600)
    alive = [p for p in procs if p.is_alive()]
    for p in alive:
        p.kill()
    out = []
    while not q.empty():
        out.append(q.get())
    assert not alive, f"{len(alive)} rank processes did not finish: {out}"
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    return out


@pytest.mark.parametrize("R", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("bits", [3, 4, 6, 8])
def test_one_process_driving_every_rank(bits, R):
    """The per-rank calls issued for all R ranks from one process on one
    stream (every send, then every reduce, then every decode): every output
    and every gathered wire equals the oracle's, ragged tail included, and
    fewer tiles than ranks at the small size."""
    import oracle
    import bit_quantized_all_gb300 as qr
    from bit_quantized_all_gb300.peer import twoshot_peer_local
    for n in (2048 * 13 + 77, 1500):
        dtype = 1 if bits in (3, 4) else 0
        xs = _inputs(R, n, dtype, 50 * bits + R + n)
        tdt = {0: torch.float16, 1: torch.bfloat16}[dtype]
        dev = [torch.from_numpy(x.view(np.int16)).cuda().view(tdt) for x in xs]
        ys, ws = twoshot_peer_local(bits, dev)
        torch.cuda.synchronize()
        ref = oracle.allreduce(bits, dtype, xs)
        red_ref = oracle.segment_reduce(bits, [oracle.encode(bits, dtype, x) for x in xs], n)
        T = -(-n // 2048)
        seg = -(-T // R)
        tb = qr.qr_tile_bytes(bits)
        for j in range(R):
            got = ys[j].view(torch.int16).cpu().numpy().view(np.uint16)
            assert np.array_equal(got, ref), (bits, R, n, j)
            g = R * seg * tb
            assert np.array_equal(ws[j][g: g + T * tb].cpu().numpy(), red_ref), (bits, R, n, j)
    assert qr.qr_wait_timeouts() == 0


@pytest.mark.parametrize("R", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("codec", [("fc", 4, 4), ("fc", 4, 8), ("fc", 8, 8), "fp4"], ids=["fc44", "fc48", "fc88", "fp4"])
def test_one_process_driving_every_rank_codecs(codec, R):
    """As above for the asymmetric and the FP4 codec: every output equals the
    oracle's all-reduce and the codec's fused kernel, every gathered wire
    the oracle's Phase-1B output, ragged tail and fewer tiles than ranks
    included."""
    import bit_quantized_all_gb300 as qr
    from bit_quantized_all_gb300.peer import twoshot_peer_local
    for n in (2048 * 13 + 77, 1500):
        dtype = (R + n) % 2
        xs = _inputs(R, n, dtype, 7 * R + n + (0 if codec == "fp4" else codec[1] + 3 * codec[2]))
        tdt = {0: torch.float16, 1: torch.bfloat16}[dtype]
        dev = [torch.from_numpy(x.view(np.int16)).cuda().view(tdt) for x in xs]
        ys, ws = twoshot_peer_local(codec, dev)
        torch.cuda.synchronize()
        ref, red_ref, g, glen = _codec_refs(codec, dtype, xs, n, R)
        fused = _fused(codec, dev)
        for j in range(R):
            got = ys[j].view(torch.int16).cpu().numpy().view(np.uint16)
            assert np.array_equal(got, ref), (codec, R, n, j)
            assert np.array_equal(got, fused), (codec, R, n, j)
            assert np.array_equal(ws[j][g: g + glen].cpu().numpy(), red_ref), (codec, R, n, j)
        # the workspaces reused with other data: nothing left over matters
        xs2 = _inputs(R, n, dtype, 99 + R + n)
        dev2 = [torch.from_numpy(x.view(np.int16)).cuda().view(tdt) for x in xs2]
        ys2, _ = twoshot_peer_local(codec, dev2, workspaces=ws)
        ref2 = _codec_refs(codec, dtype, xs2, n, R)[0]
        for j in range(R):
            assert np.array_equal(ys2[j].view(torch.int16).cpu().numpy().view(np.uint16), ref2), (codec, R, n, j)
    assert qr.qr_wait_timeouts() == 0


@pytest.mark.parametrize("world,cases", [
    (2, [(4, 2048 * 40 + 37, 1), (3, 2048 * 9, 0), (8, 2048 * 3 + 1, 1), (6, 100, 0)]),
    (4, [(4, 2048 * 40 + 37, 1), (3, 2048 * 9 + 5, 1), (6, 2048 * 2, 0), (8, 700, 1)]),
    (8, [(4, 2048 * 64 + 11, 1), (3, 2048 * 5, 1)]),
    (2, [(("fc", 4, 8), 2048 * 40 + 37, 1), (("fc", 4, 4), 2048 * 9, 0), ("fp4", 2048 * 3 + 16, 1)]),
    (3, [(("fc", 8, 8), 2048 * 17 + 5, 0), ("fp4", 2048 * 11, 0), (("fc", 4, 8), 1000, 1)]),
    (8, [(("fc", 4, 8), 2048 * 64 + 11, 1), ("fp4", 2048 * 64 + 32, 1)]),
], ids=["R2", "R4", "R8", "codecs-R2", "codecs-R3", "codecs-R8"])
def test_every_rank_matches_the_oracle(world, cases):
    res = _run(world, cases)
    steps = [r for r in res if r[1] >= 0]
    assert len(steps) == world * len(cases) * 2, res
    assert all(r[3] == "ok" for r in steps), [r for r in steps if r[3] != "ok"]
    assert sorted(r[3] for r in res if r[1] == -1) == ["timeouts=0"] * world, res
    assert not [r for r in res if r[1] == -2], res


def _offset_by_16_bytes(x: torch.Tensor) -> torch.Tensor:
    """x's values in a buffer that starts 16 bytes past a 32-byte boundary."""
    buf = torch.empty(x.numel() + 16, dtype=x.dtype, device=x.device)
    v = buf[8: 8 + x.numel()]
    assert v.data_ptr() % 32 == 16
    v.copy_(x)
    return v


@pytest.mark.parametrize("codec", [4, 3, ("fc", 4, 8), ("fc", 8, 8), "fp4"], ids=["int4", "int3", "fc48", "fc88", "fp4"])
def test_sixteen_byte_aligned_inputs_and_outputs(codec):
    """The per-rank calls with every input and output 16 but not 32 bytes
    aligned (the narrower loads and stores): the same outputs as the
    oracle's."""
    from bit_quantized_all_gb300.peer import twoshot_peer_local
    R, n = 5, 2048 * 9 + 333
    xs = _inputs(R, n, 1, 4242)
    dev = [_offset_by_16_bytes(torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)) for x in xs]
    ys = [_offset_by_16_bytes(torch.zeros(n, dtype=torch.bfloat16, device="cuda")) for _ in range(R)]
    twoshot_peer_local(codec, dev, ys=ys)
    torch.cuda.synchronize()
    ref = _codec_refs(codec, 1, xs, n, R)[0]
    for j in range(R):
        assert np.array_equal(ys[j].view(torch.int16).cpu().numpy().view(np.uint16), ref), (codec, j)
