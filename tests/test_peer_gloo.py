"""The per-rank two-shot all-reduce's host protocol (bit_quantized_all_gb300.peer)
as R gloo processes on the CPU.

The GPU calls are replaced by a stand-in with the same methods (ShmOps):
each rank's workspace lives in POSIX shared memory, the handle a rank shares
is the memory's name, and the send / reduce / decode steps move bytes between
the workspaces exactly as include/qr.h lays them out (recv[s] at s*seg
tiles, the gathered wire at R*seg tiles; for the symmetric, the asymmetric
and the FP4 codec), with the oracle doing the quantization arithmetic.  So this checks the protocol itself -- handle
exchange, which rank writes where, the joins between the phases -- end to
end against the oracle's all-reduce, at world sizes 2, 3 and 4, and that a
rank which leaves between steps makes the others fail at their next join
with PeerError instead of reading a half-written workspace.  The kernels
themselves are checked on the GPU (tests/test_gpu_peer.py)."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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


def _codec(bits):
    """The oracle's (recv tile bytes, gathered tile bytes, encode, segment
    reduce, decode) for a codec as bit_quantized_all_gb300.peer names it:
    3/4/6/8, ("fc", bits_rs, bits_ag) or "fp4"."""
    import oracle
    from bit_quantized_all_gb300.peer import codec_of
    c = codec_of(bits)
    if c[0] == "fc":
        rs, ag = c[1], c[2]
        return (oracle.fc_tile_bytes(rs), oracle.fc_tile_bytes(ag), lambda dt, x: oracle.fc_encode(rs, dt, x),
                lambda ws, n: oracle.fc_segment_reduce(rs, ag, ws, n), lambda dt, w, n: oracle.fc_decode(ag, dt, w, n))
    if c[0] == "fp4":
        tb = oracle.fp4_tile_bytes()
        return tb, tb, oracle.fp4_encode, oracle.fp4_segment_reduce, oracle.fp4_decode
    b = c[1]
    tb = oracle.tile_bytes(b)
    return (tb, tb, lambda dt, x: oracle.encode(b, dt, x), lambda ws, n: oracle.segment_reduce(b, ws, n),
            lambda dt, w, n: oracle.decode(b, dt, w, n))


def _allreduce_ref(bits, dtype, xs):
    import oracle
    if bits == "fp4":
        return oracle.fp4_allreduce(dtype, xs)
    if isinstance(bits, tuple):
        return oracle.fc_allreduce(bits[1], bits[2], dtype, xs)
    return oracle.allreduce(bits, dtype, xs)


class ShmOps:
    """Host stand-ins for the per-rank library calls (see the module docstring)."""

    def __init__(self, inputs, outputs):
        self.mem = {}       # "pointer" -> (SharedMemory, uint8 view)
        self.next = 1 << 40
        self.inputs = inputs    # pointer -> host array of n 16-bit patterns
        self.outputs = outputs  # pointer -> filled by decode

    @staticmethod
    def _seg(R, n):
        T = -(-n // 2048)
        return T, -(-T // R)

    def workspace_bytes(self, bits, R, n):
        tbi, tbo = _codec(bits)[:2]
        T, seg = self._seg(R, n)
        return R * seg * (tbi + tbo)

    def _register(self, shm):
        p = self.next
        self.next += 1 << 32
        self.mem[p] = (shm, np.ndarray(shm.size, dtype=np.uint8, buffer=shm.buf))
        return p

    def alloc(self, nbytes):
        from multiprocessing import shared_memory
        shm = shared_memory.SharedMemory(create=True, size=nbytes)
        self.owned = shm
        return shm, self._register(shm)

    def get_handle(self, ptr):
        return self.mem[ptr][0].name.encode()

    def open_handle(self, handle):
        from multiprocessing import shared_memory
        return self._register(shared_memory.SharedMemory(name=handle.decode()))

    def close_handle(self, ptr):
        shm, _ = self.mem.pop(ptr)
        shm.close()

    def send(self, bits, dtype, R, rank, x_ptr, n, peers, stream):
        tb, _, encode, _, _ = _codec(bits)
        T, seg = self._seg(R, n)
        wire = encode(dtype, self.inputs[x_ptr])
        for k in range(R):
            t0, t1 = k * seg, min(T, (k + 1) * seg)
            if t0 < t1:
                self.mem[peers[k]][1][rank * seg * tb: (rank * seg + t1 - t0) * tb] = wire[t0 * tb: t1 * tb]

    def reduce(self, bits, R, rank, n, peers, stream):
        tb, tbo, _, segment_reduce, _ = _codec(bits)
        T, seg = self._seg(R, n)
        t0, t1 = rank * seg, min(T, (rank + 1) * seg)
        if t0 >= t1:
            return
        own = self.mem[peers[rank]][1]
        copies = [own[s * seg * tb: (s * seg + t1 - t0) * tb].copy() for s in range(R)]
        n_seg = min(n, t1 * 2048) - t0 * 2048
        red = segment_reduce(copies, n_seg)
        for j in range(R):
            g = R * seg * tb
            self.mem[peers[j]][1][g + t0 * tbo: g + t1 * tbo] = red

    def decode(self, bits, dtype, R, n, ws_ptr, y_ptr, stream):
        tb, tbo, _, _, decode = _codec(bits)
        T, seg = self._seg(R, n)
        g = R * seg * tb
        self.outputs[y_ptr] = decode(dtype, self.mem[ws_ptr][1][g: g + T * tbo].copy(), n)

    def stream(self, stream=None):
        return None

    def synchronize(self, stream):
        pass

    def release(self):
        for p in list(self.mem):
            self.close_handle(p)
        self.owned.unlink()


def _worker(rank, world, port, cases, leave_after, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import oracle
    from bit_quantized_all_gb300.peer import PeerError, PeerTwoShot, init_group
    oracle.build()
    group = init_group(rank, world, port, timeout_s=20.0)
    try:
        for ci, (bits, n, dtype) in enumerate(cases):
            inputs, outputs = {}, {}
            ops = ShmOps(inputs, outputs)
            peer = PeerTwoShot(bits, n, dtype, group=group, ops=ops)
            for step in range(2):
                if leave_after is not None and rank == world - 1 and step == leave_after:
                    q.put((rank, ci, step, "left"))
                    q.close()
                    q.join_thread()  # the report reaches the parent before the process ends
                    ops.release()
                    os._exit(0)  # between steps, nothing in flight
                xs = _inputs(world, n, dtype, 1000 * ci + 10 * step + 7)
                inputs[1], outputs[2] = xs[rank], None
                try:
                    peer.allreduce(1, 2)
                except PeerError as e:
                    q.put((rank, ci, step, f"peer error: {e}"))
                    ops.release()
                    return
                ref = _allreduce_ref(bits, dtype, xs)
                q.put((rank, ci, step, "ok" if np.array_equal(outputs[2], ref) else "MISMATCH"))
            peer.close()
            ops.release()
    finally:
        try:
            dist.destroy_process_group()
        except Exception:  # noqa: BLE001
            pass


def _mismatch_worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import oracle
    from bit_quantized_all_gb300.peer import PeerTwoShot, init_group
    oracle.build()
    group = init_group(rank, world, port, timeout_s=20.0)
    try:
        ops = ShmOps({}, {})
        try:
            PeerTwoShot(4, 2048 * (3 + rank), 1, group=group, ops=ops)  # every rank a different n
            q.put((rank, "constructed"))
        except ValueError as e:
            q.put((rank, f"refused: {e}"))
        q.put((rank, f"allocated={hasattr(ops, 'owned')}"))
    finally:
        dist.destroy_process_group()


def test_ranks_that_disagree_on_the_shape_are_refused_before_any_mapping():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_mismatch_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    out = []
    while not q.empty():
        out.append(q.get())
    assert len(out) == 2 * world, out
    assert all(m.startswith("refused") or m == "allocated=False" for _, m in out), out


def _run(world, cases, leave_after=None):
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, cases, leave_after, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    alive = [p for p in procs if p.is_alive()]
    for p in alive:
        p.kill()
    out = []
    while not q.empty():
        out.append(q.get())
    assert not alive, f"{len(alive)} rank processes did not finish"
    return out


@pytest.mark.parametrize("world", [2, 3, 4])
def test_every_rank_gets_the_oracle_allreduce(world):
    cases = [(4, 2048 * 5 + 37, 1), (3, 2048 * 2, 0), (8, 100, 1),  # the last: fewer tiles than ranks
             (("fc", 4, 8), 2048 * 4 + 9, 1), ("fp4", 2048 * 3 + 16, 0)]
    res = _run(world, cases)
    assert len(res) == world * len(cases) * 2, res
    assert all(r[3] == "ok" for r in res), res


def test_a_rank_that_leaves_between_steps_fails_the_next_join():
    world = 3
    res = _run(world, [(4, 2048 * 3 + 5, 1)], leave_after=1)
    by_rank = {}
    for rank, ci, step, what in res:
        by_rank.setdefault(rank, []).append((step, what))
    assert (1, "left") in by_rank[world - 1]
    for rank in range(world - 1):
        steps = dict(by_rank[rank])
        assert steps[0] == "ok", by_rank
        assert steps[1].startswith("peer error"), by_rank


def test_codec_names():
    """How the per-rank calls name a codec: a width, ("fc", rs, ag) or "fp4"."""
    from bit_quantized_all_gb300.peer import codec_of
    assert codec_of(4) == ("qr", 4) and codec_of(np.int64(3)) == ("qr", 3)
    assert codec_of(("fc", 4, 8)) == ("fc", 4, 8)
    assert codec_of("fp4") == ("fp4",)
    for bad in (True, "int4", ("fc", 4), ("qr", 4, 4), 4.0, None):
        with pytest.raises(ValueError):
            codec_of(bad)
