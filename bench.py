#!/usr/bin/env python
"""Benchmark of the fused quantize -> reduce -> dequantize all-reduce codec.

Workload: the message-size sweep's point R = 8 ranks, 2^27 bf16 values per
rank (256 MiB per rank, 2 GiB of input per call), N(0,1) viewed as rows of
4096 channels with 8 seeded outlier channels x20.
One step = one fused qr_allreduce at INT4 and one at INT3 over the same
inputs (the whole hot path: send-path quantize, Phase-1B decode + fp32 sum +
re-quantize, Phase-2 decode), two kernel launches.  The inputs (2 GiB) exceed
the 129 MB L2, so no flush is needed between steps.

Metric: input GB/s = R * N * 2 B per call / device time (1 GB = 1e9 B), and the
dominant kernel's fraction of the measured HBM bandwidth, where its bytes are
the algorithmic 2RN + 2N (every input read once, the output written once).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs N independent replicas (one per GPU, launched by torchrun); the
codec has no data-path exchange on one GPU, so there is no collective.
`--impl reference` times the CPU oracle on the host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "fused quant-reduce-dequant input GB/s & % of HBM roofline, R=8, INT4/INT3"
R = 8
N = 1 << 27
DTYPE = workloads.BF16
BITS = (4, 3)
SEED = 5
WORKLOAD = ("sweep point R=8, 2^27 bf16 values per rank (256 MiB/rank, N(0,1) + 8 outlier channels x20), "
            "fused INT4 + INT3 all-reduce per step")
FALLBACK_HBM_GBS = 6800.0


def set_values_per_rank(n: int) -> None:
    global N, WORKLOAD
    if n != N:
        if n <= 0 or n % 2048:
            raise SystemExit("--values-per-rank must be a positive multiple of 2048")
        N = n
        WORKLOAD = f"sweep point R=8, {n} bf16 values per rank (profiling case), fused INT4 + INT3 per step"


def tile_bytes(bits: int) -> int:
    return 256 * bits + 128


def config(extra=None) -> dict:
    c = {"workload": WORKLOAD, "ranks": R, "values_per_rank": N, "storage": "bf16",
         "bits": list(BITS), "data": "synthetic N(0,1) + 8 outlier channels x20, seed 5",
         "l2": "inputs larger than L2 (2 GiB per call vs 129 MB L2): no flush",
         "scaling_mode": "replicas (no data-path exchange on one GPU)"}
    if extra:
        c.update(extra)
    return c


def host_inputs(n: int | None = None) -> list[np.ndarray]:
    n = N if n is None else n
    with cf.ThreadPoolExecutor(min(R, os.cpu_count() or 1)) as ex:
        return list(ex.map(lambda r: workloads.sweep_rank(r, n, DTYPE, SEED), range(R)))


# ---------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------
def _oracle_tiles(orc, xs, bits, t0, t1):
    return orc.allreduce(bits, DTYPE, [x[t0 * 2048: t1 * 2048] for x in xs])


def oracle_run(orc, xs, tiles, threads, start=0):
    """All-reduce `tiles` consecutive tiles (from `start`, wrapping) at every
    bit width, split across `threads` threads (ctypes releases the GIL)."""
    T = N // 2048
    chunks = []
    per = -(-tiles // threads)
    for i in range(threads):
        a = i * per
        b = min(tiles, a + per)
        if a < b:
            chunks.append(((start + a) % T, (start + a) % T + (b - a)))
    chunks = [(a, min(b, T)) for a, b in chunks]

    def work(c):
        for bits in BITS:
            _oracle_tiles(orc, xs, bits, c[0], c[1])

    with cf.ThreadPoolExecutor(len(chunks)) as ex:
        list(ex.map(work, chunks))
    return sum(b - a for a, b in chunks)


def oracle_calibrate(orc, xs, threads) -> float:
    """Seconds of wall time per tile (all ranks, every bit width) on `threads` threads."""
    tiles = 4 * threads
    oracle_run(orc, xs, tiles, threads)
    t = time.perf_counter()
    done = oracle_run(orc, xs, tiles, threads, start=tiles)
    return (time.perf_counter() - t) / done


def cpu_baseline(xs, budget_s=12.0) -> dict:
    import oracle as orc
    orc.build()
    threads = os.cpu_count() or 1
    per_tile = oracle_calibrate(orc, xs, threads)
    tiles = int(max(threads, min(N // 2048, budget_s / per_tile)))
    t = time.perf_counter()
    done = oracle_run(orc, xs, tiles, threads)
    dt = time.perf_counter() - t
    gbs = done * 2048 * R * 2 * len(BITS) / dt / 1e9
    # the same oracle on one core, on a smaller sample (about 2 s)
    one = int(max(1, min(N // 2048, 2.0 / (per_tile * threads))))
    t = time.perf_counter()
    done1 = oracle_run(orc, xs, one, 1)
    dt1 = time.perf_counter() - t
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"first {done} of {N // 2048} tiles of every rank, INT4 and INT3, "
                      f"{threads} threads, {dt:.1f} s wall",
            "single_thread": {"value": round(done1 * 2048 * R * 2 * len(BITS) / dt1 / 1e9, 4), "unit": "GB/s",
                              "sample": f"first {done1} tiles of every rank, INT4 and INT3, 1 thread, "
                                        f"{dt1:.1f} s"}}


def _time_oracle(orc, xs, dtype, bits_list, tiles, threads, min_s=2.0, codec="qr"):
    """Input GB/s and values/s of the oracle's all-reduce over the first
    `tiles` tiles of every rank (every width in `bits_list`: a width for the
    symmetric codec, a (reduce-scatter, all-gather) pair for the asymmetric
    one, ignored for FP4), on `threads` threads each taking a contiguous
    share of the tiles, repeated until `min_s` seconds have passed."""
    if codec == "qr":
        def allreduce(b, part):
            orc.allreduce(b, dtype, part)
    elif codec == "fc":
        def allreduce(b, part):
            orc.fc_allreduce(b[0], b[1], dtype, part)
    else:
        def allreduce(b, part):
            orc.fp4_allreduce(dtype, part)
    R_ = len(xs)
    n = min(tiles * 2048, xs[0].size)
    per = -(-tiles // threads)
    spans = [(a * 2048, min(n, (a + per) * 2048)) for a in range(0, tiles, per)]
    spans = [sp for sp in spans if sp[0] < sp[1]]

    def work(sp):
        for b in bits_list:
            allreduce(b, [x[sp[0]:sp[1]] for x in xs])

    reps, t = 0, time.perf_counter()
    with cf.ThreadPoolExecutor(len(spans)) as ex:
        while True:
            list(ex.map(work, spans))
            reps += 1
            dt = time.perf_counter() - t
            if dt >= min_s:
                break
    values = reps * n * R_ * len(bits_list)
    return values * 2 / dt / 1e9, values / dt, reps, dt, len(spans)


def run_cpu_sweep(args) -> None:
    """The oracle as a CPU baseline on every workload, on one thread and on
    all the host's cores: one JSON line per (workload, threads).  Large
    workloads are timed on a prefix sample of their tiles (the oracle's cost
    per tile does not depend on where the tile is); the sample is drawn with
    the workload's own seeds, so it is the workload's first tiles."""
    import oracle as orc
    orc.build()
    cores = os.cpu_count() or 1
    W = workloads
    cases = [
        ("c1: R=2, 4096 fp16 values per rank, crafted blocks", W.C1, None, None),
        ("c2: R=4, 16x8192 bf16 decode-step activation", W.C2, None, None),
        ("c3: R=8, 1024x5120 bf16 prefill activation, Student-t", W.C3, None, None),
        ("c4: R=4, 32x1024x4096 fp16, N(0, 0.5)", W.C4, 4096, None),
        ("sweep: R=8, 2^27 bf16 values per rank (256 MiB)", dict(R=8, N=1 << 27, dtype=W.BF16, bits=(4, 3)),
         4096, 5),
        ("sweep: R=8, 2^29 bf16 values per rank (1 GiB)", dict(R=8, N=1 << 29, dtype=W.BF16, bits=(4, 3)),
         4096, 5),
        ("fc sweep: R=8, 2^27 bf16 values per rank, asymmetric group-128 codec",
         dict(R=8, N=1 << 27, dtype=W.BF16, bits=((4, 4), (4, 8), (8, 8))), 4096, 5, "fc"),
        ("fp4 sweep: R=8, 2^27 bf16 values per rank, E2M1 codec", dict(R=8, N=1 << 27, dtype=W.BF16, bits=(4,)),
         4096, 5, "fp4"),
    ]
    for name, cfg, sample_tiles, seed, *rest in cases:
        codec = rest[0] if rest else "qr"
        T = cfg["N"] // 2048 if cfg["N"] % 2048 == 0 else cfg["N"] // 2048 + 1
        tiles = T if sample_tiles is None else min(T, sample_tiles)
        if seed is None and sample_tiles is None:
            xs = W.ranks(cfg)
        elif seed is None:  # c4: the first tiles of each rank's draw
            xs = [W.c4_rank(r)[:tiles * 2048] for r in range(cfg["R"])]
        else:
            xs = [W.sweep_rank(r, tiles * 2048, cfg["dtype"], seed) for r in range(cfg["R"])]
        for threads in (1, cores):
            gbs, vps, reps, dt, used = _time_oracle(orc, xs, cfg["dtype"], cfg["bits"], tiles, threads, codec=codec)
            print(json.dumps({"cpu_sweep": name, "codec": codec, "R": cfg["R"], "values_per_rank": cfg["N"],
                              "bits": list(cfg["bits"]), "threads": used, "cores": cores,
                              "input_gbs": round(gbs, 4), "values_per_s": round(vps, 1),
                              "sample": f"{'all' if tiles == T else 'first'} {tiles} of {T} tiles per rank, "
                                        f"every width, {reps} passes in {dt:.1f} s",
                              "kind": "oracle"}), flush=True)


def run_reference(args) -> None:
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle as orc
    orc.build()
    xs = host_inputs()
    threads = os.cpu_count() or 1
    per_tile = oracle_calibrate(orc, xs, threads)
    budget_s = 150.0
    step_tiles = int(max(1, min(N // 2048, budget_s / (args.steps + args.warmup) / per_tile)))
    pos = 0
    for _ in range(args.warmup):
        pos += oracle_run(orc, xs, step_tiles, min(threads, step_tiles), start=pos)
    t = time.perf_counter()
    done = 0
    for _ in range(args.steps):
        k = oracle_run(orc, xs, step_tiles, min(threads, step_tiles), start=pos)
        pos += k
        done += k
    dt = time.perf_counter() - t
    gbs = done * 2048 * R * 2 * len(BITS) / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config(),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{step_tiles} consecutive tiles of every rank per step (of {N // 2048}), "
                                   f"INT4 and INT3, {threads} threads"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.proc = None
        self.out = None
        self.gpu_id = gpu_id

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [[c.strip() for c in ln.split(",")] for ln in out.splitlines() if ln.count(",") >= 7]
        if not rows:
            return None
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        smax = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((float(r[2]) for r in rows if r[2].replace(".", "").isdigit()), default=None)}


def _gpu_uuid(torch, dev) -> str | None:
    try:
        u = torch.cuda.get_device_properties(dev).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except (AttributeError, AssertionError, RuntimeError):  # no uuid property, or no such device
        return None


# ---------------------------------------------------------------------------
# replicas: every rank runs the whole workload on its own GPU; the job's time
# is the slowest rank's, its throughput the units of all ranks over that time
# ---------------------------------------------------------------------------
def max_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world: int, calls: int, bytes_per_call: int, elapsed_ms: float) -> float:
    return world * calls * bytes_per_call / (elapsed_ms / 1e3) / 1e9


# ---------------------------------------------------------------------------
# roofline helpers
# ---------------------------------------------------------------------------
def measured_hbm() -> tuple[float, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured (MEASURED_PEAKS.json hbm_gbs: copy bandwidth)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, one earlier GB300 measurement)"


# The sources that determine the benchmarked kernel's code and launch shape.
FUSED16_SOURCES = ("qr_device.cuh", "qr_kernels.cuh", "qr_pipeline.cuh", "qr_staged.cuh", "qr_allreduce16.cuh",
                   "qr_allreduce16_b3.cu", "qr_allreduce16_b4.cu", "qr_allreduce.cu", "qr_grid.cu", "qr_launch.h")


def _code_only(src: str) -> str:
    """C/CUDA source without comments and with whitespace collapsed, so that a
    comment edit does not make a capture of unchanged code look stale."""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def csrc_hash(files=None) -> str:
    h = hashlib.sha256()
    d = os.path.join(ROOT, "bit_quantized_all_gb300", "csrc")
    for f in sorted(FUSED16_SOURCES if files is None else files):
        with open(os.path.join(d, f), encoding="utf-8") as fh:
            h.update(f.encode() + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str) -> tuple[float | None, str]:
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if it
    was taken on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None, "no ncu capture committed"
    e = d.get(kernel)
    if not e:
        return None, f"no ncu capture of {kernel}"
    if e.get("csrc_hash") != csrc_hash():
        return None, "kernel sources changed since the ncu capture"
    return float(e["dram_bytes_per_launch"]), e.get("source", "profiles/traffic.json")


# ---------------------------------------------------------------------------
# message-size sweep (not the headline line): fused and unfused arms
# interleaved, median of `reps` launches, L2 flushed between launches when a
# point's bytes are below 512 MiB
# ---------------------------------------------------------------------------
SWEEP_SIZES = [1 << 14, 1 << 16, 1 << 18, 1 << 20, (1 << 20) + 37, 1 << 22, 1 << 24, 1 << 26, 1 << 27,
               1 << 28, 1 << 29, 1 << 30]


def run_sweep(args) -> None:
    import torch

    from bit_quantized_all_gb300 import build
    build.build()
    import bit_quantized_all_gb300 as qr

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    peak, peak_src = measured_hbm()
    flush = L2Flush(dev)
    sizes = [int(v) for v in args.sweep_sizes.split(",")] if args.sweep_sizes else SWEEP_SIZES
    dtypes = [{"fp16": workloads.FP16, "bf16": workloads.BF16}[d] for d in args.sweep_dtypes.split(",")]
    ranks = [int(r) for r in args.sweep_R.split(",")]
    widths = [int(b) for b in args.sweep_bits.split(",")]
    from bit_quantized_all_gb300.peer import CudaPeerOps, twoshot_peer_local
    if args.sweep_codec == "fc":
        run_sweep_fc(args, qr, dev, peak, flush, sizes, dtypes, ranks)
        return
    if args.sweep_codec == "fp4":
        run_sweep_fp4(args, qr, dev, peak, flush, sizes, dtypes, ranks)
        return
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    for dtype in dtypes:
        tdt = torch.float16 if dtype == workloads.FP16 else torch.bfloat16
        for Rs in ranks:
            for n in sizes:
                xs = [x.view(tdt) for x in workloads.device_sweep(Rs, n, dtype, seed=SEED, device=dev)]
                y = torch.empty(n, dtype=tdt, device=dev)
                y2 = torch.empty(n, dtype=tdt, device=dev)
                for bits in widths:
                    W = qr.qr_wire_bytes(bits, n)
                    wires = [torch.empty(W, dtype=torch.uint8, device=dev) for _ in range(Rs)]
                    red = torch.empty(W, dtype=torch.uint8, device=dev)
                    yu = torch.empty(n, dtype=tdt, device=dev)
                    fused_b = 2 * Rs * n + 2 * n
                    unf_b = fused_b + 2 * (Rs + 1) * W
                    do_flush = fused_b < (512 << 20)

                    def fused():
                        qr.qr_allreduce(bits, xs, y=y)

                    def unfused():
                        for r in range(Rs):
                            qr.qr_encode(bits, xs[r], wire=wires[r])
                        qr.qr_segment_reduce(bits, wires, n, out=red)
                        qr.qr_decode(bits, red, n, y=yu)

                    def encode_all():
                        for r in range(Rs):
                            qr.qr_encode(bits, xs[r], wire=wires[r])

                    def reduce_only():
                        qr.qr_segment_reduce(bits, wires, n, out=red)

                    def decode_only():
                        qr.qr_decode(bits, red, n, y=yu)

                    ws = torch.empty(qr.qr_twoshot_workspace_bytes(bits, Rs, n), dtype=torch.uint8, device=dev)
                    ys2 = [torch.empty(n, dtype=tdt, device=dev) for _ in range(Rs)]

                    def twoshot():
                        qr.qr_allreduce_twoshot(bits, xs, ys=ys2, workspace=ws)

                    wsf = torch.empty(qr.lib().qr_twoshot_flags_workspace_bytes(bits, Rs, n), dtype=torch.uint8,
                                      device=dev)
                    ys3 = [torch.empty(n, dtype=tdt, device=dev) for _ in range(Rs)]

                    def twoshot_flags():  # one cooperative launch, phases joined by per-tile flags
                        qr.qr_allreduce_twoshot(bits, xs, ys=ys3, workspace=wsf, flags=True)

                    # the per-rank two-shot (qr_twoshot_peer_*), every rank's calls
                    # issued from this process: R sends, R owner reductions, R decodes
                    wsp = [torch.empty(CudaPeerOps(dev).workspace_bytes(bits, Rs, n), dtype=torch.uint8, device=dev)
                           for _ in range(Rs)]
                    ys4 = [torch.empty(n, dtype=tdt, device=dev) for _ in range(Rs)]

                    def twoshot_peer():
                        twoshot_peer_local(bits, xs, ys=ys4, workspaces=wsp)

                    regs_ctas = 4 * 4 * sms  # forces the register-fed fused kernel (four waves)

                    def fused_regs():
                        qr.qr_allreduce(bits, xs, y=y2, ctas=regs_ctas)

                    arms = (("fused", fused), ("fused_regs", fused_regs), ("unfused", unfused),
                            ("encode", encode_all), ("reduce", reduce_only), ("decode", decode_only),
                            ("twoshot", twoshot), ("twoshot_flags", twoshot_flags), ("twoshot_peer", twoshot_peer))
                    times = time_arms(arms, args, flush if do_flush else None,
                                      warm=(fused, fused_regs, unfused, twoshot, twoshot_flags, twoshot_peer))
                    same = bool(torch.equal(y.view(torch.int16), yu.view(torch.int16))) and bool(
                        torch.equal(y.view(torch.int16), y2.view(torch.int16))) and all(
                        torch.equal(y.view(torch.int16), v.view(torch.int16)) for v in ys2 + ys3 + ys4)
                    # two-shot: R sends (2N in, W out each), R*W + W for the owners'
                    # reductions, R decodes (W in, 2N out each); the per-rank
                    # two-shot's owners store their reduced segment into all R
                    # workspaces (R*W + R*W) and every rank decodes its own copy
                    kernel_b = {"fused": fused_b, "fused_regs": fused_b, "unfused": unf_b, "encode": Rs * (2 * n + W),
                                "reduce": (Rs + 1) * W, "decode": W + 2 * n,
                                "twoshot": 4 * Rs * n + (3 * Rs + 1) * W, "twoshot_flags": 4 * Rs * n + (3 * Rs + 1) * W,
                                "twoshot_peer": 4 * Rs * n + 4 * Rs * W}
                    for name, alg in kernel_b.items():
                        if not times[name]:
                            print(json.dumps({"sweep": name, "R": Rs, "values_per_rank": n, "bits": bits,
                                              "not_captured": True}), flush=True)
                            continue
                        med = statistics.median(times[name])
                        print(json.dumps({
                            "sweep": name, "R": Rs, "values_per_rank": n, "storage": "fp16" if dtype == 0 else "bf16",
                            "bits": bits, "median_ms": round(med, 5),
                            "input_gbs": round(Rs * n * 2 / (med / 1e3) / 1e9, 2),
                            "alg_gbs": round(alg / (med / 1e3) / 1e9, 2),
                            "frac": round(alg / (med / 1e3) / 1e9 / peak, 4),
                            "l2_flushed": do_flush, "l2_flush": "write then read 256 MiB" if do_flush else None, "fused_equals_unfused": same, "reps": args.reps,
                            "burst": 1 if do_flush else args.burst, "graph": bool(args.graph)}), flush=True)
                    del wires, red, yu, ws, ys2, wsf, ys3, wsp, ys4
                del xs, y
                torch.cuda.empty_cache()


class L2Flush:
    """Evicts the L2 (129 MB) between timed samples: writes one 256 MiB buffer,
    then reads another.  The read leaves the L2 holding clean lines, so the
    next timed kernel does not pay for writing back the flush's dirty lines
    (up to 129 MB, ~19 us of HBM time, which would be charged to a kernel
    that only reads tens of MB)."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.ones(256 << 20, dtype=torch.uint8, device=dev)

    def __call__(self) -> None:
        self.w.fill_(1)
        self.r.sum()


def time_arms(arms, args, flush, warm=()):
    """Per-arm CUDA-event times (ms per launch sequence), arms interleaved.
    Before each sample the GPU is given work that outlasts the host's
    enqueueing of the sample's first call (the L2 eviction, else a short
    sleep kernel), so the events bracket device time only.
    With `flush` (an L2Flush) the L2 is evicted before every timed sample
    and each sample is one launch sequence; without it each
    sample is `args.burst` back-to-back sequences of the same arm (their mean),
    which keeps a kernel's shared-memory configuration from being switched
    by the other arms between launches."""
    import torch

    for _ in range(3):
        for fn in warm:
            fn()
    times = {name: [] for name, _ in arms}
    burst = 1 if flush is not None else max(1, args.burst)
    graphs = {}
    if getattr(args, "graph", False):
        # each arm's `burst` calls captured once and replayed: the time is the
        # GPU's alone, without the host's per-call overhead
        side = torch.cuda.Stream()
        for name, fn in arms:
            fn()  # first use of every kernel on this device happens outside the capture
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            try:
                side.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(side):
                    with torch.cuda.graph(g, stream=side):
                        for _ in range(burst):
                            fn()
                torch.cuda.synchronize()
                graphs[name] = g
            except RuntimeError:
                torch.cuda.synchronize()
                graphs[name] = None
    for _ in range(args.reps):
        for name, fn in arms:
            if graphs and graphs[name] is None:
                continue
            if flush is not None:
                flush()
            else:
                # keep the GPU busy while the host enqueues the sample's first
                # call, so that the timed interval holds device work only
                torch.cuda._sleep(1 << 18)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            if graphs:
                graphs[name].replay()
            else:
                for _ in range(burst):
                    fn()
            e1.record()
            e1.synchronize()
            times[name].append(e0.elapsed_time(e1) / burst)
    return times


def run_sweep_fc(args, qr, dev, peak, flush, sizes, dtypes, ranks) -> None:
    """The sweep for the Flash Communication codec: width pairs (4,4), (4,8)
    (the mixed "INT6") and (8,8), fused and unfused arms interleaved."""
    import torch

    from bit_quantized_all_gb300.peer import CudaPeerOps, twoshot_peer_local

    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    for dtype in dtypes:
        tdt = torch.float16 if dtype == workloads.FP16 else torch.bfloat16
        for Rs in ranks:
            for n in sizes:
                xs = [x.view(tdt) for x in workloads.device_sweep(Rs, n, dtype, seed=SEED, device=dev)]
                y = torch.empty(n, dtype=tdt, device=dev)
                yu = torch.empty(n, dtype=tdt, device=dev)
                y2 = torch.empty(n, dtype=tdt, device=dev)
                for brs, bag in qr.FC_PAIRS:
                    Wi, Wo = qr.qr_fc_wire_bytes(brs, n), qr.qr_fc_wire_bytes(bag, n)
                    wires = [torch.empty(Wi, dtype=torch.uint8, device=dev) for _ in range(Rs)]
                    red = torch.empty(Wo, dtype=torch.uint8, device=dev)
                    red2 = torch.empty(Wo, dtype=torch.uint8, device=dev)
                    fused_b = 2 * Rs * n + 2 * n
                    kernel_b = {"fused": fused_b, "fused_regs": fused_b, "unfused": fused_b + 2 * Rs * Wi + 2 * Wo,
                                "encode": Rs * (2 * n + Wi), "reduce": Rs * Wi + Wo,
                                "reduce_staged": Rs * Wi + Wo, "decode": Wo + 2 * n,
                                # R sends (2N in, Wi out), the owners' R*Wi in and Wo
                                # out, R decodes (Wo in, 2N out)
                                "twoshot": 4 * Rs * n + 2 * Rs * Wi + (Rs + 1) * Wo,
                                # the per-rank calls: R sends, R owners reading R*Wi
                                # and storing their segment into R workspaces, R decodes
                                "twoshot_peer": 4 * Rs * n + 2 * Rs * Wi + 2 * Rs * Wo}
                    do_flush = fused_b < (512 << 20)
                    wst = torch.empty(qr.qr_fc_twoshot_workspace_bytes(brs, bag, Rs, n), dtype=torch.uint8,
                                      device=dev)
                    yst = [torch.empty(n, dtype=tdt, device=dev) for _ in range(Rs)]
                    codec = ("fc", brs, bag)
                    wsp = [torch.empty(CudaPeerOps(dev).workspace_bytes(codec, Rs, n), dtype=torch.uint8, device=dev)
                           for _ in range(Rs)]
                    ysp = [torch.empty(n, dtype=tdt, device=dev) for _ in range(Rs)]

                    def twoshot():
                        qr.qr_fc_allreduce_twoshot(brs, bag, xs, ys=yst, workspace=wst)

                    def twoshot_peer():
                        twoshot_peer_local(codec, xs, ys=ysp, workspaces=wsp)

                    def fused():
                        qr.qr_fc_allreduce(brs, bag, xs, y=y)

                    def fused_regs():  # the register-fed fused kernel (four waves)
                        qr.qr_fc_allreduce(brs, bag, xs, y=y2, ctas=4 * 4 * sms)

                    def encode_all():
                        for r in range(Rs):
                            qr.qr_fc_encode(brs, xs[r], wire=wires[r])

                    def reduce_only():
                        qr.qr_fc_segment_reduce(brs, bag, wires, n, out=red)

                    def reduce_staged():  # the staged Phase-1B kernel at any size
                        qr.qr_fc_segment_reduce(brs, bag, wires, n, out=red2, staged=True)

                    def decode_only():
                        qr.qr_fc_decode(bag, red, n, y=yu)

                    def unfused():
                        encode_all()
                        reduce_only()
                        decode_only()

                    arms = (("fused", fused), ("fused_regs", fused_regs), ("unfused", unfused),
                            ("encode", encode_all), ("reduce", reduce_only), ("reduce_staged", reduce_staged),
                            ("decode", decode_only), ("twoshot", twoshot), ("twoshot_peer", twoshot_peer))
                    times = time_arms(arms, args, flush if do_flush else None,
                                      warm=(fused, fused_regs, unfused, reduce_staged, twoshot, twoshot_peer))
                    same = bool(torch.equal(y.view(torch.int16), yu.view(torch.int16))) and bool(
                        torch.equal(y.view(torch.int16), y2.view(torch.int16))) and bool(torch.equal(red, red2)) and all(
                        torch.equal(y.view(torch.int16), v.view(torch.int16)) for v in yst + ysp)
                    for name, alg in kernel_b.items():
                        med = statistics.median(times[name])
                        print(json.dumps({
                            "sweep": name, "codec": "fc", "R": Rs, "values_per_rank": n,
                            "storage": "fp16" if dtype == 0 else "bf16", "bits_rs": brs, "bits_ag": bag,
                            "median_ms": round(med, 5), "input_gbs": round(Rs * n * 2 / (med / 1e3) / 1e9, 2),
                            "alg_gbs": round(alg / (med / 1e3) / 1e9, 2),
                            "frac": round(alg / (med / 1e3) / 1e9 / peak, 4),
                            "l2_flushed": do_flush, "l2_flush": "write then read 256 MiB" if do_flush else None, "fused_equals_unfused": same, "reps": args.reps,
                            "burst": 1 if do_flush else args.burst}), flush=True)
                    del wires, red, red2, wst, yst, wsp, ysp
                del xs, y, yu, y2
                torch.cuda.empty_cache()


def run_sweep_fp4(args, qr, dev, peak, flush, sizes, dtypes, ranks) -> None:
    """The sweep for the FP4 codec (the INT4 tile with E2M1 elements): the
    fused kernel and the three unfused steps, interleaved."""
    import torch

    from bit_quantized_all_gb300.peer import CudaPeerOps, twoshot_peer_local

    for dtype in dtypes:
        tdt = torch.float16 if dtype == workloads.FP16 else torch.bfloat16
        for Rs in ranks:
            for n in sizes:
                xs = [x.view(tdt) for x in workloads.device_sweep(Rs, n, dtype, seed=SEED, device=dev)]
                y = torch.empty(n, dtype=tdt, device=dev)
                yu = torch.empty(n, dtype=tdt, device=dev)
                W = qr.qr_fp4_wire_bytes(n)
                wires = [torch.empty(W, dtype=torch.uint8, device=dev) for _ in range(Rs)]
                red = torch.empty(W, dtype=torch.uint8, device=dev)
                fused_b = 2 * Rs * n + 2 * n
                kernel_b = {"fused": fused_b, "unfused": fused_b + 2 * Rs * W + 2 * W,
                            "encode": Rs * (2 * n + W), "reduce": (Rs + 1) * W, "decode": W + 2 * n,
                            "twoshot": 4 * Rs * n + (3 * Rs + 1) * W, "twoshot_peer": 4 * Rs * n + 4 * Rs * W}
                wst = torch.empty(qr.qr_fp4_twoshot_workspace_bytes(Rs, n), dtype=torch.uint8, device=dev)
                yst = [torch.empty(n, dtype=tdt, device=dev) for _ in range(Rs)]
                wsp = [torch.empty(CudaPeerOps(dev).workspace_bytes("fp4", Rs, n), dtype=torch.uint8, device=dev)
                       for _ in range(Rs)]
                ysp = [torch.empty(n, dtype=tdt, device=dev) for _ in range(Rs)]
                do_flush = fused_b < (512 << 20)

                def fused():
                    qr.qr_fp4_allreduce(xs, y=y)

                def encode_all():
                    for r in range(Rs):
                        qr.qr_fp4_encode(xs[r], wire=wires[r])

                def reduce_only():
                    qr.qr_fp4_segment_reduce(wires, n, out=red)

                def decode_only():
                    qr.qr_fp4_decode(red, n, y=yu)

                def unfused():
                    encode_all()
                    reduce_only()
                    decode_only()

                def twoshot():
                    qr.qr_fp4_allreduce_twoshot(xs, ys=yst, workspace=wst)

                def twoshot_peer():
                    twoshot_peer_local("fp4", xs, ys=ysp, workspaces=wsp)

                arms = (("fused", fused), ("unfused", unfused), ("encode", encode_all), ("reduce", reduce_only),
                        ("decode", decode_only), ("twoshot", twoshot), ("twoshot_peer", twoshot_peer))
                times = time_arms(arms, args, flush if do_flush else None, warm=(fused, unfused, twoshot, twoshot_peer))
                same = bool(torch.equal(y.view(torch.int16), yu.view(torch.int16))) and all(
                    torch.equal(y.view(torch.int16), v.view(torch.int16)) for v in yst + ysp)
                for name, alg in kernel_b.items():
                    med = statistics.median(times[name])
                    print(json.dumps({
                        "sweep": name, "codec": "fp4", "R": Rs, "values_per_rank": n,
                        "storage": "fp16" if dtype == 0 else "bf16",
                        "median_ms": round(med, 5), "input_gbs": round(Rs * n * 2 / (med / 1e3) / 1e9, 2),
                        "alg_gbs": round(alg / (med / 1e3) / 1e9, 2),
                        "frac": round(alg / (med / 1e3) / 1e9 / peak, 4),
                        "l2_flushed": do_flush, "l2_flush": "write then read 256 MiB" if do_flush else None,
                        "fused_equals_unfused": same, "reps": args.reps,
                        "burst": 1 if do_flush else args.burst}), flush=True)
                del wires, red, wst, yst, wsp, ysp
                del xs, y, yu
                torch.cuda.empty_cache()


def _graph_times(fn, reps, burst, flush, torch):
    """CUDA-event times (ms per call) of `burst` calls of `fn` captured in one
    CUDA graph and replayed `reps` times; with `flush` the L2 is evicted
    before each replay (each sample then starts on cold data)."""
    fn()  # the first use of each kernel (per-context setup) outside the capture
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for _ in range(burst):
                fn()
    torch.cuda.synchronize()
    out = []
    for _ in range(reps):
        if flush is not None:
            flush()
        else:
            torch.cuda._sleep(1 << 16)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        e1.synchronize()
        out.append(e0.elapsed_time(e1) / burst)
    return out


def run_configs(args) -> None:
    """GPU throughput on the four named workloads (c1..c4 of workloads.py),
    every width each one lists, fused and unfused arms, with the L2 evicted
    before every call (cold: inputs come from HBM) and back to back (warm:
    inputs that fit the 129 MB L2 stay there); GPU time per call from CUDA
    graph replays, so the host's per-call overhead is not in it.  Beside each
    workload, the oracle on the host cores (one thread and all)."""
    import torch

    from bit_quantized_all_gb300 import build
    build.build()
    import bit_quantized_all_gb300 as qr
    import oracle as orc
    orc.build()

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    peak, peak_src = measured_hbm()
    flush = L2Flush(dev)
    cores = os.cpu_count() or 1
    W = workloads
    for cfg in (W.C1, W.C2, W.C3, W.C4):
        Rs, n, dtype = cfg["R"], cfg["N"], cfg["dtype"]
        tdt = torch.float16 if dtype == W.FP16 else torch.bfloat16
        xs_host = W.ranks(cfg)
        xs = [torch.from_numpy(x.view(np.int16)).to(dev).view(tdt) for x in xs_host]
        y = torch.empty(n, dtype=tdt, device=dev)
        yu = torch.empty(n, dtype=tdt, device=dev)
        in_bytes = Rs * n * 2
        for bits in cfg["bits"]:
            Wb = qr.qr_wire_bytes(bits, n)
            wires = [torch.empty(Wb, dtype=torch.uint8, device=dev) for _ in range(Rs)]
            red = torch.empty(Wb, dtype=torch.uint8, device=dev)

            def fused():
                qr.qr_allreduce(bits, xs, y=y)

            def unfused():
                for r in range(Rs):
                    qr.qr_encode(bits, xs[r], wire=wires[r])
                qr.qr_segment_reduce(bits, wires, n, out=red)
                qr.qr_decode(bits, red, n, y=yu)

            alg = {"fused": 2 * Rs * n + 2 * n, "unfused": 2 * Rs * n + 2 * n + 2 * (Rs + 1) * Wb}
            launches = {"fused": 1, "unfused": Rs + 2}
            fused()
            unfused()
            torch.cuda.synchronize()
            same = bool(torch.equal(y.view(torch.int16), yu.view(torch.int16)))
            for name, fn in (("fused", fused), ("unfused", unfused)):
                for l2 in ("cold", "warm"):
                    t = _graph_times(fn, args.reps, 1 if l2 == "cold" else args.burst,
                                     flush if l2 == "cold" else None, torch)
                    med = statistics.median(t)
                    fits = alg[name] <= 129e6
                    print(json.dumps({
                        "config": cfg["name"], "R": Rs, "values_per_rank": n,
                        "storage": "fp16" if dtype == W.FP16 else "bf16", "bits": bits, "arm": name,
                        "launches_per_call": launches[name], "l2": l2,
                        "l2_note": ("evicted before each call (write then read 256 MiB)" if l2 == "cold" else
                                    (f"{args.burst} calls back to back; the call's bytes fit the 129 MB L2"
                                     if fits else f"{args.burst} calls back to back; larger than the L2")),
                        "gpu_us_per_call": round(med * 1e3, 3),
                        "input_gbs": round(in_bytes / (med / 1e3) / 1e9, 2),
                        "alg_bytes": alg[name], "alg_gbs": round(alg[name] / (med / 1e3) / 1e9, 2),
                        "frac_of_hbm": round(alg[name] / (med / 1e3) / 1e9 / peak, 4), "peak_gbs": peak,
                        "peak_source": peak_src, "fused_equals_unfused": same, "reps": args.reps,
                        "timing": "CUDA graph replays, median"}), flush=True)
            del wires, red
        # the oracle on the host cores: the whole workload (c4: its first 2048 tiles)
        T = -(-n // 2048)
        tiles = T if cfg["name"] != "c4" else min(T, 2048)
        for threads in (1, cores):
            gbs, vps, reps, dt, used = _time_oracle(orc, xs_host, dtype, cfg["bits"], tiles, threads, min_s=1.0)
            print(json.dumps({"config": cfg["name"], "arm": "cpu_oracle", "R": Rs, "values_per_rank": n,
                              "bits": list(cfg["bits"]), "threads": used, "cores": cores,
                              "input_gbs": round(gbs, 4), "values_per_s": round(vps, 1),
                              "sample": f"{'all' if tiles == T else 'first'} {tiles} of {T} tiles per rank, "
                                        f"every width, {reps} passes in {dt:.1f} s"}), flush=True)
        del xs, y, yu, xs_host
        torch.cuda.empty_cache()


def run_medium(args) -> None:
    """Medium messages, R = 8, INT4, bf16.  (1) Back to back with every call
    reading HBM: K sets of the inputs (and K outputs) spanning at least
    640 MiB, one CUDA graph of K calls, set k by call k, and the same K
    calls launched one by one on the stream; beside it K device copies of
    9N bytes (the 18N bytes a fused call moves), the size-matched
    bandwidth.  (2) One call after an L2 eviction, for the default launch,
    the register-fed kernel at several CTA counts and the staged kernel at
    several CTA counts."""
    import torch

    from bit_quantized_all_gb300 import build
    build.build()
    import bit_quantized_all_gb300 as qr

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    peak, peak_src = measured_hbm()
    Rm = 8
    sizes = [int(v) for v in args.sweep_sizes.split(",")] if args.sweep_sizes else \
        [1 << 20, 1 << 21, 1 << 22, 5242880, 1 << 23, 1 << 24, 1 << 25]

    def graph_per_call(fns, reps):
        for f in fns:
            f()
        torch.cuda.synchronize()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                for f in fns:
                    f()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            torch.cuda._sleep(1 << 16)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            e1.synchronize()
            ts.append(e0.elapsed_time(e1))
        return statistics.median(ts) / len(fns)

    def stream_per_call(fns, reps):
        # the calls launched one by one on the stream, queued behind a sleep
        # kernel that outlasts their enqueueing, so the events time the device
        for f in fns:
            f()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            torch.cuda._sleep(1 << 22)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for f in fns:
                f()
            e1.record()
            e1.synchronize()
            ts.append(e0.elapsed_time(e1))
        return statistics.median(ts) / len(fns)

    flush = L2Flush(dev)
    for n in sizes:
        K = max(2, -(-(640 << 20) // (2 * Rm * n)))
        base = [x.view(torch.bfloat16) for x in workloads.device_sweep(Rm, n, workloads.BF16, seed=SEED, device=dev)]
        sets = [[b.clone() for b in base] for _ in range(K)]
        ys = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(K)]
        t_f = graph_per_call([(lambda k=k: qr.qr_allreduce(4, sets[k], y=ys[k])) for k in range(K)], args.reps)
        t_s = stream_per_call([(lambda k=k: qr.qr_allreduce(4, sets[k], y=ys[k])) for k in range(K)], args.reps)
        alg = 2 * Rm * n + 2 * n
        src = [torch.empty(alg // 2, dtype=torch.uint8, device=dev) for _ in range(K)]
        dst = [torch.empty(alg // 2, dtype=torch.uint8, device=dev) for _ in range(K)]
        t_c = graph_per_call([(lambda k=k: dst[k].copy_(src[k])) for k in range(K)], args.reps)
        print(json.dumps({"medium": "back_to_back", "R": Rm, "bits": 4, "values_per_rank": n, "rotated_sets": K,
                          "fused_us": round(t_f * 1e3, 2), "fused_frac": round(alg / (t_f / 1e3) / 1e9 / peak, 3),
                          "fused_stream_us": round(t_s * 1e3, 2),
                          "fused_stream_frac": round(alg / (t_s / 1e3) / 1e9 / peak, 3),
                          "copy_of_same_bytes_us": round(t_c * 1e3, 2),
                          "copy_frac": round(alg / (t_c / 1e3) / 1e9 / peak, 3),
                          "fused_over_copy": round(t_c / t_f, 3), "peak_gbs": peak}), flush=True)
        del src, dst, sets
        y = ys[0]
        arms = [("default", lambda: qr.qr_allreduce(4, base, y=y))]
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        for c in (sms // 2, sms, 2 * sms, 3 * sms, 4 * sms):
            arms.append((f"register_fed_{c}", (lambda c=c: qr.qr_allreduce(4, base, y=y, ctas=c))))
        for c in (sms // 2, 3 * sms // 4, sms):
            arms.append((f"staged_{c}", (lambda c=c: qr.qr_allreduce_staged(4, base, y=y, ctas=c))))
        for name, fn in arms:
            med = statistics.median(_graph_times(fn, args.reps, 1, flush, torch))
            print(json.dumps({"medium": "cold_single_call", "R": Rm, "bits": 4, "values_per_rank": n, "arm": name,
                              "us": round(med * 1e3, 2), "frac": round(alg / (med / 1e3) / 1e9 / peak, 3)}),
                  flush=True)
        del base, ys, y
        torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--values-per-rank", type=int, default=N,
                    help="a smaller message for profiling captures (the default is the benchmark workload)")
    ap.add_argument("--sweep", action="store_true",
                    help="run the message-size sweep (JSON line per point) instead of the benchmark")
    ap.add_argument("--sweep-sizes", default="", help="comma-separated values per rank for --sweep")
    ap.add_argument("--reps", type=int, default=100, help="launches per sweep point")
    ap.add_argument("--graph", action="store_true",
                    help="sweep: capture each arm in a CUDA graph and time replays (GPU time without host overhead)")
    ap.add_argument("--burst", type=int, default=1,
                    help="sweep: back-to-back launches of one arm per timed sample where L2 is not flushed")
    ap.add_argument("--cpu-sweep", action="store_true",
                    help="time the CPU oracle on every workload (1 thread and all cores); no GPU")
    ap.add_argument("--medium", action="store_true",
                    help="medium messages (R=8 INT4): back-to-back calls against a copy of the same bytes, "
                         "and single cold calls at several launch shapes")
    ap.add_argument("--configs", action="store_true",
                    help="GPU throughput on the named workloads c1..c4 (every width, fused and unfused, "
                         "cold and warm L2), with the oracle on the host cores beside each")
    ap.add_argument("--sweep-R", default="2,4,8", help="rank counts for --sweep")
    ap.add_argument("--sweep-bits", default="8,6,4,3", help="code widths for --sweep")
    ap.add_argument("--sweep-dtypes", default="fp16,bf16", help="storage types for --sweep")
    ap.add_argument("--sweep-codec", choices=["qr", "fc", "fp4"], default="qr",
                    help="qr: symmetric 32-value blocks; fc: asymmetric groups of 128; fp4: E2M1 blocks")
    args = ap.parse_args()
    if args.sweep:
        run_sweep(args)
        return
    if args.cpu_sweep:
        run_cpu_sweep(args)
        return
    if args.configs:
        run_configs(args)
        return
    if args.medium:
        run_medium(args)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    set_values_per_rank(args.values_per_rank)
    if args.impl == "reference":
        run_reference(args)
        return

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    from bit_quantized_all_gb300 import build
    build.build()
    import bit_quantized_all_gb300 as qr

    xs_host = host_inputs()
    tdt = torch.bfloat16
    pinned = [torch.from_numpy(x.view(np.int16)).pin_memory() for x in xs_host]
    xs = [p.to(dev, non_blocking=True).view(tdt) for p in pinned]
    ys = {b: torch.empty(N, dtype=tdt, device=dev) for b in BITS}
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)

    def step():
        for b in BITS:
            qr.qr_allreduce(b, xs, y=ys[b], stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # ---- device-timed region: K steps, per-launch events on the launching stream
    ev = {b: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)] for b in BITS}
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(_gpu_uuid(torch, dev))
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(args.steps):
        for b in BITS:
            ev[b][i][0].record(stream)
            qr.qr_allreduce(b, xs, y=ys[b], stream=stream)
            ev[b][i][1].record(stream)
    stop.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    elapsed_ms = max_over_ranks(start.elapsed_time(stop), dev)
    in_bytes_call = R * N * 2
    value = whole_job_gbs(world, args.steps * len(BITS), in_bytes_call, elapsed_ms)

    peak, peak_src = measured_hbm()
    kernels = {}
    for b in BITS:
        d = [s.elapsed_time(e) for s, e in ev[b]]
        avg = sum(d) / len(d)
        alg = R * N * 2 + N * 2
        kernels[b] = {"kernel": f"staged_allreduce_kernel<QrTile<{b},bf16>,R={R},G=5,SG=1,K=4>", "launches": len(d),
                      "avg_ms": avg,
                      "median_ms": statistics.median(d), "total_ms": sum(d),
                      "input_gbs": in_bytes_call / (avg / 1e3) / 1e9,
                      "achieved_gbs": alg / (avg / 1e3) / 1e9, "alg_bytes": alg}
    dom = max(BITS, key=lambda b: kernels[b]["total_ms"])
    k = kernels[dom]
    traffic, traffic_src = profiled_traffic(k["kernel"])
    roofline = {"bound": "hbm", "achieved": round(k["achieved_gbs"], 2), "peak": peak, "unit": "GB/s",
                "frac": round(k["achieved_gbs"] / peak, 4), "traffic": traffic,
                "kernel": k["kernel"], "alg_bytes_per_launch": k["alg_bytes"],
                "avg_launch_ms": round(k["avg_ms"], 5), "peak_source": peak_src,
                "traffic_source": traffic_src,
                "all_kernels": {f"INT{b}": {"achieved_gbs": round(kernels[b]["achieved_gbs"], 2),
                                            "frac": round(kernels[b]["achieved_gbs"] / peak, 4),
                                            "input_gbs": round(kernels[b]["input_gbs"], 2),
                                            "avg_ms": round(kernels[b]["avg_ms"], 5),
                                            "median_ms": round(kernels[b]["median_ms"], 5),
                                            "share": round(kernels[b]["total_ms"] /
                                                           sum(kk["total_ms"] for kk in kernels.values()), 4)}
                                for b in BITS}}

    # ---- end to end through the public API: every step copies its R inputs
    # pinned host -> device, runs both all-reduces and copies both results
    # device -> pinned host.  Steps are pipelined two deep on three streams
    # (inputs of step i+1 cross the link while step i computes and its
    # results come back), with two sets of device buffers; the host link,
    # not the copy engines, is the limit (one copy or eight concurrent ones
    # move the same ~210 GB/s host -> device on GB300).
    host_out = {b: torch.empty(N, dtype=tdt).pin_memory() for b in BITS}
    in_sets = [xs, [torch.empty_like(x) for x in xs]]
    out_sets = [ys, {b: torch.empty_like(ys[b]) for b in BITS}]
    h2d_stream, d2h_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_run(steps):
        h2d_stream.wait_stream(stream)
        d2h_stream.wait_stream(stream)
        inputs_free = [None, None]   # compute of the step that last read set k is done
        outputs_free = [None, None]  # results of the step that last wrote set k are home
        for i in range(steps):
            k = i & 1
            with torch.cuda.stream(h2d_stream):
                if inputs_free[k] is not None:
                    h2d_stream.wait_event(inputs_free[k])
                for r in range(R):
                    in_sets[k][r].view(torch.int16).copy_(pinned[r], non_blocking=True)
            stream.wait_stream(h2d_stream)
            if outputs_free[k] is not None:
                stream.wait_event(outputs_free[k])
            for b in BITS:
                qr.qr_allreduce(b, in_sets[k], y=out_sets[k][b], stream=stream)
            inputs_free[k] = torch.cuda.Event()
            inputs_free[k].record(stream)
            d2h_stream.wait_event(inputs_free[k])
            with torch.cuda.stream(d2h_stream):
                for b in BITS:
                    host_out[b].copy_(out_sets[k][b], non_blocking=True)
            outputs_free[k] = torch.cuda.Event()
            outputs_free[k].record(d2h_stream)
        stream.wait_stream(h2d_stream)
        stream.wait_stream(d2h_stream)

    def link_trials(k):
        """Times of k host -> device copies of the R inputs alone (ms each)."""
        out = []
        for _ in range(k):
            l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            l0.record(h2d_stream)
            with torch.cuda.stream(h2d_stream):
                for r in range(R):
                    in_sets[0][r].view(torch.int16).copy_(pinned[r], non_blocking=True)
            l1.record(h2d_stream)
            torch.cuda.synchronize()
            out.append(l0.elapsed_time(l1))
        return out

    e2e = None
    if args.e2e_steps > 0:
        e2e_run(2)
        torch.cuda.synchronize()
        link_ms = link_trials(3)
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_run(args.e2e_steps)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), dev)
        same = all(torch.equal(host_out[b].view(torch.int16), ys[b].view(torch.int16).cpu()) for b in BITS)
        e2e_value = whole_job_gbs(world, args.e2e_steps * len(BITS), in_bytes_call, e2e_ms)
        # the host link alone: the same R inputs copied pinned host -> device
        # with nothing else running (a step can not be faster than this copy),
        # three times before the timed steps and three after; the fastest
        # sets the bound (on one box the copies after the timed steps ran at
        # half the rate the steps themselves had reached)
        link_ms += link_trials(3)
        link_gbs = R * N * 2 / (min(link_ms) / 1e3) / 1e9
        e2e = {"value": round(e2e_value, 2), "unit": "GB/s",
               "h2d_bytes_per_step": R * N * 2, "d2h_bytes_per_step": len(BITS) * N * 2,
               "steps": args.e2e_steps, "gpu_launches": args.e2e_steps * len(BITS),
               "api": "qr_allreduce through the Python binding of the C ABI, pinned host buffers",
               "results_equal_device_timed_results": same,
               "h2d_link_gbs": round(link_gbs, 2),
               "h2d_link_trials_ms": [round(t, 3) for t in link_ms],
               "frac_of_link_bound": round(e2e_value / (world * len(BITS) * link_gbs), 4),
               "link_bound": "each step copies R*N*2 input bytes host -> device once and runs both all-reduces on "
                             "them, so the step takes at least that copy's time: bound = calls per step x link GB/s",
               "pipeline": "two steps in flight: host->device copies, compute and device->host copies "
                           "on three streams, two sets of device buffers"}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(xs_host)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(elapsed_ms / args.steps, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": config(),
            "gpu_launches": args.steps * len(BITS),
            "roofline": roofline,
            "e2e": e2e,
            "clocks": clk,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
