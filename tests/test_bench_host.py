"""Host logic of the benchmark that needs no GPU: the kernel-code hash that
ties a committed DRAM-traffic capture to the code it was taken on, the
timing of the CPU oracle used as the CPU baseline, and the keys of the
reference arm's JSON line."""
import json
import time

import pytest


def test_code_only_drops_comments_and_layout():
    import bench
    a = "int f(int x) {  // twice x\n  return 2 * x; /* block\n comment */ }\n"
    b = "int f(int x) {\n    return 2 * x;\n}  // reformatted, new comment\n"
    assert bench._code_only(a) == bench._code_only(b) == "int f(int x) { return 2 * x; }"
    assert bench._code_only("return 2 * x;") != bench._code_only("return 3 * x;")


def test_traffic_capture_is_tied_to_the_kernel_code(tmp_path, monkeypatch):
    import bench
    csrc = tmp_path / "bit_quantized_all_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "k.cuh").write_text("__global__ void k() {}  // v1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "FUSED16_SOURCES", ("k.cuh",))
    h = bench.csrc_hash(("k.cuh",))
    rec = {"kern": {"dram_bytes_per_launch": 1234, "csrc_hash": h, "source": "capture"}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.profiled_traffic("kern") == (1234.0, "capture")
    (csrc / "k.cuh").write_text("// a comment edit only\n__global__ void k() {}\n")
    assert bench.profiled_traffic("kern")[0] == 1234.0
    (csrc / "k.cuh").write_text("__global__ void k() { __syncthreads(); }\n")
    val, why = bench.profiled_traffic("kern")
    assert val is None and "changed" in why
    assert bench.profiled_traffic("other")[0] is None



def test_cpu_sweep_times_the_oracle_on_a_workload():
    import bench
    import oracle
    import workloads
    oracle.build()
    xs = workloads.ranks(workloads.C1)
    gbs, vps, reps, dt, threads = bench._time_oracle(oracle, xs, workloads.FP16, (4, 3), tiles=2, threads=4,
                                                     min_s=0.05)
    assert threads == 2  # one thread per tile at most
    assert reps >= 1 and dt >= 0.05
    assert vps == pytest.approx(reps * 4096 * 2 * 2 / dt)
    assert gbs == pytest.approx(vps * 2 / 1e9)


def test_reference_arm_line_carries_the_contract_keys(monkeypatch, capsys):
    """The reference arm's JSON line: every key the benchmark contract names,
    with its own value repeated as the CPU baseline and the end-to-end figure
    (the inputs and the timed oracle work are stubbed: this checks the line,
    not the oracle)."""
    import argparse

    import bench
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setattr(bench, "host_inputs", lambda *a, **k: [])
    monkeypatch.setattr(bench, "oracle_calibrate", lambda orc, xs, threads: 1e9)  # one tile per step
    def fake_run(orc, xs, tiles, threads, start=0):
        time.sleep(0.002)  # a measurable step
        return tiles

    monkeypatch.setattr(bench, "oracle_run", fake_run)
    bench.run_reference(argparse.Namespace(steps=3, warmup=3, gpus=1))
    line = json.loads(capsys.readouterr().out)
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == "GB/s"
    assert (line["n_gpus"], line["steps"], line["warmup"]) == (1, 3, 3)
    assert line["higher_is_better"] is True and line["vs_baseline"] is None
    assert "workload" in line["config"]
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1 and cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


@pytest.mark.parametrize("tiles, threads, start", [(7, 3, 0), (10, 4, 5), (1, 8, 9), (10, 1, 0), (25, 6, 3)])
def test_oracle_run_counts_the_tiles_it_reduces(monkeypatch, tiles, threads, start):
    """The CPU baseline's work accounting: every tile reported as done was
    reduced once per code width, chunks start where the step left off (modulo
    the message) and none runs past its end."""
    import threading

    import bench
    T = 10
    monkeypatch.setattr(bench, "N", T * 2048)
    seen, lock = [], threading.Lock()

    def fake_tiles(orc, xs, bits, t0, t1):
        assert 0 <= t0 < t1 <= T
        with lock:
            seen.extend((bits, t) for t in range(t0, t1))

    monkeypatch.setattr(bench, "_oracle_tiles", fake_tiles)
    done = bench.oracle_run(None, [], tiles, threads, start=start)
    assert 1 <= done <= tiles
    for bits in bench.BITS:
        got = [t for b, t in seen if b == bits]
        assert len(got) == done  # one reduction per counted tile and width
        if tiles <= T:  # the benchmark never asks for more than the message
            assert len(set(got)) == done
    assert (start % T) in {t for _, t in seen}
