"""Host-side logic of bench.py on CPU: the N > 1 path (one process per rank, barrier and
max over ranks, here on the gloo backend with world size 2), the reference arm's rank
handling, the JSON helpers and argument checks. No GPU is touched."""
import json
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    w, r, _ = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    dev = torch.device("cpu")
    bench.barrier(dist, dev)
    # each rank "measures" a different time; every rank must see the slowest one
    m = bench.max_over_ranks(dist, 10.0 + 5.0 * r, dev)
    bench.barrier(dist, dev)
    out.put((r, m))
    dist.destroy_process_group()


def test_two_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 15.0), (1, 15.0)]


def test_single_rank_needs_no_process_group(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (1, 0, 0)
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(None, 3.25, torch.device("cpu")) == 3.25
    bench.barrier(None)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main(["--impl", "reference", "--steps", "3", "--warmup", "3", "--gpus", "2"])
    assert capsys.readouterr().out == ""


def test_warmup_below_three_is_rejected():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_traffic_is_null_when_the_kernel_changed(tmp_path, monkeypatch):
    f = tmp_path / "traffic.txt"
    f.write_text("kernel_sources_sha256_16: 0000000000000000\ndram_bytes_per_full_launch: 1.0e9\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.recorded_traffic() == (None, "kernel changed since the ncu capture")
    f.write_text(f"kernel_sources_sha256_16: {bench.kernel_source_hash()}\ndram_bytes_per_full_launch: 1.5e9\n")
    assert bench.recorded_traffic() == (1.5e9, "ncu")


def test_peaks_fall_back_when_measurements_are_missing(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, src = bench.load_peaks()
    assert src == "fallback" and peaks["bf16_tflops"] == 1900.0


def test_end_to_end_figure_counts_every_call_and_its_bytes(monkeypatch):
    """The host-buffer figure: warm-up calls, then three timed batches of `steps` calls, each
    call one whole GEMM with its copies; the bytes per step are the inputs and C."""
    import types
    monkeypatch.setattr(torch.Tensor, "pin_memory", lambda self, *a, **k: self)
    w = types.SimpleNamespace(M=64, N=32, K=16, bias=True, epi_code=1, flops=2 * 64 * 32 * 16)
    calls = []
    g = types.SimpleNamespace(gemm_run_host=lambda *a: calls.append(a))
    host = (torch.zeros(64, 16, dtype=torch.float16), torch.zeros(16, 32, dtype=torch.float16),
            torch.zeros(32, dtype=torch.float16))
    r = bench.measure_e2e(g, None, w, host, None, steps=10)
    assert len(calls) == 3 + 3 * 10
    assert len(r["batches"]) == 3 and r["steps"] == 10
    assert r["h2d_bytes_per_step"] == 2 * (64 * 16 + 16 * 32) + 2 * 32
    assert r["d2h_bytes_per_step"] == 2 * 64 * 32
    assert min(r["batches"]) - 0.1 <= r["value"] <= max(r["batches"]) + 0.1   # batches rounded to 0.1


def test_clock_summary_keeps_only_samples_inside_the_window():
    """The in-process sampler's summary: samples outside [t0, t1] are dropped, the median
    clock, power and the decoded clock-event reasons describe the window only."""
    s = object.__new__(bench.NvmlSampler)
    s.sm_max = 2070.0
    s.power_source = "instant"
    # (t, sm_mhz, power_w, reason_mask, call_us)
    s.samples = [(0.0, 2070.0, 180.0, 0x1, 30.0),              # idle, before the window
                 (1.0, 1740.0, 1350.0, 0x4, 30.0),             # power cap
                 (1.002, 1720.0, 1390.0, 0x4, 30.0),
                 (1.004, 1760.0, 1380.0, 0x4 | 0x8, 30.0),     # + hw slowdown
                 (2.0, 2070.0, 200.0, 0x0, 30.0)]              # after it
    c = s.summary(0.5, 1.5)
    assert c["samples"] == 3 and c["sm_mhz"] == 1740.0 and c["sm_mhz_min"] == 1720.0
    assert c["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert c["power_w_median"] == 1380.0 and c["power_w_max"] == 1390.0
    assert c["sm_max_mhz"] == 2070.0 and c["in_timed_region"]
    assert s.summary(3.0, 4.0)["samples"] == 0


def test_benchmark_output_is_checked_against_the_oracle_rows():
    """The CPU-baseline leg times the oracle on seeded rows and checks the benchmark's own
    output on exactly those rows. Here the 'GPU output' is the oracle's full result: the
    check passes; with one element moved by 0.05 (beyond 1e-2 + 4e-3|ref| for |ref| < 10) it
    reports one violation."""
    import numpy as np
    import oracle
    from tensor_core_gemm_tcgen05_gb300 import inputs
    w = inputs.Workload("tiny", 96, 64, 32, "gelu", True, sample_rows=16, include_last=2)
    A, B, bias = inputs.make_inputs(w)
    full, _, _ = oracle.gemm(A, B, bias, w.epi_code)
    base, parity = bench.cpu_baseline(w, (A, B, bias), target_s=0.01, gpu_out=full)
    assert base["kind"] == "oracle" and parity["ok"] and parity["violations"] == 0
    assert parity["checked_elements"] % w.N == 0
    bad = full.copy()
    bad[-1, 3] = np.float16(float(bad[-1, 3]) + 0.05)   # the last row is always sampled
    _, parity = bench.cpu_baseline(w, (A, B, bias), target_s=0.01, gpu_out=bad)
    assert not parity["ok"] and parity["violations"] == 1


def test_clock_probe_summary_reads_cycles_per_nanosecond():
    """(timer ns, cycles) pairs at 100 us: 1.75 GHz for the first 10 ms, then 2.07 GHz; a
    region of 10 ms sees only the first part; unused (zero) entries are ignored."""
    t, c, rows = 1_000_000, 5_000, []
    for i in range(150):
        rows.append((t, c))
        mhz = 1750.0 if t < 1_000_000 + 10_000_000 else 2070.0
        t += 100_000
        c += int(100_000 * mhz / 1e3)
    rows += [(0, 0)] * 20
    trace = torch.tensor(rows, dtype=torch.int64).reshape(-1)
    s = bench.clock_probe_summary(trace, 10.0)
    assert s["effective_sm_mhz"] == 1750.0 and s["intervals"] == 100 and s["interval_us"] == 100.0
    assert bench.clock_probe_summary(trace, 1e9)["effective_sm_mhz_max"] == 2070.0
