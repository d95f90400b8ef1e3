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
