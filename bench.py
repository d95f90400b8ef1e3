"""Benchmark of the GB300 FP16 tensor-core GEMM with fused epilogue.

One step = one pass of the whole path (tile raster, TMA staging, tcgen05 MMA into TMEM,
bias, activation, FP16 store) over one batch: the transformer MLP up-projection
C = GELU_erf(X W + bias) with X 8200 x 4096, W 4096 x 16384 (FP16; the M tail of 8 rows
exercises the masked path), i.e. one launch of the library's kernel. Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the FP64 CPU oracle on the host cores instead (bounded row samples
of the same workload). For N > 1 (torchrun) every rank runs its own replica of the
workload (weak scaling, no collective on the data path); the timed region is bracketed
by a barrier and the slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FP16 GEMM TFLOP/s (fp32 acc, ±bias+GELU) and % of GB300 dense FP16 peak"
WORKLOAD = "mlp_up_8200x4096x16384_bias_gelu"
# Other problems timed briefly in the same run (context lines, not the headline).
SIDE_WORKLOADS = ["gemm_8192", "gemm_8192_bias_gelu", "mlp_up_8200x4096x16384_none",
                  "gemm_2048", "gemm_2048_bias_gelu", "gemm_2048_bias_relu", "gemm_256",
                  "gemm_1024x1024x8192_bias_gelu"]
L2_BYTES = 129 * 2 ** 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = ["tensor_core_gemm_tcgen05_gb300/csrc/gemm_kernel.cuh",
                  "tensor_core_gemm_tcgen05_gb300/csrc/gemm_kernel_pair.cuh",
                  "tensor_core_gemm_tcgen05_gb300/csrc/ptx.cuh",
                  "tensor_core_gemm_tcgen05_gb300/csrc/gemm_api.cu"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "gemm_tcgen05_mlp_traffic.txt")


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ---------------------------------------------------------------------------------------------
# distributed plumbing (torchrun); N = 1 needs none of it
# ---------------------------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(dist, value: float, device) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------------------------------------
# peaks, clocks, traffic
# ---------------------------------------------------------------------------------------------
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clock, power and throttle reasons during the timed region."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"]
        except Exception:
            sel = []
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", *sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception as e:  # no nvidia-smi
            self.proc = None
            self.err = str(e)

    def mark_start(self):
        self.t0 = time.time()

    def mark_stop(self):
        self.t1 = time.time()

    def finish(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "nvidia-smi unavailable"}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts, float(parts[1]), float(parts[2]), parts[3], parts[4:]))
            except Exception:
                continue
        os.unlink(self.path)
        inside = [r for r in rows if self.t0 is not None and self.t0 - 0.05 <= r[0] <= self.t1 + 0.05]
        use = inside if inside else rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["active_mask", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in use:
            for nm, v in zip(names[1:], r[4][1:]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        power = []
        for r in use:
            try:
                power.append(float(r[3]))
            except ValueError:
                pass
        return {
            "sm_mhz": statistics.median(r[1] for r in use),
            "sm_max_mhz": max(r[2] for r in use),
            "reasons": sorted(reasons),
            "samples": len(use),
            "in_timed_region": bool(inside),
            "power_w_median": statistics.median(power) if power else None,
        }


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per launch of the headline kernel from the committed ncu summary, if it
    was taken on the current kernel sources (else None)."""
    if not os.path.exists(TRAFFIC_FILE):
        return None, "no ncu traffic summary committed"
    text = open(TRAFFIC_FILE).read()
    m_hash = re.search(r"kernel_sources_sha256_16:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_full_launch:\s*([0-9.eE+]+)", text)
    if not m_hash or not m_bytes:
        return None, "summary lacks fields"
    if m_hash.group(1) != kernel_source_hash():
        return None, "kernel changed since the ncu capture"
    return float(m_bytes.group(1)), "ncu"


# ---------------------------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------------------------
def time_device(g, ctx, w, dA, dB, dbias, dC, stream, steps, warmup, dist=None, device=None):
    """CUDA-event time of `steps` back-to-back launches (after `warmup`), max over ranks."""
    import torch
    for _ in range(warmup):
        g.gemm_run(ctx, w.M, w.N, w.K, dA, dB, dbias, dC, w.epi_code, stream)
    torch.cuda.synchronize()
    barrier(dist, device)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        g.gemm_run(ctx, w.M, w.N, w.K, dA, dB, dbias, dC, w.epi_code, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    barrier(dist, device)
    return max_over_ranks(dist, ms, device)


def device_buffers(w, device):
    import torch
    from tensor_core_gemm_tcgen05_gb300 import inputs
    A, B, bias = inputs.make_inputs(w)
    dA, dB = A.to(device), B.to(device)
    dbias = bias.to(device) if bias is not None else None
    dC = torch.empty(w.M, w.N, dtype=torch.float16, device=device)
    return (A, B, bias), (dA, dB, dbias, dC)


SOFTMAX_SHAPE = (8192, 16384)   # the MLP output's shape: 268 MB in, 268 MB out


def measure_cublas_context(device, peaks, steps=20):
    """Context only, not part of this library's path: cuBLAS (through torch.matmul) on the
    plain FP16 problems, FP32 accumulation forced, same kind of timing (back-to-back launches
    after warm-up, CUDA events)."""
    import torch
    from tensor_core_gemm_tcgen05_gb300 import inputs
    prev = torch.backends.cuda.matmul.allow_fp16_reduced_precision_reduction
    torch.backends.cuda.matmul.allow_fp16_reduced_precision_reduction = False
    out = {}
    try:
        for name in ("gemm_8192", "mlp_up_8200x4096x16384_none", "gemm_2048"):
            w = inputs.WORKLOADS[name]
            A = torch.randn(w.M, w.K, device=device).half()
            B = torch.randn(w.K, w.N, device=device).half()
            C = torch.empty(w.M, w.N, device=device, dtype=torch.float16)
            n = steps if w.flops > 1e11 else 10 * steps
            for _ in range(5):
                torch.matmul(A, B, out=C)
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(n):
                torch.matmul(A, B, out=C)
            e1.record()
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) / n * 1e3
            tf = w.flops / (us * 1e-6) / 1e12
            out[f"cublas_context_{name}"] = {"tflops": round(tf, 2), "us_per_launch": round(us, 2),
                                             "pct_of_burst_peak": round(100 * tf / float(peaks["bf16_tflops"]), 2)}
            del A, B, C
    finally:
        torch.backends.cuda.matmul.allow_fp16_reduced_precision_reduction = prev
    torch.cuda.empty_cache()
    return out


def measure_softmax(g, ctx, stream, device, peaks, steps=50):
    """Row-wise softmax (the next hot-path row): HBM-bound, so GB/s against the measured copy
    bandwidth; algorithmic bytes = one read and one write of every FP16 element."""
    import torch
    from tensor_core_gemm_tcgen05_gb300 import inputs
    rows, cols = SOFTMAX_SHAPE
    X = (inputs.random_fp16((rows, cols), 4242) * 8).to(device)
    Y = torch.empty_like(X)
    for _ in range(5):
        g.gemm_row_softmax(ctx, rows, cols, X, Y, stream)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        g.gemm_row_softmax(ctx, rows, cols, X, Y, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) / steps * 1e3
    nbytes = 2 * rows * cols * 2
    gbs = nbytes / (us * 1e-6) / 1e9
    return {f"row_softmax_{rows}x{cols}": {
        "us_per_launch": round(us, 2), "GB/s": round(gbs, 1), "bound": "hbm",
        "frac_of_measured_hbm": round(gbs / float(peaks["hbm_gbs"]), 4),
        "algorithmic_bytes_per_launch": nbytes}}


def measure_fused_softmax(g, ctx, stream, device, peaks, steps=30):
    """GEMM with the row-softmax epilogue on attention-score shapes (HBM-bound: the logits
    never leave the SM), against the same result computed unfused (GEMM, then the row
    softmax in place: C is written, read and written again)."""
    import torch
    from tensor_core_gemm_tcgen05_gb300 import inputs
    res = {}
    for wname in ("scores_262144x256x128_softmax", "scores_32768x1024x128_softmax"):
        w = inputs.WORKLOADS[wname]
        _, (dA, dB, dbias, dC) = device_buffers(w, device)

        def fused():
            g.gemm_run(ctx, w.M, w.N, w.K, dA, dB, dbias, dC, g.EPI_SOFTMAX, stream)

        def unfused():
            g.gemm_run(ctx, w.M, w.N, w.K, dA, dB, dbias, dC, g.EPI_NONE, stream)
            g.gemm_row_softmax(ctx, w.M, w.N, dC, dC, stream)

        out = {}
        for name, fn in (("fused", fused), ("unfused", unfused)):
            for _ in range(5):
                fn()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(steps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            out[name] = e0.elapsed_time(e1) / steps * 1e3
        gbs = w.bytes / (out["fused"] * 1e-6) / 1e9
        res[w.name] = {
            "us_per_launch": round(out["fused"], 2), "unfused_us": round(out["unfused"], 2),
            "GB/s": round(gbs, 1), "bound": "hbm", "frac_of_measured_hbm": round(gbs / float(peaks["hbm_gbs"]), 4),
            "tflops": round(w.flops / (out["fused"] * 1e-6) / 1e12, 1), "algorithmic_bytes_per_launch": w.bytes}
        del dA, dB, dbias, dC
    return res


ATTN_SHAPE = (64, 4096)   # heads (e.g. batch 4 x 16 heads) and tokens, head dimension 128


def measure_attention(g, ctx, stream, device, peaks, steps=10):
    """FlashAttention forward (the last next-row): flops 4 * heads * S^2 * 128 (half of it
    when causal), against the dense tensor peak."""
    import math
    import torch
    from tensor_core_gemm_tcgen05_gb300 import inputs
    H, S = ATTN_SHAPE
    Q, K, V = (inputs.random_fp16((H, S, 128), 900 + i, "normal").to(device) for i in range(3))
    O = torch.empty_like(Q)
    out = {}
    for causal in (False, True):
        def fn():
            g.gemm_attention_fwd(ctx, H, S, S, 128, Q, K, V, O, 1.0 / math.sqrt(128), causal, stream)
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) / steps * 1e3
        flops = 4 * H * S * S * 128 * (0.5 if causal else 1.0)
        tf = flops / (us * 1e-6) / 1e12
        out[f"attention_fwd_{H}x{S}x128_{'causal' if causal else 'full'}"] = {
            "us_per_launch": round(us, 1), "tflops": round(tf, 1), "bound": "tensor",
            "pct_of_burst_peak": round(100 * tf / float(peaks["bf16_tflops"]), 2)}
    return out


def measure_e2e(g, ctx, w, host, stream, steps, batches=3):
    """Same metric through gemm_run_host: pinned host inputs copied in, C copied out, every
    step inside the timed region (host wall clock around synchronous calls). `batches` timed
    batches of `steps` calls; the median batch is reported (a batch of a few milliseconds is
    easily disturbed on the host side), every batch's value alongside."""
    import torch
    A, B, bias = host
    pA, pB = A.pin_memory(), B.pin_memory()
    pbias = bias.pin_memory() if bias is not None else None
    pC = torch.empty(w.M, w.N, dtype=torch.float16).pin_memory()
    for _ in range(3):
        g.gemm_run_host(ctx, w.M, w.N, w.K, pA, pB, pbias, pC, w.epi_code, stream)
    dts = []
    for _ in range(batches):
        t0 = time.perf_counter()
        for _ in range(steps):
            g.gemm_run_host(ctx, w.M, w.N, w.K, pA, pB, pbias, pC, w.epi_code, stream)
        dts.append(time.perf_counter() - t0)
    dt = statistics.median(dts)
    h2d = 2 * (w.M * w.K + w.K * w.N) + (2 * w.N if w.bias else 0)
    d2h = 2 * w.M * w.N
    return {"value": round(w.flops * steps / dt / 1e12, 3), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": round(dt * 1e3 / steps, 4),
            "batches": [round(w.flops * steps / t / 1e12, 1) for t in dts],
            "api": "gemm_run_host (pinned host buffers)"}


def cpu_baseline(w, host, target_s=12.0, max_rows=None):
    """The FP64 oracle, as it stands, on a bounded row sample of the workload."""
    import oracle
    from tensor_core_gemm_tcgen05_gb300 import inputs
    A, B, bias = host
    cores = oracle.default_threads()
    probe_rows = inputs.sample_rows(w.M, min(max(cores, 8), w.M), seed=99).numpy()
    t0 = time.perf_counter()
    _, _, used = oracle.gemm(A, B, bias, w.epi_code, rows=probe_rows)
    t_probe = time.perf_counter() - t0
    rate = len(probe_rows) / max(t_probe, 1e-6)
    nrows = int(min(max_rows or w.M, max(len(probe_rows), rate * target_s)))
    rows = inputs.sample_rows(w.M, nrows, include_last=min(w.include_last, nrows)).numpy()
    t0 = time.perf_counter()
    _, _, used = oracle.gemm(A, B, bias, w.epi_code, rows=rows)
    dt = time.perf_counter() - t0
    flops = 2.0 * len(rows) * w.N * w.K
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": used, "kind": "oracle",
            "seconds": round(dt, 3),
            "sample": f"{len(rows)} seeded full rows of C ({len(rows)} x {w.N}, K={w.K}, "
                      f"{w.epilogue} epilogue) out of M={w.M}, FP64 C oracle, {used} threads",
            "extrapolated_full_gemm_s": round(dt * w.M / len(rows), 1)}


def run_ours(args):
    import torch
    import tensor_core_gemm_tcgen05_gb300 as g
    from tensor_core_gemm_tcgen05_gb300 import _build, inputs

    world, rank, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dist = init_dist(world, "nccl")
    if rank == 0 or not os.path.exists(g.LIB_PATH):
        _build.build()
    barrier(dist, device)
    ctx = g.Context(local)
    stream = torch.cuda.Stream(device)
    w = inputs.WORKLOADS[args.workload]
    host, (dA, dB, dbias, dC) = device_buffers(w, device)
    peaks, peak_src = load_peaks()

    sampler = ClockSampler(local) if rank == 0 else None
    # warm-up, then the timed region (clock samples are kept only inside it)
    for _ in range(args.warmup):
        g.gemm_run(ctx, w.M, w.N, w.K, dA, dB, dbias, dC, w.epi_code, stream)
    torch.cuda.synchronize()
    barrier(dist, device)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if sampler:
        sampler.mark_start()
    e0.record(stream)
    for _ in range(args.steps):
        g.gemm_run(ctx, w.M, w.N, w.K, dA, dB, dbias, dC, w.epi_code, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark_stop()
    ms_local = e0.elapsed_time(e1)
    barrier(dist, device)
    ms = max_over_ranks(dist, ms_local, device)
    status, detail = g.gemm_last_device_error(ctx)
    if status != g.GEMM_OK:
        raise RuntimeError(f"device error word {detail} during the timed region")
    clocks = sampler.finish() if sampler else None
    launches = args.steps  # one kernel launch per step

    ms_step = ms / args.steps
    value = world * w.flops / (ms_step * 1e-3) / 1e12
    if rank != 0:
        ctx.close()
        if dist:
            dist.destroy_process_group()
        return

    long_region = ms >= 1000.0
    peak_key = "bf16_tflops_sustained" if long_region else "bf16_tflops"
    peak = float(peaks[peak_key])  # FP16 and BF16 share the nominal dense tensor rate (ratio 1)
    per_gpu = value / world
    traffic, traffic_src = recorded_traffic()
    roofline = {
        "bound": "tensor", "achieved": round(per_gpu, 2), "peak": peak, "unit": "TFLOP/s",
        "frac": round(per_gpu / peak, 4), "traffic": traffic,
        "peak_source": f"{peak_src} {peak_key} (FP16 = BF16 nominal rate)",
        "traffic_source": traffic_src, "algorithmic_flops_per_launch": w.flops,
        "algorithmic_bytes_per_launch": w.bytes, "kernel": "gemm_tcgen05_pair_kernel (CTA pairs, 256x256 tiles)",
    }

    side = {}
    if not args.no_side:
        for name in SIDE_WORKLOADS:
            sw = inputs.WORKLOADS[name]
            if sw.name == w.name:
                continue
            _, (a, b, bi, c) = device_buffers(sw, device)
            n = 200 if sw.flops < 1e11 else 30
            t = time_device(g, ctx, sw, a, b, bi, c, stream, n, 5)
            tf = sw.flops / (t / n * 1e-3) / 1e12
            side[name] = {"tflops": round(tf, 2), "us_per_launch": round(t / n * 1e3, 2),
                          "pct_of_burst_peak": round(100 * tf / float(peaks["bf16_tflops"]), 2)}
            del a, b, bi, c
        torch.cuda.empty_cache()
        side.update(measure_cublas_context(device, peaks))
        side.update(measure_softmax(g, ctx, stream, device, peaks))
        side.update(measure_fused_softmax(g, ctx, stream, device, peaks))
        side.update(measure_attention(g, ctx, stream, device, peaks))

    e2e = None if args.no_e2e else measure_e2e(g, ctx, w, host, stream, steps=max(3, min(args.steps, 10)))
    base = None if args.no_cpu_baseline or world > 1 else cpu_baseline(w, host)
    ctx.close()

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic, seeded: X ~ N(0,1), W ~ N(0,1/K), bias ~ U[-0.1,0.1], all FP16",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "epilogue": f"bias+{w.epilogue}",
                   "accumulate": "fp32", "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": f"inputs larger than L2 ({w.bytes / 2**20:.0f} MiB of A+B+C per step vs "
                         f"{L2_BYTES / 2**20:.0f} MiB L2), no flush"},
        "pct_of_peak": round(100 * per_gpu / float(peaks["bf16_tflops"]), 2),
        "roofline": roofline,
        "cpu_baseline": base,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
        "side_workloads": side,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------------------------
# reference arm: the FP64 CPU oracle, as it stands, on bounded samples
# ---------------------------------------------------------------------------------------------
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from tensor_core_gemm_tcgen05_gb300 import inputs
    w = inputs.WORKLOADS[args.workload]
    host = inputs.make_inputs(w)
    A, B, bias = host
    cores = oracle.default_threads()
    # size each step so that warm-up + timed steps take about 90 s in all
    probe = inputs.sample_rows(w.M, cores, seed=99).numpy()
    t0 = time.perf_counter()
    oracle.gemm(A, B, bias, w.epi_code, rows=probe)
    rate = len(probe) / max(time.perf_counter() - t0, 1e-6)
    per_step = max(1, int(rate * 90.0 / (args.steps + args.warmup)))
    per_step = min(per_step, w.M)
    samples = [inputs.sample_rows(w.M, per_step, seed=1000 + i).numpy() for i in range(args.steps + args.warmup)]
    for i in range(args.warmup):
        oracle.gemm(A, B, bias, w.epi_code, rows=samples[i])
    t0 = time.perf_counter()
    used = cores
    for i in range(args.steps):
        _, _, used = oracle.gemm(A, B, bias, w.epi_code, rows=samples[args.warmup + i])
    dt = time.perf_counter() - t0
    flops = 2.0 * per_step * w.N * w.K * args.steps
    value = flops / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64",
        "data": "synthetic, seeded: X ~ N(0,1), W ~ N(0,1/K), bias ~ U[-0.1,0.1], all FP16",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "epilogue": f"bias+{w.epilogue}",
                   "rows_per_step": per_step},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": used, "kind": "oracle",
                         "sample": f"{per_step} seeded full rows of C per step (x {w.N}, K={w.K}) out of "
                                   f"M={w.M}, FP64 C oracle, {used} threads"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-side", action="store_true", help="skip the context workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer measurement")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, _, _ = dist_env()
    if world != args.gpus:
        log(f"note: WORLD_SIZE={world} but --gpus {args.gpus}; using WORLD_SIZE")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
