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


class NvmlSampler:
    """In-process, query-only NVML polling (SM clock, power, clock-event reasons) on a
    background thread, every `period_s` seconds, each sample stamped with the host's
    perf_counter. ctypes releases the GIL during each NVML call, so the launching thread is
    not held up. `summary(t0, t1)` describes the samples inside a host-time window."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    FI_POWER_INSTANT = 186   # NVML field id of the instantaneous board power (mW)

    def __init__(self, device_index: int, period_s: float = 0.002):
        import ctypes
        import threading
        import torch
        self.ct = ctypes
        self.period = period_s
        self.samples = []   # (t, sm_mhz, power_w, reason_mask, call_us)
        self.L = ctypes.CDLL("libnvidia-ml.so.1")
        if self.L.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        uuid = str(torch.cuda.get_device_properties(device_index).uuid)
        uuid = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        self.h = ctypes.c_void_p()
        if self.L.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) != 0:
            raise RuntimeError(f"no NVML handle for {uuid}")
        mx = ctypes.c_uint(0)
        rc = self.L.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))
        self.sm_max = float(mx.value) if rc == 0 else None

        class Value(ctypes.Union):
            _fields_ = [("dVal", ctypes.c_double), ("uiVal", ctypes.c_uint), ("ulVal", ctypes.c_ulong),
                        ("ullVal", ctypes.c_ulonglong), ("sllVal", ctypes.c_longlong), ("siVal", ctypes.c_int),
                        ("usVal", ctypes.c_ushort)]

        class Field(ctypes.Structure):
            _fields_ = [("fieldId", ctypes.c_uint32), ("scopeId", ctypes.c_uint32), ("timestamp", ctypes.c_int64),
                        ("latencyUsec", ctypes.c_int64), ("valueType", ctypes.c_uint), ("nvmlReturn", ctypes.c_uint),
                        ("value", Value)]

        self.field = Field()
        self.power_source = "instant"
        if not self._power_instant():
            self.power_source = "average"
        self.stop_ev = threading.Event()
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def _power_instant(self):
        f = self.field
        f.fieldId = self.FI_POWER_INSTANT
        f.scopeId = 0
        if self.L.nvmlDeviceGetFieldValues(self.h, 1, self.ct.byref(f)) != 0 or f.nvmlReturn != 0:
            return None
        return f.value.uiVal / 1000.0

    def _sample(self):
        ct = self.ct
        t = time.perf_counter()
        clk, mw, reasons = ct.c_uint(0), ct.c_uint(0), ct.c_ulonglong(0)
        rc = self.L.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(clk))
        sm = float(clk.value) if rc == 0 else None
        if self.power_source == "instant":
            pw = self._power_instant()
        else:
            pw = mw.value / 1000.0 if self.L.nvmlDeviceGetPowerUsage(self.h, ct.byref(mw)) == 0 else None
        rs = reasons.value if self.L.nvmlDeviceGetCurrentClocksEventReasons(self.h, ct.byref(reasons)) == 0 else 0
        self.samples.append((t, sm, pw, rs, (time.perf_counter() - t) * 1e6))

    def _run(self):
        while not self.stop_ev.is_set():
            self._sample()
            time.sleep(self.period)

    def stop(self):
        self.stop_ev.set()
        self.thread.join(timeout=5)
        try:
            self.L.nvmlShutdown()
        except Exception:
            pass

    def summary(self, t0: float, t1: float) -> dict:
        use = [x for x in self.samples if t0 <= x[0] <= t1 and x[1] is not None]
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": self.sm_max, "reasons": [], "samples": 0,
                    "source": "nvml", "in_timed_region": False}
        reasons = set()
        for x in use:
            for bit, nm in self.REASONS.items():
                if x[3] & bit:
                    reasons.add(nm)
        power = [x[2] for x in use if x[2] is not None]
        return {
            "sm_mhz": statistics.median(x[1] for x in use),
            "sm_max_mhz": self.sm_max,
            "sm_mhz_min": min(x[1] for x in use),
            "reasons": sorted(reasons),
            "samples": len(use),
            "in_timed_region": True,
            "power_w_median": round(statistics.median(power), 1) if power else None,
            "power_w_max": round(max(power), 1) if power else None,
            "power_source": self.power_source,
            "period_ms": round(1e3 * (use[-1][0] - use[0][0]) / max(1, len(use) - 1), 2),
            "source": "nvml (in-process polling, query only)",
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
    for wname in ("scores_262144x256x128_softmax", "scores_32768x512x128_softmax", "scores_32768x1024x128_softmax",
                  "scores_32768x2048x128_softmax", "scores_16384x4096x128_softmax",
                  "scores_8192x16384x128_softmax"):
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
            "kernel": g.gemm_describe(ctx, w.M, w.N, w.K, g.EPI_SOFTMAX),
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


# Parity rule of the GEMM path against the FP64 oracle (the one the tests apply): per element
# |C - ref| <= 1e-2 + 4e-3 |ref|, relative Frobenius error <= 1e-3, no NaN/Inf.
PARITY_ATOL, PARITY_RTOL, PARITY_FRO = 1e-2, 4e-3, 1e-3


def parity_stats(got, ref) -> dict:
    import numpy as np
    g = np.asarray(got, dtype=np.float16).astype(np.float64)
    r = np.asarray(ref, dtype=np.float16).astype(np.float64)
    err = np.abs(g - r)
    viol = int((err > PARITY_ATOL + PARITY_RTOL * np.abs(r)).sum())
    fro = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30))
    finite = bool(np.all(np.isfinite(g)))
    return {"checked_elements": int(err.size), "max_abs": float(err.max()), "fro_rel": fro, "violations": viol,
            "finite": finite, "ok": finite and viol == 0 and fro <= PARITY_FRO,
            "tolerance": f"|C-ref| <= {PARITY_ATOL} + {PARITY_RTOL}|ref|, fro <= {PARITY_FRO}"}


def cpu_baseline(w, host, target_s=12.0, max_rows=None, gpu_out=None):
    """The FP64 oracle, as it stands, on a bounded row sample of the workload. When the GPU's
    output of the timed launches (host copy) is given, the same oracle rows check it: the
    benchmark's own output is verified against the oracle in the same run."""
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
    ref, _, used = oracle.gemm(A, B, bias, w.epi_code, rows=rows)
    dt = time.perf_counter() - t0
    flops = 2.0 * len(rows) * w.N * w.K
    res = {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": used, "kind": "oracle",
           "seconds": round(dt, 3),
           "sample": f"{len(rows)} seeded full rows of C ({len(rows)} x {w.N}, K={w.K}, "
                     f"{w.epilogue} epilogue) out of M={w.M}, FP64 C oracle, {used} threads",
           "extrapolated_full_gemm_s": round(dt * w.M / len(rows), 1)}
    parity = None
    if gpu_out is not None:
        parity = parity_stats(gpu_out[rows], ref)
        parity["rows"] = f"the {len(rows)} oracle rows above (including the last {min(w.include_last, nrows)})"
        parity["of"] = "C of the timed launches"
    return res, parity


def start_clock_probe(g, ctx, device, region_ms, interval_us=100.0, max_samples=32768):
    """Start the library's SM-clock sampler on a stream of its own, for about `region_ms`
    (plus a margin): one thread beside the timed kernels reads the SM cycle counter and the
    global timer every `interval_us`."""
    import torch
    n = int(min(max_samples, region_ms * 1.3 * 1e3 / interval_us + 64))
    trace = torch.zeros(2 * n, dtype=torch.int64, device=device)
    side = torch.cuda.Stream(device)
    g.gemm_clock_trace(ctx, trace, n, int(interval_us * 1e3), int((region_ms * 1.3 + 1.0) * 1e6), side)
    return trace


def clock_probe_summary(trace, region_ms) -> dict:
    """SM clock over the first `region_ms` of the trace (the timed launches start right after
    the sampler): cycles / ns between consecutive samples."""
    import numpy as np
    t = trace.view(-1, 2).cpu().numpy()
    t = t[t[:, 0] > 0]
    if len(t) < 3:
        return {"samples": int(len(t))}
    ts, cs = t[:, 0].astype(np.float64), t[:, 1].astype(np.float64)
    end = ts[0] + region_ms * 1e6
    ok = ts[1:] <= end
    mhz = (np.diff(cs) / np.diff(ts) * 1e3)[ok]
    if len(mhz) == 0:
        return {"samples": int(len(t))}
    return {"effective_sm_mhz": round(float(np.median(mhz)), 1), "effective_sm_mhz_min": round(float(mhz.min()), 1),
            "effective_sm_mhz_max": round(float(mhz.max()), 1), "intervals": int(len(mhz)),
            "interval_us": round(float(np.median(np.diff(ts))) / 1e3, 1),
            "source": "gemm_clock_trace: clock64 / globaltimer on one SM beside the timed launches"}


def time_sustained(g, ctx, w, bufs, stream, step_ms, sampler, seconds=2.0):
    """The same launches back to back for about `seconds` (at least 1.5 s), right after the
    headline: the steady state at the board's power limit, with its own clock record."""
    import torch
    dA, dB, dbias, dC = bufs
    n = max(50, int(math.ceil(seconds * 1e3 / max(step_ms, 1e-3))))
    torch.cuda.synchronize()
    trace = start_clock_probe(g, ctx, dA.device, n * step_ms, interval_us=1000.0)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record(stream)
    for _ in range(n):
        g.gemm_run(ctx, w.M, w.N, w.K, dA, dB, dbias, dC, w.epi_code, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    ms = e0.elapsed_time(e1)
    clocks = sampler.summary(t0, t1) if sampler else None
    # the last half alone: after the clocks have settled at the power limit
    clocks_late = sampler.summary(t0 + 0.5 * (t1 - t0), t1) if sampler else None
    probe = clock_probe_summary(trace, ms)
    if clocks is not None:
        clocks.update(probe)
    else:
        clocks = probe
    return n, ms, clocks, clocks_late


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
    schedule = g.gemm_describe(ctx, w.M, w.N, w.K, w.epi_code)

    sampler = None
    sampler_note = None
    if rank == 0:
        try:
            sampler = NvmlSampler(local)
        except Exception as e:   # no NVML: fall back to nvidia-smi at 100 ms
            sampler_note = f"NVML unavailable ({e}); nvidia-smi sampling"
    smi = ClockSampler(local) if rank == 0 and sampler is None else None
    # warm-up (its duration sizes the clock sampler), then the timed region (clock samples
    # are kept only inside it)
    w0 = torch.cuda.Event(enable_timing=True)
    w1 = torch.cuda.Event(enable_timing=True)
    w0.record(stream)
    for _ in range(args.warmup):
        g.gemm_run(ctx, w.M, w.N, w.K, dA, dB, dbias, dC, w.epi_code, stream)
    w1.record(stream)
    torch.cuda.synchronize()
    est_region_ms = w0.elapsed_time(w1) / args.warmup * args.steps
    barrier(dist, device)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    trace = start_clock_probe(g, ctx, device, est_region_ms) if rank == 0 else None
    if smi:
        smi.mark_start()
    t_start = time.perf_counter()
    e0.record(stream)
    for _ in range(args.steps):
        g.gemm_run(ctx, w.M, w.N, w.K, dA, dB, dbias, dC, w.epi_code, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    t_stop = time.perf_counter()
    if smi:
        smi.mark_stop()
    ms_local = e0.elapsed_time(e1)
    barrier(dist, device)
    ms = max_over_ranks(dist, ms_local, device)
    status, detail = g.gemm_last_device_error(ctx)
    if status != g.GEMM_OK:
        raise RuntimeError(f"device error word {detail} during the timed region")
    launches = args.steps  # one kernel launch per step

    ms_step = ms / args.steps
    value = world * w.flops / (ms_step * 1e-3) / 1e12
    if rank != 0:
        ctx.close()
        if dist:
            dist.destroy_process_group()
        return
    if sampler:
        clocks = sampler.summary(t_start, t_stop)
        clocks["note"] = ("NVML's clock and power readings refresh more slowly than a region of a "
                          "few tens of milliseconds; effective_sm_mhz is the clock the SMs counted")
    else:
        clocks = smi.finish()
        clocks["note"] = sampler_note
    clocks.update(clock_probe_summary(trace, ms_local))
    mhz = clocks.get("effective_sm_mhz") or clocks.get("sm_mhz")
    if mhz:
        # cycles of one launch at the clock measured inside the timed region
        clocks["cycles_per_launch"] = round(ms_step * 1e-3 * mhz * 1e6)
    c_out = dC.cpu().numpy() if not args.no_cpu_baseline and world == 1 else None   # outputs of the timed launches

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
        "algorithmic_bytes_per_launch": w.bytes, "kernel": schedule.split(" ")[0], "schedule": schedule,
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
                          "pct_of_burst_peak": round(100 * tf / float(peaks["bf16_tflops"]), 2),
                          "kernel": g.gemm_describe(ctx, sw.M, sw.N, sw.K, sw.epi_code)}
            del a, b, bi, c
        torch.cuda.empty_cache()
        side.update(measure_cublas_context(device, peaks))
        side.update(measure_softmax(g, ctx, stream, device, peaks))
        side.update(measure_fused_softmax(g, ctx, stream, device, peaks))
        side.update(measure_attention(g, ctx, stream, device, peaks))

    e2e = None if args.no_e2e else measure_e2e(g, ctx, w, host, stream, steps=max(3, min(args.steps, 10)))
    # the seconds-long leg last, so that it does not heat the GPU before the short lines
    sustained = None
    if not args.no_sustained:
        n_s, ms_s, clk_s, clk_late = time_sustained(g, ctx, w, (dA, dB, dbias, dC), stream, ms_step, sampler)
        v_s = w.flops * n_s / (ms_s * 1e-3) / 1e12
        peak_s = float(peaks["bf16_tflops_sustained"])
        sustained = {"value": round(v_s, 2), "unit": "TFLOP/s", "launches": n_s, "seconds": round(ms_s * 1e-3, 3),
                     "ms_per_launch": round(ms_s / n_s, 5), "peak": peak_s,
                     "peak_source": f"{peak_src} bf16_tflops_sustained (FP16 = BF16 nominal rate)",
                     "frac": round(v_s / peak_s, 4), "clocks": clk_s, "clocks_last_half": clk_late}
        mhz_s = clk_s and (clk_s.get("effective_sm_mhz") or clk_s.get("sm_mhz"))
        if mhz_s:
            sustained["cycles_per_launch"] = round(ms_s / n_s * 1e-3 * mhz_s * 1e6)
        status, detail = g.gemm_last_device_error(ctx)
        if status != g.GEMM_OK:
            raise RuntimeError(f"device error word {detail} during the sustained run")

    base, parity = (None, None)
    if not args.no_cpu_baseline and world == 1:
        base, parity = cpu_baseline(w, host, gpu_out=c_out)
    ctx.close()
    if sampler:
        sampler.stop()

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
        "parity": parity,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
        "sustained": sustained,
        "side_workloads": side,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    if parity is not None and not parity["ok"]:
        log(f"parity check of the benchmark's output FAILED: {parity}")
        sys.exit(1)


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
    ap.add_argument("--no-sustained", action="store_true", help="skip the seconds-long sustained leg")
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
