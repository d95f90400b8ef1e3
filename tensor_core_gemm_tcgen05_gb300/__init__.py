"""GB300 (sm_103a) FP16 tensor-core GEMM with a fused bias + GELU / ReLU epilogue.

A thin ctypes binding over the C ABI in ``include/gemm.h`` (``libgb300gemm.so``, built by
``tensor_core_gemm_tcgen05_gb300._build``). Every step of the computation runs in the CUDA
kernels of that library; this module only marshals arguments. There is no CPU fallback:
if the library is missing, every call raises.

    ctx = gemm_create(0)
    gemm_run(ctx, M, N, K, A, B, bias, C, EPI_GELU, stream)   # device tensors or pointers
    gemm_destroy(ctx)

Names follow the C ABI. Tensor arguments may be ``torch.Tensor`` (their ``data_ptr()`` is
passed) or integer addresses; ``stream`` may be a ``torch.cuda.Stream``, an integer handle or
None (None means the current torch stream of the context's device when torch is loaded).
"""
from __future__ import annotations

import ctypes
import os
import threading

from .inputs import EPI_GELU, EPI_NONE, EPI_RELU, EPI_SOFTMAX  # noqa: F401  (C ABI epilogue codes)

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgb300gemm.so")

GEMM_EPI_NONE, GEMM_EPI_GELU, GEMM_EPI_RELU, GEMM_EPI_SOFTMAX = EPI_NONE, EPI_GELU, EPI_RELU, EPI_SOFTMAX
GEMM_OK = 0
GEMM_ERR_ARG = -1
GEMM_ERR_ALIGN = -2
GEMM_ERR_DEVICE = -3
GEMM_ERR_LAUNCH = -4
GEMM_ERR_TIMEOUT = -5
GEMM_ERR_NOMEM = -6
GEMM_DEBUG_NONE = 0
GEMM_DEBUG_WITHHOLD_FIRST_LOAD = 1
GEMM_DEBUG_FORCE_SINGLE = 2
GEMM_DEBUG_FORCE_PAIR = 4
GEMM_DEBUG_FORCE_STREAMK = 8
GEMM_DEBUG_FORCE_SPLITK = 16

# Every symbol include/gemm.h declares (the CPU tests check the library exports them).
EXPORTS = (
    "gemm_create", "gemm_run", "gemm_run_host", "gemm_last_device_error",
    "gemm_last_cuda_error", "gemm_destroy", "gemm_status_string", "gemm_num_sms",
    "gemm_set_timeout_ns", "gemm_set_debug", "gemm_run_noalloc", "gemm_num_pairs",
    "gemm_row_softmax", "gemm_attention_fwd", "gemm_describe", "gemm_clock_trace",
)
GEMM_NOALLOC_SCRATCH_BYTES = 256

_lock = threading.Lock()
_lib = None


class GemmError(RuntimeError):
    """A non-zero status returned by the C ABI."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {gemm_status_string(status)} ({status})")


def lib() -> ctypes.CDLL:
    """Load ``libgb300gemm.so`` (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m tensor_core_gemm_tcgen05_gb300._build` (no CPU fallback exists)")
            L = ctypes.CDLL(LIB_PATH)
            vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            L.gemm_create.argtypes = [ctypes.POINTER(vp), i32]
            run_args = [vp, i64, i64, i64, vp, vp, vp, vp, i32, vp]
            L.gemm_run.argtypes = run_args
            L.gemm_run_host.argtypes = run_args
            L.gemm_last_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
            L.gemm_last_cuda_error.argtypes = [vp]
            L.gemm_destroy.argtypes = [vp]
            L.gemm_status_string.argtypes = [i32]
            L.gemm_status_string.restype = ctypes.c_char_p
            L.gemm_num_sms.argtypes = [vp]
            L.gemm_num_pairs.argtypes = [vp]
            L.gemm_row_softmax.argtypes = [vp, i64, i64, vp, vp, vp]
            L.gemm_attention_fwd.argtypes = [vp, i64, i64, i64, i64, vp, vp, vp, vp, ctypes.c_float, i32, vp]
            L.gemm_set_timeout_ns.argtypes = [vp, ctypes.c_uint64]
            L.gemm_set_debug.argtypes = [vp, i32]
            L.gemm_run_noalloc.argtypes = [i64, i64, i64, vp, vp, vp, vp, i32, vp]
            L.gemm_describe.argtypes = [vp, i64, i64, i64, i32, ctypes.c_char_p, i64]
            L.gemm_clock_trace.argtypes = [vp, vp, i32, ctypes.c_uint64, ctypes.c_uint64, vp]
            for name in EXPORTS:
                if name != "gemm_status_string":
                    getattr(L, name).restype = i32
            _lib = L
    return _lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    return int(x)


def _stream(s, device: int | None) -> int | None:
    if s is None:
        import sys
        torch = sys.modules.get("torch")
        if torch is not None and torch.cuda.is_available() and device is not None:
            return int(torch.cuda.current_stream(device).cuda_stream)
        return None
    if hasattr(s, "cuda_stream"):
        return int(s.cuda_stream)
    return int(s)


def _check(rc: int, where: str) -> int:
    if rc != GEMM_OK:
        raise GemmError(rc, where)
    return rc


class Context:
    """Owns one ``gemm_ctx``; usable as a context manager."""

    def __init__(self, device: int = 0):
        self.device = device
        self.handle = gemm_create(device)

    def close(self):
        if self.handle:
            gemm_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _h(ctx):
    return ctx.handle if isinstance(ctx, Context) else ctx


def _dev(ctx):
    return ctx.device if isinstance(ctx, Context) else None


def gemm_create(device: int = 0) -> int:
    h = ctypes.c_void_p()
    _check(lib().gemm_create(ctypes.byref(h), int(device)), "gemm_create")
    return h.value


def gemm_run(ctx, M, N, K, A, B, bias, C, epilogue=EPI_NONE, stream=None) -> int:
    rc = lib().gemm_run(_h(ctx), M, N, K, _ptr(A), _ptr(B), _ptr(bias), _ptr(C), int(epilogue),
                        _stream(stream, _dev(ctx)))
    return _check(rc, "gemm_run")


def gemm_run_host(ctx, M, N, K, A, B, bias, C, epilogue=EPI_NONE, stream=None) -> int:
    rc = lib().gemm_run_host(_h(ctx), M, N, K, _ptr(A), _ptr(B), _ptr(bias), _ptr(C), int(epilogue),
                             _stream(stream, _dev(ctx)))
    return _check(rc, "gemm_run_host")


def gemm_run_noalloc(M, N, K, A, B, bias, C, epilogue=EPI_NONE, stream=None, device=None) -> int:
    """The allocation-free variant (no context; device pointers on the current device)."""
    rc = lib().gemm_run_noalloc(M, N, K, _ptr(A), _ptr(B), _ptr(bias), _ptr(C), int(epilogue),
                                _stream(stream, device))
    return _check(rc, "gemm_run_noalloc")


def gemm_last_device_error(ctx) -> tuple[int, int]:
    """Returns ``(status, detail)``; status is GEMM_OK or GEMM_ERR_TIMEOUT."""
    d = ctypes.c_uint32(0)
    rc = lib().gemm_last_device_error(_h(ctx), ctypes.byref(d))
    if rc not in (GEMM_OK, GEMM_ERR_TIMEOUT):
        raise GemmError(rc, "gemm_last_device_error")
    return rc, int(d.value)


def gemm_last_cuda_error(ctx) -> int:
    return int(lib().gemm_last_cuda_error(_h(ctx)))


def gemm_destroy(ctx) -> int:
    return _check(lib().gemm_destroy(_h(ctx)), "gemm_destroy")


def gemm_status_string(status: int) -> str:
    return lib().gemm_status_string(int(status)).decode()


def gemm_num_sms(ctx) -> int:
    return int(lib().gemm_num_sms(_h(ctx)))


def gemm_num_pairs(ctx) -> int:
    return int(lib().gemm_num_pairs(_h(ctx)))


def gemm_describe(ctx, M, N, K, epilogue=EPI_NONE) -> str:
    """The kernel instance, grid, cluster size and tile count gemm_run would use."""
    buf = ctypes.create_string_buffer(256)
    _check(lib().gemm_describe(_h(ctx), M, N, K, int(epilogue), buf, len(buf)), "gemm_describe")
    return buf.value.decode()


def gemm_clock_trace(ctx, trace, max_samples, interval_ns, duration_ns, stream=None) -> int:
    """Launch the SM-clock sampler into ``trace`` (device, 2 * max_samples int64/uint64)."""
    rc = lib().gemm_clock_trace(_h(ctx), _ptr(trace), int(max_samples), int(interval_ns), int(duration_ns),
                                _stream(stream, _dev(ctx)))
    return _check(rc, "gemm_clock_trace")


def gemm_row_softmax(ctx, rows, cols, X, Y, stream=None) -> int:
    rc = lib().gemm_row_softmax(_h(ctx), rows, cols, _ptr(X), _ptr(Y), _stream(stream, _dev(ctx)))
    return _check(rc, "gemm_row_softmax")


def row_softmax(ctx, X, out=None, stream=None):
    """Row-wise softmax of a 2-D torch CUDA FP16 tensor through ``gemm_row_softmax``."""
    import torch

    rows, cols = X.shape
    if out is None:
        out = torch.empty_like(X)
    for t in (X, out):
        if t.dtype != torch.float16 or not t.is_contiguous():
            raise ValueError("X and out must be contiguous float16 tensors")
    if stream is None:
        stream = torch.cuda.current_stream(X.device)
    gemm_row_softmax(ctx, rows, cols, X, out, stream)
    return out


def gemm_attention_fwd(ctx, heads, seq_q, seq_k, head_dim, Q, K, V, O, scale, causal, stream=None) -> int:
    rc = lib().gemm_attention_fwd(_h(ctx), heads, seq_q, seq_k, head_dim, _ptr(Q), _ptr(K), _ptr(V), _ptr(O),
                                  float(scale), int(bool(causal)), _stream(stream, _dev(ctx)))
    return _check(rc, "gemm_attention_fwd")


def attention(ctx, Q, K, V, scale=None, causal=False, out=None, stream=None):
    """FlashAttention forward on torch CUDA FP16 tensors [heads, seq, 128] through
    ``gemm_attention_fwd`` (``scale`` defaults to 1/sqrt(128))."""
    import math

    import torch

    H, Sq, D = Q.shape
    Sk = K.shape[1]
    if out is None:
        out = torch.empty_like(Q)
    for t in (Q, K, V, out):
        if t.dtype != torch.float16 or not t.is_contiguous():
            raise ValueError("Q, K, V and out must be contiguous float16 tensors")
    if stream is None:
        stream = torch.cuda.current_stream(Q.device)
    gemm_attention_fwd(ctx, H, Sq, Sk, D, Q, K, V, out, 1.0 / math.sqrt(D) if scale is None else scale, causal,
                       stream)
    return out


def gemm_set_timeout_ns(ctx, ns: int) -> int:
    return _check(lib().gemm_set_timeout_ns(_h(ctx), int(ns)), "gemm_set_timeout_ns")


def gemm_set_debug(ctx, flags: int) -> int:
    return _check(lib().gemm_set_debug(_h(ctx), int(flags)), "gemm_set_debug")


def gemm(ctx, A, B, bias=None, epilogue=EPI_NONE, out=None, stream=None):
    """``act(A @ B + bias)`` on torch CUDA FP16 tensors through ``gemm_run``.

    Allocates ``out`` with torch when it is not given (plumbing; the product is computed
    by the library's kernel). Returns ``out``.
    """
    import torch

    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"shape mismatch {tuple(A.shape)} @ {tuple(B.shape)}")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=A.device)
    for t in (A, B, bias, out):
        if t is not None and (t.dtype != torch.float16 or not t.is_contiguous()):
            raise ValueError("A, B, bias and out must be contiguous float16 tensors")
    if stream is None:
        stream = torch.cuda.current_stream(A.device)
    gemm_run(ctx, M, N, K, A, B, bias, out, epilogue, stream)
    return out
