"""FP64 CPU oracle for ``C = act(A @ B + bias)`` (FP16 in, FP16 out).

TEST INFRASTRUCTURE ONLY: the plain, slow, obviously correct definition that the CUDA
kernels are checked against. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline legs of ``bench.py`` may import it; the library's product path never does. It
shares no code with the CUDA path (its arithmetic lives in ``oracle.c``, compiled with the
host C compiler; this module only builds it and marshals arguments).

Every function is pinned by ``tests/test_oracle.py``; see the header of ``oracle.c`` for
what is computed and which passage of the tutorial pages each part follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

ACT_NONE, ACT_GELU, ACT_RELU, ACT_SOFTMAX = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` beside it (host C compiler only)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O3", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, _SRC,
               "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_half_to_double.restype = ctypes.c_double
            lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_double_to_half.restype = ctypes.c_uint16
            lib.oracle_double_to_half.argtypes = [ctypes.c_double]
            lib.oracle_act.restype = ctypes.c_double
            lib.oracle_act.argtypes = [ctypes.c_double, ctypes.c_int]
            lib.oracle_default_threads.restype = ctypes.c_int
            lib.oracle_softmax_rows.restype = ctypes.c_int
            lib.oracle_softmax_rows.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.oracle_attention_rows.restype = ctypes.c_int
            lib.oracle_attention_rows.argtypes = [
                ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_double, ctypes.c_int, ctypes.c_void_p,
                ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.oracle_gemm_rows.restype = ctypes.c_int
            lib.oracle_gemm_rows.argtypes = [
                ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
            _lib = lib
    return _lib


def half_to_double(bits: int) -> float:
    return _load().oracle_half_to_double(int(bits))


def double_to_half(x: float) -> int:
    return int(_load().oracle_double_to_half(float(x)))


def act(x: float, code: int) -> float:
    return _load().oracle_act(float(x), int(code))


def default_threads() -> int:
    return int(_load().oracle_default_threads())


def _u16(t) -> np.ndarray:
    """FP16 data (numpy float16/uint16 array or CPU torch.float16 tensor) as uint16 bits."""
    if t is None:
        return None
    if hasattr(t, "detach"):  # torch tensor
        t = t.detach().cpu().contiguous().view(dtype=__import__("torch").int16).numpy()
    a = np.ascontiguousarray(t)
    if a.dtype == np.float16 or a.dtype == np.int16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected FP16 bits, got {a.dtype}")
    return a


def gemm(A, B, bias=None, act_code: int = ACT_NONE, rows=None, threads: int = 0,
         want_f64: bool = False):
    """Oracle ``act(A @ B + bias)`` for the given output rows (all rows when ``rows`` is None).

    ``A`` is M x K and ``B`` K x N FP16 (numpy float16/uint16 or CPU torch.float16);
    ``bias`` has N entries or is None. Returns ``(out_fp16 [nrows, N] as numpy float16,
    out_f64 [nrows, N] or None, threads_used)``.
    """
    a, b, bi = _u16(A), _u16(B), _u16(bias)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[0]:
        raise ValueError(f"shape mismatch {a.shape} @ {b.shape}")
    M, K = a.shape
    N = b.shape[1]
    if bi is not None and bi.shape != (N,):
        raise ValueError(f"bias must have {N} entries")
    if rows is None:
        r = None
        nrows = M
    else:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = r.shape[0]
    out_h = np.empty((nrows, N), dtype=np.uint16)
    out_d = np.empty((nrows, N), dtype=np.float64) if want_f64 else None
    used = ctypes.c_int(0)
    rc = _load().oracle_gemm_rows(
        M, N, K, a.ctypes.data, b.ctypes.data, None if bi is None else bi.ctypes.data,
        int(act_code), None if r is None else r.ctypes.data, nrows, out_h.ctypes.data,
        None if out_d is None else out_d.ctypes.data, int(threads), ctypes.byref(used))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_rows failed with code {rc}")
    return out_h.view(np.float16), out_d, used.value


def softmax_rows(X, threads: int = 0, want_f64: bool = False):
    """Oracle row-wise softmax of a 2-D FP16 array: returns ``(Y fp16, Y_f64 or None)``."""
    x = _u16(X)
    if x.ndim != 2:
        raise ValueError("X must be 2-D")
    rows, cols = x.shape
    y = np.empty((rows, cols), dtype=np.uint16)
    yd = np.empty((rows, cols), dtype=np.float64) if want_f64 else None
    rc = _load().oracle_softmax_rows(rows, cols, x.ctypes.data, y.ctypes.data,
                                     None if yd is None else yd.ctypes.data, int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle_softmax_rows failed with code {rc}")
    return y.view(np.float16), yd


def attention(Q, K, V, scale: float, causal: bool, rows=None, threads: int = 0, want_f64: bool = False):
    """Oracle attention output ``softmax(scale * Q K^T [+ causal mask]) V`` per head.

    Q is [H, Sq, D], K and V are [H, Sk, D] (FP16). ``rows`` is a list of (head, query)
    pairs (all of them when None). Returns ``(out fp16 [nrows, D], out_f64 or None)``.
    """
    q, k, v = _u16(Q), _u16(K), _u16(V)
    if q.ndim != 3 or k.ndim != 3 or v.shape != k.shape or q.shape[0] != k.shape[0] or q.shape[2] != k.shape[2]:
        raise ValueError("Q [H,Sq,D], K and V [H,Sk,D] expected")
    H, Sq, D = q.shape
    Sk = k.shape[1]
    if rows is None:
        rows = [(h, i) for h in range(H) for i in range(Sq)]
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 2))
    n = r.shape[0]
    out = np.empty((n, D), dtype=np.uint16)
    outd = np.empty((n, D), dtype=np.float64) if want_f64 else None
    rc = _load().oracle_attention_rows(H, Sq, Sk, D, q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                       float(scale), int(bool(causal)), r.ctypes.data, n,
                                       out.ctypes.data, None if outd is None else outd.ctypes.data,
                                       int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle_attention_rows failed with code {rc}")
    return out.view(np.float16), outd
