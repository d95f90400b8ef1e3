"""The parity rule between the CUDA path and the FP64 oracle.

Both sides start from the same FP16 bits. The GPU accumulates in FP32 (in any order) and
rounds once to FP16; the oracle sums in FP64 and rounds once. Per checked element:
    |C - ref| <= 1e-2 + 4e-3 * |ref|
and over all checked elements the relative Frobenius error ||C - ref|| / ||ref|| <= 1e-3.
Any NaN or Inf in C fails.
"""
import numpy as np

ATOL, RTOL, FRO = 1e-2, 4e-3, 1e-3


def compare(got, ref):
    """Return error statistics of FP16 ``got`` against FP16 ``ref`` (same shape)."""
    g = np.asarray(got, dtype=np.float16).astype(np.float64)
    r = np.asarray(ref, dtype=np.float16).astype(np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    finite = bool(np.all(np.isfinite(g)))
    err = np.abs(g - r)
    bound = ATOL + RTOL * np.abs(r)
    viol = err > bound
    worst = np.unravel_index(int(np.argmax(err - bound)), err.shape) if err.size else None
    nr = float(np.linalg.norm(r))
    fro = float(np.linalg.norm(g - r)) / nr if nr > 0 else float(np.linalg.norm(g - r))
    return {
        "finite": finite,
        "max_abs": float(err.max()) if err.size else 0.0,
        "max_rel": float((err / np.maximum(np.abs(r), 1e-30)).max()) if err.size else 0.0,
        "fro_rel": fro,
        "violations": int(viol.sum()),
        "worst": tuple(int(i) for i in worst) if worst is not None else None,
        "n": int(err.size),
    }


def assert_parity(got, ref, what=""):
    s = compare(got, ref)
    assert s["finite"], f"{what}: NaN/Inf in result {s}"
    assert s["violations"] == 0, f"{what}: {s['violations']} elements outside tolerance {s}"
    assert s["fro_rel"] <= FRO, f"{what}: relative Frobenius error too large {s}"
    return s
