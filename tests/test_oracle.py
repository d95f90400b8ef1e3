"""Pins for the FP64 CPU oracle, each against something other than the oracle itself.

The tutorial pages print no worked numbers for the GEMM, so the oracle is pinned by the
format definition of FP16 (checked exhaustively against numpy), hand-worked products in
``tests/golden/gemm_textbook.txt``, standard-normal table values for GELU in
``tests/golden/normal_cdf_table.txt``, identities, brute-force loops on tiny shapes and a
library float64 matmul. Each pin is chosen so that a plausible mistake in the oracle (a
transposed operand, a per-row bias, bias after the activation, a wrong GELU constant or
sign, a wrong rounding mode) fails at least one test.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from tensor_core_gemm_tcgen05_gb300 import inputs


def _read_textbook(path):
    cases, cur = [], None
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        tag, *rest = line.split()
        if tag == "case":
            cur = {"name": rest[0], "M": int(rest[1]), "N": int(rest[2]), "K": int(rest[3]),
                   "act": rest[4]}
            cases.append(cur)
        elif tag == "bias" and rest == ["none"]:
            cur["bias"] = None
        else:
            cur[tag] = [float(v) for v in rest]
    return cases


# ---- FP16 decoding / encoding ----------------------------------------------------------

def test_half_to_double_exhaustive():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signs of zeros and infinities too
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def _np_rne(x: float) -> int:
    with np.errstate(over="ignore"):
        return int(np.array([x], dtype=np.float64).astype(np.float16).view(np.uint16)[0])


def test_double_to_half_round_trip_exhaustive():
    for b in range(65536):
        v = np.uint16(b).view(np.float16)
        if np.isnan(v):
            assert oracle.double_to_half(float(v)) & 0x7C00 == 0x7C00
            continue
        assert oracle.double_to_half(float(v)) == b, hex(b)


def test_double_to_half_ties_to_even():
    # Midpoints between consecutive finite FP16 values: ties go to the even code.
    finite = [b for b in range(0x7C00)]  # positive finite codes, 0 .. 65504
    for b in finite[:-1]:
        lo = float(np.uint16(b).view(np.float16))
        hi = float(np.uint16(b + 1).view(np.float16))
        mid = (lo + hi) / 2.0  # exact in double
        want = b if b % 2 == 0 else b + 1
        assert oracle.double_to_half(mid) == want, (b, mid)
        assert oracle.double_to_half(-mid) == want | 0x8000
        # just off the midpoint rounds to the nearer value
        assert oracle.double_to_half(np.nextafter(mid, -np.inf)) == b
        assert oracle.double_to_half(np.nextafter(mid, np.inf)) == b + 1


def test_double_to_half_specials():
    assert oracle.double_to_half(65504.0) == 0x7BFF
    assert oracle.double_to_half(65519.99) == 0x7BFF
    assert oracle.double_to_half(65520.0) == 0x7C00      # the tie above 65504 goes to inf
    assert oracle.double_to_half(-1e9) == 0xFC00
    assert oracle.double_to_half(float("inf")) == 0x7C00
    assert oracle.double_to_half(2.0 ** -25) == 0x0000   # tie between 0 and 2^-24 -> even
    assert oracle.double_to_half(3 * 2.0 ** -25) == 0x0002
    assert oracle.double_to_half(2.0 ** -24) == 0x0001
    assert oracle.double_to_half(1e-9) == 0x0000
    assert oracle.double_to_half(-0.0) == 0x8000
    assert oracle.double_to_half(1.0) == 0x3C00
    assert oracle.double_to_half(1.0 + 2.0 ** -11) == 0x3C00
    assert oracle.double_to_half(1.0 + 3 * 2.0 ** -11) == 0x3C02


def test_double_to_half_random_vs_numpy():
    rng = np.random.default_rng(7)
    xs = np.concatenate([
        rng.uniform(-1, 1, 20000),
        rng.normal(0, 300, 20000),
        rng.uniform(-1, 1, 10000) * 2.0 ** rng.integers(-30, 17, 10000),
    ])
    for x in xs:
        assert oracle.double_to_half(float(x)) == _np_rne(float(x)), x


# ---- activation ------------------------------------------------------------------------

def test_gelu_against_normal_table(golden_dir):
    rows = [l.split() for l in open(os.path.join(golden_dir, "normal_cdf_table.txt"))
            if l.strip() and not l.startswith("#")]
    for xs, ps in rows:
        x, phi = float(xs), float(ps)
        if x == 0.0:
            assert oracle.act(0.0, oracle.ACT_GELU) == 0.0
            continue
        assert abs(oracle.act(x, oracle.ACT_GELU) / x - phi) <= 5.01e-5, x
        # Phi(-x) = 1 - Phi(x)
        assert abs(oracle.act(-x, oracle.ACT_GELU) / (-x) - (1.0 - phi)) <= 5.01e-5, -x


def test_gelu_identities_and_limits():
    g = lambda x: oracle.act(x, oracle.ACT_GELU)
    for x in np.linspace(-8, 8, 161):
        # x*Phi(x) - (-x)*Phi(-x) = x*(Phi(x) + 1 - Phi(x)) = x
        assert abs(g(x) - g(-x) - x) <= 1e-14 * max(1.0, abs(x))
    for x in [6.0, 8.0, 20.0, 1000.0]:
        assert abs(g(x) - x) < 1e-8 * x
    for x in [-10.0, -20.0, -1000.0]:
        assert -1e-20 < g(x) <= 0.0
    assert g(0.0) == 0.0
    # the minimum of x*Phi(x) is about -0.17 near x = -0.75
    vals = [g(x) for x in np.linspace(-3, 0, 3001)]
    assert -0.1701 < min(vals) < -0.1699


def test_relu_and_identity():
    r = lambda x: oracle.act(x, oracle.ACT_RELU)
    assert r(3.5) == 3.5 and r(-3.5) == 0.0 and r(0.0) == 0.0 and r(1e-300) == 1e-300
    assert oracle.act(-2.25, oracle.ACT_NONE) == -2.25


# ---- the product -----------------------------------------------------------------------

def test_textbook_examples(golden_dir):
    acts = {"none": oracle.ACT_NONE, "gelu": oracle.ACT_GELU, "relu": oracle.ACT_RELU,
            "softmax": oracle.ACT_SOFTMAX}
    cases = _read_textbook(os.path.join(golden_dir, "gemm_textbook.txt"))
    assert len(cases) >= 8
    for c in cases:
        A = np.array(c["A"], dtype=np.float16).reshape(c["M"], c["K"])
        B = np.array(c["B"], dtype=np.float16).reshape(c["K"], c["N"])
        bias = None if c["bias"] is None else np.array(c["bias"], dtype=np.float16)
        want = np.array(c["C"], dtype=np.float16).reshape(c["M"], c["N"])
        got, _, _ = oracle.gemm(A, B, bias, acts[c["act"]])
        assert np.array_equal(got.view(np.uint16), want.view(np.uint16)), (c["name"], got, want)


def test_identity_products():
    A = inputs.random_fp16((48, 48), seed=11).numpy()
    eye = np.eye(48, dtype=np.float16)
    got, _, _ = oracle.gemm(eye, A)
    assert np.array_equal(got.view(np.uint16), A.view(np.uint16))
    R = inputs.random_fp16((40, 48), seed=12).numpy()
    got, _, _ = oracle.gemm(R, eye)
    assert np.array_equal(got.view(np.uint16), R.view(np.uint16))


@pytest.mark.parametrize("K", [1, 7, 256, 2048, 4096])
def test_all_ones_gives_k(K):
    A = np.ones((3, K), dtype=np.float16)
    B = np.ones((K, 5), dtype=np.float16)
    got, f64, _ = oracle.gemm(A, B, want_f64=True)
    assert np.all(f64 == K)
    assert np.all(got == np.float16(K))  # K up to 2048 and powers of two are exact in FP16


def _brute(A, B, bias, act):
    M, K = A.shape
    N = B.shape[1]
    a = A.astype(np.float64)
    b = B.astype(np.float64)
    out = np.zeros((M, N), dtype=np.float64)
    for m in range(M):
        for n in range(N):
            s = 0.0
            for k in range(K):
                s += float(a[m, k]) * float(b[k, n])
            if bias is not None:
                s += float(bias[n])
            if act == oracle.ACT_GELU:
                s = 0.5 * s * (1.0 + math.erf(s / math.sqrt(2.0)))
            elif act == oracle.ACT_RELU:
                s = max(s, 0.0)
            out[m, n] = s
    return out


def test_brute_force_tiny_shapes():
    seed = 100
    for M in range(1, 8):
        for N in (1, 2, 3, 5):
            for K in (1, 2, 3):
                for act in (oracle.ACT_NONE, oracle.ACT_GELU, oracle.ACT_RELU):
                    seed += 1
                    A = inputs.random_fp16((M, K), seed).numpy() * np.float16(4)
                    B = inputs.random_fp16((K, N), seed + 1000).numpy()
                    bias = inputs.random_fp16((N,), seed + 2000).numpy() if seed % 2 else None
                    want = _brute(A, B, bias, act)
                    got, f64, _ = oracle.gemm(A, B, bias, act, want_f64=True)
                    # the sum is bit-identical (same order, exact products); GELU may differ
                    # in the last bits (x/sqrt(2) here, x*(1/sqrt(2)) in the oracle; 1+erf(x) cancels
                    # for x << 0, so compare absolutely there)
                    if act == oracle.ACT_GELU:
                        assert np.allclose(f64, want, rtol=1e-14, atol=1e-15)
                    else:
                        assert np.array_equal(f64, want)
                    with np.errstate(over="ignore"):
                        wh = want.astype(np.float16)
                    assert np.array_equal(got.view(np.uint16), wh.view(np.uint16))


@pytest.mark.parametrize("shape", [(64, 64, 64), (130, 96, 200), (257, 136, 512)])
@pytest.mark.parametrize("act", [0, 1, 2])
def test_against_numpy_matmul(shape, act):
    M, N, K = shape
    A = inputs.random_fp16((M, K), 21).numpy()
    B = inputs.random_fp16((K, N), 22).numpy()
    bias = inputs.random_fp16((N,), 23).numpy()
    s = A.astype(np.float64) @ B.astype(np.float64) + bias.astype(np.float64)[None, :]
    if act == oracle.ACT_GELU:
        from scipy.special import erf
        s = 0.5 * s * (1.0 + erf(s / np.sqrt(2.0)))
    elif act == oracle.ACT_RELU:
        s = np.maximum(s, 0.0)
    got, f64, _ = oracle.gemm(A, B, bias, act, want_f64=True)
    scale = np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64)) + 1.0
    assert np.all(np.abs(f64 - s) <= 1e-13 * scale)
    # FP16 rounding agrees except where the two sums straddle a rounding boundary
    wh = s.astype(np.float16).view(np.uint16)
    mism = got.view(np.uint16) != wh
    assert mism.sum() <= 2


def test_row_sample_equals_full():
    A = inputs.random_fp16((300, 160), 31).numpy()
    B = inputs.random_fp16((160, 72), 32).numpy()
    bias = inputs.random_fp16((72,), 33).numpy()
    full, _, _ = oracle.gemm(A, B, bias, oracle.ACT_GELU)
    rows = inputs.sample_rows(300, 37, seed=5, include_last=8).numpy()
    part, _, _ = oracle.gemm(A, B, bias, oracle.ACT_GELU, rows=rows, threads=3)
    assert np.array_equal(part.view(np.uint16), full[rows].view(np.uint16))
    assert rows[-8:].tolist() == list(range(292, 300))


def test_threads_do_not_change_results():
    A = inputs.random_fp16((33, 40), 41).numpy()
    B = inputs.random_fp16((40, 24), 42).numpy()
    one, _, used1 = oracle.gemm(A, B, threads=1)
    many, _, used = oracle.gemm(A, B, threads=5)
    assert used1 == 1 and used == 5
    assert np.array_equal(one.view(np.uint16), many.view(np.uint16))


def test_bad_arguments_rejected():
    A = np.zeros((4, 4), np.float16)
    with pytest.raises(RuntimeError):
        oracle.gemm(A, A, rows=[0, 4])
    with pytest.raises(RuntimeError):
        oracle.gemm(A, A, act_code=7)
    with pytest.raises(ValueError):
        oracle.gemm(A, np.zeros((3, 4), np.float16))


def test_empty_shapes():
    got, _, _ = oracle.gemm(np.zeros((0, 4), np.float16), np.zeros((4, 3), np.float16))
    assert got.shape == (0, 3)
    # K = 0: the sum is empty, only the bias (then the activation) remains
    bias = np.array([1.5, -2.0], np.float16)
    got, _, _ = oracle.gemm(np.zeros((2, 0), np.float16), np.zeros((0, 2), np.float16), bias,
                            oracle.ACT_RELU)
    assert got.tolist() == [[1.5, 0.0], [1.5, 0.0]]


# ---- input generators (shared by both sides; no arithmetic of the method) --------------

def test_inputs_are_seeded_and_fp16():
    w = inputs.WORKLOADS["gemm_2048_bias_gelu"]
    small = inputs.Workload("t", 64, 48, 32, "gelu", True)
    A1, B1, b1 = inputs.make_inputs(small)
    A2, B2, b2 = inputs.make_inputs(small)
    assert A1.dtype == torch.float16 and A1.shape == (64, 32) and B1.shape == (32, 48)
    assert torch.equal(A1, A2) and torch.equal(B1, B2) and torch.equal(b1, b2)
    assert float(A1.abs().max()) <= 1.0 and w.flops == 2 * 2048 ** 3
    mlp = inputs.WORKLOADS["mlp_up_8200x4096x16384_bias_gelu"]
    rows = inputs.sample_rows(mlp.M, mlp.sample_rows, include_last=mlp.include_last)
    assert rows.numel() == 512 and rows.unique().numel() == 512
    assert rows[-8:].tolist() == list(range(8192, 8200))


# ---- row-wise softmax ------------------------------------------------------------------

def test_softmax_textbook_examples(golden_dir):
    n = 0
    for line in open(os.path.join(golden_dir, "softmax_textbook.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        xs, ys = line.split("|")
        x = np.array([float(v) for v in xs.split()], dtype=np.float16)[None, :]
        want = np.array([float(v) for v in ys.split()])
        got, f64 = oracle.softmax_rows(x, want_f64=True)
        # x is rounded to FP16 first (ln 3 is not exact in FP16); allow that shift
        assert np.allclose(f64[0], want, rtol=0, atol=2e-4 if "1.0986" in xs else 1e-9), (line, f64)
        assert np.array_equal(got[0].view(np.uint16), f64[0].astype(np.float16).view(np.uint16))
        n += 1
    assert n == 4


def test_softmax_invariants():
    rng = np.random.default_rng(3)
    x = (np.round(rng.uniform(-4, 4, (37, 50)) * 64) / 64).astype(np.float16)
    y, f64 = oracle.softmax_rows(x, want_f64=True)
    assert np.allclose(f64.sum(axis=1), 1.0, rtol=0, atol=1e-13)
    assert np.all(f64 > 0)
    # adding a constant to a row changes nothing (x + 8 is exact in FP16 here)
    y2, f2 = oracle.softmax_rows((x.astype(np.float64) + 8.0).astype(np.float16), want_f64=True)
    assert np.array_equal(f64, f2) and np.array_equal(y.view(np.uint16), y2.view(np.uint16))
    # the largest entry of a row gets the largest probability; order is preserved
    assert np.array_equal(np.argmax(f64, axis=1), np.argmax(x.astype(np.float64), axis=1))
    # a uniform row is 1/n everywhere
    u, fu = oracle.softmax_rows(np.full((2, 16), 3.5, np.float16), want_f64=True)
    assert np.all(fu == 1.0 / 16)


def test_softmax_against_scipy_and_brute_force():
    from scipy.special import softmax as sp_softmax
    x = inputs.random_fp16((64, 300), 91, scale=1.0).numpy() * np.float16(6)
    _, f64 = oracle.softmax_rows(x, want_f64=True)
    assert np.allclose(f64, sp_softmax(x.astype(np.float64), axis=1), rtol=1e-13, atol=1e-300)
    small = x[:3, :5]
    _, fs = oracle.softmax_rows(small, want_f64=True)
    for r in range(3):
        e = [math.exp(float(v)) for v in small[r].astype(np.float64)]
        s = sum(e)
        assert np.allclose(fs[r], [v / s for v in e], rtol=1e-14, atol=0)


def test_softmax_extremes_and_empty():
    x = np.full((1, 8), -11.0, np.float16)
    x[0, 3] = 11.0
    y, f64 = oracle.softmax_rows(x, want_f64=True)
    assert abs(f64[0, 3] - 1.0) < 1e-8 and np.all(f64[0, np.arange(8) != 3] < 3e-10)
    assert float(y[0, 3]) == 1.0
    y0, _ = oracle.softmax_rows(np.zeros((0, 5), np.float16))
    assert y0.shape == (0, 5)


def test_gemm_softmax_epilogue_against_numpy():
    from scipy.special import softmax as sp_softmax
    for (M, N, K) in [(37, 8, 5), (64, 200, 96), (130, 256, 300)]:
        A = inputs.random_fp16((M, K), 51 + N).numpy()
        B = inputs.random_fp16((K, N), 52 + N).numpy()
        bias = inputs.random_fp16((N,), 53 + N).numpy()
        logits = A.astype(np.float64) @ B.astype(np.float64) + bias.astype(np.float64)
        got, f64, _ = oracle.gemm(A, B, bias, oracle.ACT_SOFTMAX, want_f64=True)
        assert np.allclose(f64, sp_softmax(logits, axis=1), rtol=1e-12, atol=1e-300)
        assert np.allclose(f64.sum(axis=1), 1.0, atol=1e-13)
        # the logits are not rounded to FP16 before the softmax: compare with the rounded path
        rounded, _ = oracle.softmax_rows(logits.astype(np.float16))
        assert np.abs(rounded.astype(np.float64) - got.astype(np.float64)).max() < 0.05
        # row sampling agrees with the full computation
        rows = [0, M // 2, M - 1]
        part, _, _ = oracle.gemm(A, B, bias, oracle.ACT_SOFTMAX, rows=rows)
        assert np.array_equal(part.view(np.uint16), got[rows].view(np.uint16))


# ---- attention forward -------------------------------------------------------------------

def _np_attention(Q, K, V, scale, causal):
    from scipy.special import softmax as sp_softmax
    q, k, v = (t.astype(np.float64) for t in (Q, K, V))
    s = scale * np.einsum("hid,hjd->hij", q, k)
    if causal:
        Sq, Sk = s.shape[1], s.shape[2]
        s = np.where(np.arange(Sk)[None, None, :] <= np.arange(Sq)[None, :, None], s, -np.inf)
    return np.einsum("hij,hjd->hid", sp_softmax(s, axis=2), v)


@pytest.mark.parametrize("causal", [False, True])
def test_attention_against_scipy_composition(causal):
    rng = np.random.default_rng(5 + causal)
    H, S, D = 3, 67, 32
    Q, K, V = (rng.normal(0, 1, (H, S, D)).astype(np.float16) for _ in range(3))
    out, f64 = oracle.attention(Q, K, V, 1 / np.sqrt(D), causal, want_f64=True)
    want = _np_attention(Q, K, V, 1 / np.sqrt(D), causal).reshape(H * S, D)
    assert np.allclose(f64, want, rtol=1e-12, atol=1e-13)
    assert np.array_equal(out.view(np.uint16), f64.astype(np.float16).view(np.uint16))


def test_attention_special_cases():
    rng = np.random.default_rng(9)
    H, S, D = 2, 9, 8
    V = rng.uniform(-1, 1, (H, S, D)).astype(np.float16)
    K = rng.uniform(-1, 1, (H, S, D)).astype(np.float16)
    # one key: the output is that key's value row, exactly
    out, f = oracle.attention(rng.normal(0, 1, (H, 1, D)).astype(np.float16), K[:, :1], V[:, :1], 0.3, False,
                              want_f64=True)
    assert np.array_equal(f, V[:, 0].astype(np.float64))
    # causal: the first query sees only the first key
    Q = rng.normal(0, 1, (H, S, D)).astype(np.float16)
    _, f = oracle.attention(Q, K, V, 0.3, True, rows=[(0, 0), (1, 0)], want_f64=True)
    assert np.array_equal(f, V[:, 0].astype(np.float64))
    # zero queries: every score is equal, so the output is the mean (causal: prefix mean)
    Z = np.zeros((H, S, D), np.float16)
    _, f = oracle.attention(Z, K, V, 0.3, False, want_f64=True)
    assert np.allclose(f.reshape(H, S, D), V.astype(np.float64).mean(axis=1, keepdims=True).repeat(S, 1), atol=1e-15)
    _, f = oracle.attention(Z, K, V, 0.3, True, want_f64=True)
    pref = np.cumsum(V.astype(np.float64), axis=1) / np.arange(1, S + 1)[None, :, None]
    assert np.allclose(f.reshape(H, S, D), pref, atol=1e-15)
    # a very large scale makes the softmax one-hot on the best-matching key
    _, f = oracle.attention(K, K, V, 200.0, False, rows=[(0, 4)], want_f64=True)
    best = np.argmax(K[0].astype(np.float64) @ K[0, 4].astype(np.float64))
    assert np.allclose(f[0], V[0, best].astype(np.float64), atol=1e-6)


def test_attention_brute_force_tiny():
    rng = np.random.default_rng(2)
    H, S, D = 1, 4, 3
    Q, K, V = (rng.uniform(-2, 2, (H, S, D)).astype(np.float16) for _ in range(3))
    _, f = oracle.attention(Q, K, V, 0.7, True, want_f64=True)
    for i in range(S):
        s = [0.7 * sum(float(Q[0, i, d]) * float(K[0, j, d]) for d in range(D)) for j in range(i + 1)]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        for d in range(D):
            want = sum(e[j] * float(V[0, j, d]) for j in range(i + 1)) / sum(e)
            assert abs(f[i, d] - want) < 1e-14
