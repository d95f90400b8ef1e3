"""Parity of the FlashAttention forward kernel (through the C ABI) with the FP64 oracle.

Tolerance: the kernel rounds each probability p to FP16 before the P V product (relative
error at most 2^-12 per term, unbiased) while it divides by the FP32 sum of the unrounded p;
the resulting error in O is at most about 2^-12 * max|V| and typically far smaller, plus
one FP16 rounding of O (at most 2^-11 * |O|). Checked: elementwise
|O - ref| <= 3e-3 + 4e-3 * |ref| and relative Frobenius error <= 2e-3, no NaN/Inf.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import tensor_core_gemm_tcgen05_gb300 as g
from tensor_core_gemm_tcgen05_gb300 import inputs

pytestmark = pytest.mark.gpu
D = 128


@pytest.fixture(scope="module")
def ctx():
    from tensor_core_gemm_tcgen05_gb300 import _build
    _build.build()
    c = g.Context(0)
    yield c
    c.close()


def qkv(H, Sq, Sk, seed, dist="normal"):
    Q = inputs.random_fp16((H, Sq, D), seed, dist)
    K = inputs.random_fp16((H, Sk, D), seed + 1, dist)
    V = inputs.random_fp16((H, Sk, D), seed + 2, dist)
    return Q, K, V


def run(ctx, Q, K, V, scale, causal):
    dev = torch.device("cuda:0")
    H, Sq, _ = Q.shape
    guard = torch.full((H * Sq * D + 64,), 0x7E00, dtype=torch.int16, device=dev)
    O = guard[: H * Sq * D].view(torch.float16).view(H, Sq, D)
    g.attention(ctx, Q.to(dev), K.to(dev), V.to(dev), scale=scale, causal=causal, out=O)
    torch.cuda.synchronize()
    assert g.gemm_last_device_error(ctx) == (g.GEMM_OK, 0)
    assert torch.all(guard[H * Sq * D:] == 0x7E00), "wrote past the end of O"
    return O.cpu()


def check(got, ref, what):
    got = np.asarray(got, dtype=np.float16).astype(np.float64)
    ref = np.asarray(ref, dtype=np.float16).astype(np.float64)
    assert np.all(np.isfinite(got)), what
    err = np.abs(got - ref)
    bad = err > 3e-3 + 4e-3 * np.abs(ref)
    assert not bad.any(), (what, int(bad.sum()), float(err.max()))
    fro = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert fro <= 2e-3, (what, fro)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,Sq,Sk", [(1, 128, 128), (2, 256, 256), (3, 200, 200), (2, 1000, 1000), (1, 64, 64),
                                     (1, 8, 8)], ids=lambda v: str(v))
def test_attention_matches_oracle(ctx, H, Sq, Sk, causal):
    Q, K, V = qkv(H, Sq, Sk, 10 * Sq + H)
    scale = 1.0 / math.sqrt(D)
    O = run(ctx, Q, K, V, scale, causal)
    ref, _ = oracle.attention(Q, K, V, scale, causal)
    check(O.reshape(H * Sq, D).numpy(), ref, f"attention H={H} Sq={Sq} Sk={Sk} causal={causal}")


def test_attention_unequal_lengths_non_causal(ctx):
    Q, K, V = qkv(2, 100, 300, 77)
    O = run(ctx, Q, K, V, 0.09, False)
    ref, _ = oracle.attention(Q, K, V, 0.09, False)
    check(O.reshape(200, D).numpy(), ref, "Sq=100 Sk=300")


@pytest.mark.parametrize("Sq,Sk", [(100, 300), (300, 100), (128, 1000), (1000, 128), (257, 513)],
                         ids=lambda v: str(v))
def test_attention_unequal_lengths_causal(ctx, Sq, Sk):
    """Causal with seq_q != seq_k: query i sees keys 0 .. min(i, seq_k - 1), the mask aligned
    at the first key as the ABI and the oracle define it. With seq_q < seq_k the keys past the
    last query are never seen; with seq_q > seq_k every query from seq_k on sees all keys."""
    Q, K, V = qkv(2, Sq, Sk, 7 * Sq + Sk)
    O = run(ctx, Q, K, V, 0.09, True)
    ref, _ = oracle.attention(Q, K, V, 0.09, True)
    check(O.reshape(2 * Sq, D).numpy(), ref, f"causal Sq={Sq} Sk={Sk}")


def test_attention_long_sequence_sampled_rows(ctx):
    H, S = 4, 4096
    Q, K, V = qkv(H, S, S, 5)
    for causal in (False, True):
        O = run(ctx, Q, K, V, 1.0 / math.sqrt(D), causal)
        rows = [(h, int(i)) for h in range(H) for i in inputs.sample_rows(S, 64, seed=h + 3 * causal, include_last=2)]
        ref, _ = oracle.attention(Q, K, V, 1.0 / math.sqrt(D), causal, rows=rows)
        got = np.stack([O[h, i].numpy() for h, i in rows])
        check(got, ref, f"S=4096 causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_attention_full_size_every_head(ctx, causal):
    """The benchmark's shape, 64 heads x 4096 tokens: a full grid of CTAs, so that races
    between the kernel's warps (which small grids can hide) show. Every head against the
    FP64 oracle on sampled rows, and every row against plain FP32 PyTorch arithmetic on the
    GPU (softmax of the FP32 scores, times V): same elementwise bar."""
    H, S = 64, 4096
    Q, K, V = qkv(H, S, S, 17)
    scale = 1.0 / math.sqrt(D)
    O = run(ctx, Q, K, V, scale, causal)
    rows = [(h, int(i)) for h in range(H) for i in inputs.sample_rows(S, 4, seed=100 + h, include_last=1)]
    ref, _ = oracle.attention(Q, K, V, scale, causal, rows=rows)
    check(np.stack([O[h, i].numpy() for h, i in rows]), ref, f"every head, causal={causal}")
    dev = torch.device("cuda:0")
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        mask = torch.ones(S, S, dtype=torch.bool, device=dev).tril() if causal else None
        worst = 0.0
        for h in range(H):
            s_ = (Q[h].to(dev).float() @ K[h].to(dev).float().T) * scale
            if mask is not None:
                s_ = s_.masked_fill(~mask, float("-inf"))
            ref_h = torch.softmax(s_, dim=1) @ V[h].to(dev).float()
            err = (O[h].to(dev).float() - ref_h).abs()
            bad = err > 3e-3 + 4e-3 * ref_h.abs()
            assert not bool(bad.any()), (h, int(bad.sum()), float(err.max()))
            worst = max(worst, float(err.max()))
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    assert worst < 3e-3


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,Sq,Sk", [(200, 256, 256), (160, 300, 700), (170, 520, 130), (4, 8192, 8192)],
                         ids=lambda v: str(v))
def test_attention_several_items_per_cta(ctx, H, Sq, Sk, causal):
    """More work items (a head and a block of 256 queries) than SMs: each CTA of the
    persistent grid runs several items in turn, and when causal their key counts differ from
    one item to the next. Every row against plain FP32 PyTorch on the GPU, sampled rows of
    every head against the FP64 oracle, same elementwise bar."""
    Q, K, V = qkv(H, Sq, Sk, 3 * H + Sq + Sk)
    scale = 0.09
    O = run(ctx, Q, K, V, scale, causal)
    rows = [(h, int(i)) for h in range(H) for i in inputs.sample_rows(Sq, 6, seed=h, include_last=1)]
    ref, _ = oracle.attention(Q, K, V, scale, causal, rows=rows)
    check(np.stack([O[h, i].numpy() for h, i in rows]), ref, f"H={H} Sq={Sq} Sk={Sk} causal={causal}")
    dev = torch.device("cuda:0")
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        # query i sees keys 0 .. min(i, Sk - 1) when causal
        mask = (torch.arange(Sk, device=dev)[None, :] <= torch.arange(Sq, device=dev)[:, None]) if causal else None
        for h in range(H):
            s_ = (Q[h].to(dev).float() @ K[h].to(dev).float().T) * scale
            if mask is not None:
                s_ = s_.masked_fill(~mask, float("-inf"))
            ref_h = torch.softmax(s_, dim=1) @ V[h].to(dev).float()
            err = (O[h].to(dev).float() - ref_h).abs()
            bad = err > 3e-3 + 4e-3 * ref_h.abs()
            assert not bool(bad.any()), (h, int(bad.sum()), float(err.max()))
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


def test_attention_special_cases(ctx):
    H, S = 2, 384
    _, K, V = qkv(H, S, S, 31)
    # zero queries: uniform attention, so O is the mean of the visible values
    Z = torch.zeros(H, S, D, dtype=torch.float16)
    O = run(ctx, Z, K, V, 0.1, True).double()
    pref = torch.cumsum(V.double(), dim=1) / torch.arange(1, S + 1, dtype=torch.float64)[None, :, None]
    assert torch.allclose(O, pref, atol=2e-3, rtol=4e-3)
    O = run(ctx, Z, K, V, 0.1, False).double()
    assert torch.allclose(O, V.double().mean(dim=1, keepdim=True).expand(H, S, D), atol=2e-3, rtol=4e-3)
    # causal: the first query sees only the first key, so its output is V[h][0]
    Q = inputs.random_fp16((H, S, D), 32, "normal")
    O = run(ctx, Q, K, V, 0.1, True)
    assert torch.equal(O[:, 0], V[:, 0])


def test_attention_rejects_bad_arguments(ctx):
    dev = torch.device("cuda:0")
    X = torch.zeros(1, 128, 128, dtype=torch.float16, device=dev)
    Y = torch.zeros(1, 128, 128, dtype=torch.float16, device=dev)
    L, h = g.lib(), ctx.handle
    p = X.data_ptr()
    assert L.gemm_attention_fwd(h, 1, 128, 128, 64, p, p, p, Y.data_ptr(), 0.1, 0, None) == g.GEMM_ERR_ARG
    assert L.gemm_attention_fwd(h, 1, 128, 0, 128, p, p, p, Y.data_ptr(), 0.1, 0, None) == g.GEMM_ERR_ARG
    assert L.gemm_attention_fwd(h, 1, 128, 128, 128, p, p, p, p, 0.1, 0, None) == g.GEMM_ERR_ARG   # O overlaps Q
    assert L.gemm_attention_fwd(h, 1, 128, 128, 128, p + 2, p, p, Y.data_ptr(), 0.1, 0, None) == g.GEMM_ERR_ALIGN
    assert L.gemm_attention_fwd(h, 0, 128, 128, 128, None, None, None, None, 0.1, 0, None) == g.GEMM_OK
    torch.cuda.synchronize()
