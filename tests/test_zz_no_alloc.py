"""gemm_run_noalloc, the entry point for callers that cannot allocate device memory.

Callers such as inference-engine plugins (the engine owns all device memory), real-time
loops that forbid allocation after start-up, or code that must not touch the allocator
cannot call gemm_create, which allocates the kernel's error word with cudaMalloc. For them
gemm_run_noalloc keeps that scratch in a fixed __device__ array inside the library.

The tests call it through the C ABI, several times in a row on different shapes and
epilogues (every call reuses the one array, so a call that depended on a fresh array would
show), and check every result both against gemm_run's output for the same inputs and
against the FP64 oracle, with the tolerance of the other parity tests (the softmax
epilogue: within one FP16 ulp of the oracle, rows summing to 1). The cases cover each path
of the kernel this entry point runs: ragged M and N, bias and no bias under every
activation, the single-tile row softmax (N <= 256), K = 0 (the activation of the bias),
and more tiles than SMs (every CTA loops over several tiles through both accumulators).
The file is collected last; it passes alone in a fresh process as well as after the rest
of the suite.
"""
import numpy as np
import pytest
import torch

import oracle
import tensor_core_gemm_tcgen05_gb300 as g
from tensor_core_gemm_tcgen05_gb300 import inputs
from parity import assert_parity

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def ctx():
    from tensor_core_gemm_tcgen05_gb300 import _build
    _build.build()
    torch.cuda.set_device(DEV)
    c = g.Context(0)
    yield c
    c.close()


def noalloc(M, N, K, A, B, bias, epi):
    """One call through the C ABI into a NaN-filled C; returns C on the host."""
    out = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
    stream = torch.cuda.current_stream(DEV)
    rc = g.lib().gemm_run_noalloc(M, N, K, None if A is None else A.data_ptr(), None if B is None else B.data_ptr(),
                                  None if bias is None else bias.data_ptr(), out.data_ptr(), epi, stream.cuda_stream)
    assert rc == g.GEMM_OK, g.gemm_status_string(rc)
    torch.cuda.synchronize()
    return out.cpu()


def reference(ctx, M, N, K, A, B, bias, epi):
    ref = torch.empty(M, N, dtype=torch.float16, device=DEV)
    g.gemm_run(ctx, M, N, K, A, B, bias, ref, epi)
    torch.cuda.synchronize()
    return ref.cpu()


def check_softmax(got, ref, N):
    ulp = np.maximum(np.spacing(np.abs(ref)).astype(np.float64), 2.0 ** -24)
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    assert np.all(np.isfinite(got.astype(np.float64)))
    assert np.all(err <= ulp), (float(err.max()), int((err > ulp).sum()))
    assert np.all(np.abs(got.astype(np.float64).sum(axis=1) - 1) <= N * 2.0 ** -11)


# (M, N, K, epilogue, bias?, oracle rows: None = all)
CASES = [
    (300, 512, 256, g.EPI_GELU, True, None),
    (1000, 264, 1000, g.EPI_RELU, False, None),
    (129, 200, 64, g.EPI_GELU, False, None),          # GELU without a bias, ragged N
    (300, 256, 128, g.EPI_SOFTMAX, False, None),      # one tile spans the row
    (129, 136, 64, g.EPI_SOFTMAX, True, None),        # ragged row inside one tile
    (70, 264, 0, g.EPI_GELU, True, None),             # K = 0: GELU of the bias
    (4096, 4096, 256, g.EPI_RELU, True, 256),         # 512 tiles on fewer SMs
]


def test_noalloc_matches_gemm_run_and_the_oracle_on_calls_in_a_row(ctx):
    for i, (M, N, K, epi, with_bias, nrows) in enumerate(CASES):
        dist = "normal" if epi == g.EPI_SOFTMAX else "uniform"
        A = inputs.random_fp16((M, K), 500 + i, dist)
        B = inputs.random_fp16((K, N), 600 + i, "normal_inv_k" if epi == g.EPI_SOFTMAX else "uniform", k=max(K, 1))
        bias = inputs.random_fp16((N,), 700 + i) if with_bias else None
        dA = A.to(DEV) if K > 0 else None
        dB = B.to(DEV) if K > 0 else None
        dbias = bias.to(DEV) if bias is not None else None
        got = noalloc(M, N, K, dA, dB, dbias, epi)
        what = f"noalloc call {i + 1}: {M}x{N}x{K} epi={epi} bias={with_bias}"
        # against the existing entry point
        assert_parity(got.numpy(), reference(ctx, M, N, K, dA, dB, dbias, epi).numpy(), what + " vs gemm_run")
        # against the oracle
        rows = None if nrows is None else inputs.sample_rows(M, nrows, seed=40 + i, include_last=4).numpy()
        ref, _, _ = oracle.gemm(A, B, bias, epi, rows=rows)
        sel = got.numpy() if rows is None else got.numpy()[rows]
        if epi == g.EPI_SOFTMAX:
            check_softmax(sel, ref, N)
        else:
            assert_parity(sel, ref, what + " vs oracle")
