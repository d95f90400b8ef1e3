"""gemm_run_noalloc, the entry point for callers that cannot allocate device memory.

Callers such as inference-engine plugins (the engine owns all device memory), real-time
loops that forbid allocation after start-up, or code that must not touch the allocator
cannot call gemm_create, which allocates the kernel's error word with cudaMalloc. For them
gemm_run_noalloc keeps that scratch in a fixed __device__ array inside the library. This
test calls it through the C ABI twice in a row (different shapes and epilogues, so the
second call starts from the first call's leftover scratch) and checks each result against
gemm_run's output for the same inputs, with the tolerance of the other parity tests.
It lives in its own file, collected last, and passes alone in a fresh process as well as
after the rest of the suite.
"""
import pytest
import torch

import tensor_core_gemm_tcgen05_gb300 as g
from tensor_core_gemm_tcgen05_gb300 import inputs
from parity import assert_parity

pytestmark = pytest.mark.gpu


def test_noalloc_matches_gemm_run_on_two_calls_in_a_row():
    from tensor_core_gemm_tcgen05_gb300 import _build
    _build.build()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    L = g.lib()
    cases = [(300, 512, 256, g.EPI_GELU, True), (1000, 264, 1000, g.EPI_RELU, False)]
    with g.Context(0) as ctx:
        for i, (M, N, K, epi, with_bias) in enumerate(cases):
            A = inputs.random_fp16((M, K), 500 + i).to(dev)
            B = inputs.random_fp16((K, N), 600 + i).to(dev)
            bias = inputs.random_fp16((N,), 700 + i).to(dev) if with_bias else None
            ref = torch.empty(M, N, dtype=torch.float16, device=dev)
            g.gemm(ctx, A, B, bias, epi, out=ref)
            out = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
            stream = torch.cuda.current_stream(dev)
            rc = L.gemm_run_noalloc(M, N, K, A.data_ptr(), B.data_ptr(),
                                    None if bias is None else bias.data_ptr(), out.data_ptr(), epi,
                                    stream.cuda_stream)
            assert rc == g.GEMM_OK, g.gemm_status_string(rc)
            torch.cuda.synchronize()
            assert g.gemm_last_device_error(ctx) == (g.GEMM_OK, 0)
            assert_parity(out.cpu().numpy(), ref.cpu().numpy(), f"noalloc call {i + 1}")
