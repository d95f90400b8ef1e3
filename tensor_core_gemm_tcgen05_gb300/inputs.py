"""Seeded synthetic inputs for the FP16 GEMM ``C = act(A @ B + bias)``.

This module only draws random numbers, rounds them to FP16 once (round-to-nearest-even,
done by ``torch.Tensor.half``) and picks seeded row samples. It holds none of the GEMM's
arithmetic. The CUDA path and the CPU oracle are both fed from here: callers copy the
same FP16 bits to the device and hand them to the oracle.

The workloads are the ones the tutorial's tensor-core GEMM and fused-epilogue sections
describe, sized for one GB300:

* "TileLang: Criando Kernels de GPU ... (noticiai.com.br)", section "GEMM com Tensor
  Cores": row-major ``A[i:i+128, k:k+32]`` and ``B[k:k+32, j:j+128]`` tiles, so A is
  M x K and B is K x N, both row-major.
* "Designing High-Performance GPU Kernels with TileLang (spaxe.top)", GEMM paragraph:
  a 2048 x 2048 FP16 GEMM (read here as M = N = K = 2048).
* "TileLang ... (pro.edgex.exchange)", fused-epilogue paragraph: bias add then GELU on
  the accumulator; "noticiai.com.br", section "GEMM com epilogo fundido": ReLU.
"""
from __future__ import annotations

import dataclasses
import math

import torch

# Epilogue codes of the C ABI (bias is applied whenever a bias vector is passed).
EPI_NONE, EPI_GELU, EPI_RELU, EPI_SOFTMAX = 0, 1, 2, 3
EPILOGUES = {"none": EPI_NONE, "gelu": EPI_GELU, "relu": EPI_RELU, "softmax": EPI_SOFTMAX}

SEED_A, SEED_B, SEED_BIAS, SEED_ROWS = 1, 2, 3, 1234


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic GEMM problem: shapes, value distributions and the epilogue."""

    name: str
    M: int
    N: int
    K: int
    epilogue: str = "none"          # "none" | "gelu" | "relu" | "softmax"
    bias: bool = False
    a_dist: str = "uniform"         # "uniform": U[-1,1]; "normal": N(0,1)
    b_dist: str = "uniform"         # "uniform": U[-1,1]; "normal_inv_k": N(0,1/K)
    bias_range: float = 1.0         # bias ~ U[-bias_range, bias_range]
    sample_rows: int | None = None  # oracle checks this many seeded full rows (None: all)
    include_last: int = 0           # ... always including the last rows of C

    @property
    def flops(self) -> int:
        """Algorithmic flops, 2*M*N*K (epilogue flops are not counted)."""
        return 2 * self.M * self.N * self.K

    @property
    def bytes(self) -> int:
        """Algorithmic DRAM bytes: read A, B (and bias) once, write C once, all FP16."""
        b = 2 * (self.M * self.K + self.K * self.N + self.M * self.N)
        return b + (2 * self.N if self.bias else 0)

    @property
    def epi_code(self) -> int:
        return EPILOGUES[self.epilogue]


# The five benchmark problems, plus the epilogue-overhead variants.
WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("gemm_256", 256, 256, 256),
        Workload("gemm_2048", 2048, 2048, 2048),
        Workload("gemm_2048_bias_gelu", 2048, 2048, 2048, "gelu", True),
        Workload("gemm_2048_bias_relu", 2048, 2048, 2048, "relu", True),
        Workload("gemm_8192", 8192, 8192, 8192, sample_rows=512),
        Workload("mlp_up_8200x4096x16384_bias_gelu", 8200, 16384, 4096, "gelu", True,
                 a_dist="normal", b_dist="normal_inv_k", bias_range=0.1,
                 sample_rows=512, include_last=8),
        # Epilogue-overhead companions of the two large problems.
        Workload("gemm_8192_bias_gelu", 8192, 8192, 8192, "gelu", True, sample_rows=512),
        Workload("mlp_up_8200x4096x16384_none", 8200, 16384, 4096, "none", False,
                 a_dist="normal", b_dist="normal_inv_k", bias_range=0.1,
                 sample_rows=512, include_last=8),
        # GEMM with the row-softmax epilogue, shaped like attention scores: 262144 query rows
        # (e.g. 128 heads x 2048 tokens) against 256 keys of dimension 128; queries N(0,1),
        # keys N(0,1/K) so the logits are about N(0,1).
        Workload("scores_262144x256x128_softmax", 262144, 256, 128, "softmax", False,
                 a_dist="normal", b_dist="normal_inv_k", sample_rows=512, include_last=8),
        # The same over rows wider than one tile: 32768 queries against 512 to 2048 keys,
        # 16384 against 4096 and 8192 against 16384.
        Workload("scores_32768x512x128_softmax", 32768, 512, 128, "softmax", False,
                 a_dist="normal", b_dist="normal_inv_k", sample_rows=256, include_last=8),
        Workload("scores_32768x1024x128_softmax", 32768, 1024, 128, "softmax", False,
                 a_dist="normal", b_dist="normal_inv_k", sample_rows=256, include_last=8),
        Workload("scores_32768x2048x128_softmax", 32768, 2048, 128, "softmax", False,
                 a_dist="normal", b_dist="normal_inv_k", sample_rows=256, include_last=8),
        Workload("scores_16384x4096x128_softmax", 16384, 4096, 128, "softmax", False,
                 a_dist="normal", b_dist="normal_inv_k", sample_rows=128, include_last=8),
        Workload("scores_8192x16384x128_softmax", 8192, 16384, 128, "softmax", False,
                 a_dist="normal", b_dist="normal_inv_k", sample_rows=64, include_last=4),
        # Few output tiles, long K: 32 tiles of 128 x 256 for ~150 SMs, the stream-K case.
        Workload("gemm_1024x1024x8192_bias_gelu", 1024, 1024, 8192, "gelu", True,
                 a_dist="normal", b_dist="normal_inv_k", bias_range=0.1, sample_rows=128, include_last=2),
    ]
}


def _draw(shape, dist: str, gen: torch.Generator, k: int, scale: float = 1.0) -> torch.Tensor:
    if dist == "uniform":
        x = torch.rand(shape, generator=gen, dtype=torch.float32) * (2.0 * scale) - scale
    elif dist == "normal":
        x = torch.randn(shape, generator=gen, dtype=torch.float32)
    elif dist == "normal_inv_k":
        x = torch.randn(shape, generator=gen, dtype=torch.float32) * (1.0 / math.sqrt(k))
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return x.half()


def make_inputs(w: Workload, seeds=(SEED_A, SEED_B, SEED_BIAS)):
    """Return host FP16 tensors (A [M,K], B [K,N], bias [N] or None), contiguous."""
    ga = torch.Generator().manual_seed(seeds[0])
    gb = torch.Generator().manual_seed(seeds[1])
    A = _draw((w.M, w.K), w.a_dist, ga, w.K)
    B = _draw((w.K, w.N), w.b_dist, gb, w.K)
    bias = None
    if w.bias:
        gbias = torch.Generator().manual_seed(seeds[2])
        bias = _draw((w.N,), "uniform", gbias, w.K, scale=w.bias_range)
    return A.contiguous(), B.contiguous(), bias


def random_fp16(shape, seed: int, dist: str = "uniform", k: int = 1, scale: float = 1.0):
    """A seeded FP16 host tensor for ad-hoc shapes (tests of ragged and tiny sizes)."""
    g = torch.Generator().manual_seed(seed)
    return _draw(tuple(shape), dist, g, k, scale).contiguous()


def sample_rows(M: int, n: int | None, seed: int = SEED_ROWS, include_last: int = 0) -> torch.Tensor:
    """Sorted int64 row indices: ``n`` distinct seeded rows of ``range(M)`` (all rows when
    ``n`` is None or >= M), always containing the last ``include_last`` rows."""
    if n is None or n >= M:
        return torch.arange(M, dtype=torch.int64)
    last = torch.arange(M - include_last, M, dtype=torch.int64)
    g = torch.Generator().manual_seed(seed)
    pool = torch.randperm(M - include_last, generator=g)[: n - include_last].to(torch.int64)
    return torch.sort(torch.cat([pool, last])).values
