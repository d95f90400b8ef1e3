"""Parity of the row-wise softmax kernel (through the C ABI) with the FP64 oracle.

Bound: every output within one FP16 ulp of the oracle's FP16 result (the GPU rounds an
FP32 value, the oracle an FP64 one; ex2.approx / exp2f and the FP32 sum add a few 1e-7
relative), with the ulp of the subnormal range (2^-24) for the smallest outputs. Guard
bands around Y must stay untouched.
"""
import numpy as np
import pytest
import torch

import oracle
import tensor_core_gemm_tcgen05_gb300 as g
from tensor_core_gemm_tcgen05_gb300 import inputs

pytestmark = pytest.mark.gpu
GUARD = 0x7E00


@pytest.fixture(scope="module")
def ctx():
    from tensor_core_gemm_tcgen05_gb300 import _build
    _build.build()
    c = g.Context(0)
    yield c
    c.close()


def assert_softmax_close(got, ref, what):
    got = np.asarray(got, dtype=np.float16)
    ref = np.asarray(ref, dtype=np.float16)
    assert np.all(np.isfinite(got.astype(np.float64))), what
    ulp = np.maximum(np.spacing(np.abs(ref)).astype(np.float64), 2.0 ** -24)
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    bad = err > ulp
    assert not bad.any(), (what, int(bad.sum()), float(err.max()))


def run(ctx, X, inplace=False):
    rows, cols = X.shape
    dev = torch.device("cuda:0")
    if inplace:
        Y = X.to(dev).clone()
        g.row_softmax(ctx, Y, out=Y)
        torch.cuda.synchronize()
        return Y.cpu()
    buf = torch.full(((rows + 2) * cols + 24,), GUARD, dtype=torch.int16, device=dev)
    Y = buf[: rows * cols].view(torch.float16).view(rows, cols)
    g.row_softmax(ctx, X.to(dev), out=Y)
    torch.cuda.synchronize()
    assert torch.all(buf[rows * cols:] == GUARD), "wrote past the end of Y"
    return Y.cpu()


# Every dispatch path and its edges: rows in registers with a warp per row and 1/2/4/8
# vectors per lane (up to 256, 512, 1024, 2048 columns) or a 256-thread CTA per row and
# 2/4/8 vectors per thread (up to 4096, 8192, 16384), and the two-pass streaming kernel
# beyond; full and ragged last vectors.
@pytest.mark.parametrize("shape", [(1, 8), (3, 16), (1000, 264), (5, 520), (77, 2048), (64, 2056), (17, 6144),
                                   (513, 16384), (33, 16392), (3, 24576), (9, 32768), (4, 32776), (5, 65536),
                                   (2, 8), (300, 1000)],
                         ids=lambda s: "x".join(map(str, s)))
def test_row_softmax_matches_oracle(ctx, shape):
    rows, cols = shape
    X = inputs.random_fp16(shape, 4000 + rows + cols, scale=1.0) * 8
    Y = run(ctx, X)
    ref, _ = oracle.softmax_rows(X)
    assert_softmax_close(Y.numpy(), ref, f"softmax {shape}")
    sums = Y.double().sum(dim=1)
    assert torch.all((sums - 1).abs() <= cols * 2.0 ** -11)


def test_row_softmax_textbook_row_padded_with_minus_inf(ctx):
    X = torch.full((2, 8), float("-inf"), dtype=torch.float16)
    X[0, :3] = torch.tensor([1.0, 2.0, 3.0])
    X[1, :4] = torch.tensor([0.0, 0.0, 0.0, 0.0])
    Y = run(ctx, X).double()
    assert torch.allclose(Y[0, :3], torch.tensor([0.0900305732, 0.2447284711, 0.6652409558], dtype=torch.float64),
                          atol=3e-4, rtol=0)
    assert torch.all(Y[0, 3:] == 0) and torch.all(Y[1, :4] == 0.25) and torch.all(Y[1, 4:] == 0)


@pytest.mark.parametrize("cols", [2048, 16384, 40000])
def test_row_softmax_masked_prefix(ctx, cols):
    """Rows whose leading columns are -inf (a masked prefix): the streamed kernel meets whole
    steps of -inf before the first finite value; they must add nothing (no NaN)."""
    X = inputs.random_fp16((3, cols), 91, scale=1.0) * 8
    X[0, : cols - 16] = float("-inf")    # only the last 16 columns are finite
    X[1, : cols // 2] = float("-inf")
    Y = run(ctx, X)
    ref, _ = oracle.softmax_rows(X)
    assert_softmax_close(Y.numpy(), ref, f"masked prefix, {cols} columns")
    assert torch.all(Y[0, : cols - 16] == 0) and torch.all(Y[1, : cols // 2] == 0)


def test_row_softmax_in_place_and_large_values(ctx):
    X = inputs.random_fp16((40, 4096), 77) * 60   # logits up to +-60: exp would overflow without the max
    Y = run(ctx, X, inplace=True)
    ref, _ = oracle.softmax_rows(X)
    assert_softmax_close(Y.numpy(), ref, "in place")


def test_row_softmax_rejects_bad_arguments(ctx):
    dev = torch.device("cuda:0")
    X = torch.zeros(4, 16, dtype=torch.float16, device=dev)
    L, h = g.lib(), ctx.handle
    assert L.gemm_row_softmax(h, 4, 12, X.data_ptr(), X.data_ptr(), None) == g.GEMM_ERR_ALIGN
    assert L.gemm_row_softmax(h, 4, 16, X.data_ptr() + 2, X.data_ptr() + 2, None) == g.GEMM_ERR_ALIGN
    assert L.gemm_row_softmax(h, 4, 16, X.data_ptr(), X.data_ptr() + 16, None) == g.GEMM_ERR_ARG
    assert L.gemm_row_softmax(h, -1, 16, X.data_ptr(), X.data_ptr(), None) == g.GEMM_ERR_ARG
    assert L.gemm_row_softmax(h, 0, 16, None, None, None) == g.GEMM_OK
    host = np.zeros(64, np.float16)
    hp = (host.ctypes.data + 15) // 16 * 16
    assert L.gemm_row_softmax(h, 2, 8, hp, X.data_ptr(), None) == g.GEMM_ERR_DEVICE
