"""Parity of the CUDA path (through the C ABI) with the FP64 CPU oracle, on a GB300.

Inputs come from the seeded generators in ``tensor_core_gemm_tcgen05_gb300.inputs``; the
same FP16 bits go to the device and to the oracle. The tolerance is the one in
``tests/parity.py`` (elementwise 1e-2 + 4e-3*|ref|, relative Frobenius 1e-3, no NaN/Inf).
Every output buffer carries guard rows and a guard tail filled with a NaN pattern, which
must come back untouched (nothing may be written past row M-1 or column N-1).
"""
import numpy as np
import pytest
import torch

import oracle
import tensor_core_gemm_tcgen05_gb300 as g
from tensor_core_gemm_tcgen05_gb300 import inputs
from parity import assert_parity

pytestmark = pytest.mark.gpu

GUARD = 0x7E00  # an FP16 NaN


@pytest.fixture(scope="module")
def ctx():
    from tensor_core_gemm_tcgen05_gb300 import _build
    _build.build()
    c = g.Context(0)
    yield c
    c.close()


FORCE = {
    "single": g.GEMM_DEBUG_FORCE_SINGLE,
    "pair": g.GEMM_DEBUG_FORCE_PAIR,
    "streamk": g.GEMM_DEBUG_FORCE_SINGLE | g.GEMM_DEBUG_FORCE_STREAMK,
    "splitk": g.GEMM_DEBUG_FORCE_SPLITK,
}


@pytest.fixture(params=list(FORCE))
def kctx(ctx, request):
    """The context with the kernel choice forced: one-CTA 128x256 tiles, CTA-pair 256x256
    tiles (cta_group::2), one-CTA tiles under stream-K with one k-block unit per CTA (up to
    one CTA per SM), so that most tiles are cut into several parts summed through the
    workspace, or one-CTA tiles under split-K (a cluster of 8, 4 or 2 CTAs per tile, the
    largest not above the k-blocks, partials summed over distributed shared memory; K under
    two k-blocks keeps whole tiles)."""
    if request.param == "pair" and g.gemm_num_pairs(ctx) == 0:
        pytest.skip("the pair kernel cannot run on this device")
    g.gemm_set_debug(ctx, FORCE[request.param])
    yield ctx
    g.gemm_set_debug(ctx, g.GEMM_DEBUG_NONE)


def run_guarded(ctx, A, B, bias, epi, stream=None):
    """Run the GEMM into a buffer with 3 guard rows and a 40-element guard tail; check the
    guards and return the M x N result on the host."""
    M, K = A.shape
    N = B.shape[1]
    dev = torch.device("cuda:0")
    buf = torch.full(((M + 3) * N + 40,), GUARD, dtype=torch.int16, device=dev)
    Cv = buf[: M * N].view(torch.float16).view(M, N)
    dA, dB = A.to(dev), B.to(dev)
    dbias = bias.to(dev) if bias is not None else None
    g.gemm(ctx, dA, dB, dbias, epi, out=Cv, stream=stream)
    torch.cuda.synchronize()
    assert g.gemm_last_device_error(ctx) == (g.GEMM_OK, 0)
    tail = buf[M * N:].cpu()
    assert torch.all(tail == GUARD), "kernel wrote past the end of C"
    return Cv.cpu()


def oracle_ref(A, B, bias, epi, rows=None):
    ref, _, _ = oracle.gemm(A, B, bias, epi, rows=rows)
    return ref


def check(ctx, M, N, K, epi=g.EPI_NONE, with_bias=False, seed=0, dist="uniform"):
    A = inputs.random_fp16((M, K), 1000 + seed, dist, k=K)
    B = inputs.random_fp16((K, N), 2000 + seed, dist, k=K)
    bias = inputs.random_fp16((N,), 3000 + seed) if with_bias else None
    C = run_guarded(ctx, A, B, bias, epi)
    return assert_parity(C.numpy(), oracle_ref(A, B, bias, epi), f"M={M} N={N} K={K} epi={epi}")


# ---- one tile first: pins the UMMA descriptors, TMEM layout and the mbarrier ring ---------

def test_single_tile_single_kblock(kctx):
    check(kctx, 128, 256, 64)
    check(kctx, 256, 256, 64)


def test_single_tile_identity(kctx):
    ctx = kctx
    # A = I (128 x 128) selects B's rows exactly: any descriptor or layout slip shows.
    K = 128
    A = torch.eye(128, K, dtype=torch.float16)
    B = inputs.random_fp16((K, 256), 5)
    C = run_guarded(ctx, A, B, None, g.EPI_NONE)
    assert torch.equal(C, B)
    # B = I picks A
    A2 = inputs.random_fp16((128, 256), 6)
    C2 = run_guarded(ctx, A2, torch.eye(256, dtype=torch.float16), None, g.EPI_NONE)
    assert torch.equal(C2, A2)


@pytest.mark.parametrize("K", [64, 192, 256, 320, 512])
def test_split_tail_identity(kctx, K):
    # When every tile has its own CTA, the last k-blocks (up to four) are multiplied into the
    # left 128 columns of the accumulator first and into the right 128 afterwards. With B = I
    # (K x 256, ones on the diagonal) C is A's first 256 columns exactly, whichever half and
    # whichever k-block (full-width or split) each column's ones fall in.
    A = inputs.random_fp16((256, K), 11 + K)
    B = torch.eye(K, 256, dtype=torch.float16)
    C = run_guarded(kctx, A, B, None, g.EPI_NONE)
    want = torch.zeros(256, 256, dtype=torch.float16)
    want[:, :min(K, 256)] = A[:, :256]
    assert torch.equal(C, want)


@pytest.mark.parametrize("shape", [(256, 136, 200), (130, 392, 256), (128, 256, 192), (200, 520, 4160)],
                         ids=lambda s: "x".join(map(str, s)))
def test_split_tail_epilogues(kctx, shape):
    # right halves partly or wholly past N, fewer k-blocks than the tail, a ragged last k-block
    check(kctx, *shape, epi=g.EPI_GELU, with_bias=True, seed=shape[2])


def test_all_ones_gives_k(kctx):
    ctx = kctx
    for K in (64, 2048):
        A = torch.ones(130, K, dtype=torch.float16)
        B = torch.ones(K, 264, dtype=torch.float16)
        C = run_guarded(ctx, A, B, None, g.EPI_NONE)
        assert torch.all(C == K)


# ---- ragged shapes, every epilogue -----------------------------------------------------------

SHAPES = [
    (128, 256, 128), (1, 256, 64), (8, 256, 128), (127, 256, 192), (129, 512, 64),
    (255, 768, 256), (256, 256, 512), (257, 512, 320), (300, 264, 200), (64, 8, 8),
    (200, 72, 40), (1000, 1000, 1000), (77, 320, 4096),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_ragged_shapes_plain(kctx, shape):
    check(kctx, *shape, seed=sum(shape))


@pytest.mark.parametrize("epi,with_bias", [(g.EPI_NONE, True), (g.EPI_GELU, True), (g.EPI_RELU, True),
                                           (g.EPI_GELU, False), (g.EPI_RELU, False)])
@pytest.mark.parametrize("shape", [(129, 264, 200), (300, 512, 1024), (8, 2048, 64)],
                         ids=lambda s: "x".join(map(str, s)))
def test_epilogues(kctx, shape, epi, with_bias):
    check(kctx, *shape, epi=epi, with_bias=with_bias, seed=shape[0] + 7 * epi)


def test_more_tiles_than_sms(kctx):
    # 16 x 10 = 160 tiles of 128 x 256 on ~150 SMs (8 x 10 = 80 pair tiles on ~75 pairs),
    # then 512 (256) tiles: every CTA runs several tiles, both TMEM accumulators and many
    # ring phases.
    check(kctx, 2048, 2560, 256, epi=g.EPI_GELU, with_bias=True, seed=1)
    check(kctx, 4096, 4096, 128, epi=g.EPI_RELU, with_bias=True, seed=2)
    check(kctx, 4104, 2056, 320, epi=g.EPI_GELU, with_bias=True, seed=4)


def test_k_zero_gives_activation_of_bias(kctx):
    ctx = kctx
    M, N = 70, 264
    bias = inputs.random_fp16((N,), 9)
    dev = torch.device("cuda:0")
    for epi in (g.EPI_NONE, g.EPI_GELU, g.EPI_RELU):
        C = torch.empty(M, N, dtype=torch.float16, device=dev)
        g.gemm_run(ctx, M, N, 0, None, None, bias.to(dev), C, epi)
        torch.cuda.synchronize()
        ref = oracle_ref(torch.zeros(M, 0, dtype=torch.float16), torch.zeros(0, N, dtype=torch.float16),
                         bias, epi)
        assert_parity(C.cpu().numpy(), ref, f"K=0 epi={epi}")


def test_activation_accuracy_on_every_fp16_input(ctx):
    """K = 0 gives C = act(bias), so the epilogue's activation can be checked value by value:
    every finite FP16 number in [-12, 12] goes through it. Identity and ReLU must be exact;
    GELU must be within one FP16 ulp of the FP64 oracle (or 5e-7 absolute, where the result
    is so small that FP32 rounding of 1 + erf dominates)."""
    bits = np.arange(0, 0x10000, dtype=np.uint32).astype(np.uint16)
    vals = bits.view(np.float16)
    vals = vals[np.isfinite(vals) & (np.abs(vals.astype(np.float64)) <= 12.0)]
    n = (len(vals) + 7) // 8 * 8
    bias = np.zeros(n, dtype=np.float16)
    bias[: len(vals)] = vals
    dev = torch.device("cuda:0")
    tb = torch.from_numpy(bias.view(np.int16)).view(torch.float16)
    for epi in (g.EPI_NONE, g.EPI_RELU, g.EPI_GELU):
        C = torch.empty(2, n, dtype=torch.float16, device=dev)
        g.gemm_run(ctx, 2, n, 0, None, None, tb.to(dev), C, epi)
        torch.cuda.synchronize()
        got = C.cpu().numpy().astype(np.float64)
        ref = oracle_ref(torch.zeros(2, 0, dtype=torch.float16), torch.zeros(0, n, dtype=torch.float16),
                         tb, epi).astype(np.float64)
        if epi != g.EPI_GELU:
            assert np.array_equal(got, ref)
        else:
            ulp = np.spacing(np.abs(ref).astype(np.float16)).astype(np.float64)
            err = np.abs(got - ref)
            bad = err > np.maximum(ulp, 5e-7)
            assert not bad.any(), (bias[np.nonzero(bad[0])[0][:10]], err[bad][:10])


@pytest.mark.parametrize("shape", [(300, 256, 128), (129, 200, 64), (1000, 8, 512), (64, 64, 4096),
                                   (4104, 256, 128), (5, 136, 8), (300, 256, 192), (20000, 256, 64)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("with_bias", [False, True])
def test_softmax_epilogue(kctx, shape, with_bias):
    """GEMM with the fused row softmax, rows of one tile: within one FP16 ulp of the oracle's
    softmax of the FP64 logits (the GPU's logits are FP32 sums; their error, about 1e-6
    relative, moves a probability by far less than an FP16 ulp). 20000 rows loop every CTA
    over many tiles and ring phases."""
    M, N, K = shape
    A = inputs.random_fp16((M, K), 6000 + M, "normal")
    B = inputs.random_fp16((K, N), 6100 + N, "normal_inv_k", k=K)
    bias = inputs.random_fp16((N,), 6200 + N) if with_bias else None
    C = run_guarded(kctx, A, B, bias, g.EPI_SOFTMAX).numpy()
    ref = oracle_ref(A, B, bias, g.EPI_SOFTMAX)
    ulp = np.maximum(np.spacing(np.abs(ref)).astype(np.float64), 2.0 ** -24)
    err = np.abs(C.astype(np.float64) - ref.astype(np.float64))
    assert np.all(np.isfinite(C.astype(np.float64)))
    assert np.all(err <= ulp), (shape, float(err.max()), int((err > ulp).sum()))
    assert np.all(np.abs(C.astype(np.float64).sum(axis=1) - 1) <= N * 2.0 ** -11)


WIDE_SOFTMAX = [(300, 264, 128), (129, 1000, 64), (257, 2048, 256), (200, 4096, 128), (4104, 512, 128),
                (64, 3000, 320), (7, 776, 8), (64, 4096, 128), (20000, 512, 64), (4104, 4104, 64),
                (130, 8192, 64), (40, 16384, 128), (1000, 5000, 64)]


@pytest.mark.parametrize("shape", WIDE_SOFTMAX, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("with_bias", [False, True])
def test_softmax_epilogue_wide_rows(ctx, shape, with_bias):
    """Rows wider than one tile, any width: each CTA sweeps its span of column tiles twice
    (row statistics, then outputs from recomputed logits), and a cluster of 1, 2, 4 or 8 CTAs
    per 128-row block merges the statistics through distributed shared memory. Same bar as
    the one-tile softmax: within one FP16 ulp of the oracle, rows sum to 1. Ragged last
    tiles, ragged spans (CTAs without tiles), 4104 and 20000 rows (clusters loop over row
    blocks and reuse both statistics buffers many times)."""
    M, N, K = shape
    A = inputs.random_fp16((M, K), 6300 + M, "normal")
    B = inputs.random_fp16((K, N), 6400 + N, "normal_inv_k", k=K)
    bias = inputs.random_fp16((N,), 6500 + N) if with_bias else None
    C = run_guarded(ctx, A, B, bias, g.EPI_SOFTMAX).numpy()
    ref = oracle_ref(A, B, bias, g.EPI_SOFTMAX)
    ulp = np.maximum(np.spacing(np.abs(ref)).astype(np.float64), 2.0 ** -24)
    err = np.abs(C.astype(np.float64) - ref.astype(np.float64))
    assert np.all(np.isfinite(C.astype(np.float64)))
    assert np.all(err <= ulp), (shape, float(err.max()), int((err > ulp).sum()))
    assert np.all(np.abs(C.astype(np.float64).sum(axis=1) - 1) <= N * 2.0 ** -11)


def test_wide_softmax_timeout_then_recovery(ctx):
    """Every CTA of every row cluster withholds its first load: the waits (MMA operands,
    then the row exchange of the others) run out, the kernel returns and reports a timeout,
    and the context computes a correct wide softmax afterwards."""
    g.gemm_set_timeout_ns(ctx, 20_000_000)
    g.gemm_set_debug(ctx, g.GEMM_DEBUG_WITHHOLD_FIRST_LOAD)
    try:
        dev = torch.device("cuda:0")
        A = torch.ones(256, 64, dtype=torch.float16, device=dev)
        B = torch.ones(64, 1024, dtype=torch.float16, device=dev)
        C = torch.zeros(256, 1024, dtype=torch.float16, device=dev)
        g.gemm(ctx, A, B, None, g.EPI_SOFTMAX, out=C)
        torch.cuda.synchronize()
        status, detail = g.gemm_last_device_error(ctx)
        assert status == g.GEMM_ERR_TIMEOUT and detail in (1, 2, 3, 4, 5, 7)
        assert g.gemm_last_device_error(ctx) == (g.GEMM_OK, 0)
    finally:
        g.gemm_set_debug(ctx, g.GEMM_DEBUG_NONE)
        g.gemm_set_timeout_ns(ctx, 2_000_000_000)
    test_softmax_epilogue_wide_rows(ctx, (300, 1000, 64), True)


def test_softmax_cluster_sizes_are_covered(ctx):
    """The wide-row shapes above reach every cluster size the softmax schedule uses (the
    choice minimises the busiest CTA's tile epilogues; see gemm_describe)."""
    seen = {}
    for M, N, K in WIDE_SOFTMAX:
        d = g.gemm_describe(ctx, M, N, K, g.EPI_SOFTMAX)
        assert d.startswith("gemm_softmax_kernel<SoftmaxConfig<3>,true>"), d
        seen[int(d.split("cluster=")[1].split()[0])] = (M, N, K)
    assert {1, 2, 4, 8} <= set(seen), seen
    assert g.gemm_describe(ctx, 300, 256, 128, g.EPI_SOFTMAX).startswith("gemm_softmax_kernel<SoftmaxConfig<3>,false>")


def test_softmax_epilogue_limits(ctx):
    dev = torch.device("cuda:0")
    # K = 0 over a wide row: softmax of the bias
    bias_w = inputs.random_fp16((1536,), 98).to(dev)
    Cw = torch.empty(5, 1536, dtype=torch.float16, device=dev)
    g.gemm_run(ctx, 5, 1536, 0, None, None, bias_w, Cw, g.EPI_SOFTMAX)
    torch.cuda.synchronize()
    refw, _ = oracle.softmax_rows(bias_w.cpu()[None, :].repeat(5, 1))
    ulpw = np.maximum(np.spacing(np.abs(refw)).astype(np.float64), 2.0 ** -24)
    assert np.all(np.abs(Cw.cpu().numpy().astype(np.float64) - refw.astype(np.float64)) <= ulpw)
    # K = 0: softmax of the bias row; all-zero logits give 1/N everywhere
    bias = inputs.random_fp16((256,), 99).to(dev)
    C2 = torch.empty(3, 256, dtype=torch.float16, device=dev)
    g.gemm_run(ctx, 3, 256, 0, None, None, bias, C2, g.EPI_SOFTMAX)
    C3 = torch.empty(3, 256, dtype=torch.float16, device=dev)
    g.gemm_run(ctx, 3, 256, 0, None, None, None, C3, g.EPI_SOFTMAX)
    torch.cuda.synchronize()
    ref, _ = oracle.softmax_rows(bias.cpu()[None, :].repeat(3, 1))
    ulp = np.maximum(np.spacing(np.abs(ref)).astype(np.float64), 2.0 ** -24)
    assert np.all(np.abs(C2.cpu().numpy().astype(np.float64) - ref.astype(np.float64)) <= ulp)
    assert torch.all(C3 == 1.0 / 256)


def test_empty_m_or_n_is_a_no_op(ctx):
    dev = torch.device("cuda:0")
    C = torch.full((4, 8), 3.0, dtype=torch.float16, device=dev)
    A = torch.ones(4, 8, dtype=torch.float16, device=dev)
    B = torch.ones(8, 8, dtype=torch.float16, device=dev)
    assert g.gemm_run(ctx, 0, 8, 8, A, B, None, C) == g.GEMM_OK
    assert g.gemm_run(ctx, 4, 0, 8, A, B, None, C) == g.GEMM_OK
    torch.cuda.synchronize()
    assert torch.all(C == 3.0)


# ---- the benchmark problems --------------------------------------------------------------------

@pytest.mark.parametrize("name", list(inputs.WORKLOADS))
def test_workload_parity(ctx, name):
    w = inputs.WORKLOADS[name]
    A, B, bias = inputs.make_inputs(w)
    rows = inputs.sample_rows(w.M, w.sample_rows, include_last=w.include_last)
    dev = torch.device("cuda:0")
    C = torch.empty(w.M, w.N, dtype=torch.float16, device=dev)
    g.gemm(ctx, A.to(dev), B.to(dev), None if bias is None else bias.to(dev), w.epi_code, out=C)
    torch.cuda.synchronize()
    assert g.gemm_last_device_error(ctx) == (g.GEMM_OK, 0)
    got = C[rows.to(dev)].cpu().numpy()
    ref = oracle_ref(A, B, bias, w.epi_code, rows=rows.numpy())
    s = assert_parity(got, ref, name)
    if w.sample_rows:
        # properties that hold at any size, over the whole output
        assert bool(torch.isfinite(C).all())
        if w.epilogue == "gelu":
            assert float(C.min()) >= -0.1701 - 1e-3   # GELU is bounded below by about -0.17


# ---- boundary behaviour on the device --------------------------------------------------------------

def test_bad_arguments_are_rejected_before_launch(ctx):
    dev = torch.device("cuda:0")
    A = torch.zeros(64, 64, dtype=torch.float16, device=dev)
    B = torch.zeros(64, 64, dtype=torch.float16, device=dev)
    C = torch.zeros(64, 64, dtype=torch.float16, device=dev)
    L, h = g.lib(), ctx.handle

    def rc(M=64, N=64, K=64, a=A.data_ptr(), b=B.data_ptr(), bias=None, c=C.data_ptr(), epi=0):
        return L.gemm_run(h, M, N, K, a, b, bias, c, epi, None)

    assert rc() == g.GEMM_OK
    assert rc(M=-1) == g.GEMM_ERR_ARG
    assert rc(K=2 ** 31) == g.GEMM_ERR_ARG
    assert rc(epi=4) == g.GEMM_ERR_ARG
    assert rc(a=None) == g.GEMM_ERR_ARG
    assert rc(c=None) == g.GEMM_ERR_ARG
    assert rc(N=60) == g.GEMM_ERR_ALIGN
    assert rc(K=36) == g.GEMM_ERR_ALIGN
    assert rc(a=A.data_ptr() + 2) == g.GEMM_ERR_ALIGN
    assert rc(bias=C.data_ptr() + 8) == g.GEMM_ERR_ALIGN
    assert rc(c=A.data_ptr()) == g.GEMM_ERR_ARG                        # C overlaps A
    host = np.zeros(64 * 64 + 8, dtype=np.float16)
    hp = (host.ctypes.data + 15) // 16 * 16
    assert rc(a=hp) == g.GEMM_ERR_DEVICE                                # host memory
    assert rc(c=hp) == g.GEMM_ERR_DEVICE
    torch.cuda.synchronize()
    assert g.gemm_last_device_error(ctx) == (g.GEMM_OK, 0)
    assert g.gemm_num_sms(ctx) >= 100
    assert 0 <= g.gemm_num_pairs(ctx) <= g.gemm_num_sms(ctx) // 2


def test_describe_names_the_dispatched_kernel(ctx):
    """gemm_describe reports the kernel instance gemm_run launches (the bench names the
    kernel it times with it): CTA pairs for the MLP problem, split-K clusters for few long
    tiles, row clusters for the wide softmax, nothing for an empty problem; the shape
    checks are gemm_run's."""
    d = g.gemm_describe
    assert d(ctx, 8200, 16384, 4096, g.EPI_GELU).startswith("gemm_tcgen05_pair_kernel<")
    assert "SCHED_SPLIT_K" in d(ctx, 1024, 1024, 8192, g.EPI_GELU)
    assert d(ctx, 262144, 256, 128, g.EPI_SOFTMAX).startswith("gemm_softmax_kernel<SoftmaxConfig<3>,false>")
    assert d(ctx, 32768, 1024, 128, g.EPI_SOFTMAX).startswith("gemm_softmax_kernel<SoftmaxConfig<3>,true>")
    assert d(ctx, 0, 8, 8, g.EPI_NONE).startswith("none")
    with pytest.raises(g.GemmError) as e:
        d(ctx, 8, 60, 8, g.EPI_NONE)
    assert e.value.status == g.GEMM_ERR_ALIGN
    g.gemm_set_debug(ctx, g.GEMM_DEBUG_FORCE_SINGLE | g.GEMM_DEBUG_FORCE_STREAMK)
    try:
        assert "SCHED_STREAM_K" in d(ctx, 1024, 1024, 8192, g.EPI_GELU)
    finally:
        g.gemm_set_debug(ctx, g.GEMM_DEBUG_NONE)


def test_clock_trace_beside_a_gemm(ctx):
    """The SM-clock sampler on a stream of its own while a GEMM runs on another: timestamps
    ascend at the requested interval and the cycles per nanosecond are a plausible SM clock
    (between 0.3 and 2.5 GHz); the GEMM beside it is still correct."""
    dev = torch.device("cuda:0")
    n = 200
    trace = torch.zeros(2 * n, dtype=torch.int64, device=dev)
    side = torch.cuda.Stream(dev)
    g.gemm_clock_trace(ctx, trace, n, 50_000, 5_000_000, side)
    check(ctx, 1000, 1000, 1000, epi=g.EPI_GELU, with_bias=True, seed=21)
    torch.cuda.synchronize()
    t = trace.view(-1, 2).cpu().numpy()
    t = t[t[:, 0] > 0].astype(np.float64)
    assert 50 <= len(t) <= n
    dt = np.diff(t[:, 0])
    assert np.all(dt > 0) and abs(np.median(dt) - 50_000) < 5_000
    ghz = np.diff(t[:, 1]) / dt
    assert np.all((ghz > 0.3) & (ghz < 2.5)), ghz
    with pytest.raises(g.GemmError):
        g.gemm_clock_trace(ctx, trace, n, 10, 5_000_000, side)   # interval below 1 us


@pytest.mark.parametrize("force", ["single", "pair", "pair_one_unit"])
def test_bounded_wait_reports_timeout_and_context_survives(ctx, force):
    """The producer withholds its first operand load, so the MMA warp's wait runs out:
    the kernel must return (no hang, no fault) and report GEMM_ERR_TIMEOUT; afterwards the
    same context computes correct results again. "pair" has more work units than pairs (the
    four-warp instance), "pair_one_unit" one tile (the sixteen-warp instance)."""
    pairs = g.gemm_num_pairs(ctx)
    if force != "single" and pairs == 0:
        pytest.skip("the pair kernel cannot run on this device")
    flag = g.GEMM_DEBUG_FORCE_SINGLE if force == "single" else g.GEMM_DEBUG_FORCE_PAIR
    M, N = (256 * (pairs + 1), 256) if force == "pair" else (256, 256)
    g.gemm_set_timeout_ns(ctx, 20_000_000)
    g.gemm_set_debug(ctx, g.GEMM_DEBUG_WITHHOLD_FIRST_LOAD | flag)
    try:
        desc = g.gemm_describe(ctx, M, N, 64, g.EPI_NONE)
        if force == "pair":
            assert "PairConfig<256,3,4,128>" in desc, desc
        elif force == "pair_one_unit":
            assert "PairConfig<256,3,16,128,true>" in desc, desc
        dev = torch.device("cuda:0")
        A = torch.ones(M, 64, dtype=torch.float16, device=dev)
        B = torch.ones(64, N, dtype=torch.float16, device=dev)
        C = torch.zeros(M, N, dtype=torch.float16, device=dev)
        g.gemm(ctx, A, B, None, g.EPI_NONE, out=C)
        torch.cuda.synchronize()
        status, detail = g.gemm_last_device_error(ctx)
        assert status == g.GEMM_ERR_TIMEOUT
        assert detail in (1, 2, 3, 4, 5)
        assert g.gemm_last_device_error(ctx) == (g.GEMM_OK, 0)   # cleared
    finally:
        g.gemm_set_debug(ctx, g.GEMM_DEBUG_NONE)
        g.gemm_set_timeout_ns(ctx, 2_000_000_000)
    check(ctx, 256, 512, 256, epi=g.EPI_GELU, with_bias=True, seed=3)


def test_streamk_timeout_then_recovery(ctx):
    """Stream-K with tiles cut into 16 parts: CTA 0 (owner of tile 0) withholds its first
    load and gives up, so the ready flags of its 15 contributors stay raised. The timeout
    is reported, gemm_last_device_error lowers the flags, and the next stream-K GEMM (with
    different inputs, so stale partials would show) is correct."""
    g.gemm_set_timeout_ns(ctx, 20_000_000)
    g.gemm_set_debug(ctx, g.GEMM_DEBUG_WITHHOLD_FIRST_LOAD | FORCE["streamk"])
    try:
        dev = torch.device("cuda:0")
        A = torch.ones(256, 1024, dtype=torch.float16, device=dev)
        B = torch.ones(1024, 256, dtype=torch.float16, device=dev)
        C = torch.zeros(256, 256, dtype=torch.float16, device=dev)
        g.gemm(ctx, A, B, None, g.EPI_NONE, out=C)
        torch.cuda.synchronize()
        status, detail = g.gemm_last_device_error(ctx)
        assert status == g.GEMM_ERR_TIMEOUT and detail in (1, 2, 3, 4, 5, 6)
        assert g.gemm_last_device_error(ctx) == (g.GEMM_OK, 0)
        g.gemm_set_debug(ctx, FORCE["streamk"])
        check(ctx, 256, 256, 1024, epi=g.EPI_GELU, with_bias=True, seed=12)
    finally:
        g.gemm_set_debug(ctx, g.GEMM_DEBUG_NONE)
        g.gemm_set_timeout_ns(ctx, 2_000_000_000)


def test_splitk_timeout_then_recovery(ctx):
    """Split-K in clusters of 8 with every CTA withholding its first load: every wait runs
    out, every CTA still reaches both cluster barriers (no hang), the timeout is reported,
    and the next split-K GEMM on the same context is correct."""
    g.gemm_set_timeout_ns(ctx, 20_000_000)
    g.gemm_set_debug(ctx, g.GEMM_DEBUG_WITHHOLD_FIRST_LOAD | FORCE["splitk"])
    try:
        dev = torch.device("cuda:0")
        A = torch.ones(256, 1024, dtype=torch.float16, device=dev)
        B = torch.ones(1024, 256, dtype=torch.float16, device=dev)
        C = torch.zeros(256, 256, dtype=torch.float16, device=dev)
        g.gemm(ctx, A, B, None, g.EPI_NONE, out=C)
        torch.cuda.synchronize()
        status, detail = g.gemm_last_device_error(ctx)
        assert status == g.GEMM_ERR_TIMEOUT and detail in (1, 2, 3, 4, 5)
        assert g.gemm_last_device_error(ctx) == (g.GEMM_OK, 0)
        g.gemm_set_debug(ctx, FORCE["splitk"])
        check(ctx, 256, 256, 1024, epi=g.EPI_GELU, with_bias=True, seed=13)
    finally:
        g.gemm_set_debug(ctx, g.GEMM_DEBUG_NONE)
        g.gemm_set_timeout_ns(ctx, 2_000_000_000)


@pytest.mark.parametrize("shape", [(128, 256, 1024), (200, 264, 520), (1000, 520, 8200), (384, 512, 192)],
                         ids=lambda v: "x".join(map(str, v)))
def test_splitk_cluster_sizes_and_tails(ctx, shape):
    """Split-K with 8, 4 and 2 CTAs per tile (K = 1024, 520, 8200 and 192 give 16, 9, 129 and
    3 k-blocks: uneven ranges, a ragged last k-block), rows and columns past M and N in the
    last tiles, every epilogue; bit-identical between two runs (fixed summation order)."""
    M, N, K = shape
    g.gemm_set_debug(ctx, FORCE["splitk"])
    try:
        for epi, with_bias in ((g.EPI_NONE, False), (g.EPI_GELU, True), (g.EPI_RELU, True)):
            check(ctx, M, N, K, epi=epi, with_bias=with_bias, seed=M + K + epi)
        dev = torch.device("cuda:0")
        A = inputs.random_fp16((M, K), 7).to(dev)
        B = inputs.random_fp16((K, N), 8).to(dev)
        C1 = torch.empty(M, N, dtype=torch.float16, device=dev)
        C2 = torch.empty(M, N, dtype=torch.float16, device=dev)
        g.gemm(ctx, A, B, None, g.EPI_NONE, out=C1)
        g.gemm(ctx, A, B, None, g.EPI_NONE, out=C2)
        torch.cuda.synchronize()
        assert torch.equal(C1, C2)
        assert g.gemm_last_device_error(ctx) == (g.GEMM_OK, 0)
    finally:
        g.gemm_set_debug(ctx, g.GEMM_DEBUG_NONE)


@pytest.mark.parametrize("epi,with_bias", [(g.EPI_NONE, False), (g.EPI_GELU, True)])
def test_pair_last_round_in_n_halves(ctx, epi, with_bias):
    """Pair kernel with a few more 256 x 256 tiles than pairs: the last round's tiles run as
    N-halves (256 x 128, one B box per CTA), one per pair. Ragged M, N and K put rows and
    columns past C in the split tiles; every row is checked against the oracle, and two runs
    agree bit for bit."""
    pairs = g.gemm_num_pairs(ctx)
    if pairs < 4:
        pytest.skip("the pair kernel cannot run on this device")
    n_blocks = 4
    m_blocks = (pairs + 4 + n_blocks - 1) // n_blocks   # pairs + 1 .. pairs + 7 tiles
    M, N, K = 256 * m_blocks - 100, 256 * n_blocks - 56, 520
    tiles = m_blocks * n_blocks
    assert 0 < tiles % pairs <= pairs // 2
    desc = g.gemm_describe(ctx, M, N, K, epi)
    assert "pair_kernel" in desc and f"(last {tiles % pairs} split in N-halves)" in desc, desc
    check(ctx, M, N, K, epi=epi, with_bias=with_bias, seed=77 + epi)
    dev = torch.device("cuda:0")
    A = inputs.random_fp16((M, K), 78).to(dev)
    B = inputs.random_fp16((K, N), 79).to(dev)
    C1 = torch.empty(M, N, dtype=torch.float16, device=dev)
    C2 = torch.empty(M, N, dtype=torch.float16, device=dev)
    g.gemm(ctx, A, B, None, epi, out=C1)
    g.gemm(ctx, A, B, None, epi, out=C2)
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)
    assert g.gemm_last_device_error(ctx) == (g.GEMM_OK, 0)


@pytest.mark.parametrize("shape", [(256, 256, 128), (300, 520, 1000), (700, 264, 4104)],
                         ids=lambda v: "x".join(map(str, v)))
def test_pair_instance_with_one_unit_per_pair(ctx, shape):
    """With no more work units than pairs the pair kernel runs its sixteen-warp instance,
    whose output staging lies in the operand ring: B = I gives A exactly, and GELU + bias
    matches the oracle with rows and columns past C in the last tiles."""
    if g.gemm_num_pairs(ctx) == 0:
        pytest.skip("the pair kernel cannot run on this device")
    M, N, K = shape
    g.gemm_set_debug(ctx, g.GEMM_DEBUG_FORCE_PAIR)
    try:
        assert "PairConfig<256,3,16,128,true>" in g.gemm_describe(ctx, M, N, K, g.EPI_GELU)
        if N <= K:
            A = inputs.random_fp16((M, K), 31 + K)
            C = run_guarded(ctx, A, torch.eye(K, N, dtype=torch.float16), None, g.EPI_NONE)
            assert torch.equal(C, A[:, :N])
        check(ctx, M, N, K, epi=g.EPI_GELU, with_bias=True, seed=M + N)
        assert g.gemm_last_device_error(ctx) == (g.GEMM_OK, 0)
    finally:
        g.gemm_set_debug(ctx, g.GEMM_DEBUG_NONE)


def test_long_k_one_wave_runs_on_pairs(ctx):
    """A one-wave problem with K >= 8192 and enough 256 x 256 tiles for three quarters of the
    pairs runs on the pair kernel (its main loop needs fewer L2 bytes per flop); the same
    sizes with K = 4096 stay on single SMs. Sampled rows, the last ones included, against the
    oracle, ragged M, N and K."""
    pairs = g.gemm_num_pairs(ctx)
    if pairs < 4:
        pytest.skip("the pair kernel cannot run on this device")
    n_blocks = 8
    m_blocks = max(1, (3 * pairs + 3) // 4 + n_blocks - 1) // n_blocks   # >= 3/4 of the pairs
    M, N = 256 * m_blocks - 48, 256 * n_blocks - 16
    if ((M + 127) // 128) * ((N + 255) // 256) > g.gemm_num_sms(ctx) or m_blocks * n_blocks > pairs:
        pytest.skip("no one-wave shape with that many pair tiles on this device")
    assert "pair_kernel" in g.gemm_describe(ctx, M, N, 8200, g.EPI_GELU)
    assert "pair_kernel" not in g.gemm_describe(ctx, M, N, 4096, g.EPI_GELU)
    K = 8200
    A = inputs.random_fp16((M, K), 95)
    B = inputs.random_fp16((K, N), 96)
    bias = inputs.random_fp16((N,), 97)
    C = run_guarded(ctx, A, B, bias, g.EPI_GELU)
    rows = inputs.sample_rows(M, 160, seed=11, include_last=4).numpy()
    assert_parity(C.numpy()[rows], oracle_ref(A, B, bias, g.EPI_GELU, rows=rows), "long-K pair")


def _random_shapes(seed, n, m_max, n_max, k_max):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        M = int(rng.integers(1, m_max + 1))
        N = 8 * int(rng.integers(1, n_max // 8 + 1))
        K = 8 * int(rng.integers(0, k_max // 8 + 1))
        epi = int(rng.choice([g.EPI_NONE, g.EPI_GELU, g.EPI_RELU]))
        out.append((M, N, K, epi, bool(rng.integers(0, 2))))
    return out


@pytest.mark.parametrize("schedule", ["default", "single", "pair", "splitk", "streamk"])
def test_random_shapes_against_the_oracle(ctx, schedule):
    """Seeded random problems (ragged M, N and K, K = 0 included, every epilogue, with and
    without bias) under the planner's own choice and under each forced schedule: sampled rows,
    the last ones included, against the oracle, guard rows and tail untouched."""
    if schedule == "pair" and g.gemm_num_pairs(ctx) == 0:
        pytest.skip("the pair kernel cannot run on this device")
    big = schedule == "default"
    shapes = _random_shapes({"default": 71, "single": 72, "pair": 73, "splitk": 74, "streamk": 75}[schedule],
                            40 if big else 24, 6000 if big else 1500, 6000 if big else 1500, 9000 if big else 4000)
    if schedule != "default":
        g.gemm_set_debug(ctx, FORCE[schedule])
    try:
        for i, (M, N, K, epi, with_bias) in enumerate(shapes):
            A = inputs.random_fp16((M, K), 8000 + i, k=max(K, 1))
            B = inputs.random_fp16((K, N), 8100 + i, k=max(K, 1))
            bias = inputs.random_fp16((N,), 8200 + i) if with_bias else None
            C = run_guarded(ctx, A, B, bias, epi)
            rows = inputs.sample_rows(M, 24, seed=60 + i, include_last=3).numpy()
            what = f"{schedule} {M}x{N}x{K} epi={epi} bias={with_bias}: {g.gemm_describe(ctx, M, N, K, epi)}"
            assert_parity(C.numpy()[rows], oracle_ref(A, B, bias, epi, rows=rows), what)
        assert g.gemm_last_device_error(ctx) == (g.GEMM_OK, 0)
    finally:
        g.gemm_set_debug(ctx, g.GEMM_DEBUG_NONE)


def test_splitk_in_host_column_bands(ctx):
    """Split-K inside gemm_run_host's column bands: each band's C is a slice of a wider
    matrix (row stride N, not the band's width), which split-K writes directly."""
    M, N, K = 2056, 8200, 512
    A = inputs.random_fp16((M, K), 87).pin_memory()
    B = inputs.random_fp16((K, N), 88).pin_memory()
    bias = inputs.random_fp16((N,), 89).pin_memory()
    C = torch.full((M, N), float("nan"), dtype=torch.float16).pin_memory()
    g.gemm_set_debug(ctx, FORCE["splitk"])
    try:
        g.gemm_run_host(ctx, M, N, K, A, B, bias, C, g.EPI_GELU)
    finally:
        g.gemm_set_debug(ctx, g.GEMM_DEBUG_NONE)
    assert bool(torch.isfinite(C).all())
    rows = inputs.sample_rows(M, 200, seed=10, include_last=4).numpy()
    assert_parity(C.numpy()[rows], oracle_ref(A, B, bias, g.EPI_GELU, rows=rows), "split-K column bands")


def test_streamk_graph_replays_with_new_inputs(ctx):
    """A captured stream-K GEMM replayed with new inputs each time: every owner must wait for
    this replay's partials (the flags are lowered after use, not left from the last run)."""
    dev = torch.device("cuda:0")
    M, N, K = 384, 512, 2048
    g.gemm_set_debug(ctx, FORCE["streamk"])
    try:
        dA = torch.empty(M, K, dtype=torch.float16, device=dev)
        dB = inputs.random_fp16((K, N), 91).to(dev)
        C = torch.empty(M, N, dtype=torch.float16, device=dev)
        g.gemm(ctx, dA.zero_(), dB, None, g.EPI_NONE, out=C)   # first call outside capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            g.gemm(ctx, dA, dB, None, g.EPI_NONE, out=C)
        for seed in (92, 93, 94):
            A = inputs.random_fp16((M, K), seed)
            dA.copy_(A.to(dev))
            graph.replay()
            torch.cuda.synchronize()
            assert_parity(C.cpu().numpy(), oracle_ref(A, dB.cpu(), None, g.EPI_NONE), f"replay {seed}")
        assert g.gemm_last_device_error(ctx) == (g.GEMM_OK, 0)
    finally:
        g.gemm_set_debug(ctx, g.GEMM_DEBUG_NONE)


@pytest.mark.parametrize("schedule", ["default", "streamk"])
def test_default_streamk_on_few_tiles(ctx, schedule):
    """1024 x 1024 x 8192 + bias + GELU: 32 tiles of 128 x 256 on ~150 SMs. The default
    schedule takes split-K (clusters of 4 CTAs, each a quarter of K); forced stream-K cuts
    each tile into ~5 parts. Against the oracle on sampled rows, and bit-identical between
    two runs (the parts are added in a fixed order)."""
    g.gemm_set_debug(ctx, g.GEMM_DEBUG_NONE if schedule == "default" else FORCE["streamk"])
    M, N, K = 1024, 1024, 8192
    A = inputs.random_fp16((M, K), 61, "normal")
    B = inputs.random_fp16((K, N), 62, "normal_inv_k", k=K)
    bias = inputs.random_fp16((N,), 63)
    dev = torch.device("cuda:0")
    C1 = torch.empty(M, N, dtype=torch.float16, device=dev)
    C2 = torch.empty(M, N, dtype=torch.float16, device=dev)
    dA, dB, db = A.to(dev), B.to(dev), bias.to(dev)
    g.gemm(ctx, dA, dB, db, g.EPI_GELU, out=C1)
    g.gemm(ctx, dA, dB, db, g.EPI_GELU, out=C2)
    torch.cuda.synchronize()
    assert g.gemm_last_device_error(ctx) == (g.GEMM_OK, 0)
    assert torch.equal(C1, C2)
    rows = inputs.sample_rows(M, 96, seed=5, include_last=2).numpy()
    rows = np.union1d(rows, [0, 127, 128, 511, 512, 1023])
    g.gemm_set_debug(ctx, g.GEMM_DEBUG_NONE)
    assert_parity(C1.cpu().numpy()[rows], oracle_ref(A, B, bias, g.EPI_GELU, rows=rows), f"few tiles, {schedule}")


def test_host_buffer_entry_point(ctx):
    M, N, K = 300, 512, 256
    A = inputs.random_fp16((M, K), 71).pin_memory()
    B = inputs.random_fp16((K, N), 72).pin_memory()
    bias = inputs.random_fp16((N,), 73).pin_memory()
    C = torch.empty(M, N, dtype=torch.float16).pin_memory()
    g.gemm_run_host(ctx, M, N, K, A, B, bias, C, g.EPI_GELU)
    assert_parity(C.numpy(), oracle_ref(A, B, bias, g.EPI_GELU), "gemm_run_host")
    # pageable memory works too
    C2 = torch.empty(M, N, dtype=torch.float16)
    g.gemm_run_host(ctx, M, N, K, A.clone(), B.clone(), None, C2, g.EPI_RELU)
    assert_parity(C2.numpy(), oracle_ref(A, B, None, g.EPI_RELU), "gemm_run_host pageable")
    # an output above 32 MiB is pipelined in 4 row chunks (the last one ragged)
    M, N, K = 4100, 4096, 512
    A = inputs.random_fp16((M, K), 74).pin_memory()
    B = inputs.random_fp16((K, N), 75).pin_memory()
    bias = inputs.random_fp16((N,), 76).pin_memory()
    C = torch.full((M, N), float("nan"), dtype=torch.float16).pin_memory()
    g.gemm_run_host(ctx, M, N, K, A, B, bias, C, g.EPI_GELU)
    rows = inputs.sample_rows(M, 300, seed=8, include_last=8).numpy()
    rows = np.union1d(rows, [0, 1279, 1280, 2559, 2560, 3839, 3840])
    assert bool(torch.isfinite(C).all())
    assert_parity(C.numpy()[rows], oracle_ref(A, B, bias, g.EPI_GELU, rows=rows), "gemm_run_host chunked")
    # A smaller than B: column bands of C (2304, 2304, 2304 and a ragged 1288 columns)
    M, N, K = 2056, 8200, 512
    A = inputs.random_fp16((M, K), 77).pin_memory()
    B = inputs.random_fp16((K, N), 78).pin_memory()
    bias = inputs.random_fp16((N,), 79).pin_memory()
    C = torch.full((M, N), float("nan"), dtype=torch.float16).pin_memory()
    g.gemm_run_host(ctx, M, N, K, A, B, bias, C, g.EPI_RELU)
    assert bool(torch.isfinite(C).all())
    rows = inputs.sample_rows(M, 200, seed=9, include_last=4).numpy()
    assert_parity(C.numpy()[rows], oracle_ref(A, B, bias, g.EPI_RELU, rows=rows), "gemm_run_host column bands")


def test_host_buffer_row_halves_and_column_bands(ctx):
    """gemm_run_host with A of 33.6 MB (at least 32 MiB) and smaller than B: A goes up in two
    row halves (2304 rows, then 1800) and B in four column bands, one GEMM per half and band
    (eight GEMMs, each writing a slice of C with row stride N). Sampled rows on both sides of
    the halves' boundary, against the oracle."""
    M, N, K = 4104, 8200, 4096
    A = inputs.random_fp16((M, K), 91, "normal").pin_memory()
    B = inputs.random_fp16((K, N), 92, "normal_inv_k", k=K).pin_memory()
    bias = inputs.random_fp16((N,), 93).pin_memory()
    C = torch.full((M, N), float("nan"), dtype=torch.float16).pin_memory()
    g.gemm_run_host(ctx, M, N, K, A, B, bias, C, g.EPI_GELU)
    assert bool(torch.isfinite(C).all())
    rows = inputs.sample_rows(M, 120, seed=11, include_last=4).numpy()
    rows = np.union1d(rows, [0, 2303, 2304, 2305])
    assert_parity(C.numpy()[rows], oracle_ref(A, B, bias, g.EPI_GELU, rows=rows), "row halves x column bands")


def test_side_stream_and_cuda_graph(ctx):
    dev = torch.device("cuda:0")
    M, N, K = 640, 768, 512
    A = inputs.random_fp16((M, K), 81)
    B = inputs.random_fp16((K, N), 82)
    bias = inputs.random_fp16((N,), 83)
    dA, dB, dbias = A.to(dev), B.to(dev), bias.to(dev)
    ref = oracle_ref(A, B, bias, g.EPI_GELU)
    s = torch.cuda.Stream()
    C = torch.empty(M, N, dtype=torch.float16, device=dev)
    with torch.cuda.stream(s):
        g.gemm(ctx, dA, dB, dbias, g.EPI_GELU, out=C)
    s.synchronize()
    assert_parity(C.cpu().numpy(), ref, "side stream")
    C.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        g.gemm(ctx, dA, dB, dbias, g.EPI_GELU, out=C)
    for _ in range(3):
        C.zero_()
        graph.replay()
    torch.cuda.synchronize()
    assert_parity(C.cpu().numpy(), ref, "graph replay")
