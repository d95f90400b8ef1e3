/*
 * gemm.h - C ABI of the GB300 (sm_103a) FP16 tensor-core GEMM with a fused epilogue.
 *
 *     C = act(A * B + bias)        A: M x K, B: K x N, C: M x N, all FP16, row-major
 *
 * The operation is the tensor-core GEMM of the TileLang tutorial pages:
 *  - "TileLang: Criando Kernels de GPU de Alto Desempenho ..." (noticiai.com.br), section
 *    "GEMM com Tensor Cores: onde a magica acontece": a tiled matrix multiply whose caller
 *    passes A, B, C and M, N, K (tiled_gemm(A, B, C, M, N, K)); tiles A[i:i+128, k:k+32]
 *    and B[k:k+32, j:j+128], i.e. A is M x K and B is K x N, both row-major.
 *  - same page, section "GEMM com epilogo fundido: ReLU e bias 'de graca'": ReLU (and, by
 *    the same pattern, bias and GELU) applied to the accumulator inside the one kernel,
 *    with no extra pass over C in DRAM.
 *  - "TileLang ..." (pro.edgex.exchange), fused-epilogue paragraph: bias addition, then
 *    GELU, on the register-resident accumulator before the output store.
 *  - "Designing High-Performance GPU Kernels with TileLang" (spaxe.top), GEMM paragraph:
 *    FP16 matrix multiplication on tensor cores.
 * Arithmetic: FP16 inputs, FP32 accumulation in Tensor Memory, epilogue in FP32 (bias is
 * added first, then the activation; GELU is the exact-erf form 0.5*x*(1+erf(x/sqrt(2)))),
 * one round-to-nearest-even conversion to FP16, one store.
 *
 * Threading: a context may be used by one host thread at a time (or with external
 * serialisation). Calls on different contexts are independent. GEMMs of one context that
 * take the stream-K schedule (see gemm_run) share the context's workspace, so they must not
 * run at the same time on the GPU: keep one context's GEMMs on one stream (or in stream
 * order), or give each concurrently used stream a context of its own.
 */
#ifndef GB300_GEMM_H
#define GB300_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque context: cached device properties, the tensor-map encoder, a 4-byte device
 * error word, the stream-K workspace (128 KB of FP32 partial sums and a few ready flags
 * per SM, about 19.5 MB on GB300) and (only once gemm_run_host has been called) host-path
 * staging buffers. */
typedef struct gemm_ctx gemm_ctx;

/* Epilogue selector. The bias is applied whenever `bias` is non-NULL, for every value. */
enum gemm_epilogue {
    GEMM_EPI_NONE = 0, /* C = A*B (+ bias)                                           */
    GEMM_EPI_GELU = 1, /* C = GELU_erf(A*B (+ bias))                                 */
    GEMM_EPI_RELU = 2, /* C = max(A*B (+ bias), 0)                                   */
    GEMM_EPI_SOFTMAX = 3 /* C[r][:] = softmax over the row of A*B (+ bias): the logits stay
                            in FP32 inside the kernel and are never written. Any N.
                            N <= 256: one 128 x 256 tile spans the row, one pass. Wider
                            rows: a thread-block cluster of 1, 2, 4 or 8 CTAs per block of
                            128 rows, each CTA a span of 256-column tiles, two passes
                            (running row maximum and sum over the span, merged across
                            the cluster through distributed shared memory; then the
                            logits are recomputed and the probabilities written). Returns
                            GEMM_ERR_ARG only if the device cannot run the kernel at all.
                            "Designing High-Performance GPU Kernels with TileLang"
                            (spaxe.top): row-wise softmax in the GEMM epilogue.       */
};

/* Status codes. Every error is detected before anything is enqueued: on error nothing
 * has been launched or copied, except for GEMM_ERR_LAUNCH, which wraps a CUDA error
 * reported by the launch itself. */
enum gemm_status {
    GEMM_OK = 0,
    GEMM_ERR_ARG = -1,     /* NULL context or buffer, negative or too large size,
                              epilogue out of range                                   */
    GEMM_ERR_ALIGN = -2,   /* a pointer not 16-byte aligned, or N or K not a multiple of
                              8 (row strides must be multiples of 16 bytes)           */
    GEMM_ERR_DEVICE = -3,  /* no such device, not compute capability 10.3, or a buffer
                              that is not device memory of the context's device       */
    GEMM_ERR_LAUNCH = -4,  /* a CUDA runtime call failed (see gemm_last_cuda_error)   */
    GEMM_ERR_TIMEOUT = -5, /* a bounded in-kernel wait ran out; the kernel returned
                              early and C is incomplete (see gemm_last_device_error) */
    GEMM_ERR_NOMEM = -6    /* host or device allocation failed (create, run_host)     */
};

/* Create a context for CUDA device `device` (0-based). Checks that the device has compute
 * capability 10.3 (GB300, sm_103a), reads its SM count, sets the kernel's shared-memory
 * attribute, resolves cuTensorMapEncodeTiled and allocates the 4-byte device error word and
 * the stream-K workspace.
 * On success *out receives the context (caller frees it with gemm_destroy) and GEMM_OK is
 * returned; on failure *out is set to NULL. The caller's current device is left as it was. */
int gemm_create(gemm_ctx **out, int device);

/* Enqueue C = act(A*B + bias) on `stream` (a cudaStream_t; NULL = the legacy default
 * stream) and return without waiting.
 *   M, N, K : sizes, 0 <= M, N, K <= 2^31 - 1. M = 0 or N = 0 is a no-op (GEMM_OK, nothing
 *             enqueued). K = 0 gives C = act(bias) (act(0) without a bias). M is
 *             arbitrary (rows past a tile multiple are masked); N and K must be multiples
 *             of 8.
 *   A       : device pointer, M x K FP16 row-major (K contiguous), 16-byte aligned.
 *   B       : device pointer, K x N FP16 row-major (N contiguous), 16-byte aligned.
 *             (A and B may be NULL only when K = 0.)
 *   bias    : device pointer to N FP16 values (16-byte aligned), or NULL for no bias.
 *   C       : device pointer, M x N FP16 row-major, 16-byte aligned; written, never read.
 *             C must not overlap A, B or bias.
 *   epilogue: a gemm_epilogue value.
 * Ownership: the caller owns every buffer and must keep them alive until the stream has
 * passed this call. gemm_run allocates nothing and launches exactly one kernel.
 * Schedule: 256 x 256 tiles on CTA pairs when there are at least as many as co-resident
 * pairs, or when K >= 8192, at least three quarters of the pairs get a tile and the
 * single-SM tiles would fit one wave; otherwise 128 x 256 tiles on single SMs. On pairs, a
 * last round of tiles that at most half of the pairs would work on runs as 256 x 128
 * halves, one per pair. When the single-SM tiles leave most SMs idle:
 * split-K, a cluster of S = 8, 4 or 2 CTAs per tile (the largest S with tiles x S <= SMs,
 * all clusters co-resident, and at least 8 k-blocks of 64 per CTA), each CTA summing 1/S of
 * the k-blocks; the S FP32 partials are added over distributed shared memory in a fixed
 * order and the CTA of rank r applies the epilogue to rows [r*128/S, (r+1)*128/S) of the
 * tile. Failing that, when the tiles are at most half the SMs and K gives at least twice as
 * many CTAs as tiles 16 k-blocks each, stream-K: the tiles' k-blocks are split evenly over
 * up to every SM, and a tile cut between SMs is summed in FP32 through the context's
 * workspace before its epilogue. (Both change the summation order, not the result's
 * tolerance, against the whole-tile schedule.) Never for GEMM_EPI_SOFTMAX.
 * Errors: see gemm_status. A wait that runs out inside the kernel is reported later by
 * gemm_last_device_error, not by this call. */
int gemm_run(gemm_ctx *ctx, int64_t M, int64_t N, int64_t K, const void *A, const void *B,
             const void *bias, void *C, int epilogue, void *stream);

/* The same operation on HOST buffers (pinned memory gives asynchronous copies; pageable
 * memory works but is copied synchronously). Device staging buffers, two internal copy
 * streams and their events are owned by the context (created or grown on first use, freed
 * by gemm_destroy). Outputs under 32 MiB are done in one piece; larger ones in 4 bands (8
 * from 256 MiB on) of whole 256-wide tiles whose uploads, GEMMs (one kernel launch each, on `stream`)
 * and downloads overlap: column bands of C when A is the smaller operand (A in two row halves
 * when it is 32 MiB or more, uploaded in the order the GEMMs need them: A_0, B_0, A_1, B_1,
 * B_2, ..., one GEMM per row half and column band), row bands otherwise (B whole, then A in
 * row bands); the softmax epilogue always uses row bands. Returns after C is on the host (the call
 * synchronises `stream`). Same argument rules as gemm_run, except that the pointers are
 * host pointers. Also reports a device-side timeout (GEMM_ERR_TIMEOUT), since it
 * synchronises. */
int gemm_run_host(gemm_ctx *ctx, int64_t M, int64_t N, int64_t K, const void *A,
                  const void *B, const void *bias, void *C, int epilogue, void *stream);

/* After the caller has synchronised the stream(s) that ran this context's GEMMs: return
 * GEMM_OK, or GEMM_ERR_TIMEOUT if a bounded in-kernel wait ran out since the last call.
 * `detail` (may be NULL) receives the raw error word (which wait ran out: 1 producer
 * slot, 2 MMA operands, 3 MMA accumulator, 4 epilogue accumulator, 5 teardown drain,
 * 6 stream-K partial sum from another SM, 7 row statistics from the other CTAs of a
 * softmax row cluster). Clears the word, and after an error also the
 * stream-K ready flags a kernel that gave up may have left raised (call it before the next
 * GEMM on this context once a timeout is possible). Synchronous. */
int gemm_last_device_error(gemm_ctx *ctx, uint32_t *detail);

/* The last CUDA runtime error code seen by this context (0 if none), for diagnosis of
 * GEMM_ERR_LAUNCH / GEMM_ERR_NOMEM. */
int gemm_last_cuda_error(gemm_ctx *ctx);

/* Destroy a context (NULL is accepted). Frees the error word, the stream-K workspace and
 * any staging buffers; the
 * caller must have synchronised every stream that still runs work of this context. */
int gemm_destroy(gemm_ctx *ctx);

/* A static, human-readable name for a status code. */
const char *gemm_status_string(int status);

/* Number of streaming multiprocessors the one-CTA kernel sizes its grid to. */
int gemm_num_sms(gemm_ctx *ctx);

/* Which kernel instance gemm_run would launch for an M x N x K problem with `epilogue`, with
 * the context's current debug flags: writes a NUL-terminated description of at most len - 1
 * characters to `buf` (host memory owned by the caller), of the form
 *   "<kernel instance> grid=<CTAs> cluster=<CTAs per cluster> tiles=<output tiles>",
 * e.g. "gemm_tcgen05_pair_kernel<PairConfig<256,3,4,128>> grid=152 cluster=2 tiles=2112",
 * followed by " (last <n> split in N-halves)" when the pair kernel runs its last n tiles as
 * two half-width work units each.
 * The kernel instance names the template instance as it appears in a profiler's kernel
 * list. Launches nothing and touches no device memory. Returns GEMM_OK, or the status
 * gemm_run would return for these sizes and epilogue (GEMM_ERR_ARG, GEMM_ERR_ALIGN), or
 * GEMM_ERR_ARG for a NULL `buf` or len <= 0. (No counterpart in the tutorial pages: it
 * reports the schedule choice so that measurements can name the kernel they time.) */
int gemm_describe(gemm_ctx *ctx, int64_t M, int64_t N, int64_t K, int epilogue, char *buf, int64_t len);

/* Measurement aid (no counterpart in the tutorial pages): samples the SM clock while other
 * work runs. One thread of a 32-thread CTA (no shared memory) reads the global nanosecond
 * timer and the SM cycle counter every `interval_ns` and writes trace[2i] = timer (ns),
 * trace[2i + 1] = cycles, for i < max_samples, until `duration_ns` has passed since its first
 * sample; it sleeps in between. Launched on `stream`, asynchronous: put it on a stream of its
 * own just before the kernels to be timed, and it runs beside them on one SM (one warp
 * slot); (cycles difference) / (timer difference) of consecutive samples is the SM clock in
 * GHz over that interval.
 *   trace: device memory of the context's device, 2 * max_samples uint64, 16-byte aligned,
 *          owned by the caller; entries past the last sample are not written (zero-fill it
 *          first to find the count).
 *   1 <= max_samples <= 2^20, 1000 <= interval_ns <= 1e7, duration_ns <= 1e10.
 * Returns GEMM_OK once launched, GEMM_ERR_ARG / _ALIGN / _DEVICE before launching, or
 * GEMM_ERR_LAUNCH. */
int gemm_clock_trace(gemm_ctx *ctx, uint64_t *trace, int max_samples, uint64_t interval_ns,
                     uint64_t duration_ns, void *stream);

/* Number of CTA pairs (2-SM clusters) the device can run at once with the pair kernel,
 * which takes 256 x 256 tiles; 0 if the pair kernel cannot run (then every call uses the
 * one-CTA kernel). gemm_run picks the pair kernel when the problem has at least this many
 * 256 x 256 tiles, else the one-CTA kernel (128 x 256 tiles). */
int gemm_num_pairs(gemm_ctx *ctx);

/* Row-wise softmax: Y[r][j] = exp(X[r][j] - m_r) / sum_k exp(X[r][k] - m_r), m_r the row
 * maximum ("TileLang: Criando Kernels de GPU ..." (noticiai.com.br), section "Softmax por
 * linha e FlashAttention": per row the maximum, subtraction, exponential and
 * normalisation; "TileLang ..." (pro.edgex.exchange): max and sum reductions in registers).
 *   rows, cols: 0 <= rows, 0 <= cols <= 2^31 - 1; either 0 is a no-op. cols must be a
 *               multiple of 8.
 *   X, Y      : device pointers (the context's device), rows x cols FP16 row-major,
 *               16-byte aligned. Y may be X itself (in place) but may not partly overlap it.
 * FP32 arithmetic, one RNE rounding to FP16. Entries of -inf contribute 0 (a row that is
 * all -inf gives NaN). Asynchronous on `stream`; allocates nothing; one kernel launch. */
int gemm_row_softmax(gemm_ctx *ctx, int64_t rows, int64_t cols, const void *X, void *Y, void *stream);

/* FlashAttention forward: for every head h and query i,
 *   O[h][i][:] = sum_j softmax_j(scale * Q[h][i][:] . K[h][j][:]) V[h][j][:],
 * with j restricted to j <= i when `causal` is 1 ("TileLang ..." (pro.edgex.exchange),
 * FlashAttention paragraph: query, key and value tiles, online softmax with running maxima,
 * normalising sums and rescaling, without materialising the score matrix; "Designing
 * High-Performance GPU Kernels with TileLang" (spaxe.top): causal and non-causal).
 *   heads, seq_q, seq_k: 0 <= each <= 2^31 - 1; heads = 0 or seq_q = 0 is a no-op;
 *               seq_k = 0 is an error. head_dim must be 128.
 *   Q          : device pointer, [heads][seq_q][128] FP16, contiguous, 16-byte aligned.
 *   K, V       : device pointers, [heads][seq_k][128] FP16, contiguous, 16-byte aligned.
 *   O          : device pointer, [heads][seq_q][128] FP16, written; must not overlap Q/K/V.
 *   scale      : multiplies Q.K (commonly 1/sqrt(128)); causal: 0 or 1.
 * FP32 scores and accumulation in Tensor Memory, probabilities rounded to FP16 for the P V
 * product, one RNE rounding of O. Asynchronous on `stream`; allocates nothing; one kernel
 * launch. In-kernel waits report through gemm_last_device_error like the GEMM. */
int gemm_attention_fwd(gemm_ctx *ctx, int64_t heads, int64_t seq_q, int64_t seq_k, int64_t head_dim,
                       const void *Q, const void *K, const void *V, void *O, float scale, int causal,
                       void *stream);

/* Test hooks (no effect on results when left at their defaults).
 *   gemm_set_timeout_ns: the limit of every in-kernel wait (default 2e9 ns; values below
 *     1e6 are raised to 1e6).
 *   gemm_set_debug, a bitwise OR of:
 *     GEMM_DEBUG_WITHHOLD_FIRST_LOAD: the producer (of CTA 0 of each pair, or of every
 *       CTA) holds back its first operand load, so that the MMA's wait on it runs out and
 *       the kernel must take its timeout path (a flag that nothing sets; no fault, no hang);
 *     GEMM_DEBUG_FORCE_SINGLE / GEMM_DEBUG_FORCE_PAIR: override the kernel choice, so that
 *       tests can run any shape through either kernel (FORCE_PAIR is ignored when the
 *       pair kernel cannot run);
 *     GEMM_DEBUG_FORCE_STREAMK: the one-CTA kernel always takes the stream-K schedule,
 *       with one CTA per k-block unit up to one per SM (so that tiles are cut into many
 *       parts), except for GEMM_EPI_SOFTMAX;
 *     GEMM_DEBUG_FORCE_SPLITK: the one-CTA kernel (never the pair kernel) takes the
 *       split-K schedule whenever K has at least 2 k-blocks, with the largest S of 8, 4, 2
 *       not above the k-blocks, for any number of tiles (clusters then run in several
 *       waves), except for GEMM_EPI_SOFTMAX; FORCE_STREAMK takes precedence. */
enum {
    GEMM_DEBUG_NONE = 0,
    GEMM_DEBUG_WITHHOLD_FIRST_LOAD = 1,
    GEMM_DEBUG_FORCE_SINGLE = 2,
    GEMM_DEBUG_FORCE_PAIR = 4,
    GEMM_DEBUG_FORCE_STREAMK = 8,
    GEMM_DEBUG_FORCE_SPLITK = 16
};
int gemm_set_timeout_ns(gemm_ctx *ctx, uint64_t ns);
int gemm_set_debug(gemm_ctx *ctx, int flags);

/* ---- Allocation-free variant ----------------------------------------------------------
 * The tutorial pages have no counterpart to this call; it exists for callers that cannot
 * allocate device memory. gemm_create allocates the kernel's scratch (a 4-byte device
 * error word) with cudaMalloc, which some callers may not do: plugins of an inference
 * engine that owns all device memory, real-time loops that forbid allocation after
 * start-up, code running where the allocator must not be touched.
 *
 * gemm_run_noalloc computes the same C = act(A*B + bias) with the same kernel and the
 * same argument rules as gemm_run (device pointers on the CURRENT device, N and K multiples
 * of 8, 16-byte alignment, M, N, K <= 2^31 - 1; larger sizes return GEMM_ERR_ARG), but
 * needs no context and calls no cudaMalloc, cudaFree or allocating library routine.
 * Its scratch is a file-scope __device__ array of GEMM_NOALLOC_SCRATCH_BYTES bytes that
 * every GPU loading the library holds until the process exits; this kernel needs 4 bytes
 * of it (the error word) whatever the problem size.
 *  - The first call on a device does a one-time set-up there (checks the device, sets
 *    the kernel's shared-memory limit, resolves the tensor-map encoder, looks up the
 *    array's device address). Make that first call before any stream capture.
 *  - Every call on a device shares the one array and clears the error word on `stream`
 *    before its launch. Calls whose kernels overlap on the GPU (different streams) race
 *    on the error word.
 *  - An in-kernel wait that runs out still ends the kernel cleanly, but this call has no
 *    way to report it (it returns before the kernel runs); use gemm_run and
 *    gemm_last_device_error where that report is needed.
 * Returns GEMM_OK once the work is enqueued, or an error code before anything is enqueued
 * (GEMM_ERR_LAUNCH if the launch itself fails). */
#define GEMM_NOALLOC_SCRATCH_BYTES 256
int gemm_run_noalloc(int64_t M, int64_t N, int64_t K, const void *A, const void *B,
                     const void *bias, void *C, int epilogue, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GB300_GEMM_H */
