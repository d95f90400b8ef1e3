/*
 * FP64 CPU oracle for the fused FP16 GEMM  C = act(A * B + bias).
 *
 * TEST INFRASTRUCTURE ONLY. This is the plain, slow, obviously correct definition that the
 * CUDA kernels are checked against. Only the tests, the smoke check and the benchmark's CPU
 * baseline load it; the library's product path never does. It shares no code, header,
 * helper or constant with the CUDA path.
 *
 * What it computes (the tutorial's tensor-core GEMM and its fused epilogue):
 *
 *   C[m][n] = fp16_rne( act( sum_{k} a[m][k] * b[k][n]  +  beta[n] ) )
 *
 *  - A is M x K and B is K x N, both row-major. "TileLang: Criando Kernels de GPU ..."
 *    (noticiai.com.br), section "GEMM com Tensor Cores", slices A[i:i+128, k:k+32] and
 *    B[k:k+32, j:j+128]: A's rows are output rows, B's columns are output columns.
 *  - Inputs are FP16 ("Designing High-Performance GPU Kernels with TileLang", spaxe.top,
 *    GEMM paragraph: an FP16 matrix multiply). Each input is widened exactly to double;
 *    every product of two FP16 values is exact in double and the k-sum is done in double,
 *    in the order k = 0, 1, ..., K-1.
 *  - Epilogue ("TileLang ..." pro.edgex.exchange, fused-epilogue paragraph: bias addition
 *    and GELU applied to the accumulator before the one output store; noticiai.com.br,
 *    section "GEMM com epilogo fundido": ReLU fused the same way): the bias beta[n] is
 *    added to the accumulator first (beta = 0 when no bias is given), then act is applied:
 *      identity, GELU(x) = x * Phi(x) = 0.5 * x * (1 + erf(x / sqrt(2))) (the exact erf
 *      form; the pages only say "GELU"), or ReLU(x) = max(x, 0).
 *  - The result is rounded once to FP16, round-to-nearest-even, with overflow to +-inf.
 *
 * The file also holds the row-wise softmax of the same tutorial (oracle_softmax_rows), and
 * the GEMM with a row-softmax epilogue (act = 3): softmax over each row of A*B + bias, the
 * logits kept in double (never rounded to FP16), and the attention forward result
 * (oracle_attention_rows) that the FlashAttention kernel computes.
 *
 * Parity pins (tests/test_oracle.py): exhaustive FP16 decoding and RNE encoding against
 * numpy; a textbook worked example; identity and all-ones products; brute-force loops on
 * tiny shapes; numpy float64 matmul on medium shapes; GELU against standard-normal table
 * values and its limits; ReLU sign cases; row-sample mode against full mode.
 *
 * Build: gcc -O3 -ffp-contract=off -fPIC -shared oracle.c -lm -lpthread
 * (-ffp-contract=off keeps x86 and Arm results bit-identical: no fused multiply-adds.)
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { ORACLE_ACT_NONE = 0, ORACLE_ACT_GELU = 1, ORACLE_ACT_RELU = 2, ORACLE_ACT_SOFTMAX = 3 };

/* ---- FP16 (IEEE 754 binary16) <-> double, written from the format's definition ---------
 * binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 *   exponent 0      : subnormal, value = fraction * 2^-24
 *   exponent 1..30  : normal,    value = (1024 + fraction) * 2^(exponent - 25)
 *   exponent 31     : inf (fraction 0) or NaN                                          */
double oracle_half_to_double(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int expo = (h >> 10) & 0x1f;
    const int frac = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -24);
    else if (expo == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + frac), expo - 25);
    return sign ? -v : v;
}

/* Round a double to the nearest binary16, ties to even. The quantum (spacing of binary16
 * values) at |x| is 2^(E-10) for the normal range (E = floor(log2|x|) >= -14) and 2^-24
 * below it; |x| / quantum is exact (a power-of-two scaling), rint() rounds it to the
 * nearest integer with ties to even (the default rounding mode), and the rounded value is
 * then encoded exactly. |x| >= 65520 (halfway between 65504 and 2^16) rounds to inf. */
uint16_t oracle_double_to_half(double x)
{
    const uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x))
        return 0x7e00;
    const double ax = fabs(x);
    if (ax >= 65520.0)
        return sign | 0x7c00;
    if (ax == 0.0)
        return sign;
    int e;
    frexp(ax, &e);              /* ax = f * 2^e, f in [0.5, 1) -> floor(log2 ax) = e - 1 */
    int E = e - 1;
    if (E < -14)
        E = -14;
    const double q = ldexp(1.0, E - 10);
    const double v = rint(ax / q) * q;   /* rounded magnitude, exactly representable */
    if (v == 0.0)
        return sign;
    frexp(v, &e);
    E = e - 1;
    if (E < -14)                          /* subnormal: fraction = v / 2^-24 */
        return sign | (uint16_t)ldexp(v, 24);
    const int mant = (int)(ldexp(v, 10 - E)) - 1024;  /* 0..1023 */
    return sign | (uint16_t)(((E + 15) << 10) | mant);
}

/* The epilogue's activation, in double. */
double oracle_act(double x, int act)
{
    switch (act) {
    case ORACLE_ACT_GELU:
        return 0.5 * x * (1.0 + erf(x * M_SQRT1_2));
    case ORACLE_ACT_RELU:
        return x > 0.0 ? x : 0.0;
    default:
        return x;
    }
}

int oracle_default_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/* ---- row-wise softmax ---------------------------------------------------------------------
 * Y[r][j] = fp16_rne( exp(x[r][j] - m_r) / sum_k exp(x[r][k] - m_r) ),  m_r = max_k x[r][k],
 * with x the FP16 input widened exactly to double and everything in double ("TileLang:
 * Criando Kernels de GPU ..." (noticiai.com.br), section "Softmax por linha e
 * FlashAttention": per row, the maximum, subtraction, exponentiation, normalisation).
 * Subtracting the row maximum does not change the mathematical result; it keeps exp() in
 * range. A row of length 0 has nothing to write. */
typedef struct {
    int64_t rows, cols;
    const uint16_t *X;
    uint16_t *Y;
    double *Yd;   /* rows x cols doubles before rounding, or NULL */
    int tid, nthreads;
} softmax_job_t;

static void *softmax_worker(void *arg)
{
    softmax_job_t *j = (softmax_job_t *)arg;
    for (int64_t r = j->tid; r < j->rows; r += j->nthreads) {
        const uint16_t *x = j->X + r * j->cols;
        double m = -INFINITY;
        for (int64_t c = 0; c < j->cols; ++c) {
            const double v = oracle_half_to_double(x[c]);
            if (v > m)
                m = v;
        }
        double s = 0.0;
        for (int64_t c = 0; c < j->cols; ++c)
            s += exp(oracle_half_to_double(x[c]) - m);
        for (int64_t c = 0; c < j->cols; ++c) {
            const double y = exp(oracle_half_to_double(x[c]) - m) / s;
            if (j->Yd)
                j->Yd[r * j->cols + c] = y;
            j->Y[r * j->cols + c] = oracle_double_to_half(y);
        }
    }
    return NULL;
}

/* Softmax of each of the `rows` rows of X (rows x cols FP16 bits, row-major) into Y (same
 * shape); Yd (optional) receives the values before rounding. Returns 0 or -1 (bad args). */
int oracle_softmax_rows(int64_t rows, int64_t cols, const uint16_t *X, uint16_t *Y, double *Yd, int threads)
{
    if (rows < 0 || cols < 0 || ((rows * cols > 0) && (!X || !Y)))
        return -1;
    if (rows == 0 || cols == 0)
        return 0;
    int T = threads > 0 ? threads : oracle_default_threads();
    if (T > rows)
        T = (int)rows;
    pthread_t *th = (pthread_t *)malloc((size_t)T * sizeof(pthread_t));
    softmax_job_t *jobs = (softmax_job_t *)calloc((size_t)T, sizeof(softmax_job_t));
    if (!th || !jobs) {
        free(th);
        free(jobs);
        return -2;
    }
    for (int t = 0; t < T; ++t) {
        jobs[t] = (softmax_job_t){rows, cols, X, Y, Yd, t, T};
        pthread_create(&th[t], NULL, softmax_worker, &jobs[t]);
    }
    for (int t = 0; t < T; ++t)
        pthread_join(th[t], NULL);
    free(th);
    free(jobs);
    return 0;
}

/* ---- attention forward ---------------------------------------------------------------------
 * For every head h and query row i (FlashAttention's forward result, computed the plain way:
 * "TileLang ..." (pro.edgex.exchange), FlashAttention paragraph: query, key and value tiles,
 * online softmax; the result is ordinary attention):
 *   s_j = scale * sum_d q[h][i][d] * k[h][j][d]            for keys j (j <= i when causal)
 *   O[h][i][d] = fp16_rne( sum_j exp(s_j - max_j s_j) * v[h][j][d] / sum_j exp(s_j - max s) )
 * Q is [H][Sq][D], K and V are [H][Sk][D], O is [H][Sq][D], all FP16 row-major, widened
 * exactly to double; everything in double. Causal: key j is visible to query i iff j <= i. */
typedef struct {
    int64_t H, Sq, Sk, D;
    const uint16_t *Q, *K, *V;
    double scale;
    int causal;
    const int64_t *rows;   /* (head, query) pairs: rows[2t], rows[2t+1] */
    int64_t nrows;
    uint16_t *out;         /* nrows x D */
    double *outd;
    int tid, nthreads, failed;
} attn_job_t;

static void *attn_worker(void *arg)
{
    attn_job_t *j = (attn_job_t *)arg;
    const int64_t Sk = j->Sk, D = j->D;
    double *s = (double *)malloc((size_t)(Sk > 0 ? Sk : 1) * sizeof(double));
    double *o = (double *)malloc((size_t)(D > 0 ? D : 1) * sizeof(double));
    if (!s || !o) {
        j->failed = 1;
        free(s);
        free(o);
        return NULL;
    }
    for (int64_t t = j->tid; t < j->nrows; t += j->nthreads) {
        const int64_t h = j->rows[2 * t], i = j->rows[2 * t + 1];
        const uint16_t *q = j->Q + (h * j->Sq + i) * D;
        const int64_t nk = j->causal ? (i + 1 < Sk ? i + 1 : Sk) : Sk;
        double mx = -INFINITY;
        for (int64_t k = 0; k < nk; ++k) {
            const uint16_t *kr = j->K + (h * Sk + k) * D;
            double acc = 0.0;
            for (int64_t d = 0; d < D; ++d)
                acc += oracle_half_to_double(q[d]) * oracle_half_to_double(kr[d]);
            s[k] = j->scale * acc;
            if (s[k] > mx)
                mx = s[k];
        }
        double sum = 0.0;
        for (int64_t k = 0; k < nk; ++k) {
            s[k] = exp(s[k] - mx);
            sum += s[k];
        }
        for (int64_t d = 0; d < D; ++d)
            o[d] = 0.0;
        for (int64_t k = 0; k < nk; ++k) {
            const uint16_t *vr = j->V + (h * Sk + k) * D;
            for (int64_t d = 0; d < D; ++d)
                o[d] += s[k] * oracle_half_to_double(vr[d]);
        }
        for (int64_t d = 0; d < D; ++d) {
            const double y = nk > 0 ? o[d] / sum : 0.0;
            if (j->outd)
                j->outd[t * D + d] = y;
            j->out[t * D + d] = oracle_double_to_half(y);
        }
    }
    free(s);
    free(o);
    return NULL;
}

/* Attention output rows for the (head, query) pairs in `rows` (2 * nrows int64 values).
 * Returns 0, -1 for bad arguments, -2 when memory runs out. */
int oracle_attention_rows(int64_t H, int64_t Sq, int64_t Sk, int64_t D, const uint16_t *Q, const uint16_t *K,
                          const uint16_t *V, double scale, int causal, const int64_t *rows, int64_t nrows,
                          uint16_t *out, double *outd, int threads)
{
    if (H < 0 || Sq < 0 || Sk < 0 || D < 0 || nrows < 0 || !rows || !out || !Q || !K || !V)
        return -1;
    for (int64_t t = 0; t < nrows; ++t)
        if (rows[2 * t] < 0 || rows[2 * t] >= H || rows[2 * t + 1] < 0 || rows[2 * t + 1] >= Sq)
            return -1;
    if (nrows == 0)
        return 0;
    int T = threads > 0 ? threads : oracle_default_threads();
    if (T > nrows)
        T = (int)nrows;
    pthread_t *th = (pthread_t *)malloc((size_t)T * sizeof(pthread_t));
    attn_job_t *jobs = (attn_job_t *)calloc((size_t)T, sizeof(attn_job_t));
    if (!th || !jobs) {
        free(th);
        free(jobs);
        return -2;
    }
    for (int t = 0; t < T; ++t) {
        jobs[t] = (attn_job_t){H, Sq, Sk, D, Q, K, V, scale, causal, rows, nrows, out, outd, t, T, 0};
        pthread_create(&th[t], NULL, attn_worker, &jobs[t]);
    }
    int rc = 0;
    for (int t = 0; t < T; ++t) {
        pthread_join(th[t], NULL);
        if (jobs[t].failed)
            rc = -2;
    }
    free(th);
    free(jobs);
    return rc;
}

/* ---- the GEMM --------------------------------------------------------------------------- */
typedef struct {
    int64_t N, K;
    const uint16_t *A;
    const double *Bd;      /* B widened to double, K x N row-major */
    const double *biasd;   /* N doubles, or NULL */
    int act;
    const int64_t *rows;   /* output rows to compute (nrows of them) */
    int64_t nrows;
    uint16_t *out_h;       /* nrows x N FP16 bits */
    double *out_d;         /* nrows x N doubles (value before the FP16 rounding), or NULL */
    int tid, nthreads;
    int failed;
} job_t;

static void *row_worker(void *arg)
{
    job_t *j = (job_t *)arg;
    const int64_t N = j->N, K = j->K;
    double *acc = (double *)malloc((size_t)N * sizeof(double));
    if (!acc) {
        j->failed = 1;
        return NULL;
    }
    for (int64_t i = j->tid; i < j->nrows; i += j->nthreads) {
        const int64_t m = j->rows[i];
        const uint16_t *arow = j->A + m * K;
        for (int64_t n = 0; n < N; ++n)
            acc[n] = 0.0;
        /* acc[n] = sum over k, in increasing k, of a[m][k] * b[k][n] */
        for (int64_t k = 0; k < K; ++k) {
            const double a = oracle_half_to_double(arow[k]);
            const double *brow = j->Bd + k * N;
            for (int64_t n = 0; n < N; ++n)
                acc[n] += a * brow[n];
        }
        if (j->act == ORACLE_ACT_SOFTMAX) {
            /* softmax over the whole output row of logits acc[n] + beta[n], in double
             * ("Designing High-Performance GPU Kernels with TileLang", spaxe.top: row-wise
             * softmax applied to the GEMM result in its epilogue) */
            double mx = -INFINITY, sum = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                acc[n] += (j->biasd ? j->biasd[n] : 0.0);
                if (acc[n] > mx)
                    mx = acc[n];
            }
            for (int64_t n = 0; n < N; ++n)
                sum += exp(acc[n] - mx);
            for (int64_t n = 0; n < N; ++n) {
                const double y = exp(acc[n] - mx) / sum;
                if (j->out_d)
                    j->out_d[i * N + n] = y;
                j->out_h[i * N + n] = oracle_double_to_half(y);
            }
            continue;
        }
        for (int64_t n = 0; n < N; ++n) {
            double x = acc[n] + (j->biasd ? j->biasd[n] : 0.0);
            x = oracle_act(x, j->act);
            if (j->out_d)
                j->out_d[i * N + n] = x;
            j->out_h[i * N + n] = oracle_double_to_half(x);
        }
    }
    free(acc);
    return NULL;
}

typedef struct {
    const uint16_t *src;
    double *dst;
    int64_t count;
    int tid, nthreads;
} widen_t;

static void *widen_worker(void *arg)
{
    widen_t *w = (widen_t *)arg;
    const int64_t chunk = (w->count + w->nthreads - 1) / w->nthreads;
    const int64_t lo = (int64_t)w->tid * chunk;
    const int64_t hi = lo + chunk < w->count ? lo + chunk : w->count;
    for (int64_t i = lo; i < hi; ++i)
        w->dst[i] = oracle_half_to_double(w->src[i]);
    return NULL;
}

/*
 * Compute the rows `rows[0..nrows)` of C = act(A*B + bias) (all M rows, in order, when
 * rows == NULL; then nrows must equal M).
 *   A    : M x K FP16 bits, row-major        B : K x N FP16 bits, row-major
 *   bias : N FP16 bits, or NULL (no bias)    act : 0 none, 1 GELU (erf), 2 ReLU,
 *                                             3 softmax over each output row
 *   out_h: nrows x N FP16 bits (row i of out_h is row rows[i] of C)
 *   out_d: nrows x N doubles before rounding, or NULL
 *   threads: worker threads (<= 0: all online cores); *threads_used receives the count.
 * Returns 0, -1 for bad arguments, -2 when memory runs out.
 */
int oracle_gemm_rows(int64_t M, int64_t N, int64_t K, const uint16_t *A, const uint16_t *B,
                     const uint16_t *bias, int act, const int64_t *rows, int64_t nrows,
                     uint16_t *out_h, double *out_d, int threads, int *threads_used)
{
    if (M < 0 || N < 0 || K < 0 || nrows < 0 || act < 0 || act > 3 || !out_h)
        return -1;
    if ((M * K > 0 && !A) || (K * N > 0 && !B))
        return -1;
    if (!rows && nrows != M)
        return -1;
    if (rows)
        for (int64_t i = 0; i < nrows; ++i)
            if (rows[i] < 0 || rows[i] >= M)
                return -1;
    int T = threads > 0 ? threads : oracle_default_threads();
    if (nrows > 0 && T > nrows)
        T = (int)nrows;
    if (T < 1)
        T = 1;
    if (threads_used)
        *threads_used = T;
    if (nrows == 0 || N == 0)
        return 0;

    int rc = 0;
    double *Bd = (double *)malloc((size_t)(K * N > 0 ? K * N : 1) * sizeof(double));
    double *biasd = bias ? (double *)malloc((size_t)N * sizeof(double)) : NULL;
    int64_t *allrows = rows ? NULL : (int64_t *)malloc((size_t)M * sizeof(int64_t));
    pthread_t *th = (pthread_t *)malloc((size_t)T * sizeof(pthread_t));
    job_t *jobs = (job_t *)calloc((size_t)T, sizeof(job_t));
    widen_t *wj = (widen_t *)calloc((size_t)T, sizeof(widen_t));
    if (!Bd || (bias && !biasd) || (!rows && !allrows) || !th || !jobs || !wj) {
        rc = -2;
        goto done;
    }
    for (int t = 0; t < T; ++t) {
        wj[t] = (widen_t){B, Bd, K * N, t, T};
        pthread_create(&th[t], NULL, widen_worker, &wj[t]);
    }
    for (int t = 0; t < T; ++t)
        pthread_join(th[t], NULL);
    if (bias)
        for (int64_t n = 0; n < N; ++n)
            biasd[n] = oracle_half_to_double(bias[n]);
    if (!rows) {
        for (int64_t m = 0; m < M; ++m)
            allrows[m] = m;
        rows = allrows;
    }
    for (int t = 0; t < T; ++t) {
        jobs[t] = (job_t){N, K, A, Bd, biasd, act, rows, nrows, out_h, out_d, t, T, 0};
        pthread_create(&th[t], NULL, row_worker, &jobs[t]);
    }
    for (int t = 0; t < T; ++t) {
        pthread_join(th[t], NULL);
        if (jobs[t].failed)
            rc = -2;
    }
done:
    free(Bd);
    free(biasd);
    free(allrows);
    free(th);
    free(jobs);
    free(wj);
    return rc;
}
