/*
 * CPU oracle for the dense GEMM  C = alpha * A * B + beta * C.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct
 * definition the GPU kernels are checked against.  Only the tests, the
 * package smoke check and the CPU-baseline leg of the benchmark may load or
 * run it; the library's compute path never does, and the two share no code.
 *
 * What it follows (pages cited by title and section):
 *  - "Blackwell BF16 GEMM ..." (lshu.cn), section 1.1: GEMM is
 *    C = alpha * A * B + beta * C.
 *  - "CUDA hand-written SGEMM: 0.4 -> 10.23 TFLOPS" (gtnt.cn), section 1.1:
 *    the SGEMM special case C = A * B on row-major M x K and K x N matrices,
 *    and section 2.1: one output element is the sum over k of
 *    A[row][k] * B[k][col].
 *  - "CUDA shared memory optimisation" (hdetylss.com), section 3.3: the plain
 *    CPU i/j/k triple loop.
 *  - "Blackwell BF16 GEMM ...", sections 1.2 and 6.3: BF16 operands are
 *    multiplied and accumulated in higher precision and the result is
 *    converted back to BF16 once at the end.
 *
 * Readings where the pages are silent (the BLAS conventions):
 *  - beta == 0: C is not read (it may hold NaN); the result is alpha*A*B.
 *  - alpha == 0 or K == 0: A and B are not read; the result is beta*C
 *    itself, -0 included (+0 when beta == 0).
 *  - Inputs are widened exactly to double (fp32 and bf16 are subsets of
 *    double) and every product of two widened fp32/bf16 values is exact in
 *    double; only the running sums round.  The sum runs over k in
 *    increasing order.
 *  - Rounding the double result to the output type is round to nearest,
 *    ties to even, with overflow to infinity.
 *
 * Build: plain C99, -O2 -ffp-contract=off, no fast-math, no BLAS, no
 * intrinsics, POSIX threads over rows.  Same results on x86_64 and aarch64.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F64 = 2 };

/* Exact widening of one stored element to double. */
static double load_elem(int type, const void *p, int64_t idx) {
    if (type == ORACLE_F32) return (double)((const float *)p)[idx];
    if (type == ORACLE_F64) return ((const double *)p)[idx];
    /* bf16: the 16 stored bits are the upper half of an fp32 word. */
    uint32_t w = (uint32_t)((const uint16_t *)p)[idx] << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

typedef struct {
    int64_t M, N, K;
    double alpha, beta;
    int a_type, b_type, c_type;
    const void *A, *B, *C;
    int64_t lda, ldb, ldc, ldr;
    double *R;
    int64_t row_lo, row_hi;
} gemm_job;

/* Rows row_lo..row_hi-1 of R = alpha*A*B + beta*C, loop order i, k, j. */
static void *gemm_rows(void *arg) {
    const gemm_job *g = (const gemm_job *)arg;
    double *acc = (double *)calloc((size_t)(g->N > 0 ? g->N : 1), sizeof(double));
    if (!acc) return (void *)1;
    for (int64_t i = g->row_lo; i < g->row_hi; ++i) {
        for (int64_t j = 0; j < g->N; ++j) acc[j] = 0.0;
        if (g->alpha != 0.0) {
            for (int64_t k = 0; k < g->K; ++k) {
                double a = load_elem(g->a_type, g->A, i * g->lda + k);
                for (int64_t j = 0; j < g->N; ++j)
                    acc[j] += a * load_elem(g->b_type, g->B, k * g->ldb + j);
            }
        }
        for (int64_t j = 0; j < g->N; ++j) {
            const double bc =
                (g->beta != 0.0) ? g->beta * load_elem(g->c_type, g->C, i * g->ldc + j) : 0.0;
            /* alpha == 0: the result is beta*C itself (its sign of zero too);
             * beta == 0: alpha*A*B itself */
            const double ab = g->alpha * acc[j];
            const double r = (g->alpha == 0.0) ? bc : (g->beta != 0.0) ? ab + bc : ab;
            g->R[i * g->ldr + j] = r;
        }
    }
    free(acc);
    return NULL;
}

/*
 * R (M x N, row pitch ldr, double) = alpha * A * B + beta * C.
 * A: M x K row-major, pitch lda; B: K x N, pitch ldb; C: M x N, pitch ldc.
 * *_type: 0 = fp32, 1 = bf16 (uint16 bits), 2 = double.  C may be NULL
 * when beta == 0.  nthreads <= 0 means one thread.  Returns 0, or -1 on a
 * bad argument / allocation failure.
 */
int oracle_gemm(int64_t M, int64_t N, int64_t K, double alpha,
                int a_type, const void *A, int64_t lda,
                int b_type, const void *B, int64_t ldb,
                double beta, int c_type, const void *C, int64_t ldc,
                double *R, int64_t ldr, int nthreads) {
    if (M < 0 || N < 0 || K < 0 || !R) return -1;
    if (M == 0 || N == 0) return 0;
    if (beta != 0.0 && !C) return -1;
    if (alpha != 0.0 && K > 0 && (!A || !B)) return -1;
    if (K == 0) alpha = 0.0; /* empty sum: only beta*C remains */
    if (nthreads < 1) nthreads = 1;
    if (nthreads > M) nthreads = (int)M;

    gemm_job *jobs = (gemm_job *)calloc((size_t)nthreads, sizeof(gemm_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) { free(jobs); free(tids); return -1; }
    int rc = 0;
    for (int t = 0; t < nthreads; ++t) {
        gemm_job *g = &jobs[t];
        g->M = M; g->N = N; g->K = K; g->alpha = alpha; g->beta = beta;
        g->a_type = a_type; g->b_type = b_type; g->c_type = c_type;
        g->A = A; g->B = B; g->C = C;
        g->lda = lda; g->ldb = ldb; g->ldc = ldc; g->ldr = ldr; g->R = R;
        g->row_lo = M * t / nthreads;
        g->row_hi = M * (t + 1) / nthreads;
    }
    for (int t = 1; t < nthreads; ++t)
        if (pthread_create(&tids[t], NULL, gemm_rows, &jobs[t]) != 0) rc = -1;
    if (gemm_rows(&jobs[0]) != NULL) rc = -1;
    for (int t = 1; t < nthreads; ++t) {
        void *ret = NULL;
        pthread_join(tids[t], &ret);
        if (ret != NULL) rc = -1;
    }
    free(jobs);
    free(tids);
    return rc;
}

/*
 * Selected entries only: out[e] = alpha * sum_k A[rows[e]][k] * B[k][cols[e]]
 * + beta * C[rows[e]][cols[e]], same conventions as oracle_gemm.  This is the
 * element formula evaluated one output at a time, for matrices too large to
 * multiply whole on the CPU.
 */
int oracle_gemm_entries(int64_t M, int64_t N, int64_t K, double alpha,
                        int a_type, const void *A, int64_t lda,
                        int b_type, const void *B, int64_t ldb,
                        double beta, int c_type, const void *C, int64_t ldc,
                        int64_t count, const int64_t *rows, const int64_t *cols,
                        double *out) {
    if (M < 0 || N < 0 || K < 0 || count < 0 || !rows || !cols || !out) return -1;
    if (beta != 0.0 && !C) return -1;
    if (K == 0) alpha = 0.0;
    for (int64_t e = 0; e < count; ++e) {
        int64_t i = rows[e], j = cols[e];
        if (i < 0 || i >= M || j < 0 || j >= N) return -1;
        double sum = 0.0;
        if (alpha != 0.0)
            for (int64_t k = 0; k < K; ++k)
                sum += load_elem(a_type, A, i * lda + k) * load_elem(b_type, B, k * ldb + j);
        const double bc = (beta != 0.0) ? beta * load_elem(c_type, C, i * ldc + j) : 0.0;
        const double r = (alpha == 0.0) ? bc : (beta != 0.0) ? alpha * sum + bc : alpha * sum;
        out[e] = r;
    }
    return 0;
}

/* Double -> fp32, round to nearest even (the C conversion under the default
 * rounding mode), overflow to infinity. */
void oracle_round_f32(const double *x, float *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = (float)x[i];
}

/*
 * Double -> bf16 bits, round to nearest even, overflow to infinity, taken
 * straight from the definition of the format (1 sign, 8 exponent, 7 stored
 * fraction bits, exponent bias 127, subnormal quantum 2^-133): find the
 * quantum q of the binade holding |x|, round x/q to an integer with ties to
 * even (rint under the default rounding mode), scale back, then read the
 * bits of the now exactly representable value.
 */
static uint16_t round_one_bf16(double x) {
    if (isnan(x)) return (uint16_t)(signbit(x) ? 0xFFC0 : 0x7FC0);
    if (isinf(x)) return (uint16_t)(signbit(x) ? 0xFF80 : 0x7F80);
    if (x == 0.0) return (uint16_t)(signbit(x) ? 0x8000 : 0x0000);
    int e2;
    frexp(x, &e2);                        /* |x| in [2^(e2-1), 2^e2) */
    int qexp = (e2 - 1) - 7;              /* 8 significant bits in a binade */
    if (qexp < -133) qexp = -133;         /* subnormal range */
    double r = ldexp(rint(ldexp(x, -qexp)), qexp);
    if (fabs(r) >= ldexp(1.0, 128))       /* rounded past the largest finite */
        return (uint16_t)(signbit(x) ? 0xFF80 : 0x7F80);
    float f = (float)r;                    /* exact: r is a bf16 value */
    uint32_t w;
    memcpy(&w, &f, sizeof w);
    return (uint16_t)(w >> 16);
}

void oracle_round_bf16(const double *x, uint16_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = round_one_bf16(x[i]);
}

/* Exact widening helpers, so a test can read stored operands back. */
void oracle_widen_bf16(const uint16_t *x, double *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = load_elem(ORACLE_BF16, x, i);
}

/*
 * Fused epilogue, applied to R = alpha * op(A) * op(B) computed by
 * oracle_gemm with beta = 0:  R = act(R + bias) + beta * C.
 *
 * Follows the fused "normalise, GELU, residual add" kernel of the "Z-Turbo"
 * tuning page (lanjinlin.com.cn), section 2.1: the activation is applied
 * first and the residual (here beta * C) is added after it; and the
 * epilogue customisations (GELU, residual) named by "Blackwell BF16 GEMM
 * ..." (lshu.cn), section 3.3.  The GELU is that page's tanh form,
 * 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))), here in double with the
 * exact constant sqrt(2/pi) (the page prints it as 0.79788456).
 *   bias: NULL or N values (type bias_type: 0 fp32, 1 bf16, 2 double)
 *   act:  0 none, 1 relu (max(x, 0)), 2 gelu (tanh form)
 *   beta == 0: C is not read.
 */
static double act_apply(int act, double x) {
    if (act == 1) return x > 0.0 ? x : 0.0;
    if (act == 2) {
        const double k = sqrt(2.0 / 3.14159265358979323846);
        return 0.5 * x * (1.0 + tanh(k * (x + 0.044715 * x * x * x)));
    }
    return x;
}

int oracle_epilogue(int64_t M, int64_t N, double *R, int64_t ldr, int bias_type,
                    const void *bias, int act, double beta, int c_type, const void *C,
                    int64_t ldc) {
    if (M < 0 || N < 0 || !R || act < 0 || act > 2) return -1;
    if (beta != 0.0 && !C) return -1;
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            double v = R[i * ldr + j];
            if (bias) v += load_elem(bias_type, bias, j);
            v = act_apply(act, v);
            if (beta != 0.0) v += beta * load_elem(c_type, C, i * ldc + j);
            R[i * ldr + j] = v;
        }
    return 0;
}
