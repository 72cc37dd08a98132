/*
 * gemm_oracle.c -- the CPU oracle for the dense GEMM library.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the package smoke check and the bench's
 * CPU-baseline leg do.  It shares no code, header or constant with the CUDA
 * library under dense_gemm_11_gb300/csrc.
 *
 * What it computes (plain definition, written out):
 *
 *   "SGEMM优化，从naive到warptiling", section 项目概况 / 问题与估算:
 *       C = alpha * A x B + beta * C, A is MxK, B is KxN, C is MxN, all
 *       row-major float.
 *   "第24讲 ... GEMM 分块与 Tensor Core 思维", section 0.1: the same product as
 *       the plain triple loop sum_k A[i][k] * B[k][j].
 *   "企业官网建设流程全解析" (the DeepGEMM essay), sections 1.3 and 3.2: the
 *       FP16-input / FP32-accumulate variant folds bias, scale and an
 *       activation (GELU) into the epilogue.
 *
 *   out[i][j] = act( alpha * sum_{k=0}^{K-1} A[i*lda+k] * B[k*ldb+j]
 *                    + beta * C0[i*ldc+j] + bias[j] )
 *
 * Readings where the pages are silent (BLAS convention):
 *   - beta == 0: C0 is not read (a NaN in C0 does not propagate);
 *   - alpha == 0 or K == 0: A and B are not read; the product term is 0;
 *   - bias == NULL: no bias term;  act: 0 = identity, 1 = exact GELU,
 *     GELU(x) = x * Phi(x) = 0.5 * x * (1 + erf(x / sqrt(2))); 2 = ReLU,
 *     max(x, 0); 3 = the tanh approximation of GELU (Hendrycks and Gimpel,
 *     "Gaussian Error Linear Units"), 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).
 *     The pages name "activation" and GELU in the epilogue without fixing a
 *     form; the exact form is the default, the other two are the common
 *     alternatives an inference epilogue offers.
 *
 * Arithmetic: every input arrives as double (fp32 and fp16 values are
 * exactly representable in double); the sum over k is taken in double with k
 * ascending for every (i, j).  The loop order is i, k, j (a row of partial
 * sums per i) so that B is walked along its rows; that changes no element's
 * summation order.  Alongside the value the oracle returns the per-element
 * error scale
 *
 *   S[i][j] = |alpha| * sum_k |A[i][k]| * |B[k][j]| + |beta| * |C0[i][j]|
 *
 * used by the acceptance bound |C - C_ref| <= tol * S + 1e-6.  The bias is
 * not part of S: adding it is one FP32 rounding of at most a unit in the
 * last place of |bias[j]|, which the tests allow for as a term of its own.
 *
 * Output element type (the tensor-core entry point may write C as FP16 or
 * BF16): the value above is rounded once, to nearest with ties to even, to
 * the output format; beyond the largest finite value it becomes +-inf
 * (IEEE 754 roundTiesToEven).  FP16 = binary16 (11 significand bits,
 * exponents -14..15), BF16 = 8 significand bits with binary32's exponent
 * range (-126..127).  round_format below writes that rule out for any such
 * format.
 *
 * Threads: the listed rows are split into contiguous ranges, one per thread.
 * Build with -ffp-contract=off so that x86 and Arm hosts give the same bits.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    long M, N, K;
    double alpha, beta;
    const double *A, *B, *C0, *bias;
    long lda, ldb, ldc;
    int act;
    const long *rows; /* NULL: rows r0..r1 are row numbers themselves */
    long r0, r1;      /* range of positions in the row list handled here */
    double *out, *scale;
    int status;
} oracle_job;

static double gelu_exact(double x) { return 0.5 * x * (1.0 + erf(x / sqrt(2.0))); }
static double gelu_tanh(double x) {
    const double pi = 3.14159265358979323846;
    return 0.5 * x * (1.0 + tanh(sqrt(2.0 / pi) * (x + 0.044715 * x * x * x)));
}
static double apply_act(int act, double v) {
    switch (act) {
        case 1: return gelu_exact(v);
        case 2: return v > 0.0 ? v : 0.0;
        case 3: return gelu_tanh(v);
        default: return v;
    }
}

static void *oracle_rows(void *arg) {
    oracle_job *J = (oracle_job *)arg;
    const long N = J->N, K = J->K;
    double *acc = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    double *sab = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    if (!acc || !sab) {
        free(acc);
        free(sab);
        J->status = -1;
        return NULL;
    }
    const int use_product = (J->alpha != 0.0) && (K > 0);
    for (long p = J->r0; p < J->r1; ++p) {
        const long i = J->rows ? J->rows[p] : p;
        for (long j = 0; j < N; ++j) {
            acc[j] = 0.0;
            sab[j] = 0.0;
        }
        if (use_product) {
            const double *Ai = J->A + i * J->lda;
            for (long k = 0; k < K; ++k) {
                const double a = Ai[k];
                const double aa = fabs(a);
                const double *Bk = J->B + k * J->ldb;
                for (long j = 0; j < N; ++j) {
                    acc[j] += a * Bk[j];
                    sab[j] += aa * fabs(Bk[j]);
                }
            }
        }
        double *o = J->out + p * N;
        double *s = J->scale ? J->scale + p * N : NULL;
        for (long j = 0; j < N; ++j) {
            double v = use_product ? J->alpha * acc[j] : 0.0;
            double sc = use_product ? fabs(J->alpha) * sab[j] : 0.0;
            if (J->beta != 0.0) {
                const double c = J->C0[i * J->ldc + j];
                v += J->beta * c;
                sc += fabs(J->beta) * fabs(c);
            }
            if (J->bias) v += J->bias[j];
            v = apply_act(J->act, v);
            o[j] = v;
            if (s) s[j] = sc;
        }
    }
    free(acc);
    free(sab);
    J->status = 0;
    return NULL;
}

/*
 * oracle_gemm_f64: evaluate the rows listed in rows[0..nrows) (or rows
 * 0..nrows-1 when rows == NULL) of out = act(alpha*A*B + beta*C0 + bias).
 * out and scale (scale may be NULL) are nrows x N, row-major, contiguous.
 * Returns 0 on success, -1 on a bad argument or allocation failure.
 */
int oracle_gemm_f64(long M, long N, long K, double alpha, const double *A, long lda,
                    const double *B, long ldb, double beta, const double *C0, long ldc,
                    const double *bias, int act, const long *rows, long nrows, double *out,
                    double *scale, int nthreads) {
    if (M < 0 || N < 0 || K < 0 || nrows < 0 || !out) return -1;
    if (act < 0 || act > 3) return -1;
    if (nrows == 0 || N == 0) return 0;
    if (alpha != 0.0 && K > 0 && (!A || !B || lda < K || ldb < N)) return -1;
    if (beta != 0.0 && (!C0 || ldc < N)) return -1;
    for (long p = 0; p < nrows; ++p) {
        const long i = rows ? rows[p] : p;
        if (i < 0 || i >= M) return -1;
    }
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (nthreads > nrows) nthreads = (int)nrows;

    oracle_job jobs[256];
    pthread_t tid[256];
    int started[256];
    for (int t = 0; t < nthreads; ++t) {
        oracle_job *J = &jobs[t];
        J->M = M; J->N = N; J->K = K;
        J->alpha = alpha; J->beta = beta;
        J->A = A; J->B = B; J->C0 = C0; J->bias = bias;
        J->lda = lda; J->ldb = ldb; J->ldc = ldc;
        J->act = act;
        J->rows = rows;
        J->r0 = nrows * t / nthreads;
        J->r1 = nrows * (t + 1) / nthreads;
        J->out = out; J->scale = scale;
        J->status = -1;
        started[t] = 0;
    }
    for (int t = 1; t < nthreads; ++t)
        started[t] = pthread_create(&tid[t], NULL, oracle_rows, &jobs[t]) == 0;
    oracle_rows(&jobs[0]);
    int status = jobs[0].status;
    for (int t = 1; t < nthreads; ++t) {
        if (started[t]) {
            pthread_join(tid[t], NULL);
        } else {
            oracle_rows(&jobs[t]); /* could not spawn: do the range here */
        }
        if (jobs[t].status != 0) status = -1;
    }
    return status;
}

/*
 * Round x to the nearest number of a binary floating-point format with p
 * significand bits (the leading bit included), smallest normal exponent emin
 * and largest exponent emax; ties go to the even neighbour; results past the
 * largest finite number are +-inf.  The last kept bit of x has weight 2^q,
 * q = max(exponent of x's leading bit, emin) - (p - 1) (below emin the
 * spacing stays that of the subnormals); x / 2^q is rounded to an integer in
 * the default rounding mode (nearest, ties to even) and scaled back.  Both
 * scalings are exact.
 */
static double round_format(double x, int p, int emin, int emax) {
    if (x == 0.0 || !isfinite(x)) return x;
    int e;
    frexp(x, &e); /* |x| = m * 2^e with m in [0.5, 1): the leading bit is 2^(e-1) */
    int lead = e - 1;
    if (lead < emin) lead = emin;
    const int q = lead - (p - 1);
    double r = ldexp(nearbyint(ldexp(x, -q)), q);
    const double max_finite = ldexp(2.0 - ldexp(1.0, 1 - p), emax);
    if (fabs(r) > max_finite) r = copysign(INFINITY, x);
    return r;
}

/*
 * oracle_round_f64: out[i] = x[i] rounded to the output type (0 = FP32,
 * 1 = FP16, 2 = BF16).  Returns 0, or -1 for an unknown type.
 */
int oracle_round_f64(int type, const double *x, double *out, long n) {
    int p, emin, emax;
    switch (type) {
        case 0: p = 24; emin = -126; emax = 127; break;
        case 1: p = 11; emin = -14; emax = 15; break;
        case 2: p = 8; emin = -126; emax = 127; break;
        default: return -1;
    }
    for (long i = 0; i < n; ++i) out[i] = round_format(x[i], p, emin, emax);
    return 0;
}

/* The activations alone, exposed so that their special values can be pinned. */
double oracle_gelu_f64(double x) { return gelu_exact(x); }
double oracle_act_f64(int act, double x) { return apply_act(act, x); }
