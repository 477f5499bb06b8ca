/*
 * Oracle for dense GEMM:  C = alpha * op(A) * op(B) + beta * C, row-major.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct CPU
 * statement of what the GPU library computes.  It is compiled into its own
 * shared object (liboracle_gemm.so) and is used only by the tests, the smoke
 * check and the CPU baseline of the bench.  The product library never links,
 * loads or calls it, and it shares no code with the product library.
 *
 * What it follows (citations are to the pages the method is taken from):
 *   - "Optimizing GEMM on Apple's M5 from scratch, Part 1: Basics", section
 *     "Introduction" (the sidenote defining full SGEMM as C = alpha*A*B + beta*C)
 *     and section "Kernel 1: Naive Implementation" (the three nested loops:
 *     one dot product along K per element of C).
 *   - "From a C loop to a GPU kernel", section "The first loop" (the ijk loop
 *     over row-major storage and the worked C[1][2] expansion), and the
 *     observation there that loops which keep each output's contributions in
 *     strict increasing-k order while vectorising across j (the ikj order)
 *     reproduce the plain loop exactly.
 *   - "Metal GEMM Kernels for LoRA Training on Apple Silicon", section 2
 *     "GEMM structure", variant table: nn A[M,K]@B[K,N], tn A[K,M]^T@B[K,N],
 *     nt A[M,K]@B[N,K]^T; fp16 operands with fp32 accumulation (section 1,
 *     whose type table also lists bfloat16 operands -- emulated on that GPU,
 *     native on this one).
 *
 * Arithmetic: every input element is widened exactly to double (fp32, fp16 and
 * bfloat16 values are exactly representable in double), every product of two
 * such values is exact in double (at most 24+24 significant bits), and the sum for
 * each output element is accumulated in double in strict increasing k.  The
 * file is built with -ffp-contract=off so no multiply is fused into an add.
 *
 * Besides ref[i][j] the oracle returns mag[i][j] = |alpha| * sum_k |a_ik b_kj|
 * + |beta * C_in[i][j]|, the scale against which the GPU result's error is
 * bounded.
 *
 * beta == 0 means C_in is not read at all (the BLAS convention; the pages do
 * not say), so NaN in C_in does not reach the result.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_F16 1
#define ORACLE_BF16 2

/* ---------------------------------------------------------------------------
 * IEEE 754 binary16 <-> double, written from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits; exponent field 0
 * encodes zero and subnormals (fraction * 2^-24), 31 encodes inf and NaN.
 * ------------------------------------------------------------------------- */
double oracle_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25);
    }
    return sign ? -v : v;
}

/* Round-half-to-even of a non-negative double to an integer-valued double. */
static double rne_integer(double n) {
    double fl = floor(n);
    double d = n - fl; /* exact: n and fl share the exponent range */
    if (d > 0.5) return fl + 1.0;
    if (d < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* double -> binary16 with round-to-nearest, ties to even; overflow gives inf. */
uint16_t oracle_double_to_half_rne(double x) {
    uint16_t s = signbit(x) ? 0x8000 : 0;
    if (isnan(x)) return (uint16_t)(s | 0x7e00);
    double a = fabs(x);
    if (a == 0.0) return s;
    if (isinf(a)) return (uint16_t)(s | 0x7c00);
    int ex;
    frexp(a, &ex);   /* a = m * 2^ex, m in [0.5, 1) */
    int e = ex - 1;  /* a in [2^e, 2^(e+1)) */
    if (e < -14) {
        /* subnormal range: quantum 2^-24; r == 1024 is the smallest normal,
         * whose encoding 0x0400 is exactly r. */
        double r = rne_integer(ldexp(a, 24));
        return (uint16_t)(s | (uint16_t)r);
    }
    double r = rne_integer(ldexp(a, 10 - e)); /* in [1024, 2048] */
    if (r == 2048.0) { r = 1024.0; e += 1; }
    if (e > 15) return (uint16_t)(s | 0x7c00);
    return (uint16_t)(s | (uint16_t)((e + 15) << 10) | (uint16_t)((int)r - 1024));
}

/* ---------------------------------------------------------------------------
 * bfloat16 <-> double.  bfloat16 is the upper half of an IEEE binary32: 1 sign
 * bit, 8 exponent bits (bias 127), 7 fraction bits.  Widening puts the 16 bits
 * on top of a binary32 with zero low bits, which is exact.
 * ------------------------------------------------------------------------- */
double oracle_bf16_to_double(uint16_t b) {
    const uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* double -> bfloat16, round to nearest, ties to even; overflow gives inf. */
uint16_t oracle_double_to_bf16_rne(double x) {
    uint16_t s = signbit(x) ? 0x8000 : 0;
    if (isnan(x)) return (uint16_t)(s | 0x7fc0);
    double a = fabs(x);
    if (a == 0.0) return s;
    if (isinf(a)) return (uint16_t)(s | 0x7f80);
    int ex;
    frexp(a, &ex);
    int e = ex - 1; /* a in [2^e, 2^(e+1)) */
    if (e < -126) {
        /* subnormal range: quantum 2^-133; r == 128 is the smallest normal */
        double r = rne_integer(ldexp(a, 133));
        return (uint16_t)(s | (uint16_t)r);
    }
    double r = rne_integer(ldexp(a, 7 - e)); /* in [128, 256] */
    if (r == 256.0) { r = 128.0; e += 1; }
    if (e > 127) return (uint16_t)(s | 0x7f80);
    return (uint16_t)(s | (uint16_t)((e + 127) << 7) | (uint16_t)((int)r - 128));
}

static inline double load_elem(const void* p, int dtype, int64_t idx) {
    if (dtype == ORACLE_F16) return oracle_half_to_double(((const uint16_t*)p)[idx]);
    if (dtype == ORACLE_BF16) return oracle_bf16_to_double(((const uint16_t*)p)[idx]);
    return (double)((const float*)p)[idx];
}

/* op(A)(i,k) and op(B)(k,j) as in the variant table: a transposed operand is
 * stored with the other index contiguous. */
static inline double opA(const void* A, int dtype, int transA, int64_t lda, int64_t i, int64_t k) {
    return transA ? load_elem(A, dtype, k * lda + i) : load_elem(A, dtype, i * lda + k);
}
static inline double opB(const void* B, int dtype, int transB, int64_t ldb, int64_t k, int64_t j) {
    return transB ? load_elem(B, dtype, j * ldb + k) : load_elem(B, dtype, k * ldb + j);
}

int oracle_version(void) { return 1; }

/* ------------------------------------------------------------------------- */
/* Full product.                                                              */
/* ------------------------------------------------------------------------- */
typedef struct {
    int64_t M, N, K;
    double alpha, beta;
    const double* Ad; /* op(A) widened, [M][K] */
    const double* Bd; /* op(B) widened, [K][N] */
    const void* Cin;
    int64_t ldc;
    int dtype;
    double* ref;
    double* mag;
    int tid, nthreads;
    int err;
} full_job_t;

static void* full_worker(void* arg) {
    full_job_t* j = (full_job_t*)arg;
    int64_t N = j->N, K = j->K;
    double* acc = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    double* macc = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    if (!acc || !macc) { j->err = 1; free(acc); free(macc); return NULL; }
    /* rows are dealt round-robin to the threads */
    for (int64_t i = j->tid; i < j->M; i += j->nthreads) {
        for (int64_t c = 0; c < N; ++c) { acc[c] = 0.0; macc[c] = 0.0; }
        const double* arow = j->Ad + i * K;
        for (int64_t k = 0; k < K; ++k) {          /* strict increasing k */
            const double a = arow[k];
            const double* brow = j->Bd + k * N;
            for (int64_t c = 0; c < N; ++c) {      /* every output of row i */
                const double p = a * brow[c];      /* exact */
                acc[c] += p;
                macc[c] += fabs(p);
            }
        }
        for (int64_t c = 0; c < N; ++c) {
            double r = j->alpha * acc[c];
            double m = fabs(j->alpha) * macc[c];
            if (j->beta != 0.0) {
                double cin = load_elem(j->Cin, j->dtype, i * j->ldc + c);
                r += j->beta * cin;
                m += fabs(j->beta * cin);
            }
            j->ref[i * N + c] = r;
            j->mag[i * N + c] = m;
        }
    }
    free(acc);
    free(macc);
    return NULL;
}

/*
 * ref, mag: caller-owned arrays of M*N doubles, row-major with row length N.
 * Cin may be NULL when beta == 0.  nthreads <= 0 means 1.
 * Returns 0 on success, 1 on bad arguments, 2 on allocation failure.
 */
int oracle_gemm(int transA, int transB, int64_t M, int64_t N, int64_t K, int dtype,
                double alpha, double beta, const void* A, int64_t lda, const void* B,
                int64_t ldb, const void* Cin, int64_t ldc, double* ref, double* mag,
                int nthreads) {
    if (M < 0 || N < 0 || K < 0) return 1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_F16 && dtype != ORACLE_BF16) return 1;
    if (M == 0 || N == 0) return 0;
    if (!ref || !mag) return 1;
    if (K > 0 && (!A || !B)) return 1;
    if (beta != 0.0 && !Cin) return 1;
    if (nthreads <= 0) nthreads = 1;
    if (nthreads > 256) nthreads = 256;

    /* op(A) and op(B) written out as plain double matrices (exact widening);
     * this changes no arithmetic, it only makes the k loop read rows. */
    double* Ad = (double*)malloc(sizeof(double) * (size_t)(M * (K > 0 ? K : 1)));
    double* Bd = (double*)malloc(sizeof(double) * (size_t)((K > 0 ? K : 1) * N));
    if (!Ad || !Bd) { free(Ad); free(Bd); return 2; }
    for (int64_t i = 0; i < M; ++i)
        for (int64_t k = 0; k < K; ++k) Ad[i * K + k] = opA(A, dtype, transA, lda, i, k);
    for (int64_t k = 0; k < K; ++k)
        for (int64_t c = 0; c < N; ++c) Bd[k * N + c] = opB(B, dtype, transB, ldb, k, c);

    full_job_t* jobs = (full_job_t*)calloc((size_t)nthreads, sizeof(full_job_t));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(Ad); free(Bd); free(jobs); free(th); return 2; }
    int started = 0, rc = 0;
    for (int t = 0; t < nthreads; ++t) {
        full_job_t jb = {M, N, K, alpha, beta, Ad, Bd, Cin, ldc, dtype, ref, mag, t, nthreads, 0};
        jobs[t] = jb;
    }
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, full_worker, &jobs[t]) != 0) break;
        started = t;
    }
    /* threads that failed to start: their rows are done here instead */
    for (int t = started + 1; t < nthreads; ++t) full_worker(&jobs[t]);
    full_worker(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    for (int t = 0; t < nthreads; ++t) rc |= jobs[t].err;
    free(Ad);
    free(Bd);
    free(jobs);
    free(th);
    return rc ? 2 : 0;
}

/* ------------------------------------------------------------------------- */
/* Fused epilogue: bias and activation.                                       */
/* ------------------------------------------------------------------------- */
/*
 * "From a C loop to a GPU kernel", section "Fusion": after C = A @ B the fused
 * kernel adds a learned per-output offset (bias) and applies gelu before the
 * single write.  Per output column j (the output feature):
 *     out[i][j] = act(x[i][j] + bias[j])
 * with act one of
 *     ORACLE_ACT_NONE  identity
 *     ORACLE_ACT_RELU  max(v, 0)
 *     ORACLE_ACT_GELU  v * Phi(v) = v/2 * (1 + erf(v / sqrt(2))), the exact
 *                      form (the page names gelu without a formula; the
 *                      defining expression is taken, not a tanh fit).
 * x is rows x cols, row pitch ldx, rewritten in place; bias (cols doubles) may
 * be NULL for no bias.  erf is the C library's.
 */
enum { ORACLE_ACT_NONE = 0, ORACLE_ACT_RELU = 1, ORACLE_ACT_GELU = 2 };

double oracle_gelu(double v) { return 0.5 * v * (1.0 + erf(v / sqrt(2.0))); }

int oracle_bias_act(double* x, int64_t rows, int64_t cols, int64_t ldx, const double* bias,
                    int act) {
    if (rows < 0 || cols < 0 || (rows > 0 && !x) || ldx < cols) return 1;
    if (act != ORACLE_ACT_NONE && act != ORACLE_ACT_RELU && act != ORACLE_ACT_GELU) return 1;
    for (int64_t i = 0; i < rows; ++i)
        for (int64_t j = 0; j < cols; ++j) {
            double v = x[i * ldx + j] + (bias ? bias[j] : 0.0);
            if (act == ORACLE_ACT_RELU) v = v > 0.0 ? v : 0.0;
            else if (act == ORACLE_ACT_GELU) v = oracle_gelu(v);
            x[i * ldx + j] = v;
        }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Selected elements only (for products too large to form in full).          */
/* ------------------------------------------------------------------------- */
typedef struct {
    int transA, transB, dtype;
    int64_t K;
    double alpha, beta;
    const void *A, *B, *Cin;
    int64_t lda, ldb, ldc;
    const int64_t *rows, *cols;
    int64_t npts;
    double *ref, *mag;
    int tid, nthreads;
} pts_job_t;

static void* pts_worker(void* arg) {
    pts_job_t* j = (pts_job_t*)arg;
    for (int64_t p = j->tid; p < j->npts; p += j->nthreads) {
        int64_t i = j->rows[p], c = j->cols[p];
        double acc = 0.0, macc = 0.0;
        for (int64_t k = 0; k < j->K; ++k) { /* strict increasing k */
            const double prod = opA(j->A, j->dtype, j->transA, j->lda, i, k) *
                                opB(j->B, j->dtype, j->transB, j->ldb, k, c);
            acc += prod;
            macc += fabs(prod);
        }
        double r = j->alpha * acc;
        double m = fabs(j->alpha) * macc;
        if (j->beta != 0.0) {
            double cin = load_elem(j->Cin, j->dtype, i * j->ldc + c);
            r += j->beta * cin;
            m += fabs(j->beta * cin);
        }
        j->ref[p] = r;
        j->mag[p] = m;
    }
    return NULL;
}

/* Same definition as oracle_gemm, evaluated only at (rows[p], cols[p]).
 * ref, mag: npts doubles each.  Indices must lie inside the M x N output. */
int oracle_gemm_points(int transA, int transB, int64_t M, int64_t N, int64_t K, int dtype,
                       double alpha, double beta, const void* A, int64_t lda, const void* B,
                       int64_t ldb, const void* Cin, int64_t ldc, const int64_t* rows,
                       const int64_t* cols, int64_t npts, double* ref, double* mag,
                       int nthreads) {
    if (M < 0 || N < 0 || K < 0 || npts < 0) return 1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_F16 && dtype != ORACLE_BF16) return 1;
    if (npts == 0) return 0;
    if (!rows || !cols || !ref || !mag) return 1;
    if (K > 0 && (!A || !B)) return 1;
    if (beta != 0.0 && !Cin) return 1;
    for (int64_t p = 0; p < npts; ++p)
        if (rows[p] < 0 || rows[p] >= M || cols[p] < 0 || cols[p] >= N) return 1;
    if (nthreads <= 0) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pts_job_t* jobs = (pts_job_t*)calloc((size_t)nthreads, sizeof(pts_job_t));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return 2; }
    for (int t = 0; t < nthreads; ++t) {
        pts_job_t jb = {transA, transB, dtype, K, alpha, beta, A, B, Cin, lda, ldb, ldc,
                        rows, cols, npts, ref, mag, t, nthreads};
        jobs[t] = jb;
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, pts_worker, &jobs[t]) != 0) break;
        started = t;
    }
    for (int t = started + 1; t < nthreads; ++t) pts_worker(&jobs[t]);
    pts_worker(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    free(jobs);
    free(th);
    return 0;
}

/* Elementwise conversions over arrays (used by the checker). */
void oracle_half_array_to_double(const uint16_t* h, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_half_to_double(h[i]);
}
void oracle_double_array_to_half_rne(const double* x, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_double_to_half_rne(x[i]);
}
void oracle_bf16_array_to_double(const uint16_t* h, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_double(h[i]);
}
void oracle_double_array_to_bf16_rne(const double* x, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_double_to_bf16_rne(x[i]);
}
