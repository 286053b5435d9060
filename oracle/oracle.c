/*
 * CPU oracle for the mixed-precision GEMM  C = alpha * A * B + beta * C.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the correctness reference that the
 * CUDA library is checked against. Only the test suite, the smoke check and
 * the benchmark's CPU-baseline leg may load it. The library never calls it
 * and shares no code with it.
 *
 * What it computes (the plain definition, element by element, in double):
 *
 *   out[i][j] = alpha * sum_{k=0}^{K-1} dec(A[i*lda + k]) * dec(B(k, j))
 *             + beta  * C[i*ldc + j]                      (term dropped if beta == 0)
 *
 *   S[i][j]   = sum_{k=0}^{K-1} |dec(A[i*lda + k]) * dec(B(k, j))|
 *
 * with B(k, j) = B[k*ldb + j] for row-major B (K x N, the default) or
 * B[j*ldb + k] for column-major B ("Day 80, Capstone 4", "Independent gate":
 * the gate's solve() takes B column-major).
 *
 * Sources:
 *  - "Day 80, Capstone 4: a tensor-core GEMM", sections "Capability" and
 *    "Minimal model": FP16 inputs A and B, FP32 accumulation and FP32 C,
 *    because FP16 has no finite value above 65,504.
 *  - Same page, "Compare like with like": every element is checked against a
 *    double-precision CPU result; "Independent gate": the harness reference
 *    is float64 with Kahan summation (the `kahan` flag below).
 *  - "Day 72: Tensor cores with WMMA", "Why this program calls cuBLAS twice":
 *    the double CPU reference the WMMA kernels are gated on.
 *  - alpha/beta follow the BLAS GEMM convention that the pages' matched
 *    cublasGemmEx baseline uses: beta == 0 means C is not read (so a NaN
 *    poisoned C does not propagate), alpha == 0 or K == 0 means A and B are
 *    not read.
 *
 * dec() is this file's own IEEE 754 binary16 decoder (sign, 5-bit exponent
 * with bias 15, 10-bit fraction; subnormals, infinities and NaN included).
 *
 * Each product of two binary16 values has at most 22 significant bits, so it
 * is exact in double; the double sum has error at most about K * 2^-53 * S.
 *
 * The element loops follow the definition directly. The only liberty taken
 * is memory order: a column of B is decoded once into a contiguous buffer
 * (oracle_gemm) and rows are split across threads. Every element is still
 * summed over k = 0 .. K-1 in order, so the result is the same for any
 * thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------------ */
/* binary16 -> double                                                        */
/* ------------------------------------------------------------------------ */

double oracle_half_to_double(uint16_t h) {
    const int sign = (h >> 15) & 1;
    const int exponent = (h >> 10) & 0x1f;
    const int fraction = h & 0x3ff;
    double v;
    if (exponent == 0) {
        /* zero or subnormal: fraction * 2^-24 */
        v = ldexp((double)fraction, -24);
    } else if (exponent == 31) {
        v = fraction ? NAN : INFINITY;
    } else {
        /* normal: (1 + fraction/1024) * 2^(exponent-15) */
        v = ldexp((double)(1024 + fraction), exponent - 25);
    }
    return sign ? -v : v;
}

static double g_table[65536];
static pthread_once_t g_table_once = PTHREAD_ONCE_INIT;

static void build_table(void) {
    for (uint32_t h = 0; h < 65536u; ++h) g_table[h] = oracle_half_to_double((uint16_t)h);
}

static const double* table(void) {
    pthread_once(&g_table_once, build_table);
    return g_table;
}

/* ------------------------------------------------------------------------ */
/* one element                                                               */
/* ------------------------------------------------------------------------ */

typedef struct {
    int64_t M, N, K;
    double alpha, beta;
    const uint16_t* A; int64_t lda;
    const uint16_t* B; int64_t ldb;
    const float* C;    int64_t ldc;
    int kahan;
    int64_t b_sk, b_sj;   /* B(k, j) = B[k*b_sk + j*b_sj] */
} problem_t;

/* sum_k dec(A[i,k]) * dec(B[k,j]) with B's column j given as a strided
 * pointer (bcol[k*bstride]) or an already-decoded contiguous column. */
static void dot_row(const problem_t* p, const double* dec, int64_t i,
                    const uint16_t* bcol, int64_t bstride, const double* bdec,
                    double* sum_out, double* abs_out) {
    const uint16_t* arow = p->A + i * p->lda;
    double sum = 0.0, comp = 0.0, sabs = 0.0;
    for (int64_t k = 0; k < p->K; ++k) {
        const double a = dec[arow[k]];
        const double b = bdec ? bdec[k] : dec[bcol[k * bstride]];
        const double prod = a * b;
        if (p->kahan) {
            const double y = prod - comp;
            const double t = sum + y;
            comp = (t - sum) - y;
            sum = t;
        } else {
            sum += prod;
        }
        sabs += fabs(prod);
    }
    *sum_out = sum;
    *abs_out = sabs;
}

static double finish(const problem_t* p, int64_t i, int64_t j, double sum) {
    double v = (p->alpha == 0.0) ? 0.0 : p->alpha * sum;
    if (p->beta != 0.0) v += p->beta * (double)p->C[i * p->ldc + j];
    return v;
}

/* ------------------------------------------------------------------------ */
/* threading                                                                 */
/* ------------------------------------------------------------------------ */

static int resolve_threads(int nthreads) {
    if (nthreads > 0) return nthreads;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

typedef struct {
    const problem_t* p;
    int64_t begin, end;          /* range of columns (full) or elements (sampled) */
    const int64_t* I; const int64_t* J;
    double* out; double* S;      /* full: M x N row-major; sampled: n entries */
    int status;
} job_t;

static void* run_columns(void* arg) {
    job_t* job = (job_t*)arg;
    const problem_t* p = job->p;
    const double* dec = table();
    double* bdec = (double*)malloc((size_t)(p->K > 0 ? p->K : 1) * sizeof(double));
    if (!bdec) { job->status = -1; return NULL; }
    for (int64_t j = job->begin; j < job->end; ++j) {
        for (int64_t k = 0; k < p->K; ++k) bdec[k] = dec[p->B[k * p->b_sk + j * p->b_sj]];
        for (int64_t i = 0; i < p->M; ++i) {
            double sum = 0.0, sabs = 0.0;
            if (p->alpha != 0.0) dot_row(p, dec, i, NULL, 0, bdec, &sum, &sabs);
            job->out[i * p->N + j] = finish(p, i, j, sum);
            if (job->S) job->S[i * p->N + j] = sabs;
        }
    }
    free(bdec);
    job->status = 0;
    return NULL;
}

static void* run_elements(void* arg) {
    job_t* job = (job_t*)arg;
    const problem_t* p = job->p;
    const double* dec = table();
    for (int64_t e = job->begin; e < job->end; ++e) {
        const int64_t i = job->I[e], j = job->J[e];
        double sum = 0.0, sabs = 0.0;
        if (p->alpha != 0.0) dot_row(p, dec, i, p->B + j * p->b_sj, p->b_sk, NULL, &sum, &sabs);
        job->out[e] = finish(p, i, j, sum);
        if (job->S) job->S[e] = sabs;
    }
    job->status = 0;
    return NULL;
}

static int run_parallel(void* (*fn)(void*), const problem_t* p, int64_t count,
                        const int64_t* I, const int64_t* J, double* out, double* S,
                        int nthreads) {
    (void)table();
    int nt = resolve_threads(nthreads);
    if (count < nt) nt = (int)(count > 0 ? count : 1);
    job_t* jobs = (job_t*)calloc((size_t)nt, sizeof(job_t));
    pthread_t* tids = (pthread_t*)calloc((size_t)nt, sizeof(pthread_t));
    if (!jobs || !tids) { free(jobs); free(tids); return -1; }
    int status = 0;
    for (int t = 0; t < nt; ++t) {
        jobs[t].p = p;
        jobs[t].begin = count * t / nt;
        jobs[t].end = count * (t + 1) / nt;
        jobs[t].I = I; jobs[t].J = J; jobs[t].out = out; jobs[t].S = S;
        jobs[t].status = -1;
    }
    for (int t = 1; t < nt; ++t)
        if (pthread_create(&tids[t], NULL, fn, &jobs[t]) != 0) { tids[t] = 0; fn(&jobs[t]); }
    fn(&jobs[0]);
    for (int t = 1; t < nt; ++t)
        if (tids[t]) pthread_join(tids[t], NULL);
    for (int t = 0; t < nt; ++t) status |= jobs[t].status;
    free(jobs); free(tids);
    return status;
}

static int check(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                 const void* A, const void* B, const void* C, double alpha, double beta,
                 int b_col_major) {
    const int64_t b_min = b_col_major ? K : N;
    if (M < 0 || N < 0 || K < 0) return -2;
    if (lda < (K > 1 ? K : 1) || ldb < (b_min > 1 ? b_min : 1) || ldc < (N > 1 ? N : 1)) return -2;
    if (M > 0 && N > 0) {
        if (alpha != 0.0 && K > 0 && (!A || !B)) return -2;
        if (beta != 0.0 && !C) return -2;
    }
    return 0;
}

static problem_t make_problem(int64_t M, int64_t N, int64_t K, double alpha, const uint16_t* A,
                              int64_t lda, const uint16_t* B, int64_t ldb, double beta,
                              const float* C, int64_t ldc, int kahan, int b_col_major) {
    problem_t p = {M, N, K, alpha, beta, A, lda, B, ldb, C, ldc, kahan,
                   b_col_major ? 1 : ldb, b_col_major ? ldb : 1};
    return p;
}

/* Every element: out and S are M x N, row-major with leading dimension N.
 * b_col_major selects B(k, j) = B[j*ldb + k] (ldb >= K) instead of
 * B[k*ldb + j] (ldb >= N). Returns 0 on success, -2 on invalid arguments,
 * -1 on allocation failure. */
int oracle_gemm_ex(int64_t M, int64_t N, int64_t K, double alpha,
                   const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
                   double beta, const float* C, int64_t ldc,
                   double* out, double* S, int kahan, int nthreads, int b_col_major) {
    int rc = check(M, N, K, lda, ldb, ldc, A, B, C, alpha, beta, b_col_major);
    if (rc) return rc;
    if (M == 0 || N == 0) return 0;
    problem_t p = make_problem(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, kahan, b_col_major);
    return run_parallel(run_columns, &p, N, NULL, NULL, out, S, nthreads);
}

/* The listed elements (I[e], J[e]) only: out[e] and S[e]. */
int oracle_elements_ex(int64_t M, int64_t N, int64_t K, double alpha,
                       const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
                       double beta, const float* C, int64_t ldc,
                       int64_t count, const int64_t* I, const int64_t* J,
                       double* out, double* S, int kahan, int nthreads, int b_col_major) {
    int rc = check(M, N, K, lda, ldb, ldc, A, B, C, alpha, beta, b_col_major);
    if (rc) return rc;
    for (int64_t e = 0; e < count; ++e)
        if (I[e] < 0 || I[e] >= M || J[e] < 0 || J[e] >= N) return -2;
    if (count == 0) return 0;
    problem_t p = make_problem(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, kahan, b_col_major);
    return run_parallel(run_elements, &p, count, I, J, out, S, nthreads);
}

/* Row-major B. */
int oracle_gemm(int64_t M, int64_t N, int64_t K, double alpha,
                const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
                double beta, const float* C, int64_t ldc,
                double* out, double* S, int kahan, int nthreads) {
    return oracle_gemm_ex(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, out, S, kahan, nthreads, 0);
}

int oracle_elements(int64_t M, int64_t N, int64_t K, double alpha,
                    const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
                    double beta, const float* C, int64_t ldc,
                    int64_t count, const int64_t* I, const int64_t* J,
                    double* out, double* S, int kahan, int nthreads) {
    return oracle_elements_ex(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, count, I, J, out, S,
                              kahan, nthreads, 0);
}
