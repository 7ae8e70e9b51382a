/*
 * gemm_oracle.c -- the CPU oracle for the pipelined GEMM (TEST INFRASTRUCTURE).
 *
 * This file is test infrastructure, not product code.  Only tests/,
 * __graft_entry__.smoke() and bench.py's cpu_baseline / reference legs load it.
 * It shares no code, header, table or helper with the CUDA path under
 * stage_software_pipelining_gb300/csrc, and it includes nothing from there.
 *
 * What it computes (the plain definition, evaluated in fp64):
 *
 *     C[i][j] = alpha * sum_k A[i][k] * B[k][j]  +  beta * C0[i][j]
 *     Abs[i][j] =        sum_k |A[i][k]| * |B[k][j]|
 *
 * Sources for the definition:
 *  - "CUTLASS-CuTe 初步(6)" (hxf0223.github.io), section 2 "Thread Block Tile":
 *    the problem is stated as C += A * B, accumulated over K by summing the
 *    products of the K tiles.  The page's own GEMM formula did not survive
 *    extraction, so the BLAS form alpha*A*B + beta*C is taken (the plain
 *    reading of the problem the GEMM library entry point states).
 *  - "Software Pipelining and Double Buffering" (andriisonsiadlo.github.io),
 *    section "Double buffering with shared memory": the kernel accumulates
 *    acc += As[row][k] * Bs[k][col] over all k and stores C = acc.
 *
 * Readings where the pages are silent:
 *  - beta == 0: C0 is not read at all (BLAS convention), so NaN/Inf in C0 do
 *    not reach the result.
 *  - alpha is applied to the full K sum, then beta*C0 is added.
 *  - Inputs are decoded exactly to fp64 from their storage format (IEEE
 *    binary32, IEEE binary16, or bfloat16 = the top half of a binary32); every
 *    such value is exactly representable in a double.
 *  - Layout: A is row-major M x K with leading dimension lda; B is K x N,
 *    row-major (element (k,j) at B[k*ldb + j]) or column-major (element (k,j)
 *    at B[j*ldb + k]); C0 is row-major M x N with leading dimension ldc0.
 *
 * The loop is the plain i-k-j triple loop.  Rows of C are independent, so an
 * OpenMP loop over rows changes nothing about the arithmetic of any entry.
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC (no FMA contraction,
 * so x86 and Arm hosts give the same bits).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Storage formats the oracle decodes. */
#define ORACLE_T_F32 0
#define ORACLE_T_F16 1
#define ORACLE_T_BF16 2

/* Status codes. */
#define ORACLE_OK 0
#define ORACLE_EARG -1
#define ORACLE_ENOMEM -2

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * Subnormals (exponent field 0) are fraction * 2^-24. */
double oracle_decode_f16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);
    } else if (e == 31) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + f), e - 25);
    }
    return sign ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double oracle_decode_bf16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xff;
    int f = h & 0x7f;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -133);
    } else if (e == 255) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(128 + f), e - 134);
    }
    return sign ? -v : v;
}

/* IEEE 754 binary32: 1 sign bit, 8 exponent bits (bias 127), 23 fraction bits. */
double oracle_decode_f32(uint32_t w) {
    int sign = (w >> 31) & 1;
    int e = (w >> 23) & 0xff;
    int32_t f = (int32_t)(w & 0x7fffff);
    double v;
    if (e == 0) {
        v = ldexp((double)f, -149);
    } else if (e == 255) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)((1 << 23) + f), e - 150);
    }
    return sign ? -v : v;
}

/* Element idx (in elements) of an array stored in format t. */
static double load(const void* p, int t, int64_t idx) {
    if (t == ORACLE_T_F32) return oracle_decode_f32(((const uint32_t*)p)[idx]);
    if (t == ORACLE_T_F16) return oracle_decode_f16(((const uint16_t*)p)[idx]);
    return oracle_decode_bf16(((const uint16_t*)p)[idx]);
}

static int64_t b_index(int64_t k, int64_t j, int64_t ldb, int b_col_major) {
    return b_col_major ? j * ldb + k : k * ldb + j;
}

static int check_args(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, int a_type,
                      const void* B, int64_t ldb, int b_type, int b_col_major, const void* C0,
                      int64_t ldc0, int c0_type, double beta) {
    if (M < 0 || N < 0 || K < 0) return ORACLE_EARG;
    if (a_type < 0 || a_type > 2 || b_type < 0 || b_type > 2 || c0_type < 0 || c0_type > 2)
        return ORACLE_EARG;
    if (M > 0 && K > 0 && (A == NULL || lda < K)) return ORACLE_EARG;
    if (N > 0 && K > 0 && (B == NULL || ldb < (b_col_major ? K : N))) return ORACLE_EARG;
    if (beta != 0.0 && M > 0 && N > 0 && (C0 == NULL || ldc0 < N)) return ORACLE_EARG;
    return ORACLE_OK;
}

/*
 * Rows [row_begin, row_end) of C = alpha*A*B + beta*C0 (and Abs if non-NULL).
 * The output arrays hold only those rows: row i of the result goes to
 * C[(i - row_begin)*ldc + j] and Abs[(i - row_begin)*ldabs + j].
 * nthreads <= 0 means "OpenMP default".
 */
int oracle_gemm_rows(int64_t M, int64_t N, int64_t K,
                     const void* A, int64_t lda, int a_type,
                     const void* B, int64_t ldb, int b_type, int b_col_major,
                     const void* C0, int64_t ldc0, int c0_type,
                     double alpha, double beta,
                     double* C, int64_t ldc, double* Abs, int64_t ldabs,
                     int64_t row_begin, int64_t row_end, int nthreads) {
    int st = check_args(M, N, K, A, lda, a_type, B, ldb, b_type, b_col_major, C0, ldc0, c0_type,
                        beta);
    if (st != ORACLE_OK) return st;
    if (row_begin < 0 || row_end > M || row_begin > row_end) return ORACLE_EARG;
    if (N > 0 && row_end > row_begin && (C == NULL || ldc < N)) return ORACLE_EARG;
    if (Abs != NULL && ldabs < N) return ORACLE_EARG;
    if (N == 0 || row_end == row_begin) return ORACLE_OK;

    int nt = 1;
#ifdef _OPENMP
    nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#endif
    /* One pair of row accumulators per thread. */
    double* acc_all = (double*)malloc((size_t)nt * (size_t)N * sizeof(double));
    double* aacc_all = (double*)malloc((size_t)nt * (size_t)N * sizeof(double));
    int failed = (acc_all == NULL || aacc_all == NULL);
    if (!failed) {
#ifdef _OPENMP
#pragma omp parallel for num_threads(nt) schedule(dynamic, 1)
#endif
        for (int64_t i = row_begin; i < row_end; ++i) {
            int tid = 0;
#ifdef _OPENMP
            tid = omp_get_thread_num();
#endif
            double* acc = acc_all + (size_t)tid * (size_t)N;
            double* aacc = aacc_all + (size_t)tid * (size_t)N;
            for (int64_t j = 0; j < N; ++j) {
                acc[j] = 0.0;
                aacc[j] = 0.0;
            }
            /* acc[j] = sum over k of A[i][k] * B[k][j] */
            for (int64_t k = 0; k < K; ++k) {
                double a = load(A, a_type, i * lda + k);
                for (int64_t j = 0; j < N; ++j) {
                    double b = load(B, b_type, b_index(k, j, ldb, b_col_major));
                    acc[j] += a * b;
                    aacc[j] += fabs(a) * fabs(b);
                }
            }
            for (int64_t j = 0; j < N; ++j) {
                double out = alpha * acc[j];
                if (beta != 0.0) out += beta * load(C0, c0_type, i * ldc0 + j);
                C[(i - row_begin) * ldc + j] = out;
                if (Abs != NULL) Abs[(i - row_begin) * ldabs + j] = aacc[j];
            }
        }
    }
    free(acc_all);
    free(aacc_all);
    return failed ? ORACLE_ENOMEM : ORACLE_OK;
}

/* The whole of C (and Abs): rows [0, M). */
int oracle_gemm(int64_t M, int64_t N, int64_t K,
                const void* A, int64_t lda, int a_type,
                const void* B, int64_t ldb, int b_type, int b_col_major,
                const void* C0, int64_t ldc0, int c0_type,
                double alpha, double beta,
                double* C, int64_t ldc, double* Abs, int64_t ldabs, int nthreads) {
    return oracle_gemm_rows(M, N, K, A, lda, a_type, B, ldb, b_type, b_col_major, C0, ldc0,
                            c0_type, alpha, beta, C, ldc, Abs, ldabs, 0, M, nthreads);
}

/*
 * Selected entries only: out[t] = C[rows[t]][cols[t]], abs_out[t] = Abs[...]
 * (abs_out may be NULL).  Each entry is the same sum over k as above, taken
 * in increasing k.  Used where the full product is too large for the CPU.
 */
int oracle_gemm_entries(int64_t M, int64_t N, int64_t K,
                        const void* A, int64_t lda, int a_type,
                        const void* B, int64_t ldb, int b_type, int b_col_major,
                        const void* C0, int64_t ldc0, int c0_type,
                        double alpha, double beta,
                        const int64_t* rows, const int64_t* cols, int64_t count,
                        double* out, double* abs_out, int nthreads) {
    int st = check_args(M, N, K, A, lda, a_type, B, ldb, b_type, b_col_major, C0, ldc0, c0_type,
                        beta);
    if (st != ORACLE_OK) return st;
    if (count < 0 || (count > 0 && (rows == NULL || cols == NULL || out == NULL)))
        return ORACLE_EARG;
    for (int64_t t = 0; t < count; ++t)
        if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N) return ORACLE_EARG;
#ifdef _OPENMP
    int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#pragma omp parallel for num_threads(nt) schedule(dynamic, 16)
#else
    (void)nthreads;
#endif
    for (int64_t t = 0; t < count; ++t) {
        int64_t i = rows[t], j = cols[t];
        double acc = 0.0, aacc = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double a = load(A, a_type, i * lda + k);
            double b = load(B, b_type, b_index(k, j, ldb, b_col_major));
            acc += a * b;
            aacc += fabs(a) * fabs(b);
        }
        double v = alpha * acc;
        if (beta != 0.0) v += beta * load(C0, c0_type, i * ldc0 + j);
        out[t] = v;
        if (abs_out != NULL) abs_out[t] = aacc;
    }
    return ORACLE_OK;
}

/*
 * The streaming-copy counter-example (the grid-stride copy of
 * "learn-kernels.com, Matrix multiplication", listing after "Overlap needs
 * stages"): its result is defined as byte i of dst = byte i of src.
 */
int oracle_copy_bytes(unsigned char* dst, const unsigned char* src, int64_t n) {
    if (n < 0 || (n > 0 && (dst == NULL || src == NULL))) return ORACLE_EARG;
    for (int64_t i = 0; i < n; ++i) dst[i] = src[i];
    return ORACLE_OK;
}

/* Threads an OpenMP region would use with nthreads <= 0 (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
