/*
 * CPU oracle for the FP32 GEMM C = A*B.  TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference
 * arm may load this library.  The product path (the CUDA library under
 * software_pipelined_gb300/) never calls it, shares no header, helper or
 * constant with it, and fails loudly when its own extension is missing.
 *
 * What it computes is the plain definition of the matrix product that the
 * pages' tiled, double-buffered K-loop evaluates ("Double Buffering" technique
 * page and "Case Study: The Double-Buffered GEMM": each output tile is the sum
 * over K tiles of the products of A's row panel and B's column panel), and the
 * full-output check is against an FP64 oracle ("Dependence-aware group
 * synchronization on M1 Max", section "Controlled implementation comparison":
 * every run checks the complete output against an FP64 oracle):
 *
 *     C[i][j] = sum_{k=0}^{K-1} (double)A[i*lda+k] * (double)B[k*ldb+j]
 *     S[i][j] = sum_{k=0}^{K-1} |A[i*lda+k]| * |B[k*ldb+j]|
 *
 * Both sums run in FP64 in ascending k.  A product of two FP32 values is exact
 * in FP64 (24+24 significant bits < 53), so the only rounding is that of the
 * FP64 additions.  S is the scale of the accuracy bound
 * |C_gpu - C| <= 2*K*2^-24*S.
 *
 * Loop order is i-k-j: row i's FP64 accumulators are updated for every j at
 * each k, so every element is still summed in ascending k; the j loop has no
 * cross-iteration dependence.  Rows are independent and are split over OpenMP
 * threads.  Build with -O2 -ffp-contract=off and without -ffast-math, so no
 * reassociation takes place.
 *
 * Row-major, leading dimensions in elements: A is M x K (lda >= K), B is K x N
 * (ldb >= N), C and S are M x N (ldc >= N).  Padding columns are never read.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_get_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Full product: C (and, when S is not NULL, S) for all M x N outputs. */
void oracle_gemm_f64(int64_t M, int64_t N, int64_t K,
                     const float* A, int64_t lda,
                     const float* B, int64_t ldb,
                     double* C, double* S, int64_t ldc)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i) {
        double* c = C + i * ldc;
        double* s = S ? S + i * ldc : NULL;
        for (int64_t j = 0; j < N; ++j) c[j] = 0.0;
        if (s)
            for (int64_t j = 0; j < N; ++j) s[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double a = (double)A[i * lda + k];
            const float* b = B + k * ldb;
            if (s) {
                for (int64_t j = 0; j < N; ++j) {
                    const double p = a * (double)b[j];
                    c[j] += p;
                    s[j] += fabs(p);
                }
            } else {
                for (int64_t j = 0; j < N; ++j) c[j] += a * (double)b[j];
            }
        }
    }
}

/* Selected outputs, one dot product each: c[t] = C[rows[t]][cols[t]] and
 * s[t] = S[rows[t]][cols[t]], summed in ascending k exactly as above.  Used for
 * sampled checks of products too large to form whole on the host. */
void oracle_gemm_f64_entries(int64_t n, const int64_t* rows, const int64_t* cols,
                             int64_t K,
                             const float* A, int64_t lda,
                             const float* B, int64_t ldb,
                             double* c, double* s)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        const float* a = A + rows[t] * lda;
        const float* b = B + cols[t];
        double acc = 0.0, mag = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double p = (double)a[k] * (double)b[k * ldb];
            acc += p;
            mag += fabs(p);
        }
        c[t] = acc;
        if (s) s[t] = mag;
    }
}
