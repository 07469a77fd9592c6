/*
 * CPU oracle for the dense product C = A.B.
 *
 * TEST INFRASTRUCTURE ONLY. The tests, the package's smoke check and the
 * bench's CPU-baseline leg are the only callers. The CUDA library never links,
 * loads or calls this file, and this file shares nothing with it.
 *
 * What it computes is the plain definition that every register-tiling page
 * starts from: one output element is the dot product of a row of A with a
 * column of B,
 *
 *     C[i][j] = sum_{k=0}^{K-1} A[i][k] * B[k][j]
 *
 * ("【infra之路】理解 Register Tiling", section "先看 Shared Memory 版本里，一个
 * 线程在做什么": the per-thread loop accumulating sA[row][k]*sB[k][col];
 * "寄存器Tiling跨架构解析", section 1.1: tiling at the global, shared and
 * register levels only re-groups this sum, it does not change it).
 *
 * Reading of the pages (they fix no precision): inputs are fp32 values (bf16
 * inputs are widened to fp32 exactly by the caller), widened again exactly to
 * fp64; each product is rounded to fp64 and added to an fp64 accumulator in
 * increasing k. This file must be compiled with -ffp-contract=off so that no
 * fused multiply-add changes that rounding. Beside C it returns
 *
 *     S[i][j] = sum_k |A[i][k] * B[k][j]|      (fp64, same order)
 *
 * the scale against which the GPU result's rounding error is bounded.
 *
 * No blocking, no reordering: the k loop is the innermost loop and runs in
 * increasing order. Rows (or sampled entries) are split across OpenMP threads,
 * which changes no sum.
 */
#include <math.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* One entry of C and of S, by the definition. */
static void dot_entry(int64_t N, int64_t K, const float *A, const float *B,
                      int64_t i, int64_t j, double *c_out, double *s_out)
{
    double c = 0.0;
    double s = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double p = (double)A[i * K + k] * (double)B[k * N + j];
        c += p;
        s += fabs(p);
    }
    *c_out = c;
    *s_out = s;
}

/* Every entry: C and S are M x N row-major fp64 arrays owned by the caller.
 * nthreads <= 0 uses the OpenMP default. */
void oracle_gemm(int64_t M, int64_t N, int64_t K, const float *A, const float *B,
                 double *C, double *S, int nthreads)
{
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(static) num_threads(nthreads)
#else
    (void)nthreads;
#endif
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j)
            dot_entry(N, K, A, B, i, j, &C[i * N + j], &S[i * N + j]);
}

/* Only the listed entries: C[t], S[t] receive entry (rows[t], cols[t]). */
void oracle_gemm_sampled(int64_t M, int64_t N, int64_t K, const float *A, const float *B,
                         int64_t count, const int64_t *rows, const int64_t *cols,
                         double *C, double *S, int nthreads)
{
    (void)M;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(static) num_threads(nthreads)
#else
    (void)nthreads;
#endif
    for (int64_t t = 0; t < count; ++t)
        dot_entry(N, K, A, B, rows[t], cols[t], &C[t], &S[t]);
}
