/*
 * FP64 oracle for C = A*B and y = A*x -- TEST INFRASTRUCTURE ONLY.
 * See oracle.c for the definitions followed and their sources.
 *
 * All pointers are host pointers to row-major FP64 arrays owned by the caller.
 * Return 0 on success, 1 on invalid arguments, 2 on allocation failure.
 */
#ifndef GTG_ORACLE_H
#define GTG_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* C = A*B (M x N), A is M x K (lda >= K), B is K x N (ldb >= N), ldc >= N.
 * If E is non-NULL it receives sum_k |A[i][k]*B[k][j]| (lde >= N).
 * nthreads <= 0 uses every online core. */
int oracle_gemm_f64(int64_t M, int64_t N, int64_t K,
                    const double *A, int64_t lda,
                    const double *B, int64_t ldb,
                    double *C, int64_t ldc,
                    double *E, int64_t lde,
                    int nthreads);

/* y = A*x, A is M x N (lda >= N), x has N entries, y has M.
 * If E is non-NULL it receives sum_j |A[i][j]*x[j]|. Single-threaded. */
int oracle_gemv_f64(int64_t M, int64_t N,
                    const double *A, int64_t lda,
                    const double *x,
                    double *y, double *E);

/* In place: C[i][j] = act(C[i][j] + bias), bias[j] when bias_per_column
 * (GEMM: one bias per output column), else bias[i] (GEMV: one per row);
 * bias may be NULL. act: 0 = identity, 1 = ReLU, max(v, 0). */
int oracle_bias_act_f64(int64_t M, int64_t N, double *C, int64_t ldc,
                        const double *bias, int bias_per_column, int act);

/* 2-D convolution of a batch of images (cross-correlation, as in
 * convolutional layers), zero padding:
 *   Y[n][oh][ow][co] = sum_{kh<KH} sum_{kw<KW} sum_{ci<C}
 *                      X[n][oh*sh - ph + kh*dh][ow*sw - pw + kw*dw][ci] * Wt[kh][kw][ci][co]
 * where terms whose input row or column falls outside the image are zero.
 * X is N x H x W x C (channels last), Wt is KH x KW x C x CO, Y is
 * N x OH x OW x CO with OH = (H + 2 ph - dh (KH - 1) - 1) / sh + 1 (floor),
 * OW likewise. E (optional, same shape as Y) receives the sum of |X * Wt|
 * over the same terms. Strides and dilations >= 1, paddings >= 0, and OH, OW
 * must be >= 1 (else 1 is returned). nthreads <= 0 uses every online core. */
int oracle_conv2d_f64(int64_t N, int64_t H, int64_t W, int64_t C, int64_t CO,
                      int64_t KH, int64_t KW, int64_t sh, int64_t sw, int64_t ph, int64_t pw,
                      int64_t dh, int64_t dw, const double *X, const double *Wt,
                      double *Y, double *E, int nthreads);

/* Number of threads nthreads <= 0 resolves to. */
int oracle_threads_default(void);

#ifdef __cplusplus
}
#endif

#endif
