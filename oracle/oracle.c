/*
 * FP64 oracle for dense matrix products -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the bench's CPU-baseline leg load this
 * library. The product path (the CUDA kernels behind libgtg) never calls it,
 * and this file shares no code, header or helper with that path.
 *
 * What it computes is the plain definition of each product, nothing more:
 *
 *   GEMM  C[i][j] = sum_{k=0}^{K-1} A[i][k] * B[k][j]
 *         ("Matrix Operations", Vulkan ML-inference tutorial, section
 *          "Matrix-Matrix Multiplication (GEMM)"; restated as C_ij =
 *          sum_k A_ik B_kj in "GPU Matrix Multiplication: Tiling and Shared
 *          Memory", section 1, with K the inner dimension).
 *
 *   GEMV  y[i] = sum_{j=0}^{N-1} A[i][j] * x[j]
 *         ("Matrix Operations", section "Matrix-Vector Multiplication").
 *
 * Beside each result it also returns the error magnitude
 *   E[i][j] = sum_k |A[i][k] * B[k][j]|     (E[i] = sum_j |A[i][j] x[j]|)
 * which scales the per-element acceptance bounds used by the tests.
 *
 * A fully connected layer adds a bias to each output and applies an
 * activation ("Matrix Operations": fully connected layers are the
 * matrix-vector products, activation functions add the non-linearity):
 *
 *   out = act(product + bias),  act = identity or ReLU(v) = max(v, 0),
 *
 * with one bias per output column for the GEMM (C = X * W^T, a batch of
 * inputs in the rows of X) and one per output row for the GEMV (y = W x).
 *
 * A convolutional layer is reduced to a matrix product by the pages
 * ("GPU Matrix Multiplication: Tiling and Shared Memory", closing section:
 * convolutions map to matrix multiplication through im2col; "Matrix
 * Operations", introduction). The oracle does not take that route: it
 * computes the convolution from its definition, a sum over the kernel window
 * of input times weight with zero padding outside the image,
 *
 *   Y[n][oh][ow][co] = sum_{kh, kw, ci} X[n][oh*sh - ph + kh*dh]
 *                                       [ow*sw - pw + kw*dw][ci] * W[kh][kw][ci][co],
 *
 * taken kh, then kw, then ci ascending, one FP64 accumulator per output.
 *
 * Every matrix is row-major with an explicit leading dimension (the pages
 * index A[row*K + k], B[k*N + col], C[row*N + col]; a leading dimension
 * larger than the row length only skips padding).
 *
 * Arithmetic: IEEE binary64, each output's K products added in ascending k
 * order into its own accumulator (built with -ffp-contract=off so that no
 * multiply-add is fused). The loop nest is i, k, j: for a fixed output
 * element this is the same ascending-k sum as the textbook i, j, k nest; the
 * order only decides which element is worked on next. Rows are split across
 * POSIX threads; each output has a single owner, so results do not depend on
 * the thread count.
 */
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    int64_t row_begin, row_end;
    int64_t N, K;
    const double *A; int64_t lda;
    const double *B; int64_t ldb;
    double *C; int64_t ldc;
    double *E; int64_t lde;
} gemm_job;

/* Rows [row_begin, row_end) of C (and E). */
static void gemm_rows(const gemm_job *j)
{
    for (int64_t i = j->row_begin; i < j->row_end; ++i) {
        double *c = j->C + i * j->ldc;
        double *e = j->E ? j->E + i * j->lde : NULL;
        for (int64_t col = 0; col < j->N; ++col) c[col] = 0.0;
        if (e) for (int64_t col = 0; col < j->N; ++col) e[col] = 0.0;
        for (int64_t k = 0; k < j->K; ++k) {
            const double a = j->A[i * j->lda + k];
            const double *b = j->B + k * j->ldb;
            for (int64_t col = 0; col < j->N; ++col) {
                const double p = a * b[col];
                c[col] += p;
                if (e) e[col] += fabs(p);
            }
        }
    }
}

static void *gemm_thread(void *arg)
{
    gemm_rows((const gemm_job *)arg);
    return NULL;
}

static int resolve_threads(int nthreads, int64_t rows)
{
    if (nthreads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = n > 0 ? (int)n : 1;
    }
    if (nthreads > 1024) nthreads = 1024;
    if (rows < nthreads) nthreads = rows > 0 ? (int)rows : 1;
    return nthreads;
}

int oracle_threads_default(void)
{
    return resolve_threads(0, 1 << 30);
}

int oracle_gemm_f64(int64_t M, int64_t N, int64_t K,
                    const double *A, int64_t lda,
                    const double *B, int64_t ldb,
                    double *C, int64_t ldc,
                    double *E, int64_t lde,
                    int nthreads)
{
    if (M < 0 || N < 0 || K < 0) return 1;
    if (M == 0 || N == 0) return 0;
    if (!C || lda < K || ldb < N || ldc < N) return 1;
    if (K > 0 && (!A || !B)) return 1;
    if (E && lde < N) return 1;

    int nt = resolve_threads(nthreads, M);
    gemm_job *jobs = (gemm_job *)calloc((size_t)nt, sizeof(gemm_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nt, sizeof(pthread_t));
    if (!jobs || !tids) { free(jobs); free(tids); return 2; }

    for (int t = 0; t < nt; ++t) {
        gemm_job *j = &jobs[t];
        j->row_begin = M * t / nt;
        j->row_end = M * (t + 1) / nt;
        j->N = N; j->K = K;
        j->A = A; j->lda = lda; j->B = B; j->ldb = ldb;
        j->C = C; j->ldc = ldc; j->E = E; j->lde = lde;
    }
    int started = 0;
    for (int t = 1; t < nt; ++t) {
        if (pthread_create(&tids[t], NULL, gemm_thread, &jobs[t]) != 0) break;
        started = t;
    }
    /* threads that could not be started are run here, in order */
    gemm_rows(&jobs[0]);
    for (int t = started + 1; t < nt; ++t) gemm_rows(&jobs[t]);
    for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
    free(jobs);
    free(tids);
    return 0;
}

int oracle_gemv_f64(int64_t M, int64_t N,
                    const double *A, int64_t lda,
                    const double *x,
                    double *y, double *E)
{
    if (M < 0 || N < 0) return 1;
    if (M == 0) return 0;
    if (!y || lda < N) return 1;
    if (N > 0 && (!A || !x)) return 1;
    for (int64_t i = 0; i < M; ++i) {
        double sum = 0.0, mag = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            const double p = A[i * lda + j] * x[j];
            sum += p;
            mag += fabs(p);
        }
        y[i] = sum;
        if (E) E[i] = mag;
    }
    return 0;
}

int oracle_bias_act_f64(int64_t M, int64_t N, double *C, int64_t ldc,
                        const double *bias, int bias_per_column, int act)
{
    if (M < 0 || N < 0 || (M > 0 && N > 0 && (!C || ldc < N))) return 1;
    if (act != 0 && act != 1) return 1;
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double v = C[i * ldc + j];
            if (bias) v += bias_per_column ? bias[j] : bias[i];
            if (act == 1 && v < 0.0) v = 0.0;
            C[i * ldc + j] = v;
        }
    }
    return 0;
}

typedef struct {
    int64_t row_begin, row_end;   /* rows of the output = (n, oh) pairs */
    int64_t H, W, C, CO, KH, KW, sh, sw, ph, pw, dh, dw, OH, OW;
    const double *X, *Wt;
    double *Y, *E;
} conv_job;

static void conv_rows(const conv_job *j)
{
    for (int64_t r = j->row_begin; r < j->row_end; ++r) {
        const int64_t n = r / j->OH, oh = r % j->OH;
        for (int64_t ow = 0; ow < j->OW; ++ow) {
            double *y = j->Y + ((n * j->OH + oh) * j->OW + ow) * j->CO;
            double *e = j->E ? j->E + ((n * j->OH + oh) * j->OW + ow) * j->CO : NULL;
            for (int64_t co = 0; co < j->CO; ++co) {
                double sum = 0.0, mag = 0.0;
                for (int64_t kh = 0; kh < j->KH; ++kh) {
                    const int64_t ih = oh * j->sh - j->ph + kh * j->dh;
                    if (ih < 0 || ih >= j->H) continue;   /* zero padding */
                    for (int64_t kw = 0; kw < j->KW; ++kw) {
                        const int64_t iw = ow * j->sw - j->pw + kw * j->dw;
                        if (iw < 0 || iw >= j->W) continue;
                        const double *x = j->X + ((n * j->H + ih) * j->W + iw) * j->C;
                        const double *w = j->Wt + (kh * j->KW + kw) * j->C * j->CO + co;
                        for (int64_t ci = 0; ci < j->C; ++ci) {
                            const double p = x[ci] * w[ci * j->CO];
                            sum += p;
                            mag += fabs(p);
                        }
                    }
                }
                y[co] = sum;
                if (e) e[co] = mag;
            }
        }
    }
}

static void *conv_thread(void *arg)
{
    conv_rows((const conv_job *)arg);
    return NULL;
}

int oracle_conv2d_f64(int64_t N, int64_t H, int64_t W, int64_t C, int64_t CO,
                      int64_t KH, int64_t KW, int64_t sh, int64_t sw, int64_t ph, int64_t pw,
                      int64_t dh, int64_t dw, const double *X, const double *Wt,
                      double *Y, double *E, int nthreads)
{
    if (N < 0 || H < 1 || W < 1 || C < 0 || CO < 0 || KH < 1 || KW < 1) return 1;
    if (sh < 1 || sw < 1 || dh < 1 || dw < 1 || ph < 0 || pw < 0) return 1;
    const int64_t span_h = H + 2 * ph - dh * (KH - 1) - 1, span_w = W + 2 * pw - dw * (KW - 1) - 1;
    if (span_h < 0 || span_w < 0) return 1;
    const int64_t OH = span_h / sh + 1, OW = span_w / sw + 1;
    if (N == 0 || CO == 0) return 0;
    if (!Y || (C > 0 && (!X || !Wt))) return 1;
    const int64_t rows = N * OH;
    const int t = resolve_threads(nthreads, rows);
    conv_job *jobs = (conv_job *)calloc((size_t)t, sizeof(conv_job));
    pthread_t *tid = (pthread_t *)calloc((size_t)t, sizeof(pthread_t));
    if (!jobs || !tid) {
        free(jobs);
        free(tid);
        return 2;
    }
    for (int i = 0; i < t; ++i) {
        conv_job *j = &jobs[i];
        j->row_begin = rows * i / t;
        j->row_end = rows * (i + 1) / t;
        j->H = H; j->W = W; j->C = C; j->CO = CO; j->KH = KH; j->KW = KW;
        j->sh = sh; j->sw = sw; j->ph = ph; j->pw = pw; j->dh = dh; j->dw = dw;
        j->OH = OH; j->OW = OW;
        j->X = X; j->Wt = Wt; j->Y = Y; j->E = E;
    }
    int started = 0;
    for (int i = 1; i < t; ++i) {
        if (pthread_create(&tid[i], NULL, conv_thread, &jobs[i]) != 0) break;
        started = i;
    }
    for (int i = started + 1; i < t; ++i) conv_rows(&jobs[i]);   /* threads that did not start */
    conv_rows(&jobs[0]);
    for (int i = 1; i <= started; ++i) pthread_join(tid[i], NULL);
    free(jobs);
    free(tid);
    return 0;
}
