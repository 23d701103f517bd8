// The pages' own kernel designs, built for sm_103a so that their claims can
// be measured on this GPU against the library's kernels. They compute the
// same products (FP32, ascending k per output) and are checked against the
// same oracle; they are not on any product path.
//
//   gemv naive   one thread per output row, the whole vector read from global
//                memory by every thread ("Matrix Operations", Matrix-Vector
//                Multiplication, "Naive Implementation");
//   gemv shared  the vector staged in shared memory 256 entries at a time,
//                with a barrier on each side of every chunk, one thread per
//                row ("Optimized Implementation with Shared Memory" with
//                "Handling Large Vectors");
//   gemm naive   one thread per output, T x T threads per block, A and B read
//                from global memory for every multiply-add ("Naive
//                Implementation"; "CUDA Programming (6)" section 3.1);
//   gemm tiled   T x T tiles of A and B in shared memory, zero-padded at the
//                edges, two barriers per tile, one output per thread
//                ("Tiled Implementation with Shared Memory"; section 3.2).
#include "internal.h"

namespace gtg {
namespace {

constexpr int kVecThreads = 256;

__global__ void __launch_bounds__(kVecThreads) gemv_naive_kernel(int M, int N, const float *A, long long lda,
                                                                 const float *x, float *y) {
    const int row = blockIdx.x * kVecThreads + threadIdx.x;
    if (row >= M) return;   // no barrier in this kernel, so an early exit is safe
    const float *a = A + static_cast<long long>(row) * lda;
    float sum = 0.f;
    for (int j = 0; j < N; ++j) sum = fmaf(a[j], x[j], sum);
    y[row] = sum;
}

__global__ void __launch_bounds__(kVecThreads) gemv_shared_kernel(int M, int N, const float *A, long long lda,
                                                                  const float *x, float *y) {
    __shared__ float chunk[kVecThreads];
    const int row = blockIdx.x * kVecThreads + threadIdx.x;
    const bool active = row < M;   // every thread reaches every barrier
    const float *a = A + static_cast<long long>(active ? row : 0) * lda;
    float sum = 0.f;
    for (int base = 0; base < N; base += kVecThreads) {
        const int len = min(kVecThreads, N - base);
        if (static_cast<int>(threadIdx.x) < len) chunk[threadIdx.x] = x[base + threadIdx.x];
        __syncthreads();
        if (active)
            for (int j = 0; j < len; ++j) sum = fmaf(a[base + j], chunk[j], sum);
        __syncthreads();
    }
    if (active) y[row] = sum;
}

template <int T>
__global__ void __launch_bounds__(T *T) gemm_naive_kernel(int M, int N, int K, const float *A, long long lda,
                                                          const float *B, long long ldb, float *C, long long ldc) {
    const int row = blockIdx.y * T + threadIdx.y;
    const int col = blockIdx.x * T + threadIdx.x;
    if (row >= M || col >= N) return;   // no barrier in this kernel
    float sum = 0.f;
    for (int k = 0; k < K; ++k)
        sum = fmaf(A[static_cast<long long>(row) * lda + k], B[static_cast<long long>(k) * ldb + col], sum);
    C[static_cast<long long>(row) * ldc + col] = sum;
}

template <int T>
__global__ void __launch_bounds__(T *T) gemm_tiled_kernel(int M, int N, int K, const float *A, long long lda,
                                                          const float *B, long long ldb, float *C, long long ldc) {
    __shared__ float As[T][T];
    __shared__ float Bs[T][T];
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int row = blockIdx.y * T + ty;
    const int col = blockIdx.x * T + tx;
    float sum = 0.f;
    for (int k0 = 0; k0 < K; k0 += T) {
        // out-of-range elements are padded with zeros
        As[ty][tx] = (row < M && k0 + tx < K) ? A[static_cast<long long>(row) * lda + k0 + tx] : 0.f;
        Bs[ty][tx] = (k0 + ty < K && col < N) ? B[static_cast<long long>(k0 + ty) * ldb + col] : 0.f;
        __syncthreads();   // the tiles are complete
#pragma unroll
        for (int k = 0; k < T; ++k) sum = fmaf(As[ty][k], Bs[k][tx], sum);
        __syncthreads();   // everyone is done before the next tiles overwrite them
    }
    if (row < M && col < N) C[static_cast<long long>(row) * ldc + col] = sum;
}

template <int T>
void gemm_dims(int M, int N, dim3 &grid, dim3 &block) {
    grid = dim3(static_cast<unsigned>((N + T - 1) / T), static_cast<unsigned>((M + T - 1) / T));
    block = dim3(T, T);
}

}  // namespace

cudaError_t ablation_gemm_launch(int variant, const GemmArgs &g, cudaStream_t stream) {
    dim3 grid, block;
    const int M = static_cast<int>(g.M), N = static_cast<int>(g.N), K = static_cast<int>(g.K);
    const auto *A = static_cast<const float *>(g.A);
    const auto *B = static_cast<const float *>(g.B);
    if (grid_too_large(g.M, g.N, variant == GTG_ABL_GEMM_NAIVE_16 || variant == GTG_ABL_GEMM_TILED_16 ? 16 : 32))
        return cudaErrorInvalidConfiguration;
    switch (variant) {
        case GTG_ABL_GEMM_NAIVE_16:
            gemm_dims<16>(M, N, grid, block);
            gemm_naive_kernel<16><<<grid, block, 0, stream>>>(M, N, K, A, g.lda, B, g.ldb, g.C, g.ldc);
            break;
        case GTG_ABL_GEMM_NAIVE_32:
            gemm_dims<32>(M, N, grid, block);
            gemm_naive_kernel<32><<<grid, block, 0, stream>>>(M, N, K, A, g.lda, B, g.ldb, g.C, g.ldc);
            break;
        case GTG_ABL_GEMM_TILED_16:
            gemm_dims<16>(M, N, grid, block);
            gemm_tiled_kernel<16><<<grid, block, 0, stream>>>(M, N, K, A, g.lda, B, g.ldb, g.C, g.ldc);
            break;
        case GTG_ABL_GEMM_TILED_32:
            gemm_dims<32>(M, N, grid, block);
            gemm_tiled_kernel<32><<<grid, block, 0, stream>>>(M, N, K, A, g.lda, B, g.ldb, g.C, g.ldc);
            break;
        default:
            return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t ablation_gemv_launch(int variant, const GemvArgs &g, cudaStream_t stream) {
    const unsigned blocks = static_cast<unsigned>((g.M + kVecThreads - 1) / kVecThreads);
    const int M = static_cast<int>(g.M), N = static_cast<int>(g.N);
    const auto *A = static_cast<const float *>(g.A);
    switch (variant) {
        case GTG_ABL_GEMV_NAIVE:
            gemv_naive_kernel<<<blocks, kVecThreads, 0, stream>>>(M, N, A, g.lda, g.x, g.y);
            break;
        case GTG_ABL_GEMV_SHARED:
            gemv_shared_kernel<<<blocks, kVecThreads, 0, stream>>>(M, N, A, g.lda, g.x, g.y);
            break;
        default:
            return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

bool grid_too_large(int64_t M, int64_t N, int tile) {
    return (M + tile - 1) / tile > 65535 || (N + tile - 1) / tile > 2147483647ll;
}

}  // namespace gtg
