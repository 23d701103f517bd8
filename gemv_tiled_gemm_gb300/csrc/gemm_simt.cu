// SIMT GEMM with exact FP32 arithmetic: C = A * B, FP32 (or BF16, widened
// exactly) operands, IEEE FP32 fused multiply-adds on the CUDA cores.
//
// This is the shared-memory tiled GEMM of "CUDA Programming (6)" (section
// 3.2) and "Matrix Operations" ("Tiled Implementation with Shared Memory"),
// with the refinements those pages list as next steps:
//   * register blocking ("Register Blocking"; section 3.4 "thread-level
//     tiling"): each thread owns an 8 x 8 block of C, so every value read
//     from shared memory feeds 8 multiply-adds;
//   * vectorised 128-bit global loads ("Vectorization");
//   * prefetching ("Prefetching"): the next K-slice is loaded into registers
//     while the current one is multiplied from the other shared buffer, so
//     one barrier per slice suffices;
//   * the multiply-adds are issued as packed two-wide FP32 FMAs (sm_100
//     family), two IEEE fused multiply-adds per instruction, which halves
//     the instruction count of the inner loop without changing any result;
//   * boundary handling as on the pages: out-of-range tile elements are
//     zero-filled, out-of-range outputs are not stored, and no thread leaves
//     before the barriers.
// A is stored transposed in shared memory (k-major) so that a thread's 8 rows
// are two 16-byte reads; B keeps its row-major layout.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace gtg {
namespace {

constexpr int kBK = 16;

template <typename T>
struct Load;

template <>
struct Load<float> {
    static __device__ __forceinline__ float4 vec4(const float *p) {
        return __ldg(reinterpret_cast<const float4 *>(p));
    }
    static __device__ __forceinline__ float one(const float *p) { return __ldg(p); }
};

// BF16 stored as 16-bit patterns; widening to FP32 is exact.
template <>
struct Load<uint16_t> {
    static __device__ __forceinline__ float bf(uint32_t bits) { return __uint_as_float(bits << 16); }
    static __device__ __forceinline__ float4 vec4(const uint16_t *p) {
        const uint2 v = __ldg(reinterpret_cast<const uint2 *>(p));
        return make_float4(bf(v.x & 0xFFFFu), bf(v.x >> 16), bf(v.y & 0xFFFFu), bf(v.y >> 16));
    }
    static __device__ __forceinline__ float one(const uint16_t *p) { return bf(__ldg(p)); }
};

// FP16 stored as 16-bit patterns; widening to FP32 is exact.
template <>
struct Load<__half> {
    static __device__ __forceinline__ float h(uint32_t bits) {
        return __half2float(__ushort_as_half(static_cast<unsigned short>(bits)));
    }
    static __device__ __forceinline__ float4 vec4(const __half *p) {
        const uint2 v = __ldg(reinterpret_cast<const uint2 *>(p));
        return make_float4(h(v.x & 0xFFFFu), h(v.x >> 16), h(v.y & 0xFFFFu), h(v.y >> 16));
    }
    static __device__ __forceinline__ float one(const __half *p) {
        return h(__ldg(reinterpret_cast<const unsigned short *>(p)));
    }
};

// Each thread owns TM rows x TN columns of the tile: 8 x 8; 8 x 4 (twice the
// threads on the same tile when tiles are few); 16 x 8 (256 x 128 tiles for
// large products: more multiply-adds per shared-memory read).
template <typename T, int BM, int BN, bool VEC, int TN = 8, int TM = 8>
struct SimtTile {
    static constexpr int TX = BN / TN;             // threads along N
    static constexpr int TY = BM / TM;             // threads along M
    static constexpr int THREADS = TX * TY;

    static constexpr int A_V4 = BM * kBK / 4 / THREADS;   // 4-element A groups per thread
    static constexpr int B_V4 = BN * kBK / 4 / THREADS;
    static_assert(A_V4 >= 1 && B_V4 >= 1, "tile too small for its thread count");
};

// gridDim.z has one of two meanings.
// Strided batch (batched != 0): the CTA at blockIdx.z = b multiplies item b,
// whose operands and output start sA, sB, sC elements after those of item 0;
// every item of the batch runs in this one launch.
// Split K (batched == 0, gridDim.z = S > 1): the CTA at blockIdx.z = z
// multiplies the K range [z * k_per, (z + 1) * k_per) and writes its FP32
// partial product to the workspace slice ws + z * M * N (leading dimension N)
// instead of C; split_reduce_kernel then adds the S slices in order z = 0 .. S-1.
template <typename T, int BM, int BN, bool VEC, int TN, int TM>
__global__ void __launch_bounds__(SimtTile<T, BM, BN, VEC, TN, TM>::THREADS)
    simt_gemm_kernel(int M, int N, int K, const T *__restrict__ A, long long lda,
                     const T *__restrict__ B, long long ldb, float *__restrict__ C, long long ldc,
                     int c_vec, int k_per, float *__restrict__ ws, const float *__restrict__ bias, int act,
                     int batched, long long sA, long long sB, long long sC) {
    using L = SimtTile<T, BM, BN, VEC, TN, TM>;
    constexpr int QN = TN / 2;   // column pairs per thread
    constexpr int PM = TM / 2;   // row pairs per thread
    constexpr int RQ = TM / 4;   // row quads per thread, BM / RQ rows apart
    // a following dependent launch (the split reduction) may be scheduled now;
    // it waits for this grid before reading anything this grid writes
    ptx::allow_next_grid();
    if (batched) {
        A += blockIdx.z * sA;
        B += blockIdx.z * sB;
        C += blockIdx.z * sC;
    } else if (gridDim.z > 1) {
        bias = nullptr;   // partial products: the reduction applies the epilogue
        act = 0;
        const int z = blockIdx.z;
        A += static_cast<long long>(z) * k_per;
        B += static_cast<long long>(z) * k_per * ldb;
        K = max(0, min(k_per, K - z * k_per));
        C = ws + static_cast<long long>(z) * M * N;
        ldc = N;
        c_vec = (N & 3) == 0;
    }
    __shared__ __align__(16) float As[2][kBK][BM];
    __shared__ __align__(16) float Bs[2][kBK][BN];

    const int tid = threadIdx.x;
    const int tx = tid % L::TX, ty = tid / L::TX;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;

    float4 ra[L::A_V4], rb[L::B_V4];

    // A: group g covers row (g % BM), k-quad (g / BM): consecutive threads take
    // consecutive rows so the transposed shared-memory stores hit distinct banks.
    auto load_a = [&](int k0) {
#pragma unroll
        for (int i = 0; i < L::A_V4; ++i) {
            const int g = tid + i * L::THREADS;
            const int r = g % BM, kq = g / BM;
            const int row = m0 + r, k = k0 + kq * 4;
            const T *p = A + static_cast<long long>(row) * lda + k;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (row < M) {
                if (VEC && k + 3 < K) {
                    v = Load<T>::vec4(p);
                } else {
                    if (k < K) v.x = Load<T>::one(p);
                    if (k + 1 < K) v.y = Load<T>::one(p + 1);
                    if (k + 2 < K) v.z = Load<T>::one(p + 2);
                    if (k + 3 < K) v.w = Load<T>::one(p + 3);
                }
            }
            ra[i] = v;
        }
    };
    auto store_a = [&](int buf) {
#pragma unroll
        for (int i = 0; i < L::A_V4; ++i) {
            const int g = tid + i * L::THREADS;
            const int r = g % BM, kq = g / BM;
            As[buf][kq * 4 + 0][r] = ra[i].x;
            As[buf][kq * 4 + 1][r] = ra[i].y;
            As[buf][kq * 4 + 2][r] = ra[i].z;
            As[buf][kq * 4 + 3][r] = ra[i].w;
        }
    };
    // B: group g covers k-row (g / (BN/4)), columns 4*(g % (BN/4)) .. +3.
    auto load_b = [&](int k0) {
#pragma unroll
        for (int i = 0; i < L::B_V4; ++i) {
            const int g = tid + i * L::THREADS;
            const int kr = g / (BN / 4), c4 = g % (BN / 4);
            const int k = k0 + kr, col = n0 + c4 * 4;
            const T *p = B + static_cast<long long>(k) * ldb + col;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (k < K) {
                if (VEC && col + 3 < N) {
                    v = Load<T>::vec4(p);
                } else {
                    if (col < N) v.x = Load<T>::one(p);
                    if (col + 1 < N) v.y = Load<T>::one(p + 1);
                    if (col + 2 < N) v.z = Load<T>::one(p + 2);
                    if (col + 3 < N) v.w = Load<T>::one(p + 3);
                }
            }
            rb[i] = v;
        }
    };
    auto store_b = [&](int buf) {
#pragma unroll
        for (int i = 0; i < L::B_V4; ++i) {
            const int g = tid + i * L::THREADS;
            const int kr = g / (BN / 4), c4 = g % (BN / 4);
            *reinterpret_cast<float4 *>(&Bs[buf][kr][c4 * 4]) = rb[i];
        }
    };

    // The 8 x 8 accumulators in pairs for the packed two-wide FMA: for row
    // pair p (rows 2p, 2p+1 of the thread's block) and column pair q,
    // d[p][q][0] = (acc[2p][2q], acc[2p+1][2q+1]) takes (a[2p], a[2p+1]) times
    // (b[2q], b[2q+1]), and d[p][q][1] = (acc[2p][2q+1], acc[2p+1][2q]) takes
    // (a[2p], a[2p+1]) times the exchanged columns (b[2q+1], b[2q]). Each lane
    // of a packed FMA is one IEEE fused multiply-add, so every output sees the
    // same operations in the same K order as with scalar FMAs (and the same
    // result).
    float2 d[PM][QN][2];
#pragma unroll
    for (int p = 0; p < PM; ++p)
#pragma unroll
        for (int q = 0; q < QN; ++q) d[p][q][0] = d[p][q][1] = make_float2(0.f, 0.f);

    const int ntiles = (K + kBK - 1) / kBK;
    if (ntiles > 0) {
        load_a(0);
        load_b(0);
        store_a(0);
        store_b(0);
    }
    __syncthreads();

    for (int t = 0; t < ntiles; ++t) {
        const int cur = t & 1;
        if (t + 1 < ntiles) {
            load_a((t + 1) * kBK);
            load_b((t + 1) * kBK);
        }
#pragma unroll
        for (int k = 0; k < kBK; ++k) {
            float2 ap[PM];
#pragma unroll
            for (int rq = 0; rq < RQ; ++rq) {
                const float4 a = *reinterpret_cast<const float4 *>(&As[cur][k][rq * (BM / RQ) + ty * 4]);
                ap[2 * rq] = make_float2(a.x, a.y);
                ap[2 * rq + 1] = make_float2(a.z, a.w);
            }
            const float4 b0 = *reinterpret_cast<const float4 *>(&Bs[cur][k][tx * 4]);
            const float4 b1 = TN == 8 ? *reinterpret_cast<const float4 *>(&Bs[cur][k][BN / 2 + tx * 4]) : b0;
            const float2 bp[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w), make_float2(b1.x, b1.y),
                                  make_float2(b1.z, b1.w)};
            const float2 bs[4] = {make_float2(b0.y, b0.x), make_float2(b0.w, b0.z), make_float2(b1.y, b1.x),
                                  make_float2(b1.w, b1.z)};
#pragma unroll
            for (int p = 0; p < PM; ++p)
#pragma unroll
                for (int q = 0; q < QN; ++q) {
                    d[p][q][0] = __ffma2_rn(ap[p], bp[q], d[p][q][0]);
                    d[p][q][1] = __ffma2_rn(ap[p], bs[q], d[p][q][1]);
                }
        }
        if (t + 1 < ntiles) {
            store_a(cur ^ 1);
            store_b(cur ^ 1);
        }
        __syncthreads();
    }

    float acc[TM][TN];
#pragma unroll
    for (int p = 0; p < PM; ++p)
#pragma unroll
        for (int q = 0; q < QN; ++q) {
            acc[2 * p][2 * q] = d[p][q][0].x;
            acc[2 * p + 1][2 * q + 1] = d[p][q][0].y;
            acc[2 * p][2 * q + 1] = d[p][q][1].x;
            acc[2 * p + 1][2 * q] = d[p][q][1].y;
        }
    // rows (i / 4) * (BM / RQ) + ty*4 + i % 4; columns tx*4 + j and (TN = 8)
    // BN/2 + tx*4 + j.
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int row = m0 + (i / 4) * (BM / RQ) + ty * 4 + (i % 4);
        if (row >= M) continue;
        float *crow = C + static_cast<long long>(row) * ldc;
#pragma unroll
        for (int h = 0; h < TN / 4; ++h) {
            const int col = n0 + (h == 0 ? tx * 4 : BN / 2 + tx * 4);
            float v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                v[j] = apply_epilogue(acc[i][h * 4 + j], col + j < N ? bias : nullptr, col + j, act);
            if (c_vec && col + 3 < N) {
                *reinterpret_cast<float4 *>(crow + col) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (col + j < N) crow[col + j] = v[j];
            }
        }
    }
}

// C[i][j] = sum over z = 0 .. S-1 of ws[z][i][j], in that order. One thread
// per 4 consecutive columns of a row (16-byte accesses when they are aligned).
__global__ void split_reduce_kernel(const float *__restrict__ ws, int splits, int M, int N,
                                    float *__restrict__ C, long long ldc, int vec,
                                    const float *__restrict__ bias, int act) {
    ptx::wait_prior_grid();   // a dependent launch: the partial products are complete
    const int n4 = (N + 3) / 4;
    const long long slice = static_cast<long long>(M) * N;
    for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
         t < static_cast<long long>(M) * n4; t += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int row = static_cast<int>(t / n4);
        const int col = static_cast<int>(t - static_cast<long long>(row) * n4) * 4;
        const long long src = static_cast<long long>(row) * N + col;
        float *dst = C + static_cast<long long>(row) * ldc + col;
        if (vec && col + 3 < N) {
            float4 v = *reinterpret_cast<const float4 *>(ws + src);
            for (int z = 1; z < splits; ++z) {
                const float4 w = *reinterpret_cast<const float4 *>(ws + z * slice + src);
                v.x += w.x;
                v.y += w.y;
                v.z += w.z;
                v.w += w.w;
            }
            v.x = apply_epilogue(v.x, bias, col, act);
            v.y = apply_epilogue(v.y, bias, col + 1, act);
            v.z = apply_epilogue(v.z, bias, col + 2, act);
            v.w = apply_epilogue(v.w, bias, col + 3, act);
            *reinterpret_cast<float4 *>(dst) = v;
        } else {
            for (int c = 0; c < 4 && col + c < N; ++c) {
                float v = ws[src + c];
                for (int z = 1; z < splits; ++z) v += ws[z * slice + src + c];
                dst[c] = apply_epilogue(v, bias, col + c, act);
            }
        }
    }
}

__global__ void epilogue_fill_kernel(float *C, long long M, long long N, long long ldc, const float *bias,
                                     int per_column, int act) {
    const long long total = M * N;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long r = i / N, c = i % N;
        C[r * ldc + c] = apply_epilogue(0.f, bias, static_cast<int>(per_column ? c : r), act);
    }
}

__global__ void zero_fill_kernel(float *C, long long M, long long N, long long ldc) {
    const long long total = M * N;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x)
        C[(i / N) * ldc + (i % N)] = 0.f;
}

template <typename T, int BM, int BN, bool VEC, int TN, int TM = 8>
cudaError_t launch_one(const GemmArgs &g, int splits, cudaStream_t stream) {
    using L = SimtTile<T, BM, BN, VEC, TN, TM>;
    const dim3 tiles(static_cast<unsigned>((g.N + BN - 1) / BN), static_cast<unsigned>((g.M + BM - 1) / BM));
    if (g.batch > 1) {
        // a strided batch: every item in one launch (blockIdx.z), in chunks of
        // at most 65535 items (the grid's z limit); no K split
        const int c_vec = ((reinterpret_cast<uintptr_t>(g.C) & 15) == 0 && (g.ldc & 3) == 0 && (g.strideC & 3) == 0)
                              ? 1 : 0;
        for (int64_t b0 = 0; b0 < g.batch; b0 += 65535) {
            const dim3 grid(tiles.x, tiles.y, static_cast<unsigned>(std::min<int64_t>(g.batch - b0, 65535)));
            simt_gemm_kernel<T, BM, BN, VEC, TN, TM><<<grid, L::THREADS, 0, stream>>>(
                static_cast<int>(g.M), static_cast<int>(g.N), static_cast<int>(g.K),
                static_cast<const T *>(g.A) + b0 * g.strideA, g.lda, static_cast<const T *>(g.B) + b0 * g.strideB,
                g.ldb, g.C + b0 * g.strideC, g.ldc, c_vec, 0, nullptr, g.bias, g.act, 1, g.strideA, g.strideB,
                g.strideC);
            const cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    const dim3 grid(tiles.x, tiles.y, static_cast<unsigned>(splits));
    const int c_vec = ((reinterpret_cast<uintptr_t>(g.C) & 15) == 0 && (g.ldc & 3) == 0) ? 1 : 0;
    const int k_per = static_cast<int>(((g.K + kBK - 1) / kBK + splits - 1) / splits * kBK);
    float *ws = nullptr;
    cudaError_t e;
    if (splits > 1) {
        e = ws_alloc(reinterpret_cast<void **>(&ws), static_cast<size_t>(splits) * g.M * g.N * sizeof(float), stream);
        if (e != cudaSuccess) return e;
    }
    simt_gemm_kernel<T, BM, BN, VEC, TN, TM><<<grid, L::THREADS, 0, stream>>>(
        static_cast<int>(g.M), static_cast<int>(g.N), static_cast<int>(g.K),
        static_cast<const T *>(g.A), g.lda, static_cast<const T *>(g.B), g.ldb, g.C, g.ldc, c_vec, k_per, ws,
        g.bias, g.act, 0, 0, 0, 0);
    e = cudaGetLastError();
    if (splits > 1) {
        if (e == cudaSuccess) e = split_reduce_launch(ws, splits, g.M, g.N, g.C, g.ldc, g.bias, g.act, stream);
        const cudaError_t f = cudaFreeAsync(ws, stream);   // stream-ordered: after the reduction
        if (e == cudaSuccess) e = f;
    }
    return e;
}

template <typename T, bool VEC>
cudaError_t launch_typed(const GemmArgs &g, const gtg_plan &plan, cudaStream_t stream) {
    if (plan.bm == 256) return launch_one<T, 256, 128, VEC, 8, 16>(g, plan.splits, stream);
    if (plan.bm == 128) return launch_one<T, 128, 128, VEC, 8>(g, plan.splits, stream);
    return launch_one<T, 64, 64, VEC, 4>(g, plan.splits, stream);
}

bool vec_ok(const GemmArgs &g) {
    // 4 consecutive elements per load: 16 bytes for FP32, 8 for BF16 / FP16;
    // in a batch every item keeps the alignment of the first
    const uintptr_t mask = (g.prec == GTG_PREC_BF16 || g.prec == GTG_PREC_F16) ? 7 : 15;
    return (reinterpret_cast<uintptr_t>(g.A) & mask) == 0 && (reinterpret_cast<uintptr_t>(g.B) & mask) == 0 &&
           (g.lda % 4) == 0 && (g.ldb % 4) == 0 && (g.batch == 1 || ((g.strideA % 4) == 0 && (g.strideB % 4) == 0));
}

}  // namespace

// Tile: 128 x 128 (8 warps, 8 x 8 outputs per thread) when there are enough
// such tiles for every SM, or 256 x 128 (8 warps, 16 x 8 per thread) when
// their waves come out ahead. Otherwise, when K is long enough, 128 x 128 tiles
// split in K so that the CTAs fill at least three quarters of the SMs once
// (one CTA of 8 warps per SM); else 64 x 64 tiles of 4 warps (8 x 4 outputs
// per thread), whose small grids split K (plan->splits) so that about six
// CTAs run on every SM, each split keeping at least two 16-deep K slices; the
// partial products go through a workspace. Measured (FP32, CUDA events):
// 1024^3 96.5 us with the earlier 2-warp 64 x 64 tiles, 76 us with 4-warp
// ones, 65.7 us as 128 x 128 tiles in two K ranges; the 4-warp tiles are as
// fast or faster on every small shape tried (256^3 to 2048^3, 1000 x 700 x
// 1500, 1024^2 x 4096).
void simt_plan(const DeviceInfo &dev, const GemmArgs &g, gtg_plan *plan) {
    // a strided batch runs all its items in one launch: tiles count over the
    // whole batch, and K is never split (the items fill the GPU instead)
    const int64_t items = std::max<int64_t>(g.batch, 1);
    const int64_t big_tiles = items * ((g.M + 127) / 128) * ((g.N + 127) / 128);
    const int64_t kslices = (g.K + kBK - 1) / kBK;
    const bool big = big_tiles >= dev.sms;
    plan->kernel = GTG_KERNEL_SIMT;
    plan->bk = kBK;
    plan->smem = 0;
    plan->cluster = 1;
    plan->stages = 2;   // double-buffered shared-memory slices
    if (!big && big_tiles > 0 && items == 1) {
        int64_t fill = std::min<int64_t>(dev.sms / big_tiles, kslices / 32);
        if (fill >= 2 && 4 * big_tiles * fill >= 3 * dev.sms) {
            const int64_t k_per = (kslices + fill - 1) / fill;   // every split owns K slices
            fill = (kslices + k_per - 1) / k_per;
            plan->bm = plan->bn = 128;
            plan->threads = 256;
            plan->splits = static_cast<int>(fill);
            plan->grid = static_cast<int>(big_tiles * fill);
            return;
        }
    }
    plan->bm = plan->bn = big ? 128 : 64;
    plan->threads = big ? 256 : 128;
    if (big) {
        // 256 x 128 tiles (16 x 8 outputs per thread) do a 128 x 128 tile's work
        // about 8 % faster but come in half as many units: take them when their
        // wave count says so (measured, FP32: 8192^2 x 4096 46.4 -> 50.0,
        // 3000^3 43.9 -> 47.0, 4096 x 2048 x 4096 39.3 -> 43.5 TFLOP/s; kept at
        // 128 x 128 for 4096^3 and 2560^2 x 2048, where they were slower)
        const int64_t t256 = items * ((g.M + 255) / 256) * ((g.N + 127) / 128);
        const int64_t t128 = items * ((g.M + 127) / 128) * ((g.N + 127) / 128);
        const double w256 = static_cast<double>((t256 + dev.sms - 1) / dev.sms) * 2.0 / 1.08;
        const double w128 = static_cast<double>((t128 + dev.sms - 1) / dev.sms);
        if (t256 >= dev.sms && w256 < w128) plan->bm = 256;
    }
    const int64_t tiles = items * ((g.M + plan->bm - 1) / plan->bm) * ((g.N + plan->bn - 1) / plan->bn);
    int64_t splits = 1;
    if (!big && items == 1) {
        // the busiest SM's K work: ceil(CTAs / SMs) CTAs of ceil(slices / S)
        // slices each; a split must save more than a fixed allowance for the
        // extra partial-product traffic and the reduction launch
        auto work = [&](int64_t sp) {
            const int64_t per = (kslices + sp - 1) / sp;
            return static_cast<double>((tiles * sp + dev.sms - 1) / dev.sms) * per + (sp > 1 ? 0.25 * kslices + 4 : 0);
        };
        double best = work(1);
        for (int64_t sp = 2; sp <= 16 && sp <= kslices / 2; ++sp) {
            const double w = work(sp);
            if (w < best) {
                best = w;
                splits = sp;
            }
        }
        // every split must own at least one K slice
        const int64_t k_per = (kslices + splits - 1) / splits;
        splits = (kslices + k_per - 1) / k_per;
    }
    plan->splits = static_cast<int>(splits);
    plan->grid = static_cast<int>(tiles * splits);
}

cudaError_t simt_launch(const DeviceInfo &dev, const GemmArgs &g, const gtg_plan &plan,
                        cudaStream_t stream) {
    (void)dev;
    // a strided batch is one launch over all items (blockIdx.z), see launch_one
    const bool vec = vec_ok(g);
    if (g.prec == GTG_PREC_BF16)
        return vec ? launch_typed<uint16_t, true>(g, plan, stream) : launch_typed<uint16_t, false>(g, plan, stream);
    if (g.prec == GTG_PREC_F16)
        return vec ? launch_typed<__half, true>(g, plan, stream) : launch_typed<__half, false>(g, plan, stream);
    return vec ? launch_typed<float, true>(g, plan, stream) : launch_typed<float, false>(g, plan, stream);
}

cudaError_t epilogue_fill_launch(float *C, int64_t M, int64_t N, int64_t ldc, const float *bias, int per_column,
                                 int act, cudaStream_t stream) {
    const long long total = M * N;
    long long blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    epilogue_fill_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(C, M, N, ldc, bias, per_column, act);
    return cudaGetLastError();
}

cudaError_t split_reduce_launch(const float *ws, int splits, int64_t M, int64_t N, float *C, int64_t ldc,
                                const float *bias, int act, cudaStream_t stream) {
    const long long quads = M * ((N + 3) / 4);
    const unsigned blocks = static_cast<unsigned>(std::min<long long>((quads + 255) / 256, 8192));
    // ws is a pool allocation (256-byte aligned) of rows of N floats: 16-byte
    // accesses need N % 4 == 0, and C a 16-byte aligned base and ldc % 4 == 0
    const int vec = ((N & 3) == 0 && (reinterpret_cast<uintptr_t>(C) & 15) == 0 && (ldc & 3) == 0) ? 1 : 0;
    // scheduled while the GEMM that wrote ws finishes (programmatic dependent
    // launch); the kernel waits for it before reading
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, split_reduce_kernel, ws, splits, static_cast<int>(M), static_cast<int>(N), C, ldc,
                              vec, bias, act);
}

cudaError_t zero_fill_launch(float *C, int64_t M, int64_t N, int64_t ldc, cudaStream_t stream) {
    const long long total = M * N;
    long long blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    zero_fill_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(C, M, N, ldc);
    return cudaGetLastError();
}

}  // namespace gtg
