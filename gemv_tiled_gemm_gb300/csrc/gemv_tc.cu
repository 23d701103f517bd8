// Batched GEMV of a BF16 matrix on the tensor cores: y_b = act(A x_b + bias)
// for b < batch (3..8), A (M x N) BF16, x and y FP32 ("Matrix Operations",
// Matrix-Vector Multiplication; fully connected layers applied to a batch of
// inputs).
//
// With eight vectors the product is a dense contraction of A with an N x 8
// matrix, and on the CUDA cores every matrix element costs eight FMAs and a
// share of the vector reads: the CUDA-core kernel reaches only about half of
// the HBM rate. Here A streams through TMA into the A operand of
// tcgen05.mma (kind::f16, M = 128), so the kernel is bound by reading A once.
//
// Precision: the MMA multiplies BF16 by BF16. Each FP32 vector entry is
// written as the sum of three BF16 pieces, x = x1 + x2 + x3 + r with
// x1 = bf16(x), x2 = bf16(x - x1), x3 = bf16(x - x1 - x2) (each difference
// exact in FP32) and |r| <= 2^-27 |x|; every product of a BF16 matrix element
// with a piece is exact in FP32 and the tensor core adds them in FP32, so the
// result meets the FP32 GEMV bound. A first kernel writes the pieces of
// vector b as rows 3b, 3b+1, 3b+2 of a small K-major matrix, read by TMA as
// the MMA's 32-row B operand (rows past 3 * batch are the tensor map's zero
// fill), so y_b = D[3b] + D[3b+1] + D[3b+2], added in that order. (Writing
// the pieces inside the product kernel, two warps converting each slice of x
// into its B slot, was slower: at batch 8 0.31 / 0.46 / 0.53 of the copy
// peak at 4096^2 / 8192^2 / 16384^2 against 0.40 / 0.67 / 0.88.)
//
// Work division: tiles of 128 rows, each of ks K slices of 64 columns; the
// tiles x ks slices are cut into one contiguous range per CTA of a persistent
// grid (one CTA per SM), so every SM reads the same share of A whatever the
// tile count. A CTA's range covers parts of one or more tiles; a tile it
// covers whole is written to y directly, the parts of a tile shared by CTAs
// go to a workspace, and whichever CTA finishes its part last adds them all
// in CTA order (each epilogue warp for its 32 rows, counted by an atomic per
// tile and warp), so the result does not depend on scheduling.
//
// Roles (192 threads): warp 0 issues the TMA loads, warp 1 owns TMEM (two 32-
// column accumulators) and issues the MMAs, warps 2-5 read the accumulator
// of a finished tile part (each its 32 TMEM lanes = rows) and write it out.
// The product kernel is a dependent launch after the kernel that writes the
// vector pieces, scheduled while that kernel finishes.
// Every wait is bounded; on time-out the kernel latches GTG_ERR_TIMEOUT,
// drains what it issued, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace gtg {
namespace {

constexpr int kThreads = 192;
constexpr int kBM = 128;                       // matrix rows per tile (MMA M)
constexpr int kBK = 64;                        // BF16 columns per K slice (128 bytes)
constexpr int kNP = 32;                        // MMA N: 3 pieces x up to 8 vectors, padded
constexpr int kStages = 8;
constexpr int kABytes = kBM * 128;             // 16 KB
constexpr int kBBytes = kNP * 128;             // 4 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kNBars = 2 * kStages + 5;
constexpr int kSmem = 1024 + kStages * kStageBytes + kNBars * 8 + 16;
constexpr int kTmemCols = 2 * kNP;
constexpr uint32_t kIdesc = ptx::make_idesc(1u /* BF16 */, 0u, 0u /* B K-major */, kBM, kNP);

struct Params {
    float *y;
    long long ldy;
    float *ws;                   // [tile][part][8][kBM] partial sums of shared tiles
    int *cnt;                    // [tile][4] parts written so far, per epilogue warp (zeroed by the first kernel)
    int M, batch;
    int ks;                      // K slices per tile
    long long work;              // tiles * ks
    int maxp;                    // workspace parts per tile
    const float *bias;
    int act;
    int *status;
    unsigned long long wait_limit_ns;
    int drop_slice;              // testing hook: slice whose load CTA 0 never issues (-1: none)
};

// First unit of CTA c's range and the CTA whose range holds unit f.
__host__ __device__ __forceinline__ long long range_begin(long long c, long long work, long long grid) {
    return c * work / grid;
}
__host__ __device__ __forceinline__ int cta_of(long long f, long long work, long long grid) {
    return static_cast<int>(((f + 1) * grid - 1) / work);
}

__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag, const Params &p) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer_ns() - t0 > p.wait_limit_ns) {
            *abort_flag = 1;
            atomicCAS(p.status, 0, static_cast<int>(GTG_ERR_TIMEOUT));
            return false;
        }
    }
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag, const Params &p) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, abort_flag, p);
}

// Ignores the abort flag: lets work already issued finish. Bounded as well.
__device__ __noinline__ void wait_drain(uint32_t bar, uint32_t parity, const Params &p) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer_ns() - t0 > p.wait_limit_ns) {
            atomicCAS(p.status, 0, static_cast<int>(GTG_ERR_TIMEOUT));
            return;
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    gemv_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmX, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sA = ptx::smem_addr(smem);
    const uint32_t sB = sA + kStages * kABytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kNBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const uint32_t bar0 = ptx::smem_addr(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto accf_bar = [&](int a) { return bar0 + 8u * (2 * kStages + a); };
    auto acce_bar = [&](int a) { return bar0 + 8u * (2 * kStages + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(accf_bar(a), 1);
            ptx::mbar_init(acce_bar(a), 4);   // one arrive per epilogue warp
        }
        ptx::mbar_init(drain_bar, 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmX);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // A never depends on the kernel before this one (that kernel started only
    // after everything before it had completed), so the first stages' loads
    // of A go out before waiting for it; the vector pieces it writes, the part
    // counters it zeroes and the outputs wait for it (griddepcontrol.wait).
    ptx::allow_next_grid();

    const long long f0 = range_begin(blockIdx.x, p.work, gridDim.x);
    const long long f1 = range_begin(blockIdx.x + 1, p.work, gridDim.x);

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            const long long fp = min(f1, f0 + kStages);   // the first stages: A now, the pieces after the wait
            // unit f = (tile t, slice k), stepped without a 64-bit division per
            // unit (measured: batch 8 at 8192^2 and 16384^2 0.5 us faster)
            const int t0 = static_cast<int>(f0 / p.ks);
            const int k0 = static_cast<int>(f0 - static_cast<long long>(t0) * p.ks);
            int t = t0, k = k0;
            auto next = [&] {
                if (++k == p.ks) {
                    k = 0;
                    ++t;
                }
            };
            uint32_t it = 0;
            for (long long f = f0; f < fp; ++f, ++it, next()) {
                if (p.drop_slice == static_cast<int>(it) && blockIdx.x == 0) continue;
                ptx::mbar_arrive_expect_tx(full_bar(static_cast<int>(it)), kStageBytes);
                ptx::tma_load_3d(sA + it * kABytes, &tmA, full_bar(static_cast<int>(it)), k * kBK, t * kBM, 0);
            }
            ptx::wait_prior_grid();
            it = 0;
            for (long long f = f0, kx = k0; f < fp; ++f, ++it, kx = kx + 1 == p.ks ? 0 : kx + 1) {
                if (p.drop_slice == static_cast<int>(it) && blockIdx.x == 0) continue;
                ptx::tma_load_3d(sB + it * kBBytes, &tmX, full_bar(static_cast<int>(it)), static_cast<int>(kx) * kBK,
                                 0, 0);
            }
            bool ok = true;
            for (long long f = fp; ok && f < f1; ++f, ++it, next()) {
                const int s = static_cast<int>(it % kStages);
                const uint32_t ph = (it / kStages) & 1u;
                if (!wait_bar(empty_bar(s), ph ^ 1u, abort_flag, p)) {
                    ok = false;
                    break;
                }
                if (p.drop_slice == static_cast<int>(it) && blockIdx.x == 0) continue;
                ptx::mbar_arrive_expect_tx(full_bar(s), kStageBytes);
                ptx::tma_load_3d(sA + s * kABytes, &tmA, full_bar(s), k * kBK, t * kBM, 0);
                ptx::tma_load_3d(sB + s * kBBytes, &tmX, full_bar(s), k * kBK, 0, 0);
            }
            if (!ok) {
                const uint32_t n = it < kStages ? it : kStages;
                for (uint32_t j = 1; j <= n; ++j) {
                    const uint32_t i = it - j;
                    wait_drain(full_bar(static_cast<int>(i % kStages)), (i / kStages) & 1u, p);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t it = 0;
            int local = 0;
            bool ok = true, issued = false;
            for (long long f = f0; ok && f < f1; ++local) {
                const int t = static_cast<int>(f / p.ks);
                const long long fe = min(f1, static_cast<long long>(t + 1) * p.ks);   // end of this tile part
                const int acc = local & 1;
                const uint32_t aph = (static_cast<uint32_t>(local) >> 1) & 1u;
                if (!wait_bar(acce_bar(acc), aph ^ 1u, abort_flag, p)) break;
                ptx::tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kNP);
                for (long long g = f; g < fe; ++g, ++it) {
                    const int s = static_cast<int>(it % kStages);
                    const uint32_t ph = (it / kStages) & 1u;
                    if (!wait_bar(full_bar(s), ph, abort_flag, p)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    const uint32_t a0 = sA + s * kABytes, b0 = sB + s * kBBytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        // both operands K-major, 128-byte swizzle: a K step of 16
                        // BF16 moves the start 32 bytes inside the swizzle row
                        const uint64_t ad = ptx::smem_desc_sw128(a0 + kk * 32, 16, 1024);
                        const uint64_t bd = ptx::smem_desc_sw128(b0 + kk * 32, 16, 1024);
                        ptx::mma_bf16(d_tmem, ad, bd, kIdesc, (g > f || kk > 0) ? 1u : 0u);
                    }
                    ptx::mma_commit(empty_bar(s));
                    issued = true;
                }
                if (!ok) break;
                ptx::mma_commit(accf_bar(acc));
                f = fe;
            }
            if (issued) {
                ptx::mma_commit(drain_bar);
                wait_drain(drain_bar, 0u, p);
            }
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..5)
        ptx::wait_prior_grid();   // the part counters are zeroed by the kernel before
        const int quarter = warp & 3;
        const int rr = quarter * 32 + lane;   // row within the tile
        int local = 0;
        for (long long f = f0; f < f1; ++local) {
            const int t = static_cast<int>(f / p.ks);
            const long long tb = static_cast<long long>(t) * p.ks;
            const long long fe = min(f1, tb + p.ks);
            const bool whole = f == tb && fe == tb + p.ks;
            const int acc = local & 1;
            const uint32_t aph = (static_cast<uint32_t>(local) >> 1) & 1u;
            if (!wait_bar(accf_bar(acc), aph, abort_flag, p)) break;
            ptx::tc_fence_after_sync();
            uint32_t r[32];
            ptx::tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                        static_cast<uint32_t>(acc * kNP),
                                    r);
            ptx::tmem_ld_wait();
            const int row = t * kBM + rr;
            if (whole) {
                if (row < p.M) {
#pragma unroll
                    for (int b = 0; b < 8; ++b)
                        if (b < p.batch) {
                            const float v = (__uint_as_float(r[3 * b]) + __uint_as_float(r[3 * b + 1])) +
                                            __uint_as_float(r[3 * b + 2]);
                            p.y[b * p.ldy + row] = apply_epilogue(v, p.bias, row, p.act);
                        }
                }
            } else {
                const int c0 = cta_of(tb, p.work, gridDim.x), c1 = cta_of(tb + p.ks - 1, p.work, gridDim.x);
                const int part = static_cast<int>(blockIdx.x) - c0;
                float *parts = p.ws + static_cast<long long>(t) * p.maxp * 8 * kBM + rr;   // part j at j * 8 * kBM
#pragma unroll
                for (int b = 0; b < 8; ++b)
                    if (b < p.batch)
                        parts[(part * 8 + b) * kBM] = (__uint_as_float(r[3 * b]) + __uint_as_float(r[3 * b + 1])) +
                                                      __uint_as_float(r[3 * b + 2]);
                // the warp that completes the count for its 32 rows adds the parts
                __threadfence();
                __syncwarp();
                int last = 0;
                if (lane == 0) last = atomicAdd(p.cnt + t * 4 + quarter, 1) == c1 - c0;
                if (__shfl_sync(0xFFFFFFFFu, last, 0)) {
                    __threadfence();
                    if (row < p.M) {
                        // up to 8 parts x 8 vectors of loads in flight, then added in part order
                        const int np = c1 - c0 + 1;
                        float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                        for (int j0 = 0; j0 < np; j0 += 8) {
                            float w[8][8];
#pragma unroll
                            for (int u = 0; u < 8; ++u)
#pragma unroll
                                for (int b = 0; b < 8; ++b)
                                    w[u][b] = (j0 + u < np && b < p.batch) ? parts[((j0 + u) * 8 + b) * kBM] : 0.f;
#pragma unroll
                            for (int u = 0; u < 8; ++u)
                                if (j0 + u < np)
#pragma unroll
                                    for (int b = 0; b < 8; ++b) v[b] += w[u][b];
                        }
#pragma unroll
                        for (int b = 0; b < 8; ++b)
                            if (b < p.batch) p.y[b * p.ldy + row] = apply_epilogue(v[b], p.bias, row, p.act);
                    }
                }
            }
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(acce_bar(acc));
            f = fe;
        }
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem_base, kTmemCols);
    }
}

// The three BF16 pieces of every vector entry: rows 3b, 3b+1, 3b+2 of xp.
// It also zeroes the part counters of the product kernel.
__global__ void split_vectors_kernel(const float *__restrict__ x, long long ldx, int N, int batch,
                                     __nv_bfloat16 *__restrict__ xp, long long ldp, int *__restrict__ cnt, int ncnt) {
    ptx::wait_prior_grid();   // x may come from the previous kernel in the stream
    ptx::allow_next_grid();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < ncnt; i += gridDim.x * blockDim.x) cnt[i] = 0;
    const long long total = static_cast<long long>(batch) * N;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int b = static_cast<int>(i / N), k = static_cast<int>(i - static_cast<long long>(b) * N);
        const float v = x[b * ldx + k];
        const __nv_bfloat16 h1 = __float2bfloat16_rn(v);
        const float r1 = v - __bfloat162float(h1);
        const __nv_bfloat16 h2 = __float2bfloat16_rn(r1);
        const float r2 = r1 - __bfloat162float(h2);
        const __nv_bfloat16 h3 = __float2bfloat16_rn(r2);
        xp[(3 * b) * ldp + k] = h1;
        xp[(3 * b + 1) * ldp + k] = h2;
        xp[(3 * b + 2) * ldp + k] = h3;
    }
}

// Launch with programmatic dependent launch allowed: the product kernel is
// scheduled while the first kernel finishes and waits for it
// (griddepcontrol.wait) before reading what it wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), int grid, int threads, int smem, cudaStream_t stream,
                             Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace

bool gemv_tc_eligible(const DeviceInfo &dev, const GemvArgs &g, bool any_size) {
    if (g.a_elem != 2 || g.batch < 3 || g.batch > 8 || !tc_supported(dev)) return false;
    // Where the CUDA-core kernel is faster: below 2^25 matrix elements (batch
    // 8, 4096^2: 11.7 against 13.1 us) and below batch 6, whose per-element
    // work it carries well (8192^2: batch 5 26.7 against 29.9 us, batch 6
    // 30.3 against 30.0 us; 16384^2: batch 4 84.0 against 90.5 us, batch 6
    // 118.5 against 90.7 us).
    if (!any_size && (g.M * g.N < (int64_t{1} << 25) || g.batch < 6)) return false;
    if ((reinterpret_cast<uintptr_t>(g.A) & 15) || (g.lda * 2) % 16) return false;   // TMA base and rows
    return g.M > 0 && g.N > 0 && g.M <= INT32_MAX - kBM && g.N <= INT32_MAX - kBK;
}

void gemv_tc_plan(const DeviceInfo &dev, const GemvArgs &g, gtg_plan *plan) {
    const long long tiles = (g.M + kBM - 1) / kBM, ks = (g.N + kBK - 1) / kBK;
    plan->kernel = GTG_KERNEL_TCGEN05;
    plan->bm = kBM;
    plan->bn = kNP;
    plan->bk = kBK;
    plan->stages = kStages;
    plan->grid = static_cast<int>(std::min<long long>(dev.sms, tiles * ks));
    plan->threads = kThreads;
    plan->smem = kSmem;
    plan->cluster = 1;
    plan->splits = 0;
}

cudaError_t gemv_tc_launch(const DeviceInfo &dev, const GemvArgs &g, cudaStream_t stream) {
    // the shared-memory attribute, once per device (setting it twice is harmless)
    static std::atomic<uint64_t> attr_done{0};
    const uint64_t bit = uint64_t{1} << (dev.id & 63);
    if (!(attr_done.load() & bit)) {
        const cudaError_t e = cudaFuncSetAttribute(gemv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(bit);
    }
    const long long tiles = (g.M + kBM - 1) / kBM, ks = (g.N + kBK - 1) / kBK;
    const long long work = tiles * ks;
    const int grid = static_cast<int>(std::min<long long>(dev.sms, work));
    // parts of one tile: at most ceil(ks / q) + 1 CTAs for ranges of >= q units
    const long long q = work / grid;
    const int maxp = static_cast<int>((ks + q - 1) / q + 1);
    const long long ldp = (g.N + 7) / 8 * 8;   // 16-byte rows of pieces
    const size_t xp_bytes = static_cast<size_t>(3 * g.batch * ldp) * 2;
    const size_t ws_bytes = static_cast<size_t>(tiles * maxp) * 8 * kBM * 4;
    const size_t cnt_bytes = static_cast<size_t>(tiles) * 4 * sizeof(int);
    void *xp = nullptr, *ws = nullptr, *cnt = nullptr;
    cudaError_t e = ws_alloc(&xp, xp_bytes, stream);
    if (e == cudaSuccess) e = ws_alloc(&ws, ws_bytes, stream);
    if (e == cudaSuccess) e = ws_alloc(&cnt, cnt_bytes, stream);
    CUtensorMap ta, tx;
    if (e == cudaSuccess && (!tma_map_2d(&ta, GTG_PREC_BF16, g.A, g.N, g.M, g.lda, kBK, kBM) ||
                             !tma_map_2d(&tx, GTG_PREC_BF16, xp, g.N, 3 * g.batch, ldp, kBK, kNP)))
        e = cudaErrorInvalidValue;
    if (e == cudaSuccess) {
        const long long n = g.batch * g.N;
        const int sgrid = static_cast<int>(std::min<long long>((n + 255) / 256, dev.sms * 8ll));
        e = launch_dependent(split_vectors_kernel, sgrid, 256, 0, stream, g.x, static_cast<long long>(g.ldx),
                             static_cast<int>(g.N), static_cast<int>(g.batch), static_cast<__nv_bfloat16 *>(xp),
                             static_cast<long long>(ldp), static_cast<int *>(cnt), static_cast<int>(tiles * 4));
    }
    if (e == cudaSuccess) {
        Params p;
        p.y = g.y;
        p.ldy = g.ldy;
        p.ws = static_cast<float *>(ws);
        p.cnt = static_cast<int *>(cnt);
        p.M = static_cast<int>(g.M);
        p.batch = static_cast<int>(g.batch);
        p.ks = static_cast<int>(ks);
        p.work = work;
        p.maxp = maxp;
        p.bias = g.bias;
        p.act = g.act;
        p.status = dev.status;
        p.wait_limit_ns = wait_limit_setting();
        p.drop_slice = take_test_drop_slice();
        e = launch_dependent(gemv_tc_kernel, grid, kThreads, kSmem, stream, ta, tx, p);
    }
    // stream-ordered: released after the kernels above have used them
    if (xp) cudaFreeAsync(xp, stream);
    if (ws) cudaFreeAsync(ws, stream);
    if (cnt) cudaFreeAsync(cnt, stream);
    return e;
}

}  // namespace gtg
