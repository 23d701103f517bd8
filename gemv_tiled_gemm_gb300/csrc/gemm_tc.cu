// Tensor-core GEMM for sm_103a: C (FP32) = A * B with BF16, FP16 or TF32 operands,
// one matrix or a strided batch of them.
//
// The tiling principle is the one of "GPU Matrix Multiplication: Tiling and
// Shared Memory" (section 3) and "CUDA Programming (6)" (section 3.2): each
// output tile is accumulated from K-slices of A and B staged in shared
// memory, out-of-range elements contributing zeros and out-of-range outputs
// not being stored. On GB300 the pieces are:
//
//   * staging: TMA tensor copies (128-byte swizzled) into a ring of STAGES
//     shared-memory slots, each guarded by a pair of mbarriers (full/empty)
//     instead of the pages' two __syncthreads per tile; the copy of slice
//     k+1.. overlaps the multiply of slice k (the pages' "Prefetching");
//     TMA fills out-of-bounds box elements with zeros (the pages' padding);
//   * multiply: tcgen05.mma issued by one thread, accumulating a 128 x BN
//     FP32 tile in tensor memory (TMEM); two accumulators so that the
//     epilogue of one tile overlaps the main loop of the next;
//   * epilogue: four warps read TMEM (tcgen05.ld, one row per thread) and
//     store the rows that exist (row < M, col < N);
//   * scheduling: a persistent grid (at most one CTA per SM) walks the
//     output tiles in groups of row-tiles for L2 reuse (the CTA-pair kernel:
//     odd groups walk the columns backwards and odd waves read K from its
//     end, so that each wave starts on the operand slices the previous one
//     read last).
//
// Operand layouts: A is row-major M x K, i.e. "K-major" for the MMA; B is
// row-major K x N, i.e. "MN-major". BF16 operands are read in their given
// layouts. The TF32 MMA does not take an MN-major B on this hardware (it
// leaves the accumulator untouched), so for TF32 a transpose kernel first
// writes B^T (N x K, K-major) into a temporary buffer taken from the
// device's stream-ordered memory pool, and both operands are then K-major.
//
// TF32 rounding: the TF32 MMA ignores the 13 low mantissa bits of its FP32
// operands (truncation, up to 2^-10 relative per operand, which with both
// operands reaches the 4 * 2^-11 * sum|a*b| error bound). So both operands
// are rounded to the nearest TF32 value first, by one preparation kernel that
// writes B^T and a rounded copy of A (16-byte rows, so any layout of A
// works) into pool buffers. The entry point without allocation has no room
// for the copy of A: its single-CTA kernel (ROUND_A) rounds each A tile in
// shared memory instead, with four converter warps between the tile's TMA
// load and the MMAs that read it. (Measured: that extra wait per K slice cost
// the CTA-pair kernel more than half its rate -- TF32 8192^3 950 -> 330
// TFLOP/s -- where the copy of A costs one more pass over A in HBM.)
//
// Every mbarrier wait is bounded in time. On expiry the waiting thread
// latches GTG_ERR_TIMEOUT in the library status word, raises a shared abort
// flag that makes the other roles stop, waits (bounded) for its own copies
// and MMAs in flight, and the CTA releases its TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace gtg {
namespace {

constexpr int kThreads = 192;  // warp 0 TMA, warp 1 MMA + TMEM owner, warps 2-5 epilogue
constexpr int kConvWarps = 4;  // ROUND_A kernels: warps 6-9 round A tiles to TF32 in shared memory
__host__ __device__ constexpr int threads_for(bool round_a) { return round_a ? kThreads + 32 * kConvWarps : kThreads; }
constexpr int kBM = 128;
constexpr int kGroup = 16;     // row-tiles per raster group
constexpr int kSmemBudget = 200 * 1024;

template <bool TF32, int BN_>
struct Shape {
    static constexpr int BN = BN_;
    static constexpr int ELEM = TF32 ? 4 : 2;
    static constexpr int BM = kBM;
    static constexpr int BK = 128 / ELEM;          // K elements in one 128-byte row
    static constexpr int UK = 32 / ELEM;           // K per tcgen05.mma
    static constexpr int KSTEPS = BK / UK;
    static constexpr int A_BYTES = BM * 128;       // BM rows x 128 bytes of K
    static constexpr bool B_KMAJOR = TF32;         // B staged from its transpose
    static constexpr int BCH_N = 128 / ELEM;       // N elements per 128-byte row of B (MN-major)
    static constexpr int B_CHUNKS = B_KMAJOR ? 1 : BN / BCH_N;
    static constexpr int BCH_BYTES = BK * 128;     // one 128-byte-wide column block of B (MN-major)
    static constexpr int B_BYTES = BN * BK * ELEM; // = BN rows x 128 bytes when K-major
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES_RAW = kSmemBudget / STAGE_BYTES;
    static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
    static constexpr int TMEM_COLS = 2 * BN;       // two FP32 accumulators
    static constexpr int NBARS = (TF32 ? 3 : 2) * STAGES + 5;   // TF32: a "converted" barrier per stage
    static constexpr int SMEM = 1024 /*alignment slack*/ + STAGES * STAGE_BYTES + NBARS * 8 + 16;
    static constexpr uint32_t IDESC = ptx::make_idesc(TF32 ? 2u : 1u, 0u, B_KMAJOR ? 0u : 1u, BM, BN);
    static_assert(BN % BCH_N == 0 && BN >= 64 && BN <= 256, "tile width");
    static_assert(B_KMAJOR || B_CHUNKS * BCH_BYTES == B_BYTES, "MN-major B is whole column blocks");
    static_assert(STAGE_BYTES % 1024 == 0, "stages keep 1024-byte alignment");
    static_assert(TMEM_COLS >= 32 && TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0,
                  "TMEM allocation must be a power of two in [32, 512]");
};

struct TcParams {
    float *C;
    long long ldc;
    int M, N;
    int num_m, num_n, num_kb, num_tiles;   // num_tiles counts every item of a batch
    int tiles_per_batch;
    int splits, kps;             // K split into `splits` ranges of kps slices (1: none)
    int num_units;               // num_tiles * splits, plus the extra halves of a split tail
    int tail_start;              // pair kernel: units from here on are 128-wide halves of the last tiles
    long long strideC;           // elements between the C matrices of consecutive batch items
    uint32_t idesc;              // instruction descriptor (A/B format: FP16 or BF16) of the 16-bit kernels
    int c_vec;                   // widest store for whole rows of a tile: 2 = 32 B, 1 = 16 B, 0 = 4 B
    int c_tma;                   // pair kernel: C written by tensor stores of 32 x 32 blocks (tmC)
    int *status;
    unsigned long long wait_limit_ns;
    int drop_slice;              // testing hook: K slice whose load CTA 0 never issues (-1: none)
    const float *bias;           // epilogue: C = act(acc + bias[col]); null for none
    int act;
    // implicit-GEMM convolution (A read from the image by TMA im2col loads):
    // output width and height, 64-channel blocks per pixel, window width,
    // strides, paddings, dilations
    int cv_ow, cv_oh, cv_cb, cv_kw, cv_sw, cv_sh, cv_pw, cv_ph, cv_dw, cv_dh;
};

// Apply the layer epilogue to 32 accumulator columns starting at column col.
__device__ __forceinline__ void epilogue32(uint32_t (&r)[32], const TcParams &p, int col) {
    if (p.bias == nullptr && p.act == 0) return;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const bool in = col + j < p.N;
        const float v = apply_epilogue(__uint_as_float(r[j]), in ? p.bias : nullptr, col + j, p.act);
        r[j] = __float_as_uint(v);
    }
}

// Work unit t of a launch: a tile (batch item bi, index tt within the item)
// and its K-slice range [kb0, kb1). With p.splits > 1 (never together with a
// batch) unit t is K range s = t / num_tiles of tile t % num_tiles and its
// partial tile goes to slab s of the workspace (coff = s * strideC), to be
// added in order by the split reduction.
struct Unit {
    int bi, tt, kb0, kb1;
    long long coff;
};

__device__ __forceinline__ Unit unit_of(int t, const TcParams &p) {
    Unit u;
    int s = 0;
    if (p.splits > 1) {
        s = t / p.num_tiles;
        t -= s * p.num_tiles;
    }
    u.bi = t / p.tiles_per_batch;
    u.tt = t - u.bi * p.tiles_per_batch;
    u.kb0 = s * p.kps;
    u.kb1 = min(u.kb0 + p.kps, p.num_kb);
    u.coff = static_cast<long long>(p.splits > 1 ? s : u.bi) * p.strideC;
    return u;
}

__device__ __forceinline__ void tile_coords(int t, const TcParams &p, int &mb, int &nb) {
    const int per_group = kGroup * p.num_n;
    const int g = t / per_group;
    const int first = g * kGroup;
    const int gs = min(p.num_m - first, kGroup);
    const int r = t - g * per_group;
    mb = first + r % gs;
    nb = r / gs;
}

// Bounded wait used by the pipeline roles. Returns false if this CTA must stop.
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                       const TcParams &p) {
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

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                         const TcParams &p) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, abort_flag, p);
}

// Wait that ignores the abort flag: used only to let work already in flight
// finish before shared memory or TMEM is released. Bounded as well.
__device__ __noinline__ void wait_drain(uint32_t bar, uint32_t parity, const TcParams &p) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer_ns() - t0 > p.wait_limit_ns) {
            atomicCAS(p.status, 0, static_cast<int>(GTG_ERR_TIMEOUT));
            return;
        }
    }
}

// Rounds BYTES of FP32 values in shared memory at `addr` to TF32 in place
// (one warp; every lane loads all its 16-byte pieces first, then rounds and
// stores them), then orders the writes before the tensor cores' reads.
template <int BYTES>
__device__ __forceinline__ void round_tile_tf32(uint32_t addr, int lane) {
    constexpr int kPieces = BYTES / (32 * 16);
    static_assert(kPieces * 32 * 16 == BYTES, "whole 512-byte passes");
    uint4 v[kPieces];
#pragma unroll
    for (int i = 0; i < kPieces; ++i) v[i] = ptx::ld_shared_v4(addr + (i * 32 + lane) * 16);
#pragma unroll
    for (int i = 0; i < kPieces; ++i)
        ptx::st_shared_v4(addr + (i * 32 + lane) * 16, ptx::tf32_round(v[i].x), ptx::tf32_round(v[i].y),
                          ptx::tf32_round(v[i].z), ptx::tf32_round(v[i].w));
    ptx::fence_proxy_async_smem();
}

// A bounded wait that every lane of a warp makes and that ends the same way
// for all of them (so that the warp never diverges on an abort).
__device__ __forceinline__ bool warp_wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                              const TcParams &p) {
    const bool ok = wait_bar(bar, parity, abort_flag, p);
    return __all_sync(0xFFFFFFFFu, ok);
}

// IM2COL: A is not a matrix in memory but the patch matrix of a convolution
// (rows = output pixels in (n, oh, ow) order, K = (kh, kw, channel)); each
// 128 x 64 A tile is one TMA im2col load of 128 output pixels' 64 channels
// at one window tap, straight from the channels-last image.
//
// ROUND_A (TF32 only, the entry point without allocation): A is the caller's
// matrix, not yet rounded; warps 6-9 round each A tile in shared memory to
// TF32 before the MMAs of its stage may read it.
template <bool TF32, int BN, bool IM2COL = false, bool ROUND_A = false>
__global__ void __launch_bounds__(threads_for(ROUND_A), 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const TcParams p) {
    static_assert(!ROUND_A || TF32, "only TF32 operands are rounded");
    using S = Shape<TF32, BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sA = ptx::smem_addr(smem);
    const uint32_t sB = sA + S::STAGES * S::A_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::STAGES * S::STAGE_BYTES);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + S::NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const uint32_t bar0 = ptx::smem_addr(bars);
    // barrier map: full[s] = s, empty[s] = STAGES + s, acc_full[a] = 2*STAGES + a,
    // acc_empty[a] = 2*STAGES + 2 + a, drain = 2*STAGES + 4, TF32: conv[s] = 2*STAGES + 5 + s
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S::STAGES + s); };
    auto accf_bar = [&](int a) { return bar0 + 8u * (2 * S::STAGES + a); };
    auto acce_bar = [&](int a) { return bar0 + 8u * (2 * S::STAGES + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * S::STAGES + 4);
    auto conv_bar = [&](int s) { return bar0 + 8u * (2 * S::STAGES + 5 + s); };
    // the MMAs of a stage wait for its A tile rounded (ROUND_A) or just loaded
    auto ready_bar = [&](int s) { return ROUND_A ? conv_bar(s) : full_bar(s); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S::STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
            if constexpr (ROUND_A) ptx::mbar_init(conv_bar(s), kConvWarps);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(accf_bar(a), 1);
            ptx::mbar_init(acce_bar(a), 4);  // one arrive per epilogue warp
        }
        ptx::mbar_init(drain_bar, 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), S::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // set-up above overlaps the previous kernel's tail (dependent launch);
    // no global memory is touched before that kernel has completed
    ptx::wait_prior_grid();
    ptx::allow_next_grid();

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t it = 0;  // slices issued so far
            bool ok = true;
            for (int t = blockIdx.x; ok && t < p.num_units; t += gridDim.x) {
                int mb, nb;
                const Unit u = unit_of(t, p);
                const int bi = u.bi;
                tile_coords(u.tt, p, mb, nb);
                int w0 = 0, h0 = 0, n0 = 0;   // IM2COL: window corner of the tile's first output pixel
                if constexpr (IM2COL) {
                    const int m0 = mb * S::BM;
                    const int q = m0 / p.cv_ow;
                    w0 = (m0 - q * p.cv_ow) * p.cv_sw - p.cv_pw;
                    h0 = (q % p.cv_oh) * p.cv_sh - p.cv_ph;
                    n0 = q / p.cv_oh;
                }
                for (int kb = u.kb0; kb < u.kb1; ++kb, ++it) {
                    const int s = static_cast<int>(it % S::STAGES);
                    const uint32_t ph = (it / S::STAGES) & 1u;
                    if (!wait_bar(empty_bar(s), ph ^ 1u, abort_flag, p)) {
                        ok = false;
                        break;
                    }
                    if (p.drop_slice == static_cast<int>(it) && blockIdx.x == 0) continue;
                    ptx::mbar_arrive_expect_tx(full_bar(s), S::STAGE_BYTES);
                    if constexpr (IM2COL) {
                        // K slice kb = (kh, kw, channel block cb)
                        const int tap = kb / p.cv_cb, cb = kb - tap * p.cv_cb;
                        const int kh = tap / p.cv_kw, kw = tap - kh * p.cv_kw;
                        ptx::tma_load_im2col_4d(sA + s * S::A_BYTES, &tmA, full_bar(s), cb * S::BK, w0, h0, n0,
                                                static_cast<uint16_t>(kw * p.cv_dw), static_cast<uint16_t>(kh * p.cv_dh));
                    } else {
                        ptx::tma_load_3d(sA + s * S::A_BYTES, &tmA, full_bar(s), kb * S::BK, mb * S::BM, bi);
                    }
                    if constexpr (S::B_KMAJOR) {
                        // B^T tile: BN rows of BK elements
                        ptx::tma_load_3d(sB + s * S::B_BYTES, &tmB, full_bar(s), kb * S::BK, nb * BN, bi);
                    } else {
#pragma unroll
                        for (int c = 0; c < S::B_CHUNKS; ++c)
                            ptx::tma_load_3d(sB + s * S::B_BYTES + c * S::BCH_BYTES, &tmB, full_bar(s),
                                             nb * BN + c * S::BCH_N, kb * S::BK, bi);
                    }
                }
            }
            if (!ok) {
                // let the copies already issued land before the CTA exits
                const uint32_t n = it < S::STAGES ? it : S::STAGES;
                for (uint32_t j = 1; j <= n; ++j) {
                    const uint32_t i = it - j;
                    wait_drain(full_bar(static_cast<int>(i % S::STAGES)), (i / S::STAGES) & 1u, p);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t it = 0;
            int local = 0;
            bool ok = true, issued = false;
            for (int t = blockIdx.x; ok && t < p.num_units; t += gridDim.x, ++local) {
                const int acc = local & 1;
                const uint32_t aph = (static_cast<uint32_t>(local) >> 1) & 1u;
                if (!wait_bar(acce_bar(acc), aph ^ 1u, abort_flag, p)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                const Unit u = unit_of(t, p);
                for (int kb = u.kb0; kb < u.kb1; ++kb, ++it) {
                    const int s = static_cast<int>(it % S::STAGES);
                    const uint32_t ph = (it / S::STAGES) & 1u;
                    if (!wait_bar(ready_bar(s), ph, abort_flag, p)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    const uint32_t a0 = sA + s * S::A_BYTES;
                    const uint32_t b0 = sB + s * S::B_BYTES;
#pragma unroll
                    for (int k = 0; k < S::KSTEPS; ++k) {
                        // A, K-major, 128B swizzle: 8-row groups 1024 B apart; the K
                        // step moves the start by 32 bytes inside the swizzle row.
                        const uint64_t ad = ptx::smem_desc_sw128(a0 + k * 32, 16, 1024);
                        // B, MN-major, 128B swizzle: 128-byte-wide column blocks BCH_BYTES
                        // apart (leading offset), 8-row K groups 1024 B apart (stride
                        // offset); the K step moves UK rows of 128 bytes. K-major B
                        // (TF32) is laid out like A.
                        const uint64_t bd = S::B_KMAJOR
                                                ? ptx::smem_desc_sw128(b0 + k * 32, 16, 1024)
                                                : ptx::smem_desc_sw128(b0 + k * S::UK * 128, S::BCH_BYTES, 1024);
                        const uint32_t accum = (kb > u.kb0 || k > 0) ? 1u : 0u;
                        if constexpr (TF32)
                            ptx::mma_tf32(d_tmem, ad, bd, S::IDESC, accum);
                        else
                            ptx::mma_bf16(d_tmem, ad, bd, p.idesc, accum);
                    }
                    ptx::mma_commit(empty_bar(s));  // slot free once these MMAs have read it
                    issued = true;
                }
                if (!ok) break;
                ptx::mma_commit(accf_bar(acc));     // accumulator ready for the epilogue
            }
            if (issued) {
                // nothing may still be writing TMEM when it is released
                ptx::mma_commit(drain_bar);
                wait_drain(drain_bar, 0u, p);
            }
        }
    } else if (warp >= 6) {
        // ------------------------------------------------ ROUND_A: A tiles rounded in place (warps 6-9)
        if constexpr (ROUND_A) {
            constexpr int kPart = S::A_BYTES / kConvWarps;
            uint32_t it = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < p.num_units; t += gridDim.x) {
                const Unit u = unit_of(t, p);
                for (int kb = u.kb0; kb < u.kb1; ++kb, ++it) {
                    const int s = static_cast<int>(it % S::STAGES);
                    const uint32_t ph = (it / S::STAGES) & 1u;
                    if (!warp_wait_bar(full_bar(s), ph, abort_flag, p)) {
                        ok = false;
                        break;
                    }
                    round_tile_tf32<kPart>(sA + s * S::A_BYTES + (warp - 6) * kPart, lane);
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(conv_bar(s));
                }
            }
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..5)
        const int quarter = warp & 3;  // TMEM lanes this warp may access
        const int r_in_tile = quarter * 32 + lane;
        int local = 0;
        for (int t = blockIdx.x; t < p.num_units; t += gridDim.x, ++local) {
            int mb, nb;
            const Unit u = unit_of(t, p);
            tile_coords(u.tt, p, mb, nb);
            const int acc = local & 1;
            const uint32_t aph = (static_cast<uint32_t>(local) >> 1) & 1u;
            if (!wait_bar(accf_bar(acc), aph, abort_flag, p)) break;
            ptx::tc_fence_after_sync();
            const int row = mb * S::BM + r_in_tile;
            const int col0 = nb * BN;
            const bool row_ok = row < p.M;
            const bool whole = p.c_vec && (col0 + BN <= p.N);
            float *crow = p.C + u.coff + static_cast<long long>(row) * p.ldc + col0;
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * BN);
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                ptx::tmem_ld_32x32b_x32(taddr + c * 32, r);
                ptx::tmem_ld_wait();
                epilogue32(r, p, col0 + c * 32);
                if (row_ok) {
                    if (whole && p.c_vec == 2) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) ptx::st_global_v8(crow + c * 32 + 8 * j, r + 8 * j);
                    } else if (whole) {
                        float4 *dst = reinterpret_cast<float4 *>(crow + c * 32);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                                 __uint_as_float(r[4 * j + 2]),
                                                 __uint_as_float(r[4 * j + 3]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (col0 + c * 32 + j < p.N) crow[c * 32 + j] = __uint_as_float(r[j]);
                    }
                }
            }
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(acce_bar(acc));
        }
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem_base, S::TMEM_COLS);
    }
}

// ---------------------------------------------------------------- CTA-pair kernel
// Two CTAs of a cluster share one 256 x 256 output tile: each stages its own
// 128 rows of A and its half (128 columns) of B, and one thread of the even
// CTA issues tcgen05.mma.cta_group::2 (M = 256), which reads A and B half from
// each CTA's shared memory and writes each CTA's 128 rows of D into that CTA's
// TMEM. Per SM this moves 32 KB per 128-byte-deep K slice instead of 48 KB for
// the same multiply work, so six stages fit and operand delivery keeps up.
// 16-bit B is staged MN-major (two 64-column blocks per CTA); TF32 B is staged
// from its transpose, K-major like A (128 rows of B^T per CTA).
//
// Synchronisation across the pair: both CTAs' TMA loads complete on the even
// CTA's full barrier (which expects both CTAs' bytes); the MMA thread's
// commits are multicast to the empty / accumulator-full barriers of both
// CTAs; both CTAs' epilogue warps arrive on the even CTA's accumulator-empty
// barrier. A cluster barrier after set-up and before exit keeps either CTA
// from touching a peer that has not initialised its barriers or has left.
template <bool TF32>
struct PairShape {
    static constexpr int ELEM = TF32 ? 4 : 2;
    static constexpr int BM = 128;                 // rows per CTA (256 per pair)
    static constexpr int BN = 256;                 // columns per pair tile
    static constexpr int BK = 128 / ELEM;          // K elements in one 128-byte row
    static constexpr int UK = 32 / ELEM;           // K per tcgen05.mma
    static constexpr int KSTEPS = BK / UK;
    static constexpr int A_BYTES = BM * 128;       // 16 KB
    static constexpr bool B_KMAJOR = TF32;
    static constexpr int BCH_N = 128 / ELEM;       // MN-major B: columns per 128-byte block
    static constexpr int B_CHUNKS = B_KMAJOR ? 1 : (BN / 2) / BCH_N;
    static constexpr int BCH_BYTES = BK * 128;     // MN-major B: one column block, 8 KB
    static constexpr int B_BYTES = (BN / 2) * 128; // this CTA's half of B: 16 KB either way
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;   // 32 KB per CTA
    static constexpr int STAGES = 6;
    static constexpr int TMEM_COLS = 2 * BN;
    // epilogue staging for tensor stores: per epilogue warp two 32 x 32 FP32
    // blocks (4 KB each, 128-byte swizzled rows)
    static constexpr int EPI_BYTES = 4 * 2 * 32 * 128;
    static constexpr int NBARS = 2 * STAGES + 5;
    static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + NBARS * 8 + 16;
    static_assert(B_KMAJOR || B_CHUNKS * BCH_BYTES == B_BYTES, "MN-major B is whole column blocks");
};

// Raster of the pair kernel's tiles: groups of kPairGroup pair row-tiles,
// each walked column by column (a wave of 76 clusters covers 12 row-tiles x
// about 6 column-tiles), odd groups walking the columns right to left so that
// a group starts on the B columns the previous one ended on. With the K order
// alternating from wave to wave (see the producer), a wave starts on the A
// and B slices the previous wave read last. DRAM reads per BF16 8192^3
// launch (ncu): 1.086 GB with groups of 8 walked left to right, 0.873 with
// both reversals, 0.826 = 3.08 x (A + B) with groups of 12 (groups of 4 / 6 /
// 10 / 11 / 13 / 14 / 16: 1.106 / 1.000 / 0.915 / 0.854 / 0.881 / 0.896 /
// 0.911 GB).
constexpr int kPairGroup = 12;

__device__ __forceinline__ void pair_tile_coords(int t, const TcParams &p, int &mb, int &nb) {
    const int per_group = kPairGroup * p.num_n;
    const int g = t / per_group;
    const int first = g * kPairGroup;
    const int gs = min(p.num_m - first, kPairGroup);
    const int r = t - g * per_group;
    mb = first + r % gs;
    nb = r / gs;
    if (g & 1) nb = p.num_n - 1 - nb;
}

// Tile of pair-kernel unit tt: row tile mb, first column c0 and width w.
// Units before p.tail_start are whole 256 x 256 tiles in raster order; from
// there on each remaining tile is two units, its 128-column halves, so that
// a last wave that would leave clusters idle runs as a wave of half tiles.
__device__ __forceinline__ void pair_tile(int tt, const TcParams &p, int &mb, int &c0, int &w) {
    int tile = tt, half = -1;
    if (tt >= p.tail_start) {
        tile = p.tail_start + (tt - p.tail_start) / 2;
        half = (tt - p.tail_start) & 1;
    }
    int nb;
    pair_tile_coords(tile, p, mb, nb);
    c0 = nb * 256 + (half > 0 ? 128 : 0);
    w = half >= 0 ? 128 : 256;
}

__device__ __noinline__ void spin_ns(uint64_t ns) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (ptx::globaltimer_ns() - t0 < ns) {
    }
}

// IM2COL: A is the patch matrix of a convolution, each CTA's 128 rows of a K
// slice one TMA im2col load from the channels-last image (for TF32, the
// rounded copy of it), as in the single-CTA kernel.
template <bool TF32, bool IM2COL = false>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const TcParams p) {
    using S = PairShape<TF32>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sA = ptx::smem_addr(smem);
    const uint32_t sB = sA + S::STAGES * S::A_BYTES;
    const uint32_t sEpi = sA + S::STAGES * S::STAGE_BYTES;   // 1024-aligned
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::STAGES * S::STAGE_BYTES + S::EPI_BYTES);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + S::NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const uint32_t bar0 = ptx::smem_addr(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S::STAGES + s); };
    auto accf_bar = [&](int a) { return bar0 + 8u * (2 * S::STAGES + a); };
    auto acce_bar = [&](int a) { return bar0 + 8u * (2 * S::STAGES + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * S::STAGES + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const bool leader = rank == 0;
    const int cluster_id = static_cast<int>(blockIdx.x >> 1);
    const int nclusters = static_cast<int>(gridDim.x >> 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S::STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(accf_bar(a), 1);
            ptx::mbar_init(acce_bar(a), 8);  // 4 epilogue warps in each CTA of the pair
        }
        ptx::mbar_init(drain_bar, 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmB);
        if (p.c_tma) ptx::prefetch_tensormap(&tmC);
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(ptx::smem_addr(tmem_slot), S::TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::cluster_sync();
    ptx::tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    ptx::wait_prior_grid();
    ptx::allow_next_grid();

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            const uint32_t leader_full0 = ptx::map_to_rank(full_bar(0), 0);
            uint32_t it = 0;
            bool ok = true;
            for (int t = cluster_id; ok && t < p.num_units; t += nclusters) {
                int mb, c0, w;
                const Unit u = unit_of(t, p);
                const int bi = u.bi;
                pair_tile(u.tt, p, mb, c0, w);
                const int row0 = mb * 2 * S::BM + static_cast<int>(rank) * S::BM;
                const int col0 = c0 + static_cast<int>(rank) * (w / 2);
                int w0 = 0, h0 = 0, n0 = 0;   // IM2COL: window corner of this CTA's first output pixel
                if constexpr (IM2COL) {
                    const int q = row0 / p.cv_ow;
                    w0 = (row0 - q * p.cv_ow) * p.cv_sw - p.cv_pw;
                    h0 = (q % p.cv_oh) * p.cv_sh - p.cv_ph;
                    n0 = q / p.cv_oh;
                }
                // both CTAs' A rows and B halves: (16 KB + w/2 columns x 128 B) each
                const uint32_t stage_tx = 2u * static_cast<uint32_t>(S::A_BYTES + (w / 2) * 128);
                // odd waves read K from the end (the MMA only needs slices in
                // matching pairs; accumulation order stays fixed per tile)
                const bool rev = ((t - cluster_id) / nclusters) & 1;
                for (int ki = u.kb0; ki < u.kb1; ++ki, ++it) {
                    const int kb = rev ? u.kb1 - 1 - (ki - u.kb0) : ki;
                    const int s = static_cast<int>(it % S::STAGES);
                    const uint32_t ph = (it / S::STAGES) & 1u;
                    if (!wait_bar(empty_bar(s), ph ^ 1u, abort_flag, p)) {
                        ok = false;
                        break;
                    }
                    if (p.drop_slice == static_cast<int>(it) && cluster_id == 0 && leader) continue;
                    if (leader) ptx::mbar_arrive_expect_tx(full_bar(s), stage_tx);
                    const uint32_t fb = leader_full0 + 8u * s;
                    if constexpr (IM2COL) {
                        // K slice kb = (kh, kw, channel block cb)
                        const int tap = kb / p.cv_cb, cb = kb - tap * p.cv_cb;
                        const int kh = tap / p.cv_kw, kw = tap - kh * p.cv_kw;
                        ptx::tma_load_im2col_4d_pair(sA + s * S::A_BYTES, &tmA, fb, cb * S::BK, w0, h0, n0,
                                                     static_cast<uint16_t>(kw * p.cv_dw),
                                                     static_cast<uint16_t>(kh * p.cv_dh));
                    } else {
                        ptx::tma_load_3d_pair(sA + s * S::A_BYTES, &tmA, fb, kb * S::BK, row0, bi);
                    }
                    if constexpr (S::B_KMAJOR) {
                        // this CTA's 128 rows of B^T
                        ptx::tma_load_3d_pair(sB + s * S::B_BYTES, &tmB, fb, kb * S::BK, col0, bi);
                    } else {
                        for (int c = 0; c < (w / 2) / S::BCH_N; ++c)
                            ptx::tma_load_3d_pair(sB + s * S::B_BYTES + c * S::BCH_BYTES, &tmB, fb,
                                                  col0 + c * S::BCH_N, kb * S::BK, bi);
                    }
                }
            }
            if (!ok) {
                if (leader) {
                    const uint32_t n = it < S::STAGES ? it : S::STAGES;
                    for (uint32_t j = 1; j <= n; ++j) {
                        const uint32_t i = it - j;
                        wait_drain(full_bar(static_cast<int>(i % S::STAGES)), (i / S::STAGES) & 1u, p);
                    }
                } else {
                    // this CTA's copies complete on the even CTA's barrier, which it
                    // cannot wait on; give them ample time to land
                    spin_ns(200000);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (even CTA only)
        if (leader && lane == 0) {
            uint32_t it = 0;
            int local = 0;
            bool ok = true;
            for (int t = cluster_id; ok && t < p.num_units; t += nclusters, ++local) {
                const int acc = local & 1;
                const uint32_t aph = (static_cast<uint32_t>(local) >> 1) & 1u;
                if (!wait_bar(acce_bar(acc), aph ^ 1u, abort_flag, p)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * S::BN);
                const Unit u = unit_of(t, p);
                int mb, c0, w;
                pair_tile(u.tt, p, mb, c0, w);
                // the instruction descriptor's N (bits 17-22, N / 8) for this unit's width
                const uint32_t idesc = (p.idesc & ~(0x3Fu << 17)) | (static_cast<uint32_t>(w >> 3) << 17);
                for (int kb = u.kb0; kb < u.kb1; ++kb, ++it) {   // K order does not matter here: the stages hold it
                    const int s = static_cast<int>(it % S::STAGES);
                    const uint32_t ph = (it / S::STAGES) & 1u;
                    if (!wait_bar(full_bar(s), ph, abort_flag, p)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    const uint32_t a0 = sA + s * S::A_BYTES;
                    const uint32_t b0 = sB + s * S::B_BYTES;
#pragma unroll
                    for (int k = 0; k < S::KSTEPS; ++k) {
                        const uint64_t ad = ptx::smem_desc_sw128(a0 + k * 32, 16, 1024);
                        const uint64_t bd = S::B_KMAJOR
                                                ? ptx::smem_desc_sw128(b0 + k * 32, 16, 1024)
                                                : ptx::smem_desc_sw128(b0 + k * S::UK * 128, S::BCH_BYTES, 1024);
                        const uint32_t accum = (kb > u.kb0 || k > 0) ? 1u : 0u;
                        if constexpr (TF32)
                            ptx::mma_tf32_pair(d_tmem, ad, bd, idesc, accum);
                        else
                            ptx::mma_bf16_pair(d_tmem, ad, bd, idesc, accum);
                    }
                    ptx::mma_commit_pair(empty_bar(s), 0x3);
                }
                if (!ok) break;
                ptx::mma_commit_pair(accf_bar(acc), 0x3);
            }
            // both CTAs release TMEM only after every MMA writing it has landed
            ptx::mma_commit_pair(drain_bar, 0x3);
        }
    } else {
        // ------------------------------------------------ epilogue (both CTAs)
        const int quarter = warp & 3;
        const int r_in_tile = quarter * 32 + lane;
        const uint32_t leader_acce0 = ptx::map_to_rank(acce_bar(0), 0);
        int local = 0;
        uint32_t epi_chunks = 0;   // tensor-store blocks issued by this warp
        for (int t = cluster_id; t < p.num_units; t += nclusters, ++local) {
            int mb, col0, w;
            const Unit u = unit_of(t, p);
            pair_tile(u.tt, p, mb, col0, w);
            const int acc = local & 1;
            const uint32_t aph = (static_cast<uint32_t>(local) >> 1) & 1u;
            if (!wait_bar(accf_bar(acc), aph, abort_flag, p)) break;
            ptx::tc_fence_after_sync();
            const int row = mb * 2 * S::BM + static_cast<int>(rank) * S::BM + r_in_tile;
            const bool row_ok = row < p.M;
            const bool whole = p.c_vec && (col0 + w <= p.N);
            float *crow = p.C + u.coff + static_cast<long long>(row) * p.ldc + col0;
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * S::BN);
            if (p.c_tma) {
                // each 32 x 32 block (this warp's 32 rows) goes through a swizzled
                // shared-memory buffer to a tensor store, which clips at the
                // edges of C; two buffers per warp alternate
                const int row0 = mb * 2 * S::BM + static_cast<int>(rank) * S::BM + quarter * 32;
#pragma unroll 1
                for (int c = 0; c < w / 32; ++c) {
                    uint32_t r[32];
                    ptx::tmem_ld_32x32b_x32(taddr + c * 32, r);
                    ptx::tmem_ld_wait();
                    epilogue32(r, p, col0 + c * 32);
                    const uint32_t buf = sEpi + static_cast<uint32_t>((quarter * 2 + (epi_chunks & 1)) * 4096);
                    if (lane == 0) ptx::bulk_wait_read<1>();   // the store that last used this buffer has read it
                    __syncwarp();
                    const uint32_t rowp = buf + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        ptx::st_shared_v4(rowp + (static_cast<uint32_t>(j ^ (lane & 7)) << 4), r[4 * j], r[4 * j + 1],
                                          r[4 * j + 2], r[4 * j + 3]);
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        ptx::tma_store_3d(&tmC, buf, col0 + c * 32, row0, u.bi);
                        ptx::bulk_commit();
                    }
                    ++epi_chunks;
                }
                ptx::tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive_cluster(leader_acce0 + 8u * acc);
                continue;
            }
#pragma unroll 1
            for (int c = 0; c < w / 32; ++c) {
                uint32_t r[32];
                ptx::tmem_ld_32x32b_x32(taddr + c * 32, r);
                ptx::tmem_ld_wait();
                epilogue32(r, p, col0 + c * 32);
                if (row_ok) {
                    if (whole && p.c_vec == 2) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) ptx::st_global_v8(crow + c * 32 + 8 * j, r + 8 * j);
                    } else if (whole) {
                        float4 *dst = reinterpret_cast<float4 *>(crow + c * 32);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                                 __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (col0 + c * 32 + j < p.N) crow[c * 32 + j] = __uint_as_float(r[j]);
                    }
                }
            }
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_cluster(leader_acce0 + 8u * acc);
        }
    }

    // every tensor store has read its shared-memory block before the CTA exits
    if (p.c_tma && warp >= 2 && lane == 0) ptx::bulk_wait_read<0>();
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        if (lane == 0) wait_drain(drain_bar, 0u, p);
        __syncwarp();
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc_pair(tmem_base, S::TMEM_COLS);
    }
    __syncwarp();
    ptx::cluster_sync();
}

__device__ __forceinline__ float tf32_rounded(float v) { return __uint_as_float(ptx::tf32_round(__float_as_uint(v))); }

// B (K x N, leading dimension ldb) -> Bt (N x K, leading dimension ldbt, a
// multiple of 4) with every value rounded to the nearest TF32 value (the
// operand the TF32 MMA reads), through a 64 x 64 shared-memory tile. VEC: B's rows are
// 16-byte aligned (base and ldb), so every thread moves 16-byte pieces both
// ways (a row of B or Bt is 16 of them per tile); edges of the matrix take
// single elements. blockIdx.z walks the items of a batch (strideB apart in
// B, N * ldbt apart in Bt).
// One 64 x 64 tile of B^T: rows n0.. of Bt, columns k0.. (a whole CTA of 256
// threads; every thread reaches both barriers).
template <bool VEC>
__device__ __forceinline__ void transpose_tile(const float *__restrict__ B, long long ldb, float *__restrict__ Bt,
                                               long long ldbt, int K, int N, int n0, int k0, float (&tile)[64][65],
                                               int *status) {
#ifdef GTG_DEBUG
    // this item's B (K rows of ldb) and Bt (N rows of ldbt)
    const float *b_hi = B + (static_cast<long long>(K) - 1) * ldb + N, *bt_hi = Bt + static_cast<long long>(N) * ldbt;
#endif
    (void)status;
    {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int idx = static_cast<int>(threadIdx.x) + 256 * i;
            const int r = idx >> 4, c = (idx & 15) * 4;   // row k0 + r, columns n0 + c .. + 3
            const int k = k0 + r, n = n0 + c;
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            if (k < K) {
                const float *src = B + static_cast<long long>(k) * ldb + n;
                if (VEC && n + 3 < N && GTG_DEBUG_IN(src, 16, B, b_hi, status)) {
                    const float4 q = __ldg(reinterpret_cast<const float4 *>(src));
                    v[0] = q.x;
                    v[1] = q.y;
                    v[2] = q.z;
                    v[3] = q.w;
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (n + j < N && GTG_DEBUG_IN(src + j, 4, B, b_hi, status)) v[j] = __ldg(src + j);
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) tile[r][c + j] = v[j];
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int idx = static_cast<int>(threadIdx.x) + 256 * i;
            const int r = idx >> 4, c = (idx & 15) * 4;   // row n0 + r of Bt, columns k0 + c .. + 3
            const int n = n0 + r, k = k0 + c;
            if (n < N && k < K) {
                float *dst = Bt + static_cast<long long>(n) * ldbt + k;
                if (!GTG_DEBUG_IN(dst, 4ull * min(4, K - k), Bt, bt_hi, status)) {
                } else if (k + 3 < K) {
                    *reinterpret_cast<float4 *>(dst) = make_float4(tf32_rounded(tile[c][r]), tf32_rounded(tile[c + 1][r]),
                                                                   tf32_rounded(tile[c + 2][r]),
                                                                   tf32_rounded(tile[c + 3][r]));
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (k + j < K) dst[j] = tf32_rounded(tile[c + j][r]);
                }
            }
        }
        __syncthreads();
    }
}

template <bool VEC>
__global__ void __launch_bounds__(256) transpose_kernel(const float *__restrict__ B, long long ldb,
                                                        float *__restrict__ Bt, long long ldbt, int K, int N,
                                                        long long strideB, int *status) {
    __shared__ float tile[64][65];
    // the GEMM that reads Bt is a dependent launch: it may be scheduled now and
    // set itself up, and it waits for this grid before touching Bt
    ptx::allow_next_grid();
    B += blockIdx.z * strideB;
    Bt += blockIdx.z * static_cast<long long>(N) * ldbt;
    for (int k0 = blockIdx.y * 64; k0 < K; k0 += gridDim.y * 64)
        transpose_tile<VEC>(B, ldb, Bt, ldbt, K, N, blockIdx.x * 64, k0, tile, status);
}

// Both TF32 operands prepared by one launch: blocks [0, tiles_n * tiles_k)
// each write one 64 x 64 tile of B^T, the others copy rows of A into A'
// (rows of ldk >= K elements, zero past K, 16-byte aligned, so that any
// layout of A works), every value rounded to the nearest TF32 value.
// blockIdx.y walks the items of a batch; an operand shared by every item
// (item stride 0) is prepared once (items_a or items_b = 1).
struct Tf32Prep {
    const float *A;
    long long lda, strideA;
    float *Ap;
    long long ldk;          // row stride of A' and B^T
    int items_a;
    const float *B;
    long long ldb, strideB;
    float *Bt;
    int items_b;
    int M, N, K;
    int tiles_n, tiles_k;   // 64 x 64 tiles of B^T per item
    int a_vec;              // A's base and rows are 16-byte aligned
    int *status;
};

template <bool VEC_B>
__global__ void __launch_bounds__(256) tf32_prep_kernel(const Tf32Prep q) {
    __shared__ float tile[64][65];
    ptx::allow_next_grid();   // the GEMM is a dependent launch; it waits for this grid
    const int item = static_cast<int>(blockIdx.y);
    const int tb = q.tiles_n * q.tiles_k;
    if (static_cast<int>(blockIdx.x) < tb) {
        if (item >= q.items_b) return;   // the whole CTA: no barrier is left behind
        const int t = static_cast<int>(blockIdx.x);
        transpose_tile<VEC_B>(q.B + item * q.strideB, q.ldb, q.Bt + static_cast<long long>(item) * q.N * q.ldk, q.ldk,
                              q.K, q.N, (t % q.tiles_n) * 64, (t / q.tiles_n) * 64, tile, q.status);
        return;
    }
    if (item >= q.items_a) return;
    const float *A = q.A + item * q.strideA;
    float *Ap = q.Ap + static_cast<long long>(item) * q.M * q.ldk;
#ifdef GTG_DEBUG
    const float *a_hi = A + (static_cast<long long>(q.M) - 1) * q.lda + q.K;
    const float *ap_hi = Ap + static_cast<long long>(q.M) * q.ldk;
#endif
    const long long per_row = q.ldk / 4;   // 16-byte groups of a row of A'
    const long long groups = static_cast<long long>(q.M) * per_row;
    const long long nblk = static_cast<long long>(gridDim.x) - tb;
    for (long long i = (static_cast<long long>(blockIdx.x) - tb) * 256 + threadIdx.x; i < groups; i += nblk * 256) {
        const long long r = i / per_row;
        const int c = static_cast<int>(i - r * per_row) * 4;
        const float *src = A + r * q.lda + c;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (q.a_vec && c + 3 < q.K && GTG_DEBUG_IN(src, 16, A, a_hi, q.status)) {
            const float4 t = __ldg(reinterpret_cast<const float4 *>(src));
            v[0] = t.x;
            v[1] = t.y;
            v[2] = t.z;
            v[3] = t.w;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (c + j < q.K && GTG_DEBUG_IN(src + j, 4, A, a_hi, q.status)) v[j] = __ldg(src + j);
        }
        float *dst = Ap + r * q.ldk + c;
        if (GTG_DEBUG_IN(dst, 16, Ap, ap_hi, q.status))
            *reinterpret_cast<float4 *>(dst) = make_float4(tf32_rounded(v[0]), tf32_rounded(v[1]), tf32_rounded(v[2]),
                                                           tf32_rounded(v[3]));
    }
}

// Bt = B^T on `stream` (the TF32 kernels' K-major copy of B).
cudaError_t transpose_launch(const float *B, int64_t ldb, float *Bt, int64_t ldbt, int64_t K, int64_t N,
                             int64_t batch, int64_t strideB, int *status, cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>((N + 63) / 64), static_cast<unsigned>(std::min<int64_t>((K + 63) / 64, 65535)),
                    static_cast<unsigned>(batch));
    const bool vec = (reinterpret_cast<uintptr_t>(B) & 15) == 0 && (ldb & 3) == 0 && (batch == 1 || (strideB & 3) == 0);
    if (vec)
        transpose_kernel<true><<<grid, 256, 0, stream>>>(B, ldb, Bt, ldbt, static_cast<int>(K), static_cast<int>(N), strideB,
                                                         status);
    else
        transpose_kernel<false><<<grid, 256, 0, stream>>>(B, ldb, Bt, ldbt, static_cast<int>(K), static_cast<int>(N), strideB,
                                                          status);
    return cudaGetLastError();
}

// Both TF32 operands on `stream`, one launch (see tf32_prep_kernel).
cudaError_t tf32_prep_launch(const DeviceInfo &dev, const GemmArgs &g, float *Ap, float *Bt, int64_t ldk,
                             int64_t items_a, int64_t items_b, cudaStream_t stream) {
    Tf32Prep q;
    q.A = static_cast<const float *>(g.A);
    q.lda = g.lda;
    q.strideA = g.strideA;
    q.Ap = Ap;
    q.ldk = ldk;
    q.items_a = static_cast<int>(items_a);
    q.B = static_cast<const float *>(g.B);
    q.ldb = g.ldb;
    q.strideB = g.strideB;
    q.Bt = Bt;
    q.items_b = static_cast<int>(items_b);
    q.M = static_cast<int>(g.M);
    q.N = static_cast<int>(g.N);
    q.K = static_cast<int>(g.K);
    q.tiles_n = static_cast<int>((g.N + 63) / 64);
    q.tiles_k = static_cast<int>((g.K + 63) / 64);
    q.a_vec = (reinterpret_cast<uintptr_t>(g.A) & 15) == 0 && (g.lda & 3) == 0 && (items_a == 1 || (g.strideA & 3) == 0);
    q.status = dev.status;
    const int64_t tb = static_cast<int64_t>(q.tiles_n) * q.tiles_k;
    const int64_t a_groups = g.M * (ldk / 4);
    const int64_t a_blocks = std::max<int64_t>(1, std::min<int64_t>((a_groups + 255) / 256, 8ll * dev.sms));
    if (tb + a_blocks > INT32_MAX || std::max(items_a, items_b) > 65535) return cudaErrorInvalidValue;
    const dim3 grid(static_cast<unsigned>(tb + a_blocks), static_cast<unsigned>(std::max(items_a, items_b)));
    const bool vec_b = (reinterpret_cast<uintptr_t>(g.B) & 15) == 0 && (g.ldb & 3) == 0 &&
                       (items_b == 1 || (g.strideB & 3) == 0);
    if (vec_b)
        tf32_prep_kernel<true><<<grid, 256, 0, stream>>>(q);
    else
        tf32_prep_kernel<false><<<grid, 256, 0, stream>>>(q);
    return cudaGetLastError();
}

// Copy of a row-major matrix into rows of ldd elements (the padding is never
// read): gives the tensor memory accelerator the 16-byte aligned base and row
// stride it needs when the caller's layout has neither.
template <typename E>
__global__ void __launch_bounds__(256) repack_rows_kernel(const E *__restrict__ src, long long lds, long long sstride,
                                                         E *__restrict__ dst, long long ldd, long long rows,
                                                         long long cols, int *status) {
    ptx::allow_next_grid();   // the GEMM reading dst waits for this grid
    // blockIdx.y: item of a batch (sstride apart in src, rows * ldd apart in dst)
    src += blockIdx.y * sstride;
    dst += blockIdx.y * rows * ldd;
#ifdef GTG_DEBUG
    const E *s_hi = src + (rows - 1) * lds + cols, *d_hi = dst + rows * ldd;
#endif
    (void)status;
    // a thread gathers one 16-byte group of a destination row (ldd is a
    // multiple of the group, so every group store is aligned) with element
    // loads, which any source alignment allows; past `cols` it writes zeros
    constexpr int V = 16 / sizeof(E);
    const long long groups = (cols + V - 1) / V;
    const long long total = rows * groups;
    for (long long i = blockIdx.x * 256ll + threadIdx.x; i < total; i += gridDim.x * 256ll) {
        const long long r = i / groups, c0 = (i - r * groups) * V;
        union {
            uint4 v;
            E e[V];
        } u;
        const E *s = src + r * lds + c0;
#pragma unroll
        for (int j = 0; j < V; ++j)
            u.e[j] = c0 + j < cols && GTG_DEBUG_IN(s + j, sizeof(E), src, s_hi, status) ? s[j] : E(0);
        if (GTG_DEBUG_IN(dst + r * ldd + c0, 16, dst, d_hi, status)) *reinterpret_cast<uint4 *>(dst + r * ldd + c0) = u.v;
    }
}

cudaError_t repack_launch(const void *src, int64_t lds, int64_t sstride, void *dst, int64_t ldd, int64_t rows,
                          int64_t cols, int64_t items, int64_t elem, int *status, cudaStream_t stream) {
    const long long total = rows * ((cols + 16 / elem - 1) / (16 / elem));
    const dim3 grid(static_cast<unsigned>(std::min<long long>((total + 255) / 256, 8192)),
                    static_cast<unsigned>(items));
    if (elem == 4)
        repack_rows_kernel<float><<<grid, 256, 0, stream>>>(static_cast<const float *>(src), lds, sstride,
                                                            static_cast<float *>(dst), ldd, rows, cols, status);
    else
        repack_rows_kernel<uint16_t><<<grid, 256, 0, stream>>>(static_cast<const uint16_t *>(src), lds, sstride,
                                                               static_cast<uint16_t *>(dst), ldd, rows, cols, status);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- host side
// Testing hooks (process-wide): the pipeline-wait time limit, and one K
// slice whose load the next tensor-core launch leaves out in CTA 0 so that a
// wait runs out on purpose.
std::atomic<unsigned long long> g_wait_limit_ns{kWaitLimitNs};
std::atomic<int> g_drop_slice{-1};
// How the CTA-pair kernel writes C: 0 by its own choice, 1 always by direct
// global stores, 2 by tensor stores wherever the layout allows them.
std::atomic<int> g_c_store_mode{0};

unsigned long long wait_limit_ns() { return g_wait_limit_ns.load(); }
int take_drop_slice() { return g_drop_slice.exchange(-1); }

// Widest aligned store the epilogue may use for whole rows of C.
int c_store_width(const GemmArgs &g) {
    const auto c = reinterpret_cast<uintptr_t>(g.C);
    if ((c & 31) == 0 && (g.ldc & 7) == 0) return 2;
    if ((c & 15) == 0 && (g.ldc & 3) == 0) return 1;
    return 0;
}

// K split of a launch (plan.splits > 1, single products only): the units'
// partial tiles go to a workspace of `splits` packed M x N slabs from the
// stream-ordered pool, without the epilogue, and finish_split adds them in
// order into C and applies the epilogue. Sets the unit count either way.
cudaError_t begin_split(const GemmArgs &g, const gtg_plan &plan, TcParams &p, float **ws, cudaStream_t stream) {
    *ws = nullptr;
    p.splits = 1;
    p.kps = p.num_kb;
    if (plan.splits > 1 && g.batch == 1 && p.num_kb > 1) {
        p.kps = (p.num_kb + plan.splits - 1) / plan.splits;
        p.splits = (p.num_kb + p.kps - 1) / p.kps;   // every range non-empty
    }
    p.num_units = p.num_tiles * p.splits;
    if (p.splits == 1) return cudaSuccess;
    cudaError_t e = ws_alloc(reinterpret_cast<void **>(ws), static_cast<size_t>(p.splits) * g.M * g.N * sizeof(float), stream);
    if (e != cudaSuccess) return e;
    p.C = *ws;
    p.ldc = g.N;
    p.strideC = g.M * g.N;
    p.bias = nullptr;
    p.act = 0;
    p.c_vec = (g.N & 7) == 0 ? 2 : ((g.N & 3) == 0 ? 1 : 0);   // pool memory is 256-byte aligned
    return cudaSuccess;
}

cudaError_t finish_split(const GemmArgs &g, const TcParams &p, float *ws, cudaError_t e, cudaStream_t stream) {
    if (ws == nullptr) return e;
    if (e == cudaSuccess) e = split_reduce_launch(ws, p.splits, g.M, g.N, g.C, g.ldc, g.bias, g.act, stream);
    const cudaError_t f = cudaFreeAsync(ws, stream);   // stream-ordered: after the reduction
    return e == cudaSuccess ? f : e;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

CUtensorMapDataType tma_type(int prec) {
    switch (prec) {
        case GTG_PREC_TF32: return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
        case GTG_PREC_F16: return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
        default: return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    }
}

// A row-major matrix (outer rows of `inner` elements, ld_elems apart) as a
// 3-D tensor map whose third dimension walks `batch` matrices
// batch_stride_elems apart; boxes of box_inner x box_outer x 1, 128-byte
// swizzled, out-of-range elements read as zero.
PFN_cuTensorMapEncodeIm2col_v12000 encode_im2col_fn() {
    static PFN_cuTensorMapEncodeIm2col_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeIm2col_v12000>(p);
    });
    return fn;
}

// Bounding-box corners of the im2col map: the window corners of the output
// pixels run from -pad to (last output) * stride - pad, i.e. the box is the
// image widened by the padding below and cut by pad - (window - 1) * dilation
// above; each corner is an offset from the image's first / last position.
int im2col_lower(int64_t pad) { return static_cast<int>(-pad); }
int im2col_upper(int64_t pad, int64_t window, int64_t dil) { return static_cast<int>(pad - (window - 1) * dil); }

// X (N x H x W x C, channels last) as im2col tiles of 128 pixels x one
// 128-byte channel block (64 16-bit or 32 TF32 channels).
bool encode_im2col(CUtensorMap *map, const ConvArgs &c) {
    auto fn = encode_im2col_fn();
    if (!fn) return false;
    const uint64_t e = c.prec == GTG_PREC_TF32 ? 4 : 2;
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(c.C), static_cast<cuuint64_t>(c.W), static_cast<cuuint64_t>(c.H),
                          static_cast<cuuint64_t>(c.N)};
    cuuint64_t strides[3] = {c.C * e, c.W * c.C * e, c.H * c.W * c.C * e};
    int lower[2] = {im2col_lower(c.pw), im2col_lower(c.ph)};                   // W, then H
    int upper[2] = {im2col_upper(c.pw, c.KW, c.dw), im2col_upper(c.ph, c.KH, c.dh)};
    cuuint32_t estr[4] = {1, static_cast<cuuint32_t>(c.sw), static_cast<cuuint32_t>(c.sh), 1};
    CUresult r = fn(map, tma_type(c.prec), 4, const_cast<void *>(c.X), dims, strides, lower, upper,
                    static_cast<cuuint32_t>(128 / e), 128, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_3d(CUtensorMap *map, int prec, const void *base, uint64_t inner, uint64_t outer, uint64_t ld_elems,
               uint64_t batch, uint64_t batch_stride_elems, uint32_t box_inner, uint32_t box_outer) {
    auto fn = encode_fn();
    if (!fn) return false;
    const uint64_t elem = prec == GTG_PREC_TF32 ? 4 : 2;
    if (batch <= 1) batch_stride_elems = (ld_elems * outer * elem + 15) / 16 * 16 / elem;  // unused, but valid
    cuuint64_t dims[3] = {inner, outer, batch < 1 ? 1 : batch};
    cuuint64_t strides[2] = {ld_elems * elem, batch_stride_elems * elem};
    cuuint32_t box[3] = {box_inner, box_outer, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, tma_type(prec), 3, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Instruction descriptor of the 16-bit kernels for this call's input format.
uint32_t idesc16(int prec, uint32_t M, uint32_t N) {
    return ptx::make_idesc(prec == GTG_PREC_F16 ? 0u : 1u, 0u, 1u, M, N);
}

std::atomic<int> g_pair_enabled{1};
std::atomic<int> g_force_splits{0};   // testing / tuning hook: K splits of every eligible product

struct AttrCache {
    std::mutex mu;
    uint64_t done[64] = {};  // per device: bit per kernel instantiation
};
AttrCache &attr_cache() {
    static AttrCache c;
    return c;
}

// Launch with programmatic dependent launch allowed: the CTAs may be
// scheduled while the previous kernel in the stream finishes; the kernel
// itself waits for that kernel before touching global memory.
template <typename Kern>
cudaError_t launch_pdl(Kern kern, int grid, int threads, int smem, cudaStream_t stream, const CUtensorMap &ta,
                       const CUtensorMap &tb, const TcParams &p) {
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
    return cudaLaunchKernelEx(&cfg, kern, ta, tb, p);
}

template <bool TF32, int BN>
cudaError_t launch_impl(const DeviceInfo &dev, const GemmArgs &g, const gtg_plan &plan,
                        cudaStream_t stream, int attr_bit) {
    using S = Shape<TF32, BN>;
    auto kern = tc_gemm_kernel<TF32, BN>;
    {
        AttrCache &ac = attr_cache();
        std::lock_guard<std::mutex> lk(ac.mu);
        const int d = dev.id & 63;
        if (!(ac.done[d] >> attr_bit & 1)) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
            if (e != cudaSuccess) return e;
            ac.done[d] |= 1ull << attr_bit;
        }
    }
    CUtensorMap ta, tb;
    if (!encode_3d(&ta, g.prec, g.A, g.K, g.M, g.lda, g.batch, g.strideA, S::BK, S::BM)) return cudaErrorInvalidValue;
    if constexpr (S::B_KMAJOR) {
        // TF32: g.B is already B^T (N x K, rounded), written by the preparation kernel
        if (!encode_3d(&tb, g.prec, g.B, g.K, g.N, g.ldb, g.batch, g.strideB, S::BK, BN)) return cudaErrorInvalidValue;
    } else {
        if (!encode_3d(&tb, g.prec, g.B, g.N, g.K, g.ldb, g.batch, g.strideB, S::BCH_N, S::BK))
            return cudaErrorInvalidValue;
    }
    TcParams p{};
    p.C = g.C;
    p.ldc = g.ldc;
    p.M = static_cast<int>(g.M);
    p.N = static_cast<int>(g.N);
    p.num_m = static_cast<int>((g.M + S::BM - 1) / S::BM);
    p.num_n = static_cast<int>((g.N + BN - 1) / BN);
    p.num_kb = static_cast<int>((g.K + S::BK - 1) / S::BK);
    p.tiles_per_batch = p.num_m * p.num_n;
    p.num_tiles = static_cast<int>(p.tiles_per_batch * g.batch);
    p.strideC = g.strideC;
    p.idesc = TF32 ? S::IDESC : idesc16(g.prec, S::BM, BN);
    p.c_vec = c_store_width(g);
    p.tail_start = INT32_MAX;
    p.c_tma = 0;
    p.status = dev.status;
    p.wait_limit_ns = wait_limit_ns();
    p.drop_slice = take_drop_slice();
    p.bias = g.bias;
    p.act = g.act;
    float *ws = nullptr;
    cudaError_t e = begin_split(g, plan, p, &ws, stream);
    if (e == cudaSuccess) e = launch_pdl(kern, plan.grid, kThreads, S::SMEM, stream, ta, tb, p);
    e = finish_split(g, p, ws, e, stream);
    return e;
}

// Units of the pair kernel: whole 256 x 256 tiles, and the tiles of a last
// partial wave cut into 128-wide halves when the halves fit one wave of
// clusters (16-bit inputs, a single product, no K split). tail_start = the
// first half-tile unit, INT32_MAX when there are none.
struct PairUnits {
    int units, tail_start;
};
PairUnits pair_units(int64_t tiles, int clusters, bool allowed) {
    if (allowed && clusters > 0) {
        const int64_t tail = tiles < clusters ? tiles : tiles % clusters;
        if (tail > 0 && 2 * tail <= clusters)
            return {static_cast<int>(tiles + tail), static_cast<int>(tiles - tail)};
    }
    return {static_cast<int>(tiles), INT32_MAX};
}

bool pair_halves_allowed(const GemmArgs &g, int splits) {
    return g.prec != GTG_PREC_TF32 && splits == 1 && g.batch == 1;
}

template <bool TF32>
cudaError_t launch_pair(const DeviceInfo &dev, const GemmArgs &g, const gtg_plan &plan, cudaStream_t stream,
                        int attr_bit) {
    using S = PairShape<TF32>;
    auto kern = tc_gemm_pair_kernel<TF32>;
    {
        AttrCache &ac = attr_cache();
        std::lock_guard<std::mutex> lk(ac.mu);
        const int d = dev.id & 63;
        if (!(ac.done[d] >> attr_bit & 1)) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
            if (e != cudaSuccess) return e;
            ac.done[d] |= 1ull << attr_bit;
        }
    }
    CUtensorMap ta, tb;
    if (!encode_3d(&ta, g.prec, g.A, g.K, g.M, g.lda, g.batch, g.strideA, S::BK, S::BM)) return cudaErrorInvalidValue;
    if constexpr (S::B_KMAJOR) {
        // TF32: g.B is already B^T (N x K, rounded), written by the preparation kernel
        if (!encode_3d(&tb, g.prec, g.B, g.K, g.N, g.ldb, g.batch, g.strideB, S::BK, S::BN / 2))
            return cudaErrorInvalidValue;
    } else {
        if (!encode_3d(&tb, g.prec, g.B, g.N, g.K, g.ldb, g.batch, g.strideB, S::BCH_N, S::BK))
            return cudaErrorInvalidValue;
    }
    TcParams p{};
    p.C = g.C;
    p.ldc = g.ldc;
    p.M = static_cast<int>(g.M);
    p.N = static_cast<int>(g.N);
    p.num_m = static_cast<int>((g.M + 2 * S::BM - 1) / (2 * S::BM));
    p.num_n = static_cast<int>((g.N + S::BN - 1) / S::BN);
    p.num_kb = static_cast<int>((g.K + S::BK - 1) / S::BK);
    p.tiles_per_batch = p.num_m * p.num_n;
    p.num_tiles = static_cast<int>(p.tiles_per_batch * g.batch);
    p.strideC = g.strideC;
    p.idesc = TF32 ? ptx::make_idesc(2u, 0u, 0u, 2 * S::BM, S::BN) : idesc16(g.prec, 2 * S::BM, S::BN);
    p.c_vec = c_store_width(g);
    p.tail_start = INT32_MAX;
    p.c_tma = 0;
    p.status = dev.status;
    p.wait_limit_ns = wait_limit_ns();
    p.drop_slice = take_drop_slice();
    p.bias = g.bias;
    p.act = g.act;
    float *ws = nullptr;
    cudaError_t e = begin_split(g, plan, p, &ws, stream);
    const PairUnits pu = pair_units(p.num_tiles, dev.sms / 2, pair_halves_allowed(g, p.splits));
    p.tail_start = pu.tail_start;
    if (pu.tail_start != INT32_MAX) {
        p.num_units = pu.units;
        p.tiles_per_batch = pu.units;   // a single product: unit t is tile (or half) t
    }
    const int clusters = static_cast<int>(std::min<int64_t>(p.num_units, dev.sms / 2));
    // C by tensor stores: a single product or batch (no split-K slabs) with
    // 16-byte aligned rows and items. Measured (BF16, both forms in one
    // process): tensor stores are 13-33 % faster when the epilogue is exposed
    // (8192^2 with K <= 512; at most a few units per cluster: 2048^3, 4096^2
    // x 1024, 6000 x 5000 x 4096) and 4-8 % slower in long products of many
    // waves (8192^2 with K >= 1024, 8192^3, 16384 x 4096 x 4096), where the
    // epilogue overlaps the next tile's MMAs and only adds to the SM's load.
    const int c_mode = g_c_store_mode.load();
    const int waves = (p.num_units + clusters - 1) / std::max(clusters, 1);
    const bool c_tma_pays = p.num_kb <= 8 || waves <= 8;
    CUtensorMap tc = ta;   // not read unless c_tma
    p.c_tma = c_mode != 1 && (c_mode == 2 || c_tma_pays) && p.splits == 1 &&
              (reinterpret_cast<uintptr_t>(g.C) & 15) == 0 && (g.ldc & 3) == 0 &&
              (g.batch == 1 || (g.strideC & 3) == 0) &&
              encode_3d(&tc, GTG_PREC_TF32, g.C, g.N, g.M, g.ldc, g.batch, g.strideC, 32, 32);
    if (e == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = static_cast<size_t>(S::SMEM);
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        e = cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, p);
        e = finish_split(g, p, ws, e, stream);
    }
    return e;
}

void fill_pair_plan(const DeviceInfo &dev, const GemmArgs &g, gtg_plan *plan, int splits) {
    using S = PairShape<false>;
    const int64_t tiles = g.batch * ((g.M + 2 * S::BM - 1) / (2 * S::BM)) * ((g.N + S::BN - 1) / S::BN);
    const PairUnits pu = pair_units(tiles, dev.sms / 2, pair_halves_allowed(g, splits));
    const int64_t units = pu.tail_start != INT32_MAX ? pu.units : tiles * splits;
    const int64_t clusters = std::min<int64_t>(units, dev.sms / 2);
    plan->kernel = GTG_KERNEL_TCGEN05;
    plan->bm = 2 * S::BM;
    plan->bn = S::BN;
    plan->bk = g.prec == GTG_PREC_TF32 ? PairShape<true>::BK : S::BK;
    plan->stages = S::STAGES;
    plan->grid = static_cast<int>(2 * clusters);
    plan->threads = kThreads;
    plan->smem = S::SMEM;
    plan->cluster = 2;
    plan->splits = splits;
}

template <bool TF32, int BN>
void fill_plan(const DeviceInfo &dev, const GemmArgs &g, gtg_plan *plan, int splits) {
    using S = Shape<TF32, BN>;
    const int64_t tiles = g.batch * ((g.M + S::BM - 1) / S::BM) * ((g.N + BN - 1) / BN) * splits;
    plan->kernel = GTG_KERNEL_TCGEN05;
    plan->bm = S::BM;
    plan->bn = BN;
    plan->bk = S::BK;
    plan->stages = S::STAGES;
    plan->grid = static_cast<int>(tiles < dev.sms ? tiles : dev.sms);
    plan->threads = kThreads;
    plan->smem = S::SMEM;
    plan->cluster = 1;
    plan->splits = splits;
}

// Implicit-GEMM convolution on the single-CTA kernel: Y (N*OH*OW x CO) =
// patches(X) x Wt with the A tiles loaded by TMA in im2col mode. TF32: X and
// Wt are the rounded image and the rounded W^T (CO x K) of tc_conv_launch.
template <bool TF32, int BN>
cudaError_t conv_launch_impl(const DeviceInfo &dev, const ConvArgs &c, cudaStream_t stream, int attr_bit,
                             int splits) {
    using S = Shape<TF32, BN>;
    auto kern = tc_gemm_kernel<TF32, BN, true>;
    {
        AttrCache &ac = attr_cache();
        std::lock_guard<std::mutex> lk(ac.mu);
        const int d = dev.id & 63;
        if (!(ac.done[d] >> attr_bit & 1)) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
            if (e != cudaSuccess) return e;
            ac.done[d] |= 1ull << attr_bit;
        }
    }
    const int64_t M = c.N * c.OH * c.OW, K = c.KH * c.KW * c.C;
    CUtensorMap ta, tb;
    if (!encode_im2col(&ta, c)) return cudaErrorInvalidValue;
    if constexpr (TF32) {
        if (!encode_3d(&tb, c.prec, c.Wt, K, c.CO, K, 1, 0, S::BK, BN)) return cudaErrorInvalidValue;
    } else {
        if (!encode_3d(&tb, c.prec, c.Wt, c.CO, K, c.CO, 1, 0, S::BCH_N, S::BK)) return cudaErrorInvalidValue;
    }
    TcParams p{};
    p.C = c.Y;
    p.ldc = c.CO;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(c.CO);
    p.num_m = static_cast<int>((M + S::BM - 1) / S::BM);
    p.num_n = static_cast<int>((c.CO + BN - 1) / BN);
    p.num_kb = static_cast<int>(K / S::BK);
    p.tiles_per_batch = p.num_m * p.num_n;
    p.num_tiles = p.tiles_per_batch;
    p.splits = 1;
    p.kps = p.num_kb;
    p.num_units = p.num_tiles;
    p.strideC = 0;
    p.idesc = TF32 ? S::IDESC : idesc16(c.prec, S::BM, BN);
    const auto yaddr = reinterpret_cast<uintptr_t>(c.Y);
    p.c_vec = ((yaddr & 31) == 0 && (c.CO & 7) == 0) ? 2 : (((yaddr & 15) == 0 && (c.CO & 3) == 0) ? 1 : 0);
    p.tail_start = INT32_MAX;
    p.c_tma = 0;
    p.status = dev.status;
    p.wait_limit_ns = wait_limit_ns();
    p.drop_slice = take_drop_slice();
    p.bias = c.bias;
    p.act = c.act;
    p.cv_ow = static_cast<int>(c.OW);
    p.cv_oh = static_cast<int>(c.OH);
    p.cv_cb = static_cast<int>(c.C / S::BK);
    p.cv_kw = static_cast<int>(c.KW);
    p.cv_sw = static_cast<int>(c.sw);
    p.cv_sh = static_cast<int>(c.sh);
    p.cv_pw = static_cast<int>(c.pw);
    p.cv_ph = static_cast<int>(c.ph);
    p.cv_dw = static_cast<int>(c.dw);
    p.cv_dh = static_cast<int>(c.dh);
    // K split into ranges like a GEMM's: partial tiles to workspace slabs, then
    // the ordered reduction applies the bias and activation
    GemmArgs gg{c.prec, M, c.CO, K, nullptr, 0, nullptr, 0, c.Y, c.CO};
    gg.bias = c.bias;
    gg.act = c.act;
    gtg_plan plan{};
    plan.splits = splits;
    float *ws = nullptr;
    cudaError_t e = begin_split(gg, plan, p, &ws, stream);
    const int grid = static_cast<int>(std::min<int64_t>(p.num_units, dev.sms));
    if (e == cudaSuccess) e = launch_pdl(kern, grid, kThreads, S::SMEM, stream, ta, tb, p);
    return finish_split(gg, p, ws, e, stream);
}

// Implicit-GEMM convolution on the CTA-pair kernel: 256 x 256 tiles of Y,
// each CTA's 128 output pixels of a K slice one TMA im2col load (the map's
// 128-pixel x 64-channel box is the single-CTA kernel's), half of B per CTA.
template <bool TF32>
cudaError_t conv_launch_pair(const DeviceInfo &dev, const ConvArgs &c, cudaStream_t stream, int splits, int attr_bit) {
    using S = PairShape<TF32>;
    auto kern = tc_gemm_pair_kernel<TF32, true>;
    {
        AttrCache &ac = attr_cache();
        std::lock_guard<std::mutex> lk(ac.mu);
        const int d = dev.id & 63;
        if (!(ac.done[d] >> attr_bit & 1)) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
            if (e != cudaSuccess) return e;
            ac.done[d] |= 1ull << attr_bit;
        }
    }
    const int64_t M = c.N * c.OH * c.OW, K = c.KH * c.KW * c.C;
    CUtensorMap ta, tb;
    if (!encode_im2col(&ta, c)) return cudaErrorInvalidValue;
    if constexpr (TF32) {
        // this CTA's 128 rows of the rounded W^T
        if (!encode_3d(&tb, c.prec, c.Wt, K, c.CO, K, 1, 0, S::BK, S::BN / 2)) return cudaErrorInvalidValue;
    } else {
        if (!encode_3d(&tb, c.prec, c.Wt, c.CO, K, c.CO, 1, 0, S::BCH_N, S::BK)) return cudaErrorInvalidValue;
    }
    TcParams p{};
    p.C = c.Y;
    p.ldc = c.CO;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(c.CO);
    p.num_m = static_cast<int>((M + 2 * S::BM - 1) / (2 * S::BM));
    p.num_n = static_cast<int>((c.CO + S::BN - 1) / S::BN);
    p.num_kb = static_cast<int>(K / S::BK);
    p.tiles_per_batch = p.num_m * p.num_n;
    p.num_tiles = p.tiles_per_batch;
    p.strideC = 0;
    p.idesc = TF32 ? ptx::make_idesc(2u, 0u, 0u, 2 * S::BM, S::BN) : idesc16(c.prec, 2 * S::BM, S::BN);
    const auto yaddr = reinterpret_cast<uintptr_t>(c.Y);
    p.c_vec = ((yaddr & 31) == 0 && (c.CO & 7) == 0) ? 2 : (((yaddr & 15) == 0 && (c.CO & 3) == 0) ? 1 : 0);
    p.tail_start = INT32_MAX;
    p.c_tma = 0;
    p.status = dev.status;
    p.wait_limit_ns = wait_limit_ns();
    p.drop_slice = take_drop_slice();
    p.bias = c.bias;
    p.act = c.act;
    p.cv_ow = static_cast<int>(c.OW);
    p.cv_oh = static_cast<int>(c.OH);
    p.cv_cb = static_cast<int>(c.C / S::BK);
    p.cv_kw = static_cast<int>(c.KW);
    p.cv_sw = static_cast<int>(c.sw);
    p.cv_sh = static_cast<int>(c.sh);
    p.cv_pw = static_cast<int>(c.pw);
    p.cv_ph = static_cast<int>(c.ph);
    p.cv_dw = static_cast<int>(c.dw);
    p.cv_dh = static_cast<int>(c.dh);
    GemmArgs gg{c.prec, M, c.CO, K, nullptr, 0, nullptr, 0, c.Y, c.CO};
    gg.bias = c.bias;
    gg.act = c.act;
    gtg_plan plan{};
    plan.splits = splits;
    float *ws = nullptr;
    cudaError_t e = begin_split(gg, plan, p, &ws, stream);
    const int clusters = static_cast<int>(std::min<int64_t>(p.num_units, dev.sms / 2));
    // Y by tensor stores on the same terms as a GEMM's C (see launch_pair)
    const int waves = (p.num_units + clusters - 1) / std::max(clusters, 1);
    const int c_mode = g_c_store_mode.load();
    CUtensorMap tc = ta;   // not read unless c_tma
    p.c_tma = c_mode != 1 && (c_mode == 2 || p.num_kb <= 8 || waves <= 8) && p.splits == 1 &&
              (yaddr & 15) == 0 && (c.CO & 3) == 0 &&
              encode_3d(&tc, GTG_PREC_TF32, c.Y, c.CO, M, c.CO, 1, 0, 32, 32);
    if (e == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = static_cast<size_t>(S::SMEM);
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        e = cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, p);
    }
    return finish_split(gg, p, ws, e, stream);
}

}  // namespace


void tc_set_wait_limit_ns(unsigned long long ns) { g_wait_limit_ns.store(ns ? ns : kWaitLimitNs); }
bool tma_map_2d(CUtensorMap *map, int prec, const void *base, uint64_t inner, uint64_t outer, uint64_t ld_elems,
                uint32_t box_inner, uint32_t box_outer) {
    return encode_3d(map, prec, base, inner, outer, ld_elems, 1, 0, box_inner, box_outer);
}

int take_test_drop_slice() { return take_drop_slice(); }

unsigned long long wait_limit_setting() { return g_wait_limit_ns.load(); }
void tc_drop_next_load(int slice) { g_drop_slice.store(slice); }
void tc_force_splits(int splits) { g_force_splits.store(splits > 0 ? splits : 0); }
void tc_force_c_store(int mode) { g_c_store_mode.store(mode == 1 || mode == 2 ? mode : 0); }

bool tc_supported(const DeviceInfo &dev) {
    // tcgen05 exists on the sm_100 family; this library is built for sm_103a.
    return dev.cc_major == 10 && dev.cc_minor == 3 && encode_fn() != nullptr;
}

bool tc_eligible(const GemmArgs &g) {
    if (g.prec != GTG_PREC_TF32 && g.prec != GTG_PREC_BF16 && g.prec != GTG_PREC_F16) return false;
    const int64_t elem = g.prec == GTG_PREC_TF32 ? 4 : 2;
    // 16-bit operands are read by TMA in place; TF32 operands go through the
    // preparation kernel (a rounded copy of A, the rounded B^T) in any layout
    const bool tf32 = g.prec == GTG_PREC_TF32;
    if (g.batch > 1) {
        // batch strides are tensor-map strides
        if (!tf32 && ((g.strideA * elem) % 16 || (g.strideA * elem) >= (1ll << 40))) return false;
        if (!tf32 && ((g.strideB * elem) % 16 || (g.strideB * elem) >= (1ll << 40))) return false;
        if (g.batch > 65535 || g.batch * ((g.M + 127) / 128) * ((g.N + 63) / 64) > INT32_MAX) return false;
    }
    const auto a = reinterpret_cast<uintptr_t>(g.A), b = reinterpret_cast<uintptr_t>(g.B);
    if (!tf32 && ((a & 15) || (g.lda * elem) % 16)) return false;   // TMA base and row stride of A
    if (!tf32 && ((b & 15) || (g.ldb * elem) % 16)) return false;
    if (g.M > INT32_MAX || g.N > INT32_MAX || g.K > INT32_MAX) return false;
    if ((g.lda * elem) >= (1ll << 40) || (g.ldb * elem) >= (1ll << 40)) return false;
    return g.M > 0 && g.N > 0 && g.K > 0;
}

// Kernel, tile width and K split: minimise the estimated time
//   waves x (slices per unit + kFill) x slice time  [+ the split reduction]
// where a wave is one unit (tile x K range) on every SM (CTA pair), kFill
// counts pipeline fill, set-up and the epilogue in slice times, and a slice
// of a 128 x w tile takes w/256 of a 256-wide one divided by the tile's
// relative efficiency (with M = 128 per CTA a 256-wide tile reads 96
// shared-memory bytes per tensor-core cycle, a 128-wide one 128 -- the SM's
// limit -- and a 64-wide one 192), and a 256 x 256 pair tile 1/1.15 of the
// 128 x 256 single-CTA time (2/3 of its operand bytes per SM). A split adds
// a second kernel that reads the S partial slabs and writes C once.
namespace {
constexpr double kSliceUs = 0.30;        // one 128 x 256 x (128 bytes of K) slice on one SM
constexpr double kFillSlices = 4.0;
constexpr double kReduceFixedUs = 3.0;   // the reduction's launch and allocation
constexpr double kHbmBytesPerUs = 6.0e6;
constexpr double kConvSlice = 2.0;        // an implicit convolution's K slice against a GEMM's
constexpr double kConvPairRel = 1.0 / 1.15;   // a pair slice (256 x 256 per 2 SMs) against a 128 x 256 one
double tc_cost(const DeviceInfo &dev, const GemmArgs &g, int bm, int bn, int slots, double rel, int splits,
               int bk_elems) {
    const int64_t num_kb = (g.K + bk_elems - 1) / bk_elems;
    const int64_t kps = (num_kb + splits - 1) / splits;
    const int64_t units = g.batch * ((g.M + bm - 1) / bm) * ((g.N + bn - 1) / bn) * ((num_kb + kps - 1) / kps);
    const int64_t waves = (units + slots - 1) / slots;
    double t = static_cast<double>(waves) * (static_cast<double>(kps) + kFillSlices) * kSliceUs * rel;
    if (splits > 1) t += kReduceFixedUs + (splits + 1.0) * static_cast<double>(g.M) * g.N * 4.0 / kHbmBytesPerUs;
    (void)dev;
    return t;
}
}  // namespace

void tc_plan(const DeviceInfo &dev, const GemmArgs &g, gtg_plan *plan) {
    const bool tf32 = g.prec == GTG_PREC_TF32;
    const int bk = tf32 ? 32 : 64;               // K elements per 128-byte slice
    const int64_t num_kb = (g.K + bk - 1) / bk;
    int forced = g_force_splits.load();
    if (forced > 1 && (g.batch > 1 || num_kb < 2 * forced)) forced = 0;   // not applicable: plan as usual
    const int split_opts[6] = {1, 2, 3, 4, 6, 8};
    const int widths[3] = {256, 128, 64};
    const double rel[3] = {1.0, 0.5 / 0.8, 0.25 / 0.5};
    int best_w = 0, best_s = 1;
    bool best_pair = false;
    double best_cost = 0;
    bool first = true;
    for (int si = 0; si < 6; ++si) {
        const int sp = split_opts[si];
        const int want = forced > 0 ? forced : sp;
        if (forced > 0 && si > 0) break;             // a forced split is the only option
        if (want > 1 && (g.batch > 1 || num_kb < 2 * want)) continue;
        for (int i = 0; i < 3; ++i) {
            const double c = tc_cost(dev, g, kBM, widths[i], dev.sms, rel[i], want, bk);
            if (first || c < best_cost) {
                best_cost = c;
                best_w = i;
                best_s = want;
                best_pair = false;
                first = false;
            }
        }
        if ((dev.sms & 1) == 0 && g_pair_enabled.load()) {
            double c = tc_cost(dev, g, 2 * kBM, 256, dev.sms / 2, 1.0 / 1.15, want, bk);
            if (pair_halves_allowed(g, want)) {
                // a last partial wave cut into half tiles costs about 0.6 of a
                // wave (half the multiplies, three quarters of the operand bytes)
                const int64_t tiles = ((g.M + 2 * kBM - 1) / (2 * kBM)) * ((g.N + 255) / 256);
                if (pair_units(tiles, dev.sms / 2, true).tail_start != INT32_MAX)
                    c = (static_cast<double>(tiles / (dev.sms / 2)) + 0.6) * (static_cast<double>(num_kb) + kFillSlices) *
                        kSliceUs / 1.15;
            }
            if (c < best_cost) {
                best_cost = c;
                best_s = want;
                best_pair = true;
            }
        }
    }
    if (best_pair) {
        fill_pair_plan(dev, g, plan, best_s);
        return;
    }
    switch (widths[best_w]) {
        case 256: tf32 ? fill_plan<true, 256>(dev, g, plan, best_s) : fill_plan<false, 256>(dev, g, plan, best_s); break;
        case 128: tf32 ? fill_plan<true, 128>(dev, g, plan, best_s) : fill_plan<false, 128>(dev, g, plan, best_s); break;
        default: tf32 ? fill_plan<true, 64>(dev, g, plan, best_s) : fill_plan<false, 64>(dev, g, plan, best_s); break;
    }
}

// (The plan of gemm_tf32_noalloc: its single-CTA kernel has the four
// converter warps that round A in shared memory.)
void tc_plan_unsplit_single(const DeviceInfo &dev, const GemmArgs &g, gtg_plan *plan) {
    const bool tf32 = g.prec == GTG_PREC_TF32;
    const int bk = tf32 ? 32 : 64;
    const int widths[3] = {256, 128, 64};
    const double rel[3] = {1.0, 0.5 / 0.8, 0.25 / 0.5};
    int best = 0;
    double best_cost = 0;
    for (int i = 0; i < 3; ++i) {
        const double c = tc_cost(dev, g, kBM, widths[i], dev.sms, rel[i], 1, bk);
        if (i == 0 || c < best_cost) {
            best_cost = c;
            best = i;
        }
    }
    switch (widths[best]) {
        case 256: tf32 ? fill_plan<true, 256>(dev, g, plan, 1) : fill_plan<false, 256>(dev, g, plan, 1); break;
        case 128: tf32 ? fill_plan<true, 128>(dev, g, plan, 1) : fill_plan<false, 128>(dev, g, plan, 1); break;
        default: tf32 ? fill_plan<true, 64>(dev, g, plan, 1) : fill_plan<false, 64>(dev, g, plan, 1); break;
    }
    plan->threads = threads_for(tf32);
}

bool tc_conv_eligible(const DeviceInfo &dev, const ConvArgs &c) {
    if (!tc_supported(dev) || encode_im2col_fn() == nullptr) return false;
    if (c.prec == GTG_PREC_TF32) {
        // X and Wt are read through their rounded copies (any alignment)
        if (c.C % 32) return false;                                          // 128-byte channel blocks
    } else {
        if (c.prec != GTG_PREC_BF16 && c.prec != GTG_PREC_F16) return false;
        if (c.C % 64 || (c.CO * 2) % 16) return false;                      // 128-byte channel blocks, B rows
        if ((reinterpret_cast<uintptr_t>(c.X) & 15) || (reinterpret_cast<uintptr_t>(c.Wt) & 15)) return false;
    }
    if (c.sw > 8 || c.sh > 8) return false;                                  // TMA traversal steps
    const int64_t corners[4] = {-c.pw, -c.ph, c.pw - (c.KW - 1) * c.dw, c.ph - (c.KH - 1) * c.dh};
    for (int64_t v : corners)
        if (v < -128 || v > 127) return false;                               // 8-bit corners of a 4-D map
    if ((c.KW - 1) * c.dw > 255 || (c.KH - 1) * c.dh > 255) return false;    // im2col offsets
    if (c.N * c.OH * c.OW > INT32_MAX || c.KH * c.KW * c.C > INT32_MAX) return false;
    return true;
}

// The implicit convolution's kernel: the width of single-CTA tiles (or the
// CTA pair) and the K split, by the same estimate as the GEMM planner, with a
// K slice of im2col loads costing about twice a GEMM's (measured on 3x3
// layers of 64 to 512 channels: the estimate then picks the fastest of splits
// 1-6 and widths 64-256 on each, e.g. 512 -> 512 channels at 7x7 x 64: 3 K
// ranges, 32.6 -> 22.1 us). choice: 0 any kernel, 1 single CTAs only, 2 the
// CTA pair only. gtg_force_gemm_splits applies here too. Returns false if
// `choice` rules out every kernel.
bool tc_conv_choose(const DeviceInfo &dev, const ConvArgs &c, int choice, bool *pair, int *width, int *splits) {
    GemmArgs g{c.prec, c.N * c.OH * c.OW, c.CO, c.KH * c.KW * c.C, nullptr, 0, nullptr, 0, nullptr, 0};
    const int bk = c.prec == GTG_PREC_TF32 ? 32 : 64;   // K elements per 128-byte slice
    const int64_t num_kb = g.K / bk;
    int forced = g_force_splits.load();
    if (forced > 1 && num_kb < 2 * forced) forced = 0;
    const int split_opts[6] = {1, 2, 3, 4, 6, 8};
    const int widths[3] = {256, 128, 64};
    const double rel[3] = {1.0, 0.5 / 0.8, 0.25 / 0.5};
    const bool pair_ok = choice != 1 && (dev.sms & 1) == 0 && g_pair_enabled.load();
    bool first = true;
    double best_cost = 0;
    for (int si = 0; si < 6; ++si) {
        const int sp = forced > 0 ? forced : split_opts[si];
        if (forced > 0 && si > 0) break;
        if (sp > 1 && num_kb < 2 * sp) continue;
        if (choice != 2) {
            for (int i = 0; i < 3; ++i) {
                const double cost = tc_cost(dev, g, kBM, widths[i], dev.sms, kConvSlice * rel[i], sp, bk);
                if (first || cost < best_cost) {
                    *pair = false;
                    *width = widths[i];
                    *splits = sp;
                    best_cost = cost;
                    first = false;
                }
            }
        }
        if (pair_ok) {
            const double cost = tc_cost(dev, g, 2 * kBM, 256, dev.sms / 2, kConvSlice * kConvPairRel, sp, bk);
            if (first || cost < best_cost) {
                *pair = true;
                *width = 256;
                *splits = sp;
                best_cost = cost;
                first = false;
            }
        }
    }
    return !first;
}

cudaError_t tc_conv_launch(const DeviceInfo &dev, const ConvArgs &c, cudaStream_t stream, int choice) {
    bool pair = false;
    int width = 256, splits = 1;
    if (!tc_conv_choose(dev, c, choice, &pair, &width, &splits)) return cudaErrorNotSupported;
    if (c.prec != GTG_PREC_TF32) {
        if (pair) return conv_launch_pair<false>(dev, c, stream, splits, 14);
        switch (width) {
            case 256: return conv_launch_impl<false, 256>(dev, c, stream, 7, splits);
            case 128: return conv_launch_impl<false, 128>(dev, c, stream, 8, splits);
            default: return conv_launch_impl<false, 64>(dev, c, stream, 9, splits);
        }
    }
    // TF32: the MMA truncates its operands, so the image and the weights are
    // first rounded to the nearest TF32 value (as gemm_tf32 does), the image
    // into a copy of its own size (not the KH*KW times larger patch matrix),
    // the weights into W^T (CO x K, the K-major B of the TF32 kernels); the
    // product then reads the patches from the rounded image
    const int64_t pixels = c.N * c.H * c.W, K = c.KH * c.KW * c.C;
    const size_t x_bytes = (static_cast<size_t>(pixels * c.C) * 4 + 255) / 256 * 256;
    const size_t w_bytes = static_cast<size_t>(c.CO * K) * 4;
    void *ws = nullptr;
    cudaError_t e = ws_alloc(&ws, x_bytes + w_bytes, stream);
    if (e != cudaSuccess) return e;
    float *Xr = static_cast<float *>(ws);
    float *Wr = reinterpret_cast<float *>(static_cast<char *>(ws) + x_bytes);
    GemmArgs gx{GTG_PREC_TF32, pixels, 0, c.C, c.X, c.C, nullptr, 0, nullptr, 0};   // the image alone (no B)
    e = tf32_prep_launch(dev, gx, Xr, nullptr, c.C, 1, 1, stream);
    if (e == cudaSuccess)
        e = transpose_launch(static_cast<const float *>(c.Wt), c.CO, Wr, K, K, c.CO, 1, 0, dev.status, stream);
    ConvArgs cr = c;
    cr.X = Xr;
    cr.Wt = Wr;
    if (e == cudaSuccess) {
        if (pair) {
            e = conv_launch_pair<true>(dev, cr, stream, splits, 18);
        } else {
            switch (width) {
                case 256: e = conv_launch_impl<true, 256>(dev, cr, stream, 15, splits); break;
                case 128: e = conv_launch_impl<true, 128>(dev, cr, stream, 16, splits); break;
                default: e = conv_launch_impl<true, 64>(dev, cr, stream, 17, splits); break;
            }
        }
    }
    const cudaError_t f = cudaFreeAsync(ws, stream);   // stream-ordered: after the product has read it
    return e != cudaSuccess ? e : f;
}

bool tc_conv_plan(const DeviceInfo &dev, const ConvArgs &c, int choice, gtg_plan *plan) {
    bool pair = false;
    int width = 256, splits = 1;
    if (!tc_conv_choose(dev, c, choice, &pair, &width, &splits)) return false;
    GemmArgs g{c.prec, c.N * c.OH * c.OW, c.CO, c.KH * c.KW * c.C, nullptr, 0, nullptr, 0, nullptr, 0};
    if (pair) {
        fill_pair_plan(dev, g, plan, splits);
        // no half tiles for a convolution: every unit is a 256 x 256 tile (and K range)
        const int64_t tiles = ((g.M + 255) / 256) * ((g.N + 255) / 256) * splits;
        plan->grid = static_cast<int>(2 * std::min<int64_t>(tiles, dev.sms / 2));
        return true;
    }
    const bool tf32 = c.prec == GTG_PREC_TF32;
    switch (width) {
        case 256: tf32 ? fill_plan<true, 256>(dev, g, plan, splits) : fill_plan<false, 256>(dev, g, plan, splits); break;
        case 128: tf32 ? fill_plan<true, 128>(dev, g, plan, splits) : fill_plan<false, 128>(dev, g, plan, splits); break;
        default: tf32 ? fill_plan<true, 64>(dev, g, plan, splits) : fill_plan<false, 64>(dev, g, plan, splits); break;
    }
    plan->threads = kThreads;
    return true;
}


namespace {
cudaError_t tc_launch_aligned(const DeviceInfo &dev, const GemmArgs &g, const gtg_plan &plan,
                              cudaStream_t stream) {
    const bool tf32 = g.prec == GTG_PREC_TF32;
    if (plan.bm == 2 * PairShape<false>::BM)
        return tf32 ? launch_pair<true>(dev, g, plan, stream, 10) : launch_pair<false>(dev, g, plan, stream, 6);
    switch (plan.bn) {
        case 256:
            return tf32 ? launch_impl<true, 256>(dev, g, plan, stream, 0)
                        : launch_impl<false, 256>(dev, g, plan, stream, 1);
        case 128:
            return tf32 ? launch_impl<true, 128>(dev, g, plan, stream, 2)
                        : launch_impl<false, 128>(dev, g, plan, stream, 3);
        case 64:
            return tf32 ? launch_impl<true, 64>(dev, g, plan, stream, 4)
                        : launch_impl<false, 64>(dev, g, plan, stream, 5);
        default:
            return cudaErrorInvalidValue;
    }
}

// Base, row stride and (for batch items) item stride all on 16 bytes.
bool tma_operand_ok(const void *p, int64_t ld, int64_t stride, int64_t batch, int64_t elem) {
    return (reinterpret_cast<uintptr_t>(p) & 15) == 0 && (ld * elem) % 16 == 0 &&
           (batch == 1 || (stride * elem) % 16 == 0);
}
}  // namespace

bool tc_eligible_repacked(const GemmArgs &g) {
    if (g.prec != GTG_PREC_TF32 && g.prec != GTG_PREC_BF16 && g.prec != GTG_PREC_F16) return false;
    if (g.batch > 65535 || g.batch * ((g.M + 127) / 128) * ((g.N + 63) / 64) > INT32_MAX) return false;
    if (g.M > INT32_MAX || g.N > INT32_MAX || g.K > INT32_MAX) return false;
    const int64_t elem = g.prec == GTG_PREC_TF32 ? 4 : 2;
    const int64_t ka = (g.K + 16 / elem - 1) / (16 / elem) * (16 / elem), nb = (g.N + 7) / 8 * 8;
    if (ka * elem >= (1ll << 40) || nb * 2 >= (1ll << 40)) return false;
    return g.M > 0 && g.N > 0 && g.K > 0;
}

// Operands whose base, row stride or item stride the tensor memory
// accelerator cannot take are first copied into 16-byte rows (and items of
// whole rows) from the pool: A for every precision, B for 16-bit inputs (TF32
// B goes through its transpose in any case). A shared operand (item stride 0)
// is copied once.
cudaError_t tc_launch(const DeviceInfo &dev, const GemmArgs &g, const gtg_plan &plan, cudaStream_t stream) {
    const bool tf32 = g.prec == GTG_PREC_TF32;
    const int64_t elem = tf32 ? 4 : 2;
    if (tf32) {
        // A' (rounded copy of A) and B^T (rounded), both with rows of ldk
        // elements, in one pool buffer; a shared operand is prepared once
        const int64_t ldk = (g.K + 3) / 4 * 4;
        const int64_t items_a = g.batch > 1 && g.strideA != 0 ? g.batch : 1;
        const int64_t items_b = g.batch > 1 && g.strideB != 0 ? g.batch : 1;
        const size_t a_bytes = (static_cast<size_t>(items_a * g.M * ldk) * 4 + 255) / 256 * 256;
        const size_t b_bytes = static_cast<size_t>(items_b * g.N * ldk) * 4;
        void *ws = nullptr;
        cudaError_t e = ws_alloc(&ws, a_bytes + b_bytes, stream);
        if (e != cudaSuccess) return e;
        float *Ap = static_cast<float *>(ws);
        float *Bt = reinterpret_cast<float *>(static_cast<char *>(ws) + a_bytes);
        e = tf32_prep_launch(dev, g, Ap, Bt, ldk, items_a, items_b, stream);
        GemmArgs g2 = g;
        g2.A = Ap;
        g2.lda = ldk;
        g2.strideA = items_a > 1 ? g.M * ldk : 0;
        g2.B = Bt;
        g2.ldb = ldk;
        g2.strideB = items_b > 1 ? g.N * ldk : 0;
        if (e == cudaSuccess) e = tc_launch_aligned(dev, g2, plan, stream);
        const cudaError_t f = cudaFreeAsync(ws, stream);   // stream-ordered: after the GEMM has read it
        return e != cudaSuccess ? e : f;
    }
    const bool a_bad = !tma_operand_ok(g.A, g.lda, g.strideA, g.batch, elem);
    const bool b_bad = !tf32 && !tma_operand_ok(g.B, g.ldb, g.strideB, g.batch, elem);
    if (!a_bad && !b_bad) return tc_launch_aligned(dev, g, plan, stream);
    GemmArgs g2 = g;
    void *pa = nullptr, *pb = nullptr;
    cudaError_t e = cudaSuccess;
    if (a_bad) {
        const int64_t ld = (g.K + 16 / elem - 1) / (16 / elem) * (16 / elem);
        const int64_t items = g.batch > 1 && g.strideA != 0 ? g.batch : 1;
        e = ws_alloc(&pa, static_cast<size_t>(items * g.M * ld * elem), stream);
        if (e == cudaSuccess) e = repack_launch(g.A, g.lda, g.strideA, pa, ld, g.M, g.K, items, elem, dev.status, stream);
        g2.A = pa;
        g2.lda = ld;
        g2.strideA = items > 1 ? g.M * ld : 0;
    }
    if (e == cudaSuccess && b_bad) {
        const int64_t ld = (g.N + 7) / 8 * 8;
        const int64_t items = g.batch > 1 && g.strideB != 0 ? g.batch : 1;
        e = ws_alloc(&pb, static_cast<size_t>(items * g.K * ld * 2), stream);
        if (e == cudaSuccess) e = repack_launch(g.B, g.ldb, g.strideB, pb, ld, g.K, g.N, items, 2, dev.status, stream);
        g2.B = pb;
        g2.ldb = ld;
        g2.strideB = items > 1 ? g.K * ld : 0;
    }
    if (e == cudaSuccess) e = tc_launch_aligned(dev, g2, plan, stream);
    // stream-ordered: released once the GEMM has read them
    if (pa != nullptr) {
        const cudaError_t f = cudaFreeAsync(pa, stream);
        if (e == cudaSuccess) e = f;
    }
    if (pb != nullptr) {
        const cudaError_t f = cudaFreeAsync(pb, stream);
        if (e == cudaSuccess) e = f;
    }
    return e;
}

}  // namespace gtg

// ---------------------------------------------------------------- fixed-scratch TF32 variant
// For callers that cannot allocate device memory: the B^T staging buffer of
// the TF32 path lives in a fixed array compiled into the library instead of
// coming from the memory pool. Every device that loads the library holds the
// array until the process exits; every call shares it.
namespace gtg {
namespace {
constexpr size_t kFixedScratchBytes = static_cast<size_t>(16) << 20;   // 16 MiB
}

static __device__ __align__(256) float g_tf32_fixed_scratch[kFixedScratchBytes / sizeof(float)];

size_t tf32_fixed_scratch_bytes() { return kFixedScratchBytes; }

size_t tf32_bt_bytes(int64_t N, int64_t K) {
    return static_cast<size_t>(N) * static_cast<size_t>((K + 3) / 4 * 4) * sizeof(float);
}

namespace {

// Device address of the fixed array on `device` (which must be current). In
// host code the array's name is only a host-side stand-in, so the address is
// looked up once per device and cached.
cudaError_t fixed_scratch_address(int device, float **out) {
    static std::mutex mu;
    static float *addr[64] = {};
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    if (addr[device] == nullptr) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_tf32_fixed_scratch);
        if (e != cudaSuccess) return e;
        addr[device] = static_cast<float *>(p);
    }
    *out = addr[device];
    return cudaSuccess;
}

template <int BN>
cudaError_t launch_tf32_fixed(const DeviceInfo &dev, const GemmArgs &g, const gtg_plan &plan,
                              cudaStream_t stream, float *bt, int attr_bit) {
    using S = Shape<true, BN>;
    auto kern = tc_gemm_kernel<true, BN, false, true>;   // A rounded in shared memory (no room for a copy)
    {
        AttrCache &ac = attr_cache();
        std::lock_guard<std::mutex> lk(ac.mu);
        const int d = dev.id & 63;
        if (!(ac.done[d] >> attr_bit & 1)) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
            if (e != cudaSuccess) return e;
            ac.done[d] |= 1ull << attr_bit;
        }
    }
    CUtensorMap ta, tb;
    if (!encode_3d(&ta, GTG_PREC_TF32, g.A, g.K, g.M, g.lda, 1, 0, S::BK, S::BM)) return cudaErrorInvalidValue;
    const int64_t ldbt = (g.K + 3) / 4 * 4;
    if (!encode_3d(&tb, GTG_PREC_TF32, bt, g.K, g.N, ldbt, 1, 0, S::BK, BN)) return cudaErrorInvalidValue;
    // B^T overwrites every element the GEMM reads, so the array's previous
    // contents never matter and nothing needs clearing.
    cudaError_t e = transpose_launch(static_cast<const float *>(g.B), g.ldb, bt, ldbt, g.K, g.N, 1, 0, dev.status, stream);
    if (e != cudaSuccess) return e;
    TcParams p{};
    p.C = g.C;
    p.ldc = g.ldc;
    p.M = static_cast<int>(g.M);
    p.N = static_cast<int>(g.N);
    p.num_m = static_cast<int>((g.M + S::BM - 1) / S::BM);
    p.num_n = static_cast<int>((g.N + BN - 1) / BN);
    p.num_kb = static_cast<int>((g.K + S::BK - 1) / S::BK);
    p.tiles_per_batch = p.num_m * p.num_n;
    p.num_tiles = p.tiles_per_batch;
    p.splits = 1;             // no workspace: K is never split here
    p.kps = p.num_kb;
    p.num_units = p.num_tiles;
    p.strideC = 0;
    p.idesc = S::IDESC;
    p.c_vec = c_store_width(g);
    p.tail_start = INT32_MAX;
    p.c_tma = 0;
    p.status = dev.status;
    p.wait_limit_ns = wait_limit_ns();
    p.drop_slice = take_drop_slice();
    p.bias = g.bias;
    p.act = g.act;
    kern<<<plan.grid, threads_for(true), S::SMEM, stream>>>(ta, tb, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t tc_launch_tf32_fixed_scratch(const DeviceInfo &dev, const GemmArgs &g, const gtg_plan &plan,
                                         cudaStream_t stream) {
    if (tf32_bt_bytes(g.N, g.K) > kFixedScratchBytes) return cudaErrorInvalidValue;
    float *bt = nullptr;
    const cudaError_t e = fixed_scratch_address(dev.id, &bt);
    if (e != cudaSuccess) return e;
    switch (plan.bn) {
        // attribute-cache bits of their own: these are the ROUND_A kernels
        case 256: return launch_tf32_fixed<256>(dev, g, plan, stream, bt, 11);
        case 128: return launch_tf32_fixed<128>(dev, g, plan, stream, bt, 12);
        case 64: return launch_tf32_fixed<64>(dev, g, plan, stream, bt, 13);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gtg
