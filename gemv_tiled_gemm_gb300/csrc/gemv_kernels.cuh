// Bandwidth-bound GEMV kernels: y_b = A * x_b for up to 8 vectors at once,
// with A in FP32 or BF16 and x, y and all arithmetic in FP32.
//
// "Matrix Operations" (section "Matrix-Vector Multiplication") computes
// y[i] = sum_j A[i][j] x[j] with one thread per row and, in its optimised
// form, the vector staged in shared memory once per work group so that it
// is not re-read from global memory for every row; vectors too large for
// shared memory are staged in chunks with a barrier on each side
// ("Handling Large Vectors"). The matrix, read exactly once, is the traffic
// that sets the speed.
//
// GB300 form:
//   * a warp (not a thread) owns ROWS rows at a time (or, in the ring kernel,
//     an equal range of row segments) and streams them with
//     coalesced 128-bit loads that bypass L1 (each lane keeps U x ROWS loads
//     in flight), so a row is one contiguous burst instead of the pages'
//     one-row-per-thread pattern whose neighbouring threads are a full row
//     apart;
//   * every CTA stages x (all `batch` vectors) in shared memory once; if they
//     do not fit, chunk by chunk with the barriers of the pages' chunked
//     loop, which every thread of the CTA reaches (no early return);
//   * partial sums are combined with a warp-shuffle butterfly;
//   * the grid is persistent (a multiple of the SM count) and each CTA owns
//     one contiguous, equally sized range of rows, so every SM streams the
//     same number of bytes;
//   * each matrix element loaded is used for all `batch` vectors;
//   * a 16-byte load carries 4 FP32 or 8 BF16 matrix elements; BF16 values are
//     widened to FP32 in registers (exactly), so a BF16 matrix halves the
//     bytes that bound the kernel and changes nothing else.
//
// Included by gemv.cu (FP32 matrices, and the planner) and gemv_bf16.cu
// (BF16 matrices), so that the two sets of instantiations compile in
// parallel.
#pragma once

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace gtg {
namespace gemv {

constexpr int kSmemBudget = 200 * 1024;   // per CTA, for the staged vectors

struct Params {
    const void *A;       // M x N, row-major with leading dimension lda (elements)
    long long lda;
    const float *x;
    long long ldx;
    float *y;
    long long ldy;
    int M, N;
    int chunk;           // vector entries staged per pass (multiple of 8)
    int nchunks;
    const float *bias;   // epilogue: y = act(acc + bias[row]); null for none
    int act;
    int ublock;          // gemv_blocks_kernel over a cluster: 4-column units per column block
    int x_bulk;          // x rows 16-byte aligned, ldx and N multiples of 4: stage x by bulk copies
    int *status;         // the library's device status word (set on a timed-out wait)
    unsigned long long wait_limit_ns;   // bound of every mbarrier wait
    int skip_x;          // testing hook: announce the bulk copies of x but issue none (the wait runs out)
    int dbg_shrink;      // GTG_DEBUG builds: elements taken off the checked extent of A (testing); else 0
};

// GTG_DEBUG builds: the extents every computed address of a GEMV kernel is
// checked against: the matrix (A up to its last element, less p.dbg_shrink
// elements), the outputs (batch rows of y) and the dynamic shared memory.
#ifdef GTG_DEBUG
struct DebugBounds {
    const void *a_hi;
    const float *y_hi;
    const char *s_lo, *s_hi;
};
template <typename T, int BATCH>
__device__ __forceinline__ DebugBounds debug_bounds(const Params &p, const void *smem) {
    DebugBounds d;
    const long long a_elems = p.M > 0 ? (static_cast<long long>(p.M) - 1) * p.lda + p.N - p.dbg_shrink : 0;
    d.a_hi = static_cast<const T *>(p.A) + a_elems;
    d.y_hi = p.y + static_cast<long long>(BATCH - 1) * p.ldy + p.M;
    d.s_lo = static_cast<const char *>(smem);
    d.s_hi = d.s_lo + dynamic_smem_bytes();
    return d;
}
#define GV_BOUNDS(T, BATCH, smem) const DebugBounds dbg = debug_bounds<T, BATCH>(p, smem)
#define GV_A(ptr, bytes) GTG_DEBUG_IN((ptr), (bytes), p.A, dbg.a_hi, p.status)
#define GV_Y(ptr) GTG_DEBUG_IN((ptr), 4, p.y, dbg.y_hi, p.status)
#define GV_S(ptr, bytes) GTG_DEBUG_IN((ptr), (bytes), dbg.s_lo, dbg.s_hi, p.status)
#else
#define GV_BOUNDS(T, BATCH, smem) static_cast<void>(0)
#define GV_A(ptr, bytes) true
#define GV_Y(ptr) true
#define GV_S(ptr, bytes) true
#endif

// Matrix element types. kVec = elements per 16-byte load; widen() turns one
// such load into FP32 values in column order; one() reads a single element.
template <typename T>
struct Elem;

template <>
struct Elem<float> {
    static constexpr int kVec = 4;
    static __device__ __forceinline__ void widen(const float4 &raw, float (&a)[4]) {
        a[0] = raw.x;
        a[1] = raw.y;
        a[2] = raw.z;
        a[3] = raw.w;
    }
    static __device__ __forceinline__ float one(const float *p) { return ptx::ld_stream_f1(p); }
};

// BF16 as its 16-bit pattern: two elements per 32-bit word, the lower-addressed
// one in the low half. A BF16 value is the upper half of the FP32 value with
// the same bits, so widening is a shift (or a mask) and exact.
template <>
struct Elem<uint16_t> {
    static constexpr int kVec = 8;
    static __device__ __forceinline__ float lo(uint32_t w) { return __uint_as_float(w << 16); }
    static __device__ __forceinline__ float hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
    static __device__ __forceinline__ void widen(const float4 &raw, float (&a)[8]) {
        const uint32_t w[4] = {__float_as_uint(raw.x), __float_as_uint(raw.y), __float_as_uint(raw.z),
                               __float_as_uint(raw.w)};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            a[2 * q] = lo(w[q]);
            a[2 * q + 1] = hi(w[q]);
        }
    }
    static __device__ __forceinline__ float one(const uint16_t *p) {
        return __uint_as_float(static_cast<uint32_t>(ptx::ld_stream_u16(p)) << 16);
    }
};

// Four matrix elements per load, for gemv_blocks_kernel: 16 bytes of FP32 or
// 8 bytes of BF16. With four columns per lane the lanes of a warp read x from
// shared memory in consecutive 16-byte pieces, so a 128-bit shared load takes
// four wavefronts; eight BF16 columns per lane would spread them 32 bytes
// apart and take eight.
template <typename T>
struct Quad;

template <>
struct Quad<float> {
    using Raw = float4;
    static __device__ __forceinline__ Raw load(const float *p) { return ptx::ld_stream_f4(p); }
    static __device__ __forceinline__ Raw zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
    static __device__ __forceinline__ void widen(const Raw &raw, float (&a)[4]) {
        a[0] = raw.x;
        a[1] = raw.y;
        a[2] = raw.z;
        a[3] = raw.w;
    }
};

template <>
struct Quad<uint16_t> {
    using Raw = uint2;
    static __device__ __forceinline__ Raw load(const uint16_t *p) { return ptx::ld_stream_u2(p); }
    static __device__ __forceinline__ Raw zero() { return make_uint2(0u, 0u); }
    static __device__ __forceinline__ void widen(const Raw &raw, float (&a)[4]) {
        a[0] = Elem<uint16_t>::lo(raw.x);
        a[1] = Elem<uint16_t>::hi(raw.x);
        a[2] = Elem<uint16_t>::lo(raw.y);
        a[3] = Elem<uint16_t>::hi(raw.y);
    }
};

template <typename T>
__device__ __forceinline__ float4 ld16(const T *p) {
    return ptx::ld_stream_f4(reinterpret_cast<const float *>(p));
}

template <int BATCH, int kThreads>
__device__ __forceinline__ void stage_x(float *xs, const Params &p, int c0, int len) {
#ifdef GTG_DEBUG
    const char *s_hi = reinterpret_cast<const char *>(xs) + dynamic_smem_bytes();
#endif
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
        const float *src = p.x + static_cast<long long>(b) * p.ldx + c0;
        float *dst = xs + b * p.chunk;
        for (int j = threadIdx.x; j < len; j += kThreads)
            if (GTG_DEBUG_IN(dst + j, 4, xs, s_hi, p.status)) dst[j] = __ldg(src + j);
    }
}

// Staging of all BATCH vectors by bulk copies (one per vector, issued by one
// thread, completing on one mbarrier): no registers or load instructions are
// spent on x, and the warps issue their first matrix loads while it arrives.
// The barrier must have been initialised (count 1) and made visible.
template <int BATCH>
__device__ __forceinline__ void stage_x_bulk(float *xs, const Params &p, uint32_t bar) {
    if (threadIdx.x == 0) {
        ptx::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(BATCH * p.N * 4));
        if (!p.skip_x)
#pragma unroll
            for (int b = 0; b < BATCH; ++b)
#ifdef GTG_DEBUG
                if (GTG_DEBUG_IN(xs + b * p.chunk, 4ull * p.N, xs, reinterpret_cast<const char *>(xs) + dynamic_smem_bytes(),
                                 p.status))
#endif
                    ptx::bulk_load(ptx::smem_addr(xs + b * p.chunk), p.x + static_cast<long long>(b) * p.ldx,
                                   static_cast<uint32_t>(p.N * 4), bar);
    }
}

// Waits (bounded) for the bulk-staged vectors. On time-out the status word
// records GTG_ERR_TIMEOUT, the copies are given one more bounded wait so that
// none is left writing into shared memory, and false is returned; the caller
// then skips its arithmetic but still reaches every later barrier of the CTA.
__device__ __forceinline__ bool wait_x(uint32_t bar, const Params &p) {
    if (ptx::mbar_try_wait(bar, 0)) return true;
    uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, 0)) {
        if (ptx::globaltimer_ns() - t0 > p.wait_limit_ns) {
            atomicCAS(p.status, 0, GTG_ERR_TIMEOUT);
            t0 = ptx::globaltimer_ns();
            while (!ptx::mbar_try_wait(bar, 0) && ptx::globaltimer_ns() - t0 < p.wait_limit_ns) {
            }
            return false;
        }
    }
    return true;
}

// acc[r][b] += sum over one 16-byte unit of row r (starting at column `col`
// of the staged chunk) times vector b. The x values are read from shared
// memory once per vector and serve all ROWS rows.
template <typename T, int ROWS, int BATCH>
__device__ __forceinline__ void fma_unit(float (&acc)[ROWS][BATCH], const float4 (&raw)[ROWS], const float *xs,
                                         int chunk, int col) {
    constexpr int VE = Elem<T>::kVec;
    float a[ROWS][VE];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) Elem<T>::widen(raw[r], a[r]);
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
        float xv[VE];
        const float4 *xp = reinterpret_cast<const float4 *>(xs + b * chunk + col);
#pragma unroll
        for (int q = 0; q < VE / 4; ++q) {
            const float4 v = xp[q];
            xv[4 * q] = v.x;
            xv[4 * q + 1] = v.y;
            xv[4 * q + 2] = v.z;
            xv[4 * q + 3] = v.w;
        }
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            float s = acc[r][b];
#pragma unroll
            for (int e = 0; e < VE; ++e) s = fmaf(a[r][e], xv[e], s);
            acc[r][b] = s;
        }
    }
}

// acc[r][b] += the four elements of row r at column `col` of the staged chunk
// times vector b (gemv_blocks_kernel's unit).
template <typename T, int ROWS, int BATCH>
__device__ __forceinline__ void fma_quad(float (&acc)[ROWS][BATCH], const typename Quad<T>::Raw (&raw)[ROWS],
                                         const float *xs, int chunk, int col) {
    float a[ROWS][4];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) Quad<T>::widen(raw[r], a[r]);
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
        const float4 v = *reinterpret_cast<const float4 *>(xs + b * chunk + col);
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            float s = acc[r][b];
            s = fmaf(a[r][0], v.x, s);
            s = fmaf(a[r][1], v.y, s);
            s = fmaf(a[r][2], v.z, s);
            s = fmaf(a[r][3], v.w, s);
            acc[r][b] = s;
        }
    }
}

// fma_quad with the vectors staged interleaved (XI): the BATCH values of
// column c sit together at xg + (c % 4) * BATCH, xg the base of the lane's
// group of four columns. Two vectors go through one packed FMA (the matrix
// value in both halves, the two vectors' x values, the two sums): each sum
// still takes its products in column order, one rounding each, as in
// fma_quad.
template <typename T, int ROWS, int BATCH>
__device__ __forceinline__ void fma_quad_xi(float2 (&acc)[ROWS][BATCH / 2], const typename Quad<T>::Raw (&raw)[ROWS],
                                            const float *xg) {
    static_assert(BATCH % 4 == 0, "whole 16-byte reads of x");
    float a[ROWS][4];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) Quad<T>::widen(raw[r], a[r]);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        float2 xv[BATCH / 2];
#pragma unroll
        for (int q = 0; q < BATCH / 4; ++q) {
            const float4 v = *reinterpret_cast<const float4 *>(xg + e * BATCH + 4 * q);
            xv[2 * q] = make_float2(v.x, v.y);
            xv[2 * q + 1] = make_float2(v.z, v.w);
        }
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            const float2 ad = make_float2(a[r][e], a[r][e]);
#pragma unroll
            for (int h = 0; h < BATCH / 2; ++h) acc[r][h] = __ffma2_rn(ad, xv[h], acc[r][h]);
        }
    }
}

// XI layout: floats per group of four columns (their 4 x BATCH values and 16
// bytes of padding, so that lanes reading consecutive groups meet different
// shared-memory banks).
__host__ __device__ constexpr int xi_group_floats(int batch) { return 4 * batch + 4; }

// acc[r][b] += the four elements of row r at column h + 4j times vector b,
// staged quad-transposed (entry c at (c % 4) * q + c / 4): lane j reads word
// j (+1 past the wrap) of each of four quarter rows, so the 32 lanes read
// consecutive words (gemv_blocks_kernel with PEEL).
template <typename T, int ROWS, int BATCH>
__device__ __forceinline__ void fma_quad_peeled(float (&acc)[ROWS][BATCH], const typename Quad<T>::Raw (&raw)[ROWS],
                                                const float *xs, int chunk, int q, int h, int j) {
    float a[ROWS][4];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) Quad<T>::widen(raw[r], a[r]);
    const float *xe[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) xe[e] = xs + ((h + e) & 3) * q + ((h + e) >> 2) + j;
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = xe[e][b * chunk];
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            float s = acc[r][b];
#pragma unroll
            for (int e = 0; e < 4; ++e) s = fmaf(a[r][e], v[e], s);
            acc[r][b] = s;
        }
    }
}

// Reduce-scatter over the 32 lanes of a warp for P values per lane (P a power
// of two, at most 32). Lane offsets go 16, 8, 4, 2, 1: while a lane holds more
// than one value, each level sends half of them to the partner lane and keeps
// the sum of the other half; the remaining levels are plain butterfly
// additions. Afterwards lane L holds the warp total of value L >> (5 - log2 P)
// (31 shuffles for 32 values, against 160 for a butterfly per value).
template <int P>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[P], int lane) {
#pragma unroll
    for (int lvl = 0; lvl < 5; ++lvl) {
        const int o = 16 >> lvl;
        const int k = P >> lvl;   // values per lane before this level
        if (k > 1) {
            const bool hi = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < k / 2; ++i) {
                const float send = hi ? v[i] : v[i + k / 2];
                const float keep = hi ? v[i + k / 2] : v[i];
                v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, o);
            }
        } else {
            v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], o);
        }
    }
    return v[0];
}

__host__ __device__ constexpr int pow2_at_least(int v) { return v <= 1 ? 1 : 2 * pow2_at_least((v + 1) / 2); }
__host__ __device__ constexpr int log2_of(int v) { return v <= 1 ? 0 : 1 + log2_of(v / 2); }

// The warp totals of a task's ROWS x BATCH per-lane partial sums. Returns the
// total that this lane owns and sets `vi` to its index r * BATCH + b, or to -1
// when the lane owns none (each total is owned by exactly one lane).
template <int ROWS, int BATCH>
__device__ __forceinline__ float task_total(const float (&acc)[ROWS][BATCH], int lane, int &vi) {
    constexpr int V = ROWS * BATCH;
    constexpr int P = pow2_at_least(V);
    constexpr int SHIFT = 5 - log2_of(P);
    static_assert(P <= 32, "at most 32 totals per warp");
    float v[P];
#pragma unroll
    for (int i = 0; i < P; ++i) v[i] = i < V ? acc[i / BATCH][i % BATCH] : 0.f;
    const float tot = warp_reduce_scatter<P>(v, lane);
    vi = lane >> SHIFT;
    if ((lane & ((1 << SHIFT) - 1)) != 0 || vi >= V) vi = -1;
    return tot;
}

// The task totals stored to dst[r * BATCH + b].
template <int ROWS, int BATCH>
__device__ __forceinline__ void store_task_totals(const float (&acc)[ROWS][BATCH], float *dst, int lane) {
    int vi;
    const float tot = task_total<ROWS, BATCH>(acc, lane, vi);
    if (vi >= 0) dst[vi] = tot;
}

template <typename T, int BATCH, int ROWS, int U, bool VEC>
__device__ __forceinline__ void accumulate(float (&acc)[ROWS][BATCH], const T *const (&arow)[ROWS],
                                           const float *xs, int chunk, int c0, int len, int lane, const Params &p) {
    GV_BOUNDS(T, BATCH, xs);
    if constexpr (VEC) {
        constexpr int VE = Elem<T>::kVec;
        const int nu = len / VE;
        int j = lane;
        for (; j + 32 * (U - 1) < nu; j += 32 * U) {
            float4 a[U][ROWS];
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    const T *q = arow[r] + c0 + VE * (j + 32 * u);
                    a[u][r] = GV_A(q, 16) ? ld16(q) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
            for (int u = 0; u < U; ++u) fma_unit<T, ROWS, BATCH>(acc, a[u], xs, chunk, VE * (j + 32 * u));
        }
        for (; j < nu; j += 32) {
            float4 a[ROWS];
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                const T *q = arow[r] + c0 + VE * j;
                a[r] = GV_A(q, 16) ? ld16(q) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            fma_unit<T, ROWS, BATCH>(acc, a, xs, chunk, VE * j);
        }
        const int jt = VE * nu + lane;   // fewer than VE trailing entries
        if (jt < len) {
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                const T *q = arow[r] + c0 + jt;
                const float a = GV_A(q, sizeof(T)) ? Elem<T>::one(q) : 0.f;
#pragma unroll
                for (int b = 0; b < BATCH; ++b) acc[r][b] = fmaf(a, xs[b * chunk + jt], acc[r][b]);
            }
        }
    } else {
        int j = lane;
        for (; j + 32 * (U - 1) < len; j += 32 * U) {
            float a[U][ROWS];
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    const T *q = arow[r] + c0 + j + 32 * u;
                    a[u][r] = GV_A(q, sizeof(T)) ? Elem<T>::one(q) : 0.f;
                }
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int b = 0; b < BATCH; ++b) {
                    const float xv = xs[b * chunk + j + 32 * u];
#pragma unroll
                    for (int r = 0; r < ROWS; ++r) acc[r][b] = fmaf(a[u][r], xv, acc[r][b]);
                }
        }
        for (; j < len; j += 32) {
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                const T *q = arow[r] + c0 + j;
                const float a = GV_A(q, sizeof(T)) ? Elem<T>::one(q) : 0.f;
#pragma unroll
                for (int b = 0; b < BATCH; ++b) acc[r][b] = fmaf(a, xs[b * chunk + j], acc[r][b]);
            }
        }
    }
}

// The general kernel: any row alignment, x chunked when it does not fit.
template <typename T, int BATCH, int ROWS, int U, bool VEC, int kThreads>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const Params p) {
    constexpr int kWarps = kThreads / 32;
    extern __shared__ float4 xs_raw[];
    float *xs = reinterpret_cast<float *>(xs_raw);
    const T *A = static_cast<const T *>(p.A);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    GV_BOUNDS(T, BATCH, xs);

    // this CTA's rows: [r_begin, r_end), equal shares of M
    const int r_begin = static_cast<int>(static_cast<long long>(p.M) * blockIdx.x / gridDim.x);
    const int r_end = static_cast<int>(static_cast<long long>(p.M) * (blockIdx.x + 1) / gridDim.x);
    const int ntasks = (r_end - r_begin + ROWS - 1) / ROWS;
    const int rounds = (ntasks + kWarps - 1) / kWarps;

    ptx::wait_prior_grid();
    ptx::allow_next_grid();
    if (p.nchunks == 1) {
        stage_x<BATCH, kThreads>(xs, p, 0, p.N);
        __syncthreads();
    }
    for (int round = 0; round < rounds; ++round) {  // same trip count for every warp
        const int task = round * kWarps + warp;
        const bool active = task < ntasks;
        const int row0 = r_begin + task * ROWS;
        const T *arow[ROWS];
#pragma unroll
        for (int r = 0; r < ROWS; ++r)  // rows past the range re-read the last one; never stored
            arow[r] = A + static_cast<long long>(min(row0 + r, r_end - 1)) * p.lda;

        float acc[ROWS][BATCH];
#pragma unroll
        for (int r = 0; r < ROWS; ++r)
#pragma unroll
            for (int b = 0; b < BATCH; ++b) acc[r][b] = 0.f;

        for (int c = 0; c < p.nchunks; ++c) {
            const int c0 = c * p.chunk;
            const int len = min(p.chunk, p.N - c0);
            if (p.nchunks > 1) {
                __syncthreads();              // everyone is done with the previous chunk
                stage_x<BATCH, kThreads>(xs, p, c0, len);
                __syncthreads();              // the chunk is in place
            }
            if (active) accumulate<T, BATCH, ROWS, U, VEC>(acc, arow, xs, p.chunk, c0, len, lane, p);
        }
        if (active) {
            int vi;
            const float tot = task_total<ROWS, BATCH>(acc, lane, vi);
            if (vi >= 0) {
                const int r = vi / BATCH, b = vi - r * BATCH;
                float *dst = p.y + static_cast<long long>(b) * p.ldy + row0 + r;
                if (row0 + r < r_end && GV_Y(dst)) *dst = apply_epilogue(tot, p.bias, row0 + r, p.act);
            }
        }
    }
}

// The main case for one or two vectors: 16-byte aligned rows and all of x in
// one staging chunk. A warp's work is a flat sequence of iterations (ROWS rows
// x 32*U sixteen-byte columns each); the loads of iteration it+1 are issued
// before the FMAs of iteration it, and the first loads before x is staged, so
// the matrix stream starts at once and never drains between iterations. While
// the previous kernel in the stream is still finishing, the first 4 KB of
// each of the CTA's rows is already requested into L2 (a prefetch cannot
// observe stale data: L2 is the point of coherence).
template <typename T, int BATCH, int ROWS, int U, int kThreads>
__global__ void __launch_bounds__(kThreads, 1) gemv_stream_kernel(const Params p) {
    constexpr int kWarps = kThreads / 32;
    constexpr int VE = Elem<T>::kVec;
    extern __shared__ float4 xs_raw[];
    float *xs = reinterpret_cast<float *>(xs_raw);
    const T *A = static_cast<const T *>(p.A);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    GV_BOUNDS(T, BATCH, xs);
    const int r_begin = static_cast<int>(static_cast<long long>(p.M) * blockIdx.x / gridDim.x);
    const int r_end = static_cast<int>(static_cast<long long>(p.M) * (blockIdx.x + 1) / gridDim.x);
    const int ntasks = (r_end - r_begin + ROWS - 1) / ROWS;
    const int my_tasks = ntasks > warp ? (ntasks - warp + kWarps - 1) / kWarps : 0;
    const int nu = p.N / VE;                          // whole 16-byte units per row
    // iterations per task; at least one, whose trailing-entry step covers a
    // row shorter than one unit (N < VE with padded, aligned rows)
    const int ipr = max(1, (nu + 32 * U - 1) / (32 * U));
    const int total = my_tasks * ipr;

    if (threadIdx.x < 32) {
        const uint32_t bytes = min(4096u, static_cast<uint32_t>(nu) * 16u);
        for (int r = r_begin + static_cast<int>(threadIdx.x); bytes > 0 && r < r_end; r += 32)
            ptx::prefetch_l2(A + static_cast<long long>(r) * p.lda, bytes);
    }
    ptx::wait_prior_grid();
    ptx::allow_next_grid();

    auto row_of = [&](int t, int r) { return r_begin + (warp + t * kWarps) * ROWS + r; };
    auto load = [&](int it, float4 (&dst)[U][ROWS]) {
        const int t = it / ipr, blk = it - t * ipr;
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            const T *a = A + static_cast<long long>(min(row_of(t, r), r_end - 1)) * p.lda;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int j = blk * 32 * U + 32 * u + lane;
                dst[u][r] = j < nu && GV_A(a + VE * j, 16) ? ld16(a + VE * j) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    };

    __shared__ __align__(8) unsigned long long xbar;
    const uint32_t bar = ptx::smem_addr(&xbar);
    if (p.x_bulk) {
        if (threadIdx.x == 0) {
            ptx::mbar_init(bar, 1);
            ptx::fence_barrier_init();
        }
        __syncthreads();
        stage_x_bulk<BATCH>(xs, p, bar);
    }
    float4 nxt[U][ROWS];
    if (total > 0) load(0, nxt);
    bool ok = true;
    if (p.x_bulk) {
        ok = __all_sync(0xFFFFFFFFu, wait_x(bar, p));   // warp-uniform: shuffles follow
    } else {
        stage_x<BATCH, kThreads>(xs, p, 0, p.N);
        __syncthreads();
    }
    if (!ok) return;   // no barrier follows in this kernel

    float acc[ROWS][BATCH];
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
#pragma unroll
        for (int b = 0; b < BATCH; ++b) acc[r][b] = 0.f;

    for (int it = 0; it < total; ++it) {
        float4 cur[U][ROWS];
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int r = 0; r < ROWS; ++r) cur[u][r] = nxt[u][r];
        if (it + 1 < total) load(it + 1, nxt);
        const int t = it / ipr, blk = it - t * ipr;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = blk * 32 * U + 32 * u + lane;
            if (j < nu) fma_unit<T, ROWS, BATCH>(acc, cur[u], xs, p.chunk, VE * j);
        }
        if (blk == ipr - 1) {
            // fewer than VE trailing entries when N is not a multiple of VE
            const int jt = VE * nu + lane;
            if (jt < p.N) {
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    const T *q = A + static_cast<long long>(min(row_of(t, r), r_end - 1)) * p.lda + jt;
                    const float a = GV_A(q, sizeof(T)) ? Elem<T>::one(q) : 0.f;
#pragma unroll
                    for (int b = 0; b < BATCH; ++b) acc[r][b] = fmaf(a, xs[b * p.chunk + jt], acc[r][b]);
                }
            }
            int vi;
            const float tot = task_total<ROWS, BATCH>(acc, lane, vi);
            if (vi >= 0) {
                const int r = vi / BATCH, b = vi - r * BATCH;
                const int row = row_of(t, r);
                float *dst = p.y + static_cast<long long>(b) * p.ldy + row;
                if (row < r_end && GV_Y(dst)) *dst = apply_epilogue(tot, p.bias, row, p.act);
            }
#pragma unroll
            for (int r = 0; r < ROWS; ++r)
#pragma unroll
                for (int b = 0; b < BATCH; ++b) acc[r][b] = 0.f;
        }
    }
}

// Three or more vectors (and vectors too large for one CTA's shared memory at
// any batch): the rows are split into tasks of ROWS rows x one of WC column
// segments, so every x value read from shared memory serves ROWS rows (at
// batch 8 the x reads, not the matrix, are the per-element cost) while the
// few rows per SM still give every warp work. A task's warp totals
// (reduce-scatter) go to shared memory and are added in segment order after
// a barrier, so the result does not depend on scheduling.
//
// CLUSTER: launched as clusters of C CTAs (else C = 1, a plain launch), which
// share one block of rows: CTA c of the cluster takes column block c
// (p.ublock units of VE = 4 columns; the last block takes the rest and the N % VE
// trailing entries) and stages only its 1/C of every vector. With C > 1 each
// CTA leaves one partial sum per (row, vector) in its shared memory; after a
// cluster barrier every CTA finishes a share of the rows by adding the C
// partials, read through distributed shared memory, in rank order, and a
// second cluster barrier keeps every CTA's shared memory alive until the
// others have read it. p.chunk >= (block width + 1) * VE.
//
// XI (BATCH a multiple of 4; with or without a cluster, each CTA its own
// column block): the threads stage x interleaved, the
// BATCH values of a column side by side (groups of four columns padded by 16
// bytes, so lanes reading consecutive groups meet different banks), and the
// arithmetic takes two vectors per packed FMA (fma_quad_xi): half the FMA
// instructions, the same products in the same order, so the result is
// bit-identical to the plain staging.
//
// PEEL (C = 1): rows that do not start on a boundary of the lane load (16
// bytes FP32, 8 bytes BF16). Rows kPhase = 4 apart start 4 * lda elements
// apart, a whole number of loads, so they share their offset from a load
// boundary: a task takes ROWS rows kPhase apart (rows b + i + kPhase * r of a
// block of kPhase * ROWS rows, i = 0..kPhase-1), skips their first h = 0..3
// entries (single loads) to reach aligned loads of four entries, and meets x at
// column h + 4j. x is staged quad-transposed (entry c at (c % 4) * xq + c / 4,
// xq = p.chunk / 4), so the lanes' reads of one of the four columns of a unit
// are consecutive words whatever h is. nu counts the whole units every row has
// after its head; the at most six entries past them are single loads too.
template <typename T, int BATCH, int ROWS, int WC, int U, int kThreads, bool CLUSTER, bool PEEL = false,
          bool XI = false>
__global__ void __launch_bounds__(kThreads, 1) gemv_blocks_kernel(const Params p) {
    static_assert(!PEEL || !CLUSTER, "peeled rows: one CTA per row block");
    static_assert(!XI || (!PEEL && BATCH % 4 == 0), "interleaved vectors: aligned rows, whole 16-byte reads");
    constexpr int kPhase = 4;
    constexpr unsigned kLoadBytes = 4 * sizeof(T);   // one lane load: four entries
    constexpr int kWarps = kThreads / 32;
    using Q = Quad<T>;
    using Raw = typename Q::Raw;
    constexpr int VE = 4;   // matrix elements per lane load (see Quad)
    extern __shared__ float4 xs_raw[];
    __shared__ __align__(8) unsigned long long xbar;
    const int C = CLUSTER ? static_cast<int>(ptx::cluster_nctarank()) : 1;
    const int c = CLUSTER ? static_cast<int>(ptx::cluster_ctarank()) : 0;
    const int cid = static_cast<int>(blockIdx.x) / C, ncl = static_cast<int>(gridDim.x) / C;
    const int r_begin = static_cast<int>(static_cast<long long>(p.M) * cid / ncl);
    const int r_end = static_cast<int>(static_cast<long long>(p.M) * (cid + 1) / ncl);
    const int rows = r_end - r_begin;
    const int ngroups = PEEL ? (rows + kPhase * ROWS - 1) / (kPhase * ROWS) * kPhase : (rows + ROWS - 1) / ROWS;
    const int ntasks = ngroups * WC;
    const int nu = PEEL ? (p.N >= 3 ? (p.N - 3) / VE : 0) : p.N / VE;
    const int ub0 = min(c * p.ublock, nu);                       // this CTA's units [ub0, ub1)
    const int ub1 = c == C - 1 ? nu : min(ub0 + p.ublock, nu);
    const int nub = ub1 - ub0;
    const int tail = PEEL ? 0 : (c == C - 1 ? p.N - VE * nu : 0);   // trailing entries (last block)
    const int xlen = PEEL ? p.N : VE * nub + tail;               // staged entries per vector
    const int xq = p.chunk / 4;                                  // PEEL: quads per staged vector
    const int segu = ((nub + WC - 1) / WC + 31) / 32 * 32;
    float *xs = reinterpret_cast<float *>(xs_raw);               // [BATCH][chunk]
    float *part = xs + BATCH * p.chunk;                          // [group][segment][row][batch]
    float *mine = part + static_cast<long long>(ngroups) * WC * ROWS * BATCH;   // [row][batch]
    const T *A = static_cast<const T *>(p.A) + VE * static_cast<long long>(ub0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bar = ptx::smem_addr(&xbar);
    GV_BOUNDS(T, BATCH, xs);

    if (p.x_bulk && threadIdx.x == 0) {
        ptx::mbar_init(bar, 1);
        ptx::fence_barrier_init();
    }
    // FP32 rows: the first 4 KB of this CTA's part of each row is prefetched
    // into L2 while the vectors arrive. BF16 rows: none (this kernel is then
    // bound by its per-element arithmetic and the prefetch only added L2
    // traffic; measured at batch 8, 4096^2 to 16384^2: 0.41 / 0.49 / 0.53 of
    // the copy peak with a 4 KB prefetch, 0.43 / 0.51 / 0.58 without).
    constexpr long long kPrefetch = sizeof(T) == 2 ? 0 : 4096;
    if (kPrefetch > 0 && threadIdx.x < 32) {
        // a bulk prefetch takes a 16-byte aligned start and length, so it
        // covers the 16-byte blocks inside [start, end) of the part (rows
        // start on 16 bytes, a BF16 column block may start 8 bytes past one)
        if constexpr (PEEL) {
            // each row from its first 16-byte boundary
            const long long row_bytes = static_cast<long long>(sizeof(T)) * p.N;
            for (int r = r_begin + static_cast<int>(threadIdx.x); r < r_end; r += 32) {
                const char *rp = reinterpret_cast<const char *>(A + static_cast<long long>(r) * p.lda);
                const long long lead = static_cast<long long>((16u - (reinterpret_cast<uintptr_t>(rp) & 15u)) & 15u);
                const long long span = row_bytes - lead;
                if (span >= 16) ptx::prefetch_l2(rp + lead, static_cast<uint32_t>(min(kPrefetch, span / 16 * 16)));
            }
        } else {
            const long long skew = static_cast<long long>(VE) * ub0 * static_cast<long long>(sizeof(T)) & 15;
            const long long lead = skew ? 16 - skew : 0;
            const long long span = static_cast<long long>(VE) * nub * static_cast<long long>(sizeof(T)) - lead;
            const uint32_t bytes = span >= 16 ? static_cast<uint32_t>(min(kPrefetch, span / 16 * 16)) : 0u;
            for (int r = r_begin + static_cast<int>(threadIdx.x); bytes > 0 && r < r_end; r += 32)
                ptx::prefetch_l2(reinterpret_cast<const char *>(A + static_cast<long long>(r) * p.lda) + lead, bytes);
        }
    }
    ptx::wait_prior_grid();
    ptx::allow_next_grid();
    if (p.x_bulk) {
        __syncthreads();   // the barrier is initialised
        if (threadIdx.x == 0) {
            ptx::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(BATCH * xlen * 4));
            if (xlen > 0 && !p.skip_x)
#pragma unroll
                for (int b = 0; b < BATCH; ++b)
                    if (GV_S(xs + b * p.chunk, 4ull * xlen))
                        ptx::bulk_load(ptx::smem_addr(xs + b * p.chunk),
                                       p.x + static_cast<long long>(b) * p.ldx + VE * ub0,
                                       static_cast<uint32_t>(xlen * 4), bar);
        }
    }

    const T *arow[ROWS];
    int j0 = 0, j1 = 0, h = 0;
    // PEEL: the first row of row group rg (rows first + kPhase * r)
    auto first_row = [&](int rg) { return r_begin + rg / kPhase * (kPhase * ROWS) + rg % kPhase; };
    // a task with no row in range (PEEL, fewer than kPhase * ROWS rows left) is skipped
    auto live = [&](int task) { return !PEEL || first_row(task / WC) < r_end; };
    auto setup = [&](int task) {
        const int rg = task / WC, cs = task - rg * WC;
        if constexpr (PEEL) {
            // rows past the end repeat the last row in range with the same phase
            const int first = first_row(rg);
            const int last = (r_end - 1 - first) / kPhase;
#pragma unroll
            for (int r = 0; r < ROWS; ++r)
                arow[r] = A + static_cast<long long>(first + kPhase * min(r, last)) * p.lda;
            const unsigned mis = static_cast<unsigned>(reinterpret_cast<uintptr_t>(arow[0]) & (kLoadBytes - 1));
            h = static_cast<int>(((kLoadBytes - mis) & (kLoadBytes - 1)) / sizeof(T));
#pragma unroll
            for (int r = 0; r < ROWS; ++r) arow[r] += h;   // on a load boundary
        } else {
#pragma unroll
            for (int r = 0; r < ROWS; ++r)
                arow[r] = A + static_cast<long long>(min(r_begin + rg * ROWS + r, r_end - 1)) * p.lda;
        }
        j0 = cs * segu;
        j1 = min(j0 + segu, nub);
    };
    auto load = [&](int jb, Raw (&dst)[U][ROWS]) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = jb + 32 * u + lane;
#pragma unroll
            for (int r = 0; r < ROWS; ++r)
                dst[u][r] = j < j1 && GV_A(arow[r] + VE * j, kLoadBytes) ? Q::load(arow[r] + VE * j) : Q::zero();
        }
    };

    Raw nxt[U][ROWS];
    if (warp < ntasks && live(warp)) {
        setup(warp);
        if (j0 < j1) load(j0, nxt);
    }
    bool ok = true;
    if (p.x_bulk) {
        ok = __all_sync(0xFFFFFFFFu, wait_x(bar, p));
    } else if constexpr (XI) {
        // one thread per group of four columns: a 16-byte read of each vector
        // (single reads at the end of x or for unaligned vectors), then the
        // group's columns written out interleaved
        constexpr int GS = xi_group_floats(BATCH);
        const bool vec = (reinterpret_cast<uintptr_t>(p.x) & 15) == 0 && (p.ldx & 3) == 0;
        for (int g = threadIdx.x; 4 * g < xlen; g += kThreads) {
            const int c0 = 4 * g;
            float v[BATCH][4];
#pragma unroll
            for (int b = 0; b < BATCH; ++b) {
                const float *src = p.x + static_cast<long long>(b) * p.ldx + VE * ub0 + c0;
                if (vec && c0 + 4 <= xlen) {
                    const float4 t = __ldg(reinterpret_cast<const float4 *>(src));
                    v[b][0] = t.x;
                    v[b][1] = t.y;
                    v[b][2] = t.z;
                    v[b][3] = t.w;
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) v[b][e] = c0 + e < xlen ? __ldg(src + e) : 0.f;
                }
            }
            float *dst = xs + static_cast<long long>(g) * GS;
            if (GV_S(dst, 16ull * BATCH)) {
#pragma unroll
                for (int e = 0; e < 4; ++e)
#pragma unroll
                    for (int q = 0; q < BATCH / 4; ++q)
                        *reinterpret_cast<float4 *>(dst + e * BATCH + 4 * q) =
                            make_float4(v[4 * q][e], v[4 * q + 1][e], v[4 * q + 2][e], v[4 * q + 3][e]);
            }
        }
        __syncthreads();
    } else {
#pragma unroll
        for (int b = 0; b < BATCH; ++b) {
            const float *src = p.x + static_cast<long long>(b) * p.ldx + VE * ub0;
            for (int j = threadIdx.x; j < xlen; j += kThreads) {
                float *d = xs + b * p.chunk + (PEEL ? (j & 3) * xq + (j >> 2) : j);
                if (GV_S(d, 4)) *d = __ldg(src + j);
            }
        }
        __syncthreads();
    }

    for (int task = warp; ok && task < ntasks; task += kWarps) {
        if (!live(task)) continue;
        if (task != warp) {
            setup(task);
            if (j0 < j1) load(j0, nxt);
        }
        const int cs = task % WC;
        float acc[ROWS][BATCH];
#pragma unroll
        for (int r = 0; r < ROWS; ++r)
#pragma unroll
            for (int b = 0; b < BATCH; ++b) acc[r][b] = 0.f;
        if constexpr (XI) {
            constexpr int GS = xi_group_floats(BATCH);
            float2 acc2[ROWS][BATCH / 2];
#pragma unroll
            for (int r = 0; r < ROWS; ++r)
#pragma unroll
                for (int h = 0; h < BATCH / 2; ++h) acc2[r][h] = make_float2(0.f, 0.f);
            for (int jb = j0; jb < j1; jb += 32 * U) {
                Raw cur[U][ROWS];
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int r = 0; r < ROWS; ++r) cur[u][r] = nxt[u][r];
                if (jb + 32 * U < j1) load(jb + 32 * U, nxt);
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int j = jb + 32 * u + lane;   // group j holds columns 4j .. 4j + 3
                    if (j < j1) fma_quad_xi<T, ROWS, BATCH>(acc2, cur[u], xs + static_cast<long long>(j) * GS);
                }
            }
            if (cs == WC - 1 && lane < tail) {
                const int jt = VE * nub + lane;
                const float *xc = xs + static_cast<long long>(jt >> 2) * GS + (jt & 3) * BATCH;
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    const T *q = arow[r] + jt;
                    const float a = GV_A(q, sizeof(T)) ? Elem<T>::one(q) : 0.f;
#pragma unroll
                    for (int h = 0; h < BATCH / 2; ++h)
                        acc2[r][h] = make_float2(fmaf(a, xc[2 * h], acc2[r][h].x), fmaf(a, xc[2 * h + 1], acc2[r][h].y));
                }
            }
#pragma unroll
            for (int r = 0; r < ROWS; ++r)
#pragma unroll
                for (int h = 0; h < BATCH / 2; ++h) {
                    acc[r][2 * h] = acc2[r][h].x;
                    acc[r][2 * h + 1] = acc2[r][h].y;
                }
        }
        for (int jb = j0; !XI && jb < j1; jb += 32 * U) {
            Raw cur[U][ROWS];
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int r = 0; r < ROWS; ++r) cur[u][r] = nxt[u][r];
            if (jb + 32 * U < j1) load(jb + 32 * U, nxt);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int j = jb + 32 * u + lane;
                if constexpr (PEEL) {
                    if (j < j1) fma_quad_peeled<T, ROWS, BATCH>(acc, cur[u], xs, p.chunk, xq, h, j);
                } else {
                    if (j < j1) fma_quad<T, ROWS, BATCH>(acc, cur[u], xs, p.chunk, VE * j);
                }
            }
        }
        if constexpr (PEEL) {
            // the head [0, h) and the entries past the whole units
            if (cs == WC - 1) {
                auto single = [&](int col) {
                    const float *xc = xs + (col & 3) * xq + (col >> 2);
#pragma unroll
                    for (int r = 0; r < ROWS; ++r) {
                        const T *q = arow[r] - h + col;
                        const float a = GV_A(q, sizeof(T)) ? Elem<T>::one(q) : 0.f;
#pragma unroll
                        for (int b = 0; b < BATCH; ++b) acc[r][b] = fmaf(a, xc[b * p.chunk], acc[r][b]);
                    }
                };
                if (lane < h && lane < p.N) single(lane);
                for (int col = h + VE * nu + lane; col < p.N; col += 32) single(col);
            }
        }
        if (!XI && cs == WC - 1 && lane < tail) {
            const int jt = VE * nub + lane;
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                const T *q = arow[r] + jt;
                const float a = GV_A(q, sizeof(T)) ? Elem<T>::one(q) : 0.f;
#pragma unroll
                for (int b = 0; b < BATCH; ++b) acc[r][b] = fmaf(a, xs[b * p.chunk + jt], acc[r][b]);
            }
        }
        if (GV_S(part + static_cast<long long>(task) * ROWS * BATCH, 4ull * ROWS * BATCH))
            store_task_totals<ROWS, BATCH>(acc, part + static_cast<long long>(task) * ROWS * BATCH, lane);
    }
    __syncthreads();
    if (C == 1) {
        // one CTA holds whole rows: its segment sums are the totals
        for (int idx = threadIdx.x; idx < rows * BATCH; idx += kThreads) {
            const int rl = idx / BATCH, b = idx - rl * BATCH;
            int rg, r;
            if constexpr (PEEL) {
                const int blk = rl / (kPhase * ROWS), off = rl - blk * (kPhase * ROWS);
                rg = blk * kPhase + off % kPhase;
                r = off / kPhase;
            } else {
                rg = rl / ROWS;
                r = rl - rg * ROWS;
            }
            float v = 0.f;
#pragma unroll
            for (int cs = 0; cs < WC; ++cs) v += part[((rg * WC + cs) * ROWS + r) * BATCH + b];
            float *dst = p.y + static_cast<long long>(b) * p.ldy + r_begin + rl;
            if (GV_Y(dst)) *dst = apply_epilogue(v, p.bias, r_begin + rl, p.act);
        }
        return;
    }
    // this CTA's partial per (row, vector): its segments added in order
    for (int idx = threadIdx.x; idx < rows * BATCH; idx += kThreads) {
        const int rl = idx / BATCH, b = idx - rl * BATCH;
        const int rg = rl / ROWS, r = rl - rg * ROWS;
        float v = 0.f;
#pragma unroll
        for (int cs = 0; cs < WC; ++cs) v += part[((rg * WC + cs) * ROWS + r) * BATCH + b];
        if (GV_S(mine + idx, 4)) mine[idx] = v;
    }
    ptx::cluster_sync();   // every CTA's partials are complete and visible to the cluster
    const uint32_t mine_addr = ptx::smem_addr(mine);
    for (int idx = threadIdx.x; idx < rows * BATCH; idx += kThreads) {
        const int rl = idx / BATCH, b = idx - rl * BATCH;
        if (rl % C != c) continue;   // rows are shared out round-robin over the cluster
        float v = 0.f;
        for (int cc = 0; cc < C; ++cc) v += ptx::ld_cluster_f32(ptx::map_to_rank(mine_addr, cc) + 4u * idx);
        float *dst = p.y + static_cast<long long>(b) * p.ldy + r_begin + rl;
        if (GV_Y(dst)) *dst = apply_epilogue(v, p.bias, r_begin + rl, p.act);
    }
    ptx::cluster_sync();   // no CTA leaves while another may still read its shared memory
}

// gemv_ring_kernel: how many rows a warp's range of L steps can meet when a
// row takes spr steps (a range may start inside a row).
__host__ __device__ constexpr int ring_slots(int L, int spr) { return (L + spr - 1) / spr + 1; }

// One or two vectors, 16-byte aligned rows, all of x in one CTA: the CTA's
// rows are read in steps -- a step is U x 32 consecutive 16-byte loads of
// one row, one per lane per load -- and the CTA's rows x spr steps (spr =
// steps per row), row after row, are cut into one contiguous range per warp
// of equal length (the last shorter). Every warp streams the same bytes
// whatever the row count (one row per warp would leave 5 of 32 warps idle at
// 27 rows per SM and give others two rows at 54), and a range spans few
// rows.
//
// The loads run one ring turn ahead of the arithmetic: a ring of D register
// sets of U loads each, unrolled so that every set sits in fixed registers.
// The producer is straight-line code: each load carries its predicate on the
// instruction (loads past the row's end, or past the warp's range, read
// nothing and give zeros) and the move to the next row is a select between
// two pointer increments. Lanes past the row's end read x from a block of
// zeros. When the consumer leaves a row (or its range ends) the warp totals
// of its BATCH sums go to shared memory, in the slot of (warp, row within
// the warp's range); after a barrier each (row, vector) adds the slots of
// the warps whose ranges meet its row, in warp order, so the result does not
// depend on scheduling.
template <typename T, int BATCH, int U, int D, int kThreads>
__global__ void __launch_bounds__(kThreads, 1) gemv_ring_kernel(const Params p) {
    constexpr int kWarps = kThreads / 32;
    constexpr int VE = Elem<T>::kVec;   // entries per 16-byte load
    extern __shared__ float4 xs_raw[];
    __shared__ __align__(8) unsigned long long xbar;
    __shared__ float4 xzero[2];         // x of the lanes past the end of a row
    const T *A = static_cast<const T *>(p.A);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r_begin = static_cast<int>(static_cast<long long>(p.M) * blockIdx.x / gridDim.x);
    const int r_end = static_cast<int>(static_cast<long long>(p.M) * (blockIdx.x + 1) / gridDim.x);
    const int rows = r_end - r_begin;
    const int nu = p.N / VE;                                   // whole 16-byte loads per row
    const int spr = max(1, (nu + 32 * U - 1) / (32 * U));       // steps per row (at least one: it adds the trailing entries)
    const int L = (rows * spr + kWarps - 1) / kWarps;          // steps per warp
    const int kslots = ring_slots(L, spr);                     // rows a range can meet
    const int s_first = min(warp * L, rows * spr);
    const int mine = min(s_first + L, rows * spr) - s_first;
    float *xs = reinterpret_cast<float *>(xs_raw);   // [BATCH][chunk]
    float *part = xs + BATCH * p.chunk;              // [warp][slot][batch]
    const uint32_t bar = ptx::smem_addr(&xbar);
    GV_BOUNDS(T, BATCH, xs);

    if (threadIdx.x < 2) xzero[threadIdx.x] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (p.x_bulk && threadIdx.x == 0) {
        ptx::mbar_init(bar, 1);
        ptx::fence_barrier_init();
    }
    const int row0 = s_first / spr, st0 = s_first - row0 * spr;   // where the range starts (CTA-local row)
    // While the previous kernel in the stream drains: the start of each
    // warp's range (at most 4 KB) is requested into L2.
    if (mine > 0 && lane == 0) {
        const long long j0 = 32ll * U * st0;
        const long long span = (min(32ll * U * mine, nu - j0) * 16) & ~15ll;
        if (span > 0)
            ptx::prefetch_l2(A + static_cast<long long>(r_begin + row0) * p.lda + VE * j0,
                             static_cast<uint32_t>(min(span, 4096ll)));
    }
    ptx::wait_prior_grid();
    ptx::allow_next_grid();
    if (p.x_bulk) {
        __syncthreads();   // the barrier is initialised
        if (threadIdx.x == 0) {
            ptx::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(BATCH * p.N * 4));
            if (p.N > 0 && !p.skip_x)
#pragma unroll
                for (int b = 0; b < BATCH; ++b)
                    if (GV_S(xs + b * p.chunk, 4ull * p.N))
                        ptx::bulk_load(ptx::smem_addr(xs + b * p.chunk), p.x + static_cast<long long>(b) * p.ldx,
                                       static_cast<uint32_t>(p.N * 4), bar);
        }
    }

    // producer: step ps of the current row and the lane's load address in it
    int ps = st0;
    const T *pa = A + static_cast<long long>(r_begin + row0) * p.lda + VE * (32 * U * st0 + lane);
    const long long jump = p.lda - static_cast<long long>(VE) * 32 * U * (spr - 1);
    auto issue = [&](float4 (&dst)[U], bool valid) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const T *q = pa + VE * 32 * u;
            const bool pr = valid && 32 * (U * ps + u) + lane < nu && GV_A(q, 16);
            dst[u] = ptx::ld_stream_f4_if(q, pr);
        }
        const bool wrap = ++ps == spr;
        ps = wrap ? 0 : ps;
        pa += wrap ? jump : static_cast<long long>(VE) * 32 * U;
    };

    float4 ring[D][U];
#pragma unroll
    for (int d = 0; d < D - 1; ++d) issue(ring[d], d < mine);

    bool ok = true;
    if (p.x_bulk) {
        ok = __all_sync(0xFFFFFFFFu, wait_x(bar, p));
    } else {
#pragma unroll
        for (int b = 0; b < BATCH; ++b) {
            const float *src = p.x + static_cast<long long>(b) * p.ldx;
            for (int j = threadIdx.x; j < p.N; j += kThreads)
                if (GV_S(xs + b * p.chunk + j, 4)) xs[b * p.chunk + j] = __ldg(src + j);
        }
    }
    __syncthreads();   // x (when staged by the threads) and the zero block are in place

    // consumer: CTA-local row cr, step cs
    int cr = row0, cs = st0;
    float acc[1][BATCH];
#pragma unroll
    for (int b = 0; b < BATCH; ++b) acc[0][b] = 0.f;
    const float *zero = reinterpret_cast<const float *>(xzero);
    auto consume = [&](const float4 (&cur)[U], int k) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = 32 * (U * cs + u) + lane;
            const bool in = j < nu;
            const float4 one[1] = {cur[u]};
            fma_unit<T, 1, BATCH>(acc, one, in ? xs + VE * j : zero, in ? p.chunk : 0, 0);
        }
        const bool wrap = ++cs == spr;
        if (wrap || k == mine - 1) {
            if (wrap) {
                // fewer than VE trailing entries when N is not a multiple of
                // VE: added by the warp that holds the row's last step
                const int jt = VE * nu + lane;
                if (jt < p.N) {
                    const T *q = A + static_cast<long long>(r_begin + cr) * p.lda + jt;
                    const float a = GV_A(q, sizeof(T)) ? Elem<T>::one(q) : 0.f;
#pragma unroll
                    for (int b = 0; b < BATCH; ++b) acc[0][b] = fmaf(a, xs[b * p.chunk + jt], acc[0][b]);
                }
            }
            float *slot = part + (static_cast<long long>(warp) * kslots + (cr - row0)) * BATCH;
            if (GV_S(slot, 4ull * BATCH)) store_task_totals<1, BATCH>(acc, slot, lane);
#pragma unroll
            for (int b = 0; b < BATCH; ++b) acc[0][b] = 0.f;
        }
        cs = wrap ? 0 : cs;
        cr += wrap ? 1 : 0;
    };

    if (ok) {
        // the range rounded up to whole turns of the ring; steps past its end
        // load nothing and are not consumed
        for (int base = 0; base < mine; base += D) {
#pragma unroll
            for (int d = 0; d < D; ++d) {
                issue(ring[(d + D - 1) % D], base + d + D - 1 < mine);
                if (base + d < mine) consume(ring[d], base + d);
            }
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < rows * BATCH; idx += kThreads) {
        const int rl = idx / BATCH, b = idx - rl * BATCH;
        const int w_lo = rl * spr / L, w_hi = ((rl + 1) * spr - 1) / L;   // the warps whose ranges meet row rl
        float v = 0.f;
        for (int w = w_lo; w <= w_hi; ++w)
            v += part[(static_cast<long long>(w) * kslots + (rl - w * L / spr)) * BATCH + b];
        float *dst = p.y + static_cast<long long>(b) * p.ldy + r_begin + rl;
        if (GV_Y(dst)) *dst = apply_epilogue(v, p.bias, r_begin + rl, p.act);
    }
}

// FP32 rows that are not 16-byte aligned (lda not a multiple of 4, or A off
// 16 bytes), batch 1-2, all of x in one chunk: one row per warp, each row's
// first h = 0..3 entries (up to its first 16-byte boundary) taken by single
// loads and the rest by aligned 16-byte loads (four per lane in flight, the
// next four issued before the current ones are used). x is staged at its own
// offsets, so a 16-byte unit of the row meets x at column h + 4j and x is
// read one value at a time when h != 0. nu counts the whole units that every
// row has after its head; the entries past them are single loads too.
constexpr int kPeelThreads = 1024;

template <int BATCH>
__global__ void __launch_bounds__(kPeelThreads, 1) gemv_stream_peel_kernel(const Params p) {
    constexpr int U = 4, kWarps = kPeelThreads / 32;
    extern __shared__ float4 xs_raw[];
    float *xs = reinterpret_cast<float *>(xs_raw);
    const float *A = static_cast<const float *>(p.A);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    GV_BOUNDS(float, BATCH, xs);
    const int r_begin = static_cast<int>(static_cast<long long>(p.M) * blockIdx.x / gridDim.x);
    const int r_end = static_cast<int>(static_cast<long long>(p.M) * (blockIdx.x + 1) / gridDim.x);
    const int nu = p.N >= 3 ? (p.N - 3) / 4 : 0;
    ptx::wait_prior_grid();
    ptx::allow_next_grid();
    stage_x<BATCH, kPeelThreads>(xs, p, 0, p.N);
    __syncthreads();

    for (int row = r_begin + warp; row < r_end; row += kWarps) {
        const float *a = A + static_cast<long long>(row) * p.lda;
        const int h = static_cast<int>(((16u - (reinterpret_cast<uintptr_t>(a) & 15u)) & 15u) >> 2);
        const float *av = a + h;   // 16-byte aligned
        float acc[BATCH];
#pragma unroll
        for (int b = 0; b < BATCH; ++b) acc[b] = 0.f;
        auto load = [&](int jb, float4 (&dst)[U]) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int j = jb + 32 * u + lane;
                dst[u] = j < nu && GV_A(av + 4 * j, 16) ? ptx::ld_stream_f4(av + 4 * j)
                                                        : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        };
        float4 nxt[U];
        load(0, nxt);
        for (int jb = 0; jb < nu; jb += 32 * U) {
            float4 cur[U];
#pragma unroll
            for (int u = 0; u < U; ++u) cur[u] = nxt[u];
            if (jb + 32 * U < nu) load(jb + 32 * U, nxt);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int j = jb + 32 * u + lane;
                if (j < nu) {
                    const int col = h + 4 * j;
#pragma unroll
                    for (int b = 0; b < BATCH; ++b) {
                        const float *xp = xs + b * p.chunk + col;
                        float x0, x1, x2, x3;
                        if (h == 0) {
                            const float4 xv = *reinterpret_cast<const float4 *>(xp);
                            x0 = xv.x, x1 = xv.y, x2 = xv.z, x3 = xv.w;
                        } else {
                            x0 = xp[0], x1 = xp[1], x2 = xp[2], x3 = xp[3];
                        }
                        float t = acc[b];
                        t = fmaf(cur[u].x, x0, t);
                        t = fmaf(cur[u].y, x1, t);
                        t = fmaf(cur[u].z, x2, t);
                        t = fmaf(cur[u].w, x3, t);
                        acc[b] = t;
                    }
                }
            }
        }
        // the head [0, h) and the entries past the whole units
        if (lane < h && lane < p.N) {
            const float v = GV_A(a + lane, 4) ? ptx::ld_stream_f1(a + lane) : 0.f;
#pragma unroll
            for (int b = 0; b < BATCH; ++b) acc[b] = fmaf(v, xs[b * p.chunk + lane], acc[b]);
        }
        for (int jt = h + 4 * nu + lane; jt < p.N; jt += 32) {
            const float v = GV_A(a + jt, 4) ? ptx::ld_stream_f1(a + jt) : 0.f;
#pragma unroll
            for (int b = 0; b < BATCH; ++b) acc[b] = fmaf(v, xs[b * p.chunk + jt], acc[b]);
        }
#pragma unroll
        for (int b = 0; b < BATCH; ++b) {
            float v = acc[b];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
            float *dst = p.y + static_cast<long long>(b) * p.ldy + row;
            if (lane == 0 && GV_Y(dst)) *dst = apply_epilogue(v, p.bias, row, p.act);
        }
    }
}

// Kernel choice, for aligned rows: batch <= 2 with x in one staging chunk ->
// gemv_ring_kernel (32 warps, equal step ranges) for FP32 rows and for BF16
// rows at batch 1 from 2^25 elements, else gemv_stream_kernel (32 warps, one
// row each, two BF16 rows at batch 2); batch >= 3 with x in one CTA ->
// gemv_blocks_kernel without a cluster (16 warps, 4 rows x half the columns
// per task; at batch 8 with the vectors staged interleaved, XI); x too large
// for one CTA -> gemv_blocks_kernel over a cluster (XI as well at batch 8).
// Rows off 16 bytes with x in one chunk: FP32 batch <= 2 ->
// gemv_stream_peel_kernel; FP32 batch >= 3 and BF16 -> gemv_blocks_kernel
// with PEEL. Otherwise gemv_kernel (16 warps, two rows per task, x chunked
// if needed).
constexpr int kStreamThreads = 1024;
constexpr int kRoundThreads = 512;
constexpr int kRows = 2;
constexpr int kUnroll = 4;
constexpr int kSplitRows = 4, kSplitSegs = 2;
// Loads of four columns in flight per row in gemv_blocks_kernel: two of
// 16 bytes (FP32) or four of 8 bytes (BF16), the same bytes either way
constexpr int split_unroll(int elem_bytes) { return elem_bytes == 2 ? 4 : 2; }

enum Kind { kStream = 0, kSplit = 1, kRound = 2, kCluster = 3, kPeel = 4, kPeelSplit = 5, kRing = 6, kSplitXi = 7,
            kClusterXi = 8 };

// gemv_ring_kernel: 16-byte loads per ring set and sets in the ring.
// Measured against other shapes of the ring at batch 1-2 (one process, CUDA
// events, A rotated past L2): 4 x 2 beat 1 x 8 (0.84 against 0.95 of the copy
// peak at 4096^2 FP32 batch 1) and 2 x 4 (0.93); deeper rings with fewer
// warps (512 threads x 16 or 24 sets, 256 threads x 32) were slower still.
constexpr int kRingLoads = 4, kRingDepth = 2;

template <typename T, int BATCH>
void *pick(int kind, bool vec) {
    if constexpr (BATCH <= 2) {
        if (kind == kRing) return reinterpret_cast<void *>(gemv_ring_kernel<T, BATCH, kRingLoads, kRingDepth, kStreamThreads>);
    }



    if constexpr (BATCH <= 2 && sizeof(T) == 4) {
        if (kind == kPeel) return reinterpret_cast<void *>(gemv_stream_peel_kernel<BATCH>);
    }
    if constexpr (BATCH >= 3 || sizeof(T) == 2) {
        if (kind == kPeelSplit)
            return reinterpret_cast<void *>(
                gemv_blocks_kernel<T, BATCH, kSplitRows, kSplitSegs, split_unroll(sizeof(T)), kRoundThreads, false,
                                   true>);
    }
    if constexpr (BATCH <= 2) {
        if (kind == kStream) {
            // BF16 rows at batch 2: two rows per warp, so each x value read
            // from shared memory serves both (measured, 4096^2 / 8192^2 /
            // 16384^2: 0.45 / 0.56 / 0.61 -> 0.54 / 0.84 / 0.88 of the copy
            // peak); one row per warp everywhere else (two rows were slower
            // for BF16 at batch 1 and for FP32)
            if constexpr (sizeof(T) == 2 && BATCH == 2)
                return reinterpret_cast<void *>(gemv_stream_kernel<T, BATCH, 2, 2, kStreamThreads>);
            return reinterpret_cast<void *>(gemv_stream_kernel<T, BATCH, 1, kUnroll, kStreamThreads>);
        }
    }
    if constexpr (BATCH % 4 == 0) {
        if (kind == kSplitXi)
            return reinterpret_cast<void *>(gemv_blocks_kernel<T, BATCH, kSplitRows, kSplitSegs, split_unroll(sizeof(T)),
                                                               kRoundThreads, false, false, true>);
        if (kind == kClusterXi)
            return reinterpret_cast<void *>(gemv_blocks_kernel<T, BATCH, kSplitRows, kSplitSegs, split_unroll(sizeof(T)),
                                                               kRoundThreads, true, false, true>);
    }
    if (kind == kSplit)
        return reinterpret_cast<void *>(
            gemv_blocks_kernel<T, BATCH, kSplitRows, kSplitSegs, split_unroll(sizeof(T)), kRoundThreads, false>);
    if (kind == kCluster)
        return reinterpret_cast<void *>(
            gemv_blocks_kernel<T, BATCH, kSplitRows, kSplitSegs, split_unroll(sizeof(T)), kRoundThreads, true>);
    return vec ? reinterpret_cast<void *>(gemv_kernel<T, BATCH, kRows, kUnroll, true, kRoundThreads>)
               : reinterpret_cast<void *>(gemv_kernel<T, BATCH, kRows, kUnroll, false, kRoundThreads>);
}

template <typename T>
void *kernel_for(int batch, int kind, bool vec) {
    switch (batch) {
        case 1: return pick<T, 1>(kind, vec);
        case 2: return pick<T, 2>(kind, vec);
        case 3: return pick<T, 3>(kind, vec);
        case 4: return pick<T, 4>(kind, vec);
        case 5: return pick<T, 5>(kind, vec);
        case 6: return pick<T, 6>(kind, vec);
        case 7: return pick<T, 7>(kind, vec);
        default: return pick<T, 8>(kind, vec);
    }
}

// The BF16-matrix kernels (instantiated in gemv_bf16.cu).
void *kernel_for_bf16(int batch, int kind, bool vec);

}  // namespace gemv
}  // namespace gtg
