// Bandwidth-bound FP32 GEMV: y_b = A * x_b for up to 8 vectors at once.
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
//   * a warp (not a thread) owns ROWS rows at a time and streams them with
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
//   * each matrix element loaded is used for all `batch` vectors.
#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace gtg {
namespace {

constexpr int kSmemBudget = 200 * 1024;   // per CTA, for the staged vectors

struct GemvParams {
    const float *A;
    long long lda;
    const float *x;
    long long ldx;
    float *y;
    long long ldy;
    int M, N;
    int chunk;     // vector entries staged per pass (multiple of 4)
    int nchunks;
    const float *bias;   // epilogue: y = act(acc + bias[row]); null for none
    int act;
};

template <int BATCH, int kThreads>
__device__ __forceinline__ void stage_x(float *xs, const GemvParams &p, int c0, int len) {
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
        const float *src = p.x + static_cast<long long>(b) * p.ldx + c0;
        float *dst = xs + b * p.chunk;
        for (int j = threadIdx.x; j < len; j += kThreads) dst[j] = __ldg(src + j);
    }
}

template <int BATCH, int ROWS, int U, bool VEC>
__device__ __forceinline__ void accumulate(float (&acc)[ROWS][BATCH], const float *const (&arow)[ROWS],
                                           const float *xs, int chunk, int c0, int len, int lane) {
    if constexpr (VEC) {
        const int n4 = len >> 2;
        int j = lane;
        for (; j + 32 * (U - 1) < n4; j += 32 * U) {
            float4 a[U][ROWS];
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int r = 0; r < ROWS; ++r) a[u][r] = ptx::ld_stream_f4(arow[r] + c0 + 4 * (j + 32 * u));
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int b = 0; b < BATCH; ++b) {
                    const float4 xv = reinterpret_cast<const float4 *>(xs + b * chunk)[j + 32 * u];
#pragma unroll
                    for (int r = 0; r < ROWS; ++r) {
                        float s = acc[r][b];
                        s = fmaf(a[u][r].x, xv.x, s);
                        s = fmaf(a[u][r].y, xv.y, s);
                        s = fmaf(a[u][r].z, xv.z, s);
                        s = fmaf(a[u][r].w, xv.w, s);
                        acc[r][b] = s;
                    }
                }
        }
        for (; j < n4; j += 32) {
            float4 a[ROWS];
#pragma unroll
            for (int r = 0; r < ROWS; ++r) a[r] = ptx::ld_stream_f4(arow[r] + c0 + 4 * j);
#pragma unroll
            for (int b = 0; b < BATCH; ++b) {
                const float4 xv = reinterpret_cast<const float4 *>(xs + b * chunk)[j];
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    float s = acc[r][b];
                    s = fmaf(a[r].x, xv.x, s);
                    s = fmaf(a[r].y, xv.y, s);
                    s = fmaf(a[r].z, xv.z, s);
                    s = fmaf(a[r].w, xv.w, s);
                    acc[r][b] = s;
                }
            }
        }
        const int jt = 4 * n4 + lane;   // at most 3 trailing entries
        if (jt < len) {
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                const float a = ptx::ld_stream_f1(arow[r] + c0 + jt);
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
                for (int r = 0; r < ROWS; ++r) a[u][r] = ptx::ld_stream_f1(arow[r] + c0 + j + 32 * u);
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
                const float a = ptx::ld_stream_f1(arow[r] + c0 + j);
#pragma unroll
                for (int b = 0; b < BATCH; ++b) acc[r][b] = fmaf(a, xs[b * chunk + j], acc[r][b]);
            }
        }
    }
}

template <int BATCH, int ROWS, int U, bool VEC, int kThreads>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const GemvParams p) {
    constexpr int kWarps = kThreads / 32;
    extern __shared__ float4 xs_raw[];
    float *xs = reinterpret_cast<float *>(xs_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

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
        const float *arow[ROWS];
#pragma unroll
        for (int r = 0; r < ROWS; ++r)  // rows past the range re-read the last one; never stored
            arow[r] = p.A + static_cast<long long>(min(row0 + r, r_end - 1)) * p.lda;

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
            if (active) accumulate<BATCH, ROWS, U, VEC>(acc, arow, xs, p.chunk, c0, len, lane);
        }
        if (active) {
#pragma unroll
            for (int r = 0; r < ROWS; ++r)
#pragma unroll
                for (int b = 0; b < BATCH; ++b) {
                    float s = acc[r][b];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
                    acc[r][b] = s;
                }
            // every lane now holds every total; lane (r * BATCH + b) stores one
#pragma unroll
            for (int r = 0; r < ROWS; ++r)
#pragma unroll
                for (int b = 0; b < BATCH; ++b)
                    if (lane == (r * BATCH + b) % 32 && row0 + r < r_end)
                        p.y[static_cast<long long>(b) * p.ldy + row0 + r] =
                            apply_epilogue(acc[r][b], p.bias, row0 + r, p.act);
        }
    }
}

// The main case for one or two vectors: 16-byte aligned rows and all of x in
// one staging chunk. A warp's work is a flat sequence of iterations (ROWS rows
// x 32*U float4 columns each); the loads of iteration it+1 are issued before
// the FMAs of iteration it, and the first loads before x is staged, so the
// matrix stream starts at once and never drains between iterations. While
// the previous kernel in the stream is still finishing, the first 4 KB of
// each of the CTA's rows is already requested into L2 (a prefetch cannot
// observe stale data: L2 is the point of coherence).
template <int BATCH, int ROWS, int U, int kThreads>
__global__ void __launch_bounds__(kThreads, 1) gemv_stream_kernel(const GemvParams p) {
    constexpr int kWarps = kThreads / 32;
    extern __shared__ float4 xs_raw[];
    float *xs = reinterpret_cast<float *>(xs_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r_begin = static_cast<int>(static_cast<long long>(p.M) * blockIdx.x / gridDim.x);
    const int r_end = static_cast<int>(static_cast<long long>(p.M) * (blockIdx.x + 1) / gridDim.x);
    const int ntasks = (r_end - r_begin + ROWS - 1) / ROWS;
    const int my_tasks = ntasks > warp ? (ntasks - warp + kWarps - 1) / kWarps : 0;
    const int n4 = p.N >> 2;
    const int ipr = (n4 + 32 * U - 1) / (32 * U);    // iterations per task
    const int total = my_tasks * ipr;

    if (threadIdx.x < 32) {
        const uint32_t bytes = min(4096u, static_cast<uint32_t>(n4) * 16u);
        for (int r = r_begin + static_cast<int>(threadIdx.x); bytes > 0 && r < r_end; r += 32)
            ptx::prefetch_l2(p.A + static_cast<long long>(r) * p.lda, bytes);
    }
    ptx::wait_prior_grid();
    ptx::allow_next_grid();

    auto row_of = [&](int t, int r) { return r_begin + (warp + t * kWarps) * ROWS + r; };
    auto load = [&](int it, float4 (&dst)[U][ROWS]) {
        const int t = it / ipr, blk = it - t * ipr;
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            const float *a = p.A + static_cast<long long>(min(row_of(t, r), r_end - 1)) * p.lda;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int j = blk * 32 * U + 32 * u + lane;
                dst[u][r] = j < n4 ? ptx::ld_stream_f4(a + 4 * j) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    };

    float4 nxt[U][ROWS];
    if (total > 0) load(0, nxt);
    stage_x<BATCH, kThreads>(xs, p, 0, p.N);
    __syncthreads();

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
            if (j < n4) {
#pragma unroll
                for (int b = 0; b < BATCH; ++b) {
                    const float4 xv = reinterpret_cast<const float4 *>(xs + b * p.chunk)[j];
#pragma unroll
                    for (int r = 0; r < ROWS; ++r) {
                        float s = acc[r][b];
                        s = fmaf(cur[u][r].x, xv.x, s);
                        s = fmaf(cur[u][r].y, xv.y, s);
                        s = fmaf(cur[u][r].z, xv.z, s);
                        s = fmaf(cur[u][r].w, xv.w, s);
                        acc[r][b] = s;
                    }
                }
            }
        }
        if (blk == ipr - 1) {
            // at most 3 trailing entries when N % 4 != 0
            const int jt = 4 * n4 + lane;
            if (jt < p.N) {
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    const float a = ptx::ld_stream_f1(p.A + static_cast<long long>(min(row_of(t, r), r_end - 1)) * p.lda + jt);
#pragma unroll
                    for (int b = 0; b < BATCH; ++b) acc[r][b] = fmaf(a, xs[b * p.chunk + jt], acc[r][b]);
                }
            }
#pragma unroll
            for (int r = 0; r < ROWS; ++r)
#pragma unroll
                for (int b = 0; b < BATCH; ++b) {
                    float s = acc[r][b];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
                    acc[r][b] = s;
                }
#pragma unroll
            for (int r = 0; r < ROWS; ++r)
#pragma unroll
                for (int b = 0; b < BATCH; ++b) {
                    const int row = row_of(t, r);
                    if (lane == (r * BATCH + b) % 32 && row < r_end)
                        p.y[static_cast<long long>(b) * p.ldy + row] = apply_epilogue(acc[r][b], p.bias, row, p.act);
                    acc[r][b] = 0.f;
                }
        }
    }
}

// Three or more vectors: a warp's task is ROWS rows x one of WC column
// segments, so every x value read from shared memory serves ROWS rows (the
// x reads, not the matrix, are the per-element cost at batch 8) while the
// few rows per SM still give every warp work. Each task's per-row partial
// sums go to shared memory and are added in segment order after a barrier,
// so the result does not depend on scheduling.
template <int BATCH, int ROWS, int WC, int U, int kThreads>
__global__ void __launch_bounds__(kThreads, 1) gemv_split_kernel(const GemvParams p) {
    constexpr int kWarps = kThreads / 32;
    extern __shared__ float4 xs_raw[];
    float *xs = reinterpret_cast<float *>(xs_raw);
    float *part = xs + BATCH * p.chunk;   // [group][segment][row][batch]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r_begin = static_cast<int>(static_cast<long long>(p.M) * blockIdx.x / gridDim.x);
    const int r_end = static_cast<int>(static_cast<long long>(p.M) * (blockIdx.x + 1) / gridDim.x);
    const int rows = r_end - r_begin;
    const int ngroups = (rows + ROWS - 1) / ROWS;
    const int ntasks = ngroups * WC;
    const int n4 = p.N >> 2;
    const int seg4 = ((n4 + WC - 1) / WC + 31) / 32 * 32;   // float4 columns per segment

    if (threadIdx.x < 32) {
        const uint32_t bytes = min(4096u, static_cast<uint32_t>(n4) * 16u);
        for (int r = r_begin + static_cast<int>(threadIdx.x); bytes > 0 && r < r_end; r += 32)
            ptx::prefetch_l2(p.A + static_cast<long long>(r) * p.lda, bytes);
    }
    ptx::wait_prior_grid();
    ptx::allow_next_grid();
    stage_x<BATCH, kThreads>(xs, p, 0, p.N);
    __syncthreads();

    for (int task = warp; task < ntasks; task += kWarps) {
        const int rg = task / WC, cs = task - rg * WC;
        const float *arow[ROWS];
#pragma unroll
        for (int r = 0; r < ROWS; ++r)
            arow[r] = p.A + static_cast<long long>(min(r_begin + rg * ROWS + r, r_end - 1)) * p.lda;
        const int j0 = cs * seg4, j1 = min(j0 + seg4, n4);
        float acc[ROWS][BATCH];
#pragma unroll
        for (int r = 0; r < ROWS; ++r)
#pragma unroll
            for (int b = 0; b < BATCH; ++b) acc[r][b] = 0.f;

        auto load = [&](int jb, float4 (&dst)[U][ROWS]) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int j = jb + 32 * u + lane;
#pragma unroll
                for (int r = 0; r < ROWS; ++r)
                    dst[u][r] = j < j1 ? ptx::ld_stream_f4(arow[r] + 4 * j) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        };
        float4 nxt[U][ROWS];
        if (j0 < j1) load(j0, nxt);
        for (int jb = j0; jb < j1; jb += 32 * U) {
            float4 cur[U][ROWS];
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int r = 0; r < ROWS; ++r) cur[u][r] = nxt[u][r];
            if (jb + 32 * U < j1) load(jb + 32 * U, nxt);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int j = jb + 32 * u + lane;
                if (j < j1) {
#pragma unroll
                    for (int b = 0; b < BATCH; ++b) {
                        const float4 xv = reinterpret_cast<const float4 *>(xs + b * p.chunk)[j];
#pragma unroll
                        for (int r = 0; r < ROWS; ++r) {
                            float s = acc[r][b];
                            s = fmaf(cur[u][r].x, xv.x, s);
                            s = fmaf(cur[u][r].y, xv.y, s);
                            s = fmaf(cur[u][r].z, xv.z, s);
                            s = fmaf(cur[u][r].w, xv.w, s);
                            acc[r][b] = s;
                        }
                    }
                }
            }
        }
        if (cs == WC - 1) {
            const int jt = 4 * n4 + lane;   // at most 3 trailing entries
            if (jt < p.N) {
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    const float a = ptx::ld_stream_f1(arow[r] + jt);
#pragma unroll
                    for (int b = 0; b < BATCH; ++b) acc[r][b] = fmaf(a, xs[b * p.chunk + jt], acc[r][b]);
                }
            }
        }
        float *dst = part + static_cast<long long>(task) * ROWS * BATCH;
#pragma unroll
        for (int r = 0; r < ROWS; ++r)
#pragma unroll
            for (int b = 0; b < BATCH; ++b) {
                float v = acc[r][b];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
                if (lane == (r * BATCH + b) % 32) dst[r * BATCH + b] = v;
            }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < rows * BATCH; idx += kThreads) {
        const int rl = idx / BATCH, b = idx - rl * BATCH;
        const int rg = rl / ROWS, r = rl - rg * ROWS;
        float v = 0.f;
#pragma unroll
        for (int cs = 0; cs < WC; ++cs) v += part[((rg * WC + cs) * ROWS + r) * BATCH + b];
        p.y[static_cast<long long>(b) * p.ldy + r_begin + rl] = apply_epilogue(v, p.bias, r_begin + rl, p.act);
    }
}

// Kernel choice, for aligned rows with x in one staging chunk: batch <= 2 ->
// gemv_stream_kernel (32 warps, one row each); batch >= 3 ->
// gemv_split_kernel (16 warps, 4 rows x half the columns per task).
// Otherwise gemv_kernel (16 warps, two rows per task, x chunked if needed).
constexpr int kStreamThreads = 1024;
constexpr int kRoundThreads = 512;
constexpr int kRows = 2;
constexpr int kUnroll = 4;
constexpr int kSplitRows = 4, kSplitSegs = 2, kSplitUnroll = 2;

enum class GemvKind { Stream, Split, Round };

template <int BATCH>
void *pick(GemvKind kind, bool vec) {
    if constexpr (BATCH <= 2) {
        if (kind == GemvKind::Stream)
            return reinterpret_cast<void *>(gemv_stream_kernel<BATCH, 1, kUnroll, kStreamThreads>);
    }
    if (kind == GemvKind::Split)
        return reinterpret_cast<void *>(gemv_split_kernel<BATCH, kSplitRows, kSplitSegs, kSplitUnroll, kRoundThreads>);
    return vec ? reinterpret_cast<void *>(gemv_kernel<BATCH, kRows, kUnroll, true, kRoundThreads>)
               : reinterpret_cast<void *>(gemv_kernel<BATCH, kRows, kUnroll, false, kRoundThreads>);
}

void *kernel_for(int batch, GemvKind kind, bool vec) {
    switch (batch) {
        case 1: return pick<1>(kind, vec);
        case 2: return pick<2>(kind, vec);
        case 3: return pick<3>(kind, vec);
        case 4: return pick<4>(kind, vec);
        case 5: return pick<5>(kind, vec);
        case 6: return pick<6>(kind, vec);
        case 7: return pick<7>(kind, vec);
        default: return pick<8>(kind, vec);
    }
}

bool gemv_vec(const GemvArgs &g) {
    return (reinterpret_cast<uintptr_t>(g.A) & 15) == 0 && (g.lda & 3) == 0;
}

struct Layout {
    int chunk, nchunks, smem;
    GemvKind kind;
    int threads;
};

Layout layout(const DeviceInfo &dev, const GemvArgs &g) {
    const int64_t per_entry = 4ll * g.batch;
    int64_t chunk = std::max<int64_t>(4, kSmemBudget / per_entry / 4 * 4);
    const int64_t n_pad = (g.N + 3) / 4 * 4;
    if (chunk > n_pad) chunk = n_pad;
    if (chunk < 4) chunk = 4;
    Layout l;
    l.chunk = static_cast<int>(chunk);
    l.nchunks = static_cast<int>(g.N == 0 ? 1 : (g.N + chunk - 1) / chunk);
    l.smem = static_cast<int>(chunk * per_entry);
    l.kind = GemvKind::Round;
    l.threads = kRoundThreads;
    if (gemv_vec(g) && l.nchunks == 1) {
        if (g.batch <= 2) {
            l.kind = GemvKind::Stream;
            l.threads = kStreamThreads;
        } else {
            // partial sums of one CTA's rows: groups x segments x rows x batch floats
            const int64_t rows_cta = (g.M + dev.sms - 1) / dev.sms;
            const int64_t part = (rows_cta + kSplitRows - 1) / kSplitRows * kSplitSegs * kSplitRows * g.batch * 4;
            if (l.smem + part <= dev.smem_optin) {
                l.kind = GemvKind::Split;
                l.smem = static_cast<int>(l.smem + part);
            }
        }
    }
    return l;
}

}  // namespace

void gemv_plan(const DeviceInfo &dev, const GemvArgs &g, gtg_plan *plan) {
    const Layout l = layout(dev, g);
    // One CTA per SM (it fills the register file); every CTA owns an equal
    // share of the rows.
    int64_t grid = dev.sms;
    if (grid > g.M) grid = g.M;
    plan->kernel = GTG_KERNEL_GEMV;
    plan->bm = l.kind == GemvKind::Stream ? 1 : (l.kind == GemvKind::Split ? kSplitRows : kRows);
    plan->bn = l.chunk;
    plan->bk = l.kind == GemvKind::Split ? kSplitUnroll : kUnroll;
    plan->stages = l.nchunks;
    plan->grid = static_cast<int>(std::max<int64_t>(grid, 1));
    plan->threads = l.threads;
    plan->smem = l.smem;
}

cudaError_t gemv_launch(const DeviceInfo &dev, const GemvArgs &g, const gtg_plan &plan,
                        cudaStream_t stream) {
    const Layout l = layout(dev, g);
    void *kern = kernel_for(g.batch, l.kind, gemv_vec(g));
    if (l.smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, l.smem);
        if (e != cudaSuccess) return e;
    }
    GemvParams p;
    p.A = g.A;
    p.lda = g.lda;
    p.x = g.x;
    p.ldx = g.ldx;
    p.y = g.y;
    p.ldy = g.ldy;
    p.M = static_cast<int>(g.M);
    p.N = static_cast<int>(g.N);
    p.chunk = l.chunk;
    p.nchunks = l.nchunks;
    p.bias = g.bias;
    p.act = g.act;
    void *args[] = {&p};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(plan.threads);
    cfg.dynamicSmemBytes = static_cast<size_t>(l.smem);
    cfg.stream = stream;
    // may start while the previous kernel in the stream drains; every GEMV
    // kernel waits for it (griddepcontrol.wait) before reading or writing data
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, kern, args);
}

}  // namespace gtg
