// im2col: the patch matrix of a 2-D convolution, so that the convolutional
// layer becomes one matrix product ("GPU Matrix Multiplication: Tiling and
// Shared Memory", closing section: convolutions are mapped to matrix
// multiplication through im2col; "Matrix Operations", introduction).
//
// With channels-last input X (N x H x W x C) and weights HWIO (KH x KW x C x
// CO, which read row-major are already the K x CO matrix B), row m = (n, oh,
// ow) of the patch matrix P holds, at column k = (kh*KW + kw)*C + ci, the
// input value X[n][oh*sh - ph + kh*dh][ow*sw - pw + kw*dw][ci], or zero where
// that position lies in the padding. Then Y (N x OH x OW x CO, channels last)
// = P * B, the GEMM of the tensor-core or SIMT kernels.
//
// GB300 form: a warp per output pixel (row of P). When C fills 16-byte
// chunks (8 BF16/FP16 or 4 FP32 channels) every lane writes whole chunks, so
// a warp stores 512 contiguous bytes per instruction; each CTA first builds,
// in shared memory, a table giving for every chunk of a row its offset (dy,
// dx, channel) from the window's corner, so a row needs one 32-bit decode of
// (n, oh, ow) and, per chunk, one table read and one 16-byte load. Other
// channel counts (a first layer's C = 3) take the elements one per lane along
// the row from a table of every element's offset, so a warp's loads are
// consecutive elements of each window row of X and its stores consecutive
// elements of P. Both are bound by HBM writes of P (the reads of X are mostly
// L2 hits: each input pixel is read about KH*KW / (sh*sw) times).
#include <algorithm>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace gtg {
namespace {

struct Im2col {
    const void *X;
    void *P;
    long long ldp;                 // elements per row of P (>= K, multiple of 8)
    int N, H, W, C, OH, OW, KH, KW;
    int sh, sw, ph, pw, dh, dw;
    long long M;                   // N * OH * OW rows
    int *status;                   // the library's device status word (GTG_DEBUG checks)
};

// GTG_DEBUG builds: reads of X and writes of P are checked against their extents.
#ifdef GTG_DEBUG
#define IM_X(ptr, bytes) \
    GTG_DEBUG_IN((ptr), (bytes), g.X, static_cast<const char *>(g.X) + static_cast<long long>(g.N) * g.H * g.W * g.C * ESZ_, g.status)
#define IM_P(ptr, bytes) \
    GTG_DEBUG_IN((ptr), (bytes), g.P, static_cast<const char *>(g.P) + g.M * g.ldp * ESZ_, g.status)
#else
#define IM_X(ptr, bytes) true
#define IM_P(ptr, bytes) true
#endif

constexpr int kWarpsPerCta = 8;

// V: the unit a lane moves (uint4 = 16 bytes of channels, or one element);
// VE: elements per unit.
template <typename V, int VE>
__global__ void __launch_bounds__(32 * kWarpsPerCta) im2col_kernel(const Im2col g) {
    ptx::allow_next_grid();   // the GEMM on P may be scheduled now; it waits for this grid
    const int lane = threadIdx.x & 31;
    const long long warp0 = static_cast<long long>(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5);
    const long long nwarps = static_cast<long long>(gridDim.x) * kWarpsPerCta;
    const int cc = g.C / VE;                       // chunks per input pixel
    const int chunks = g.KH * g.KW * cc;           // chunks per row of P
    const V *X = static_cast<const V *>(g.X);
    const V zero{};
    constexpr long long ESZ_ = sizeof(V) / VE;
    for (long long m = warp0; m < g.M; m += nwarps) {
        const int ow = static_cast<int>(m % g.OW);
        const long long t = m / g.OW;
        const int oh = static_cast<int>(t % g.OH);
        const int n = static_cast<int>(t / g.OH);
        const int ih0 = oh * g.sh - g.ph, iw0 = ow * g.sw - g.pw;
        V *dst = reinterpret_cast<V *>(static_cast<char *>(g.P) + m * g.ldp * (sizeof(V) / VE));
        // this lane's first chunk, then steps of 32 chunks with carries
        int c = lane % max(cc, 1), kwh = lane / max(cc, 1);
        int kw = kwh % g.KW, kh = kwh / g.KW;
        for (int q = lane; q < chunks; q += 32) {
            const int ih = ih0 + kh * g.dh, iw = iw0 + kw * g.dw;
            const bool inside = ih >= 0 && ih < g.H && iw >= 0 && iw < g.W;
            const V *src = X + ((static_cast<long long>(n) * g.H + ih) * g.W + iw) * cc + c;
            if (IM_P(dst + q, sizeof(V))) dst[q] = inside && IM_X(src, sizeof(V)) ? *src : zero;
            c += 32;
            while (c >= cc) {   // carry into kw, then kh
                c -= cc;
                if (++kw == g.KW) {
                    kw = 0;
                    ++kh;
                }
            }
        }
    }
}

// One entry of the row table: the tap's row and column offsets from the
// window corner (oh*sh - ph, ow*sw - pw) and the element offset of the value
// from that corner pixel's first channel.
struct Tap {
    int dy_dx;   // dy in the high 16 bits, dx in the low 16 bits (both >= 0)
    int off;     // (dy * W + dx) * C + channel
};

constexpr int kMaxTaps = 6144;   // 48 KB of table

// G elements of ESZ bytes make one 16-byte output chunk; every chunk is G
// contiguous channels of one tap (C % G == 0), read with one 16-byte load.
template <int ESZ>
__global__ void __launch_bounds__(32 * kWarpsPerCta) im2col_table_kernel(const Im2col g, int K) {
    ptx::allow_next_grid();   // the GEMM on P may be scheduled now; it waits for this grid
    constexpr int G = 16 / ESZ;
    extern __shared__ Tap tab[];
    const int nchunks = (K + G - 1) / G;                 // 16-byte chunks per row (the last may run into padding)
    for (int t = threadIdx.x; t < nchunks; t += blockDim.x) {
        const int k = t * G;
        const int kh = k / (g.KW * g.C), r = k - kh * (g.KW * g.C);
        const int kw = r / g.C, ci = r - kw * g.C;
        const int dy = kh * g.dh, dx = kw * g.dw;
        tab[t].dy_dx = (dy << 16) | dx;
        tab[t].off = (dy * g.W + dx) * g.C + ci;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int nwarps = gridDim.x * kWarpsPerCta;
    const char *X = static_cast<const char *>(g.X);
    constexpr long long ESZ_ = ESZ;
    for (int m = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5); m < g.M; m += nwarps) {
        const int ow = m % g.OW, t = m / g.OW;
        const int oh = t % g.OH, n = t / g.OH;
        const int ih0 = oh * g.sh - g.ph, iw0 = ow * g.sw - g.pw;
        // element index of the window corner (it may lie in the padding; only
        // positions inside the image are read)
        const long long corner = ((static_cast<long long>(n) * g.H + ih0) * g.W + iw0) * g.C;
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<char *>(g.P) + static_cast<long long>(m) * g.ldp * ESZ);
        for (int q = lane; q < nchunks; q += 32) {
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            const Tap tp = tab[q];
            const int ih = ih0 + (tp.dy_dx >> 16), iw = iw0 + (tp.dy_dx & 0xFFFF);
            const char *src = X + (corner + tp.off) * ESZ;
            if (ih >= 0 && ih < g.H && iw >= 0 && iw < g.W && IM_X(src, 16)) v = *reinterpret_cast<const uint4 *>(src);
            if (IM_P(dst + q, 16)) dst[q] = v;
        }
    }
}

// Channel counts that do not fill 16-byte chunks (a first layer's C = 3):
// lane l of the row's warp writes elements l, l + 32, ... of the row, so the
// warp's loads are consecutive elements of X within each window row (KW * C
// values in a row of the image when dw = 1) and its stores are consecutive
// elements of P. The table holds every element's offset; elements K .. ldp-1
// of the row (padding) are written as zeros.
template <int ESZ>
__global__ void __launch_bounds__(32 * kWarpsPerCta) im2col_linear_kernel(const Im2col g, int K) {
    ptx::allow_next_grid();   // the GEMM on P may be scheduled now; it waits for this grid
    using E = typename std::conditional<ESZ == 2, uint16_t, float>::type;
    extern __shared__ Tap tab[];
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
        const int kh = k / (g.KW * g.C), r = k - kh * (g.KW * g.C);
        const int kw = r / g.C, ci = r - kw * g.C;
        const int dy = kh * g.dh, dx = kw * g.dw;
        tab[k].dy_dx = (dy << 16) | dx;
        tab[k].off = (dy * g.W + dx) * g.C + ci;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int nwarps = gridDim.x * kWarpsPerCta;
    const E *X = static_cast<const E *>(g.X);
    const int width = static_cast<int>(g.ldp);
    constexpr long long ESZ_ = ESZ;
    for (int m = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5); m < g.M; m += nwarps) {
        const int ow = m % g.OW, t = m / g.OW;
        const int oh = t % g.OH, n = t / g.OH;
        const int ih0 = oh * g.sh - g.ph, iw0 = ow * g.sw - g.pw;
        const long long corner = ((static_cast<long long>(n) * g.H + ih0) * g.W + iw0) * g.C;
        E *dst = static_cast<E *>(g.P) + static_cast<long long>(m) * g.ldp;
        // a window wholly inside the image (most rows) needs no bounds checks
        const bool interior = ih0 >= 0 && ih0 + (g.KH - 1) * g.dh < g.H && iw0 >= 0 && iw0 + (g.KW - 1) * g.dw < g.W;
        // eight steps of 32 elements: all loads first, then the stores, so a
        // row's loads are in flight together
        for (int k0 = lane; k0 < width; k0 += 32 * 8) {
            E v[8];
            if (interior) {
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int k = k0 + 32 * u;
                    v[u] = k < K && IM_X(X + corner + tab[k].off, ESZ) ? X[corner + tab[k].off] : E{};
                }
            } else {
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int k = k0 + 32 * u;
                    v[u] = E{};
                    if (k < K) {
                        const Tap tp = tab[k];
                        const int ih = ih0 + (tp.dy_dx >> 16), iw = iw0 + (tp.dy_dx & 0xFFFF);
                        if (ih >= 0 && ih < g.H && iw >= 0 && iw < g.W && IM_X(X + corner + tp.off, ESZ))
                            v[u] = X[corner + tp.off];
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (k0 + 32 * u < width && IM_P(dst + k0 + 32 * u, ESZ)) dst[k0 + 32 * u] = v[u];
        }
    }
}

template <typename V, int VE>
cudaError_t launch_typed(const DeviceInfo &dev, const Im2col &g, cudaStream_t stream) {
    const long long ctas = (g.M + kWarpsPerCta - 1) / kWarpsPerCta;
    const int grid = static_cast<int>(std::min<long long>(ctas, static_cast<long long>(dev.sms) * 16));
    im2col_kernel<V, VE><<<grid, 32 * kWarpsPerCta, 0, stream>>>(g);
    return cudaGetLastError();
}

}  // namespace

cudaError_t im2col_launch(const DeviceInfo &dev, const ConvArgs &c, void *P, int64_t ldp, cudaStream_t stream) {
    Im2col g;
    g.X = c.X;
    g.P = P;
    g.ldp = ldp;
    g.N = static_cast<int>(c.N);
    g.H = static_cast<int>(c.H);
    g.W = static_cast<int>(c.W);
    g.C = static_cast<int>(c.C);
    g.OH = static_cast<int>(c.OH);
    g.OW = static_cast<int>(c.OW);
    g.KH = static_cast<int>(c.KH);
    g.KW = static_cast<int>(c.KW);
    g.sh = static_cast<int>(c.sh);
    g.sw = static_cast<int>(c.sw);
    g.ph = static_cast<int>(c.ph);
    g.pw = static_cast<int>(c.pw);
    g.dh = static_cast<int>(c.dh);
    g.dw = static_cast<int>(c.dw);
    g.M = c.N * c.OH * c.OW;
    g.status = dev.status;
    const int esz = c.elem;
    const int ve = 16 / esz;
    const int K = static_cast<int>(c.KH * c.KW * c.C);
    // window offsets addressable by the tables (16-bit dy, dx; 32-bit element offsets)
    const bool taps_ok = (c.KH - 1) * c.dh < 32768 && (c.KW - 1) * c.dw < 32768 &&
                         ((c.KH - 1) * c.dh * c.W + (c.KW - 1) * c.dw + 1) * c.C < INT32_MAX;
    const bool vec = c.C % ve == 0 && (reinterpret_cast<uintptr_t>(c.X) & 15) == 0;
    const bool p_chunks = (reinterpret_cast<uintptr_t>(P) & 15) == 0 && (ldp * esz) % 16 == 0 &&
                          ldp >= (K + ve - 1) / ve * ve;
    const long long ctas = (g.M + kWarpsPerCta - 1) / kWarpsPerCta;
    const int grid = static_cast<int>(std::min<long long>(ctas, static_cast<long long>(dev.sms) * 16));
    if (taps_ok && vec && p_chunks && (K + ve - 1) / ve <= kMaxTaps) {
        // 16-byte chunks of channels
        const size_t smem = static_cast<size_t>((K + ve - 1) / ve) * sizeof(Tap);
        if (esz == 2) im2col_table_kernel<2><<<grid, 32 * kWarpsPerCta, smem, stream>>>(g, K);
        else im2col_table_kernel<4><<<grid, 32 * kWarpsPerCta, smem, stream>>>(g, K);
        return cudaGetLastError();
    }
    if (taps_ok && !vec && K <= kMaxTaps && ldp >= K) {
        // element by element, lanes along the row
        const size_t smem = static_cast<size_t>(K) * sizeof(Tap);
        if (esz == 2) im2col_linear_kernel<2><<<grid, 32 * kWarpsPerCta, smem, stream>>>(g, K);
        else im2col_linear_kernel<4><<<grid, 32 * kWarpsPerCta, smem, stream>>>(g, K);
        return cudaGetLastError();
    }
    // otherwise: chunk by chunk with carries (very wide windows, unaligned buffers)
    const bool vchunks = vec && p_chunks;
    if (vchunks) return esz == 2 ? launch_typed<uint4, 8>(dev, g, stream) : launch_typed<uint4, 4>(dev, g, stream);
    return esz == 2 ? launch_typed<uint16_t, 1>(dev, g, stream) : launch_typed<float, 1>(dev, g, stream);
}

}  // namespace gtg
