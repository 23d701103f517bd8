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
// GB300 form: a warp per output pixel; each lane moves 16-byte chunks of
// channels (8 BF16/FP16 or 4 FP32 values) when C allows, single elements
// otherwise; consecutive lanes read consecutive chunks of one input pixel's
// channels and write consecutive chunks of the row, so both sides coalesce.
// The (kh, kw, channel) position of a lane's chunk advances by carries,
// without a division per chunk. The kernel is bound by HBM writes of P
// (the reads of X are mostly L2 hits: each input pixel is read KH*KW times).
#include <algorithm>

#include "internal.h"

namespace gtg {
namespace {

struct Im2col {
    const void *X;
    void *P;
    long long ldp;                 // elements per row of P (>= K, multiple of 8)
    int N, H, W, C, OH, OW, KH, KW;
    int sh, sw, ph, pw, dh, dw;
    long long M;                   // N * OH * OW rows
};

constexpr int kWarpsPerCta = 8;

// V: the unit a lane moves (uint4 = 16 bytes of channels, or one element);
// VE: elements per unit.
template <typename V, int VE>
__global__ void __launch_bounds__(32 * kWarpsPerCta) im2col_kernel(const Im2col g) {
    const int lane = threadIdx.x & 31;
    const long long warp0 = static_cast<long long>(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5);
    const long long nwarps = static_cast<long long>(gridDim.x) * kWarpsPerCta;
    const int cc = g.C / VE;                       // chunks per input pixel
    const int chunks = g.KH * g.KW * cc;           // chunks per row of P
    const V *X = static_cast<const V *>(g.X);
    const V zero{};
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
            dst[q] = inside ? X[((static_cast<long long>(n) * g.H + ih) * g.W + iw) * cc + c] : zero;
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
    const int esz = c.elem;
    const int ve = 16 / esz;
    // 16-byte chunks need C a multiple of the chunk and 16-byte aligned X and P rows
    const bool vec = c.C % ve == 0 && (reinterpret_cast<uintptr_t>(c.X) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(P) & 15) == 0 && (ldp * esz) % 16 == 0;
    if (vec) return esz == 2 ? launch_typed<uint4, 8>(dev, g, stream) : launch_typed<uint4, 4>(dev, g, stream);
    return esz == 2 ? launch_typed<uint16_t, 1>(dev, g, stream) : launch_typed<float, 1>(dev, g, stream);
}

}  // namespace gtg
