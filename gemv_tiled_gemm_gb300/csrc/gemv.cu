// GEMV planning and launch, and the FP32-matrix instantiations of the GEMV
// kernels (the kernels themselves and their design are in gemv_kernels.cuh).
#include <algorithm>

#include "gemv_kernels.cuh"

namespace gtg {
namespace {

using namespace gemv;

// 16-byte loads are possible when the matrix starts on a 16-byte boundary and
// every row does too.
bool gemv_vec(const GemvArgs &g) {
    return (reinterpret_cast<uintptr_t>(g.A) & 15) == 0 && (g.lda * g.a_elem) % 16 == 0;
}

struct Layout {
    int chunk, nchunks, smem;
    int kind;
    int threads;
};

Layout layout(const DeviceInfo &dev, const GemvArgs &g) {
    const int64_t per_entry = 4ll * g.batch;
    // a multiple of 8 entries keeps every chunk start on a 16-byte unit of
    // either matrix type
    int64_t chunk = std::max<int64_t>(8, kSmemBudget / per_entry / 8 * 8);
    const int64_t n_pad = (g.N + 7) / 8 * 8;
    if (chunk > n_pad) chunk = n_pad;
    if (chunk < 8) chunk = 8;
    Layout l;
    l.chunk = static_cast<int>(chunk);
    l.nchunks = static_cast<int>(g.N == 0 ? 1 : (g.N + chunk - 1) / chunk);
    l.smem = static_cast<int>(chunk * per_entry);
    l.kind = kRound;
    l.threads = kRoundThreads;
    if (gemv_vec(g) && l.nchunks == 1) {
        if (g.batch <= 2) {
            l.kind = kStream;
            l.threads = kStreamThreads;
        } else {
            // partial sums of one CTA's rows: groups x segments x rows x batch floats
            const int64_t rows_cta = (g.M + dev.sms - 1) / dev.sms;
            const int64_t part = (rows_cta + kSplitRows - 1) / kSplitRows * kSplitSegs * kSplitRows * g.batch * 4;
            if (l.smem + part <= dev.smem_optin) {
                l.kind = kSplit;
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
    plan->bm = l.kind == kStream ? 1 : (l.kind == kSplit ? kSplitRows : kRows);
    plan->bn = l.chunk;
    plan->bk = l.kind == kSplit ? split_unroll(g.a_elem) : kUnroll;
    plan->stages = l.nchunks;
    plan->grid = static_cast<int>(std::max<int64_t>(grid, 1));
    plan->threads = l.threads;
    plan->smem = l.smem;
}

cudaError_t gemv_launch(const DeviceInfo &dev, const GemvArgs &g, const gtg_plan &plan,
                        cudaStream_t stream) {
    const Layout l = layout(dev, g);
    void *kern = g.a_elem == 2 ? kernel_for_bf16(g.batch, l.kind, gemv_vec(g))
                               : kernel_for<float>(g.batch, l.kind, gemv_vec(g));
    if (l.smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, l.smem);
        if (e != cudaSuccess) return e;
    }
    Params p;
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
    // bulk copies of x need 16-byte aligned rows of a multiple of 16 bytes
    p.x_bulk = l.kind != kRound && (reinterpret_cast<uintptr_t>(g.x) & 15) == 0 && g.N % 4 == 0 &&
               (g.batch == 1 || g.ldx % 4 == 0);
    p.status = dev.status;
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
