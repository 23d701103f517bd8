// GEMV planning and launch, and the FP32-matrix instantiations of the GEMV
// kernels (the kernels themselves and their design are in gemv_kernels.cuh).
#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <tuple>

#include "gemv_kernels.cuh"

namespace gtg {

namespace {
std::atomic<int> g_gemv_skip_x{0};
}

void gemv_skip_next_x(int on) { g_gemv_skip_x.store(on ? 1 : 0); }
std::atomic<int> g_gemv_path{0};
void gemv_force_path(int mode) { g_gemv_path.store(mode >= 1 && mode <= 4 ? mode : 0); }
int take_gemv_skip_x() { return g_gemv_skip_x.exchange(0); }

namespace {

using namespace gemv;

// Room left in shared memory for the kernels' static variables (one mbarrier).
constexpr int kStaticSmemMargin = 1024;

// 16-byte loads are possible when the matrix starts on a 16-byte boundary and
// every row does too.
bool gemv_vec(const GemvArgs &g) {
    return (reinterpret_cast<uintptr_t>(g.A) & 15) == 0 && (g.lda * g.a_elem) % 16 == 0;
}

struct Layout {
    int chunk, nchunks, smem;
    int kind;
    int threads;
    int grid;
    int cluster;   // CTAs per cluster (column blocks); 1 unless kind is kCluster or kClusterXi
    int ublock;    // kCluster, kClusterXi: 4-column units per column block
};

void *kernel_of(const GemvArgs &g, int kind) {
    return g.a_elem == 2 ? kernel_for_bf16(g.batch, kind, gemv_vec(g)) : kernel_for<float>(g.batch, kind, gemv_vec(g));
}

// How many clusters of `cluster` CTAs with `smem` bytes each can be resident at
// once. Not every cluster size tiles the GPU's SMs: on a 152-SM GB300 all 76
// pairs fit but only 36 of 38 quads, so the grid is sized to what fits (a
// second wave of clusters would double the time). Cached per configuration.
int max_active_clusters(const DeviceInfo &dev, const GemvArgs &g, int kind, int cluster, int smem, int grid) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, int, int, int>, int> cache;
    const auto key = std::make_tuple(dev.id, g.a_elem, g.batch, kind, cluster, smem);
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    void *kern = kernel_of(g, kind);
    int n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(kRoundThreads);
        cfg.dynamicSmemBytes = static_cast<size_t>(smem);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = cluster;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();   // a refused query only rules this cluster size out
    std::lock_guard<std::mutex> lock(mu);
    cache[key] = n;
    return n;
}

// Shared memory of gemv_blocks_kernel over a cluster: x blocks, per-task partials, per-row partials.
int cluster_smem(const GemvArgs &g, int rows_cl, int chunk) {
    const int64_t groups = (rows_cl + kSplitRows - 1) / kSplitRows;
    return static_cast<int>((g.batch * int64_t{chunk} + groups * kSplitSegs * kSplitRows * g.batch +
                             int64_t{rows_cl} * g.batch) * 4);
}

Layout layout(const DeviceInfo &dev, const GemvArgs &g) {
    const int64_t per_entry = 4ll * g.batch;
    const int limit = dev.smem_optin - kStaticSmemMargin;
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
    l.grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(dev.sms, g.M)));
    l.cluster = 1;
    l.ublock = 0;
    if (!gemv_vec(g)) {
        // rows off 16 bytes with x in one chunk: kernels that peel each row's
        // head to reach aligned loads (FP32 batch 1-2: streaming, one row per
        // warp; FP32 batch 3-8 and BF16: row blocks of rows four apart, if
        // their partial sums fit beside x)
        if (l.nchunks == 1) {
            if (g.a_elem == 4 && g.batch <= 2) {
                l.kind = kPeel;
                l.threads = kPeelThreads;
                return l;
            }
            const int64_t rows_cta = (g.M + dev.sms - 1) / dev.sms;
            const int64_t groups = (rows_cta + 4 * kSplitRows - 1) / (4 * kSplitRows) * 4;
            const int64_t part = groups * kSplitSegs * kSplitRows * g.batch * 4;
            if (l.smem + part <= limit) {
                l.kind = kPeelSplit;
                l.smem = static_cast<int>(l.smem + part);
            }
        }
        return l;
    }
    // one or two vectors with x in one CTA: equal step ranges per warp, loads
    // in a ring (FP32 rows at batch 1-2 from any size, BF16 rows at batch 1
    // from 2^25 elements; measured against the streaming kernel: FP32 4096^2 /
    // 8192^2 / 16384^2 batch 1 0.92 / 0.97 / 1.01 -> 0.95 / 1.04 / 1.06 of the
    // copy peak, BF16 16384 x 4096 batch 1 0.75 -> 0.89; BF16 4096^2 batch 1
    // 0.65 -> 0.62 and batch 2 0.54 -> 0.42 stay on the streaming kernel)
    if (l.nchunks == 1 && g.batch <= 2 && g_gemv_path.load() != 3 &&
        (g.a_elem == 4 || (g.batch == 1 && g.M * g.N >= (int64_t{1} << 25)))) {
        const int64_t rows_cta = (g.M + l.grid - 1) / l.grid;
        const int64_t nu = g.N / (16 / g.a_elem);
        const int64_t spr = std::max<int64_t>(1, (nu + 32 * kRingLoads - 1) / (32 * kRingLoads));
        const int64_t warps = kStreamThreads / 32;
        const int64_t L = (rows_cta * spr + warps - 1) / warps;
        const int64_t part = warps * ((L + spr - 1) / spr + 1) * g.batch * 4;
        if (l.smem + part <= limit) {
            l.kind = kRing;
            l.threads = kStreamThreads;
            l.smem = static_cast<int>(l.smem + part);
            return l;
        }
    }
    if (l.nchunks == 1) {
        if (g.batch <= 2) {
            l.kind = kStream;
            l.threads = kStreamThreads;
            return l;
        }
        // partial sums of one CTA's rows: groups x segments x rows x batch floats
        const int64_t rows_cta = (g.M + dev.sms - 1) / dev.sms;
        const int64_t part = (rows_cta + kSplitRows - 1) / kSplitRows * kSplitSegs * kSplitRows * g.batch * 4;
        if (g.batch == 8 && g_gemv_path.load() != 4) {
            // the vectors staged interleaved, two per packed FMA (gemv_blocks_kernel
            // with XI). Measured against the vectors staged one after another
            // (one process, both forms, A rotated past L2, us): batch 8 FP32
            // 4096^2 13.6 -> 13.2, 16384 x 4096 43.7 -> 42.5; BF16 4096^2
            // 11.9 -> 11.3, 16384 x 4096 37.4 -> 32.4; but batch 4 FP32 / BF16
            // 4096^2 11.4 / 8.4 -> 12.2 / 9.1 (the threads' staging of x costs
            // more than the packed FMAs save), so batch 4 keeps the bulk copies
            const int64_t xi_floats = (g.N + 3) / 4 * xi_group_floats(g.batch);
            const int64_t xi_chunk = ((xi_floats + g.batch - 1) / g.batch + 3) / 4 * 4;
            const int64_t smem = xi_chunk * g.batch * 4 + part;
            if (smem <= limit) {
                l.kind = kSplitXi;
                l.chunk = static_cast<int>(xi_chunk);
                l.smem = static_cast<int>(smem);
                return l;
            }
        }
        if (l.smem + part <= limit) {
            l.kind = kSplit;
            l.smem = static_cast<int>(l.smem + part);
            return l;
        }
    }
    // x does not fit one CTA: split the columns over the CTAs of a cluster
    // (units of the blocks kernel's four-column loads)
    // (units of the blocks kernel's four-column loads); at batch 8 each CTA's
    // block of the vectors is staged interleaved (XI) where it fits, else as
    // one vector after another
    const int VE = 4;
    const int64_t nu = g.N / VE;
    const bool xi_ok = g.batch == 8 && g_gemv_path.load() != 4;
    for (int C = 2; C <= 8; C *= 2) {
        const int ub = static_cast<int>((nu + C - 1) / C);
        for (int xi = xi_ok ? 1 : 0; xi >= 0; --xi) {
            int grid = dev.sms / C * C;
            if (grid == 0) continue;
            // staged floats per vector: the block's units and the trailing entries
            const int cchunk = xi ? static_cast<int>(((int64_t{ub} + 1) * xi_group_floats(g.batch) + g.batch - 1) /
                                                     g.batch + 3) / 4 * 4
                                  : ((ub + 1) * VE + 7) / 8 * 8;
            const int kind = xi ? kClusterXi : kCluster;
            int smem = cluster_smem(g, static_cast<int>((g.M + grid / C - 1) / (grid / C)), cchunk);
            if (smem > limit) continue;
            const int fit = max_active_clusters(dev, g, kind, C, smem, grid);
            if (fit <= 0) continue;
            if (fit < grid / C) {
                grid = fit * C;
                smem = cluster_smem(g, static_cast<int>((g.M + fit - 1) / fit), cchunk);
                if (smem > limit) continue;
            }
            l.kind = kind;
            l.cluster = C;
            l.grid = grid;
            l.chunk = cchunk;
            l.nchunks = 1;
            l.ublock = ub;
            l.smem = smem;
            return l;
        }
    }
    return l;   // the round kernel, x staged chunk by chunk
}

}  // namespace

void gemv_plan(const DeviceInfo &dev, const GemvArgs &g, gtg_plan *plan) {
    const int path = g_gemv_path.load();
    if ((path == 0 || path == 2) && gemv_tc_eligible(dev, g, path == 2)) {
        gemv_tc_plan(dev, g, plan);
        return;
    }
    const Layout l = layout(dev, g);
    // One CTA per SM (it fills the register file); every CTA (cluster) owns an
    // equal share of the rows.
    plan->kernel = GTG_KERNEL_GEMV;
    plan->splits = 1;
    if (l.kind == kRing) {
        plan->bm = 1;
        plan->bn = l.chunk;
        plan->bk = kRingLoads * (kRingDepth - 1);
        plan->stages = 1;
        plan->grid = l.grid;
        plan->threads = l.threads;
        plan->smem = l.smem;
        plan->cluster = 1;
        return;
    }
    const bool two_rows = l.kind == kStream && g.a_elem == 2 && g.batch == 2;   // see pick() in gemv_kernels.cuh
    plan->bm = l.kind == kStream ? (two_rows ? 2 : 1) : (l.kind == kPeel ? 1 : (l.kind == kRound ? kRows : kSplitRows));
    plan->bn = l.chunk;
    const bool blocks = l.kind == kSplit || l.kind == kSplitXi || l.kind == kCluster || l.kind == kClusterXi ||
                        l.kind == kPeelSplit;
    plan->bk = blocks ? split_unroll(g.a_elem) : (two_rows ? 2 : kUnroll);
    plan->stages = l.nchunks;
    plan->grid = l.grid;
    plan->threads = l.threads;
    plan->smem = l.smem;
    plan->cluster = l.cluster;
}

cudaError_t gemv_launch(const DeviceInfo &dev, const GemvArgs &g, const gtg_plan &plan,
                        cudaStream_t stream) {
    if (plan.kernel == GTG_KERNEL_TCGEN05) return gemv_tc_launch(dev, g, stream);
    const Layout l = layout(dev, g);
    void *kern = kernel_of(g, l.kind);
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
    p.ublock = l.ublock;
    // bulk copies of x need 16-byte aligned rows of a multiple of 16 bytes
    // (the peeled kernels stage x themselves: at its own offsets, or quad-transposed)
    p.x_bulk = (l.kind == kStream || l.kind == kSplit || l.kind == kCluster || l.kind == kRing) &&
               (reinterpret_cast<uintptr_t>(g.x) & 15) == 0 && g.N % 4 == 0 &&
               (g.batch == 1 || g.ldx % 4 == 0);
    p.status = dev.status;
    p.wait_limit_ns = wait_limit_setting();
    p.skip_x = p.x_bulk ? take_gemv_skip_x() : 0;
    p.dbg_shrink = debug_shrink_setting();
    void *args[] = {&p};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(plan.threads);
    cfg.dynamicSmemBytes = static_cast<size_t>(l.smem);
    cfg.stream = stream;
    // may start while the previous kernel in the stream drains; every GEMV
    // kernel waits for it (griddepcontrol.wait) before reading or writing data
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = l.cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = l.kind == kCluster || l.kind == kClusterXi ? 2 : 1;
    return cudaLaunchKernelExC(&cfg, kern, args);
}

}  // namespace gtg
