// gemm_host: C = act(A * B + bias) for operands in host memory, with the
// host <-> device copies overlapped with the product.
//
// A goes to the device in blocks of rows and B in panels of columns, on one
// copy stream, in the order that keeps the rows sent and the columns sent
// about equal: every output block C[i][j] needs row block i of A and panel j
// of B, so after a fraction f of each has arrived f^2 of C can be computed,
// the most that any order allows. Each arrival makes one product possible
// (a new row block times the panels already there, or a new panel times the
// rows already there); a second stream runs it and a third copies that
// region of C back to the host while the next pieces come in. With pinned
// host memory the two copy directions and the tensor cores all work at
// once. A, B and C stay whole on the device for the duration of the call
// (buffers of the library's workspace pool),
// with leading dimensions padded to 16 bytes so that the tensor-core
// kernels can take every product.
#include <algorithm>
#include <mutex>
#include <vector>

#include "internal.h"

namespace gtg {
namespace {

// Three non-blocking streams per device, created on first use and kept.
struct HostStreams {
    cudaStream_t in = nullptr, comp = nullptr, out = nullptr;
};

cudaError_t host_streams(int device, HostStreams *hs) {
    static std::mutex mu;
    static HostStreams per_dev[64];
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    HostStreams &s = per_dev[device];
    if (s.in == nullptr) {
        cudaError_t e;
        if ((e = cudaStreamCreateWithFlags(&s.in, cudaStreamNonBlocking)) != cudaSuccess) return e;
        if ((e = cudaStreamCreateWithFlags(&s.comp, cudaStreamNonBlocking)) != cudaSuccess) return e;
        if ((e = cudaStreamCreateWithFlags(&s.out, cudaStreamNonBlocking)) != cudaSuccess) return e;
    }
    *hs = s;
    return cudaSuccess;
}

// Rows per block of A (about sixteen blocks) and columns per panel of B
// (about eight panels): whole 256-wide tiles, at least one tile.
int64_t piece(int64_t n, int64_t parts) {
    int64_t r = (n + parts - 1) / parts;
    r = (r + 255) / 256 * 256;
    return std::max<int64_t>(256, std::min<int64_t>(r, std::max<int64_t>(n, 1)));
}

int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

}  // namespace

gtg_status gemm_host_pipeline(const DeviceInfo &dev, const GemmArgs &g, gtg_status (*run)(const GemmArgs &, cudaStream_t),
                              cudaError_t *cuda_error) {
    const int64_t elem = (g.prec == GTG_PREC_BF16 || g.prec == GTG_PREC_F16) ? 2 : 4;
    gtg_status st = GTG_OK;
    HostStreams hs;
    cudaError_t e = host_streams(dev.id, &hs);
    if (e != cudaSuccess) {
        *cuda_error = e;
        return GTG_ERR_LAUNCH;
    }
    const int64_t rows = piece(g.M, 16), cols = piece(g.N, 8);
    const int64_t nblk = (g.M + rows - 1) / rows, npan = (g.N + cols - 1) / cols;
    // device copies: leading dimensions padded to 16 bytes
    const int64_t ld_a = round_up(std::max<int64_t>(g.K, 1), 16 / elem), ld_b = round_up(g.N, 16 / elem),
                  ld_c = round_up(g.N, 4);
    char *dA = nullptr, *dB = nullptr;
    float *dC = nullptr, *dbias = nullptr;
    std::vector<cudaEvent_t> evs;
    auto event = [&](cudaEvent_t *ev) {
        cudaError_t r = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
        if (r == cudaSuccess) evs.push_back(*ev);
        return r;
    };
    // stream-ordered allocations on the product stream; the copy streams wait on it
    auto alloc = [&](void **p, int64_t n) {
        return ws_alloc(p, static_cast<size_t>(std::max<int64_t>(n, 256)), hs.comp);
    };
    e = alloc(reinterpret_cast<void **>(&dA), g.M * ld_a * elem);
    if (e == cudaSuccess) e = alloc(reinterpret_cast<void **>(&dB), std::max<int64_t>(g.K, 1) * ld_b * elem);
    if (e == cudaSuccess) e = alloc(reinterpret_cast<void **>(&dC), g.M * ld_c * 4);
    if (e == cudaSuccess && g.bias) e = alloc(reinterpret_cast<void **>(&dbias), g.N * 4);
    cudaEvent_t ev_alloc;
    if (e == cudaSuccess) e = event(&ev_alloc);
    if (e == cudaSuccess) e = cudaEventRecord(ev_alloc, hs.comp);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hs.in, ev_alloc, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hs.out, ev_alloc, 0);
    if (e == cudaSuccess && g.bias)
        e = cudaMemcpyAsync(dbias, g.bias, static_cast<size_t>(g.N * 4), cudaMemcpyHostToDevice, hs.in);

    // The pieces in balanced order: a panel of B when more rows than columns
    // have been sent (or every row block is there), a block of A otherwise.
    // Every copy in is queued first, each followed by an event, so that the
    // host time of queueing the products never holds the copies back.
    struct Region {
        cudaEvent_t ready;
        int64_t r0, nr, c0, nc;
    };
    std::vector<Region> regions;
    int64_t ia = 0, jb = 0;   // pieces sent
    while (e == cudaSuccess && (ia < nblk || jb < npan)) {
        const int64_t rows_sent = std::min(ia * rows, g.M), cols_sent = std::min(jb * cols, g.N);
        const bool panel = jb < npan && (ia == nblk || (ia > 0 && rows_sent > cols_sent));
        Region r{nullptr, 0, 0, 0, 0};
        if (panel) {
            const int64_t c0 = jb * cols, nc = std::min(cols, g.N - c0);
            if (g.K > 0)
                e = cudaMemcpy2DAsync(dB + c0 * elem, static_cast<size_t>(ld_b * elem),
                                      static_cast<const char *>(g.B) + c0 * elem, static_cast<size_t>(g.ldb * elem),
                                      static_cast<size_t>(nc * elem), static_cast<size_t>(g.K), cudaMemcpyHostToDevice, hs.in);
            ++jb;
            r = Region{nullptr, 0, rows_sent, c0, nc};   // the new panel times the rows already there
        } else {
            const int64_t r0 = ia * rows, nr = std::min(rows, g.M - r0);
            if (g.K > 0)
                e = cudaMemcpy2DAsync(dA + r0 * ld_a * elem, static_cast<size_t>(ld_a * elem),
                                      static_cast<const char *>(g.A) + r0 * g.lda * elem, static_cast<size_t>(g.lda * elem),
                                      static_cast<size_t>(g.K * elem), static_cast<size_t>(nr), cudaMemcpyHostToDevice, hs.in);
            ++ia;
            r = Region{nullptr, r0, nr, 0, cols_sent};   // the new rows times the panels already there
        }
        if (e == cudaSuccess && r.nr > 0 && r.nc > 0) {
            if ((e = event(&r.ready)) == cudaSuccess) e = cudaEventRecord(r.ready, hs.in);
            regions.push_back(r);
        }
    }
    // each region's product once its pieces are in, then that region of C back
    for (size_t i = 0; i < regions.size() && e == cudaSuccess && st == GTG_OK; ++i) {
        const Region &r = regions[i];
        cudaEvent_t done;
        if ((e = cudaStreamWaitEvent(hs.comp, r.ready, 0)) != cudaSuccess) break;
        GemmArgs gb = g;
        gb.M = r.nr;
        gb.N = r.nc;
        gb.A = dA + r.r0 * ld_a * elem;
        gb.lda = ld_a;
        gb.B = dB + r.c0 * elem;
        gb.ldb = ld_b;
        gb.C = dC + r.r0 * ld_c + r.c0;
        gb.ldc = ld_c;
        gb.bias = dbias ? dbias + r.c0 : nullptr;
        if ((st = run(gb, hs.comp)) != GTG_OK) break;
        if ((e = event(&done)) != cudaSuccess || (e = cudaEventRecord(done, hs.comp)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(hs.out, done, 0)) != cudaSuccess)
            break;
        e = cudaMemcpy2DAsync(g.C + r.r0 * g.ldc + r.c0, static_cast<size_t>(g.ldc * 4), gb.C,
                              static_cast<size_t>(ld_c * 4), static_cast<size_t>(r.nc * 4), static_cast<size_t>(r.nr),
                              cudaMemcpyDeviceToHost, hs.out);
    }
    // the buffers go back to the pool after everything that uses them
    cudaEvent_t ev_in, ev_out;
    cudaError_t f = event(&ev_in);
    if (f == cudaSuccess) f = event(&ev_out);
    if (f == cudaSuccess) f = cudaEventRecord(ev_in, hs.in);
    if (f == cudaSuccess) f = cudaEventRecord(ev_out, hs.out);
    if (f == cudaSuccess) f = cudaStreamWaitEvent(hs.comp, ev_in, 0);
    if (f == cudaSuccess) f = cudaStreamWaitEvent(hs.comp, ev_out, 0);
    if (dA) cudaFreeAsync(dA, hs.comp);
    if (dB) cudaFreeAsync(dB, hs.comp);
    if (dC) cudaFreeAsync(dC, hs.comp);
    if (dbias) cudaFreeAsync(dbias, hs.comp);
    const cudaError_t s1 = cudaStreamSynchronize(hs.out), s2 = cudaStreamSynchronize(hs.comp),
                      s3 = cudaStreamSynchronize(hs.in);
    for (cudaEvent_t ev : evs) cudaEventDestroy(ev);
    if (e == cudaSuccess) e = f;
    if (e == cudaSuccess) e = s1 != cudaSuccess ? s1 : (s2 != cudaSuccess ? s2 : s3);
    if (e != cudaSuccess) {
        *cuda_error = e;
        return GTG_ERR_DEVICE;
    }
    return st;
}

}  // namespace gtg
