// C ABI of libgtg: argument validation, kernel choice and launch.
// The operations and their argument conventions are documented in gtg.h.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "gtg.h"
#include "gtg_testing.h"
#include "internal.h"

namespace gtg {
namespace {

// Device status word: kernels latch an error code here (e.g. a pipeline wait
// that ran out of time); gtg_sync_status() reads and clears it. A file-scope
// device variable, so reporting errors never needs an allocation.
__device__ int g_device_status = 0;

thread_local char t_cuda_error[256] = "no error";
std::atomic<int> g_force_simt{0};

void note_text(const char *text) {
    std::strncpy(t_cuda_error, text, sizeof(t_cuda_error) - 1);
    t_cuda_error[sizeof(t_cuda_error) - 1] = '\0';
}

void note_cuda_error(cudaError_t e) { note_text(cudaGetErrorString(e)); }

// The failure-path hooks act only when GTG_TESTING=1 is in the environment.
bool testing_enabled() {
    const char *v = std::getenv("GTG_TESTING");
    return v != nullptr && std::strcmp(v, "1") == 0;
}

// Host-side fault injection: when the countdown reaches zero, the dispatch
// that took it there fails with GTG_ERR_LAUNCH before launching anything.
// GTG_FAULT_INJECT=<n> in the environment arms it once, at the first dispatch.
std::atomic<long long> g_inject_countdown{0};
std::atomic<int> g_debug_shrink{0};   // GTG_DEBUG builds: see gtg_test_debug_shrink_extent
std::once_flag g_inject_env_once;

void read_fault_inject_env() {
    std::call_once(g_inject_env_once, [] {
        const char *v = std::getenv("GTG_FAULT_INJECT");
        if (v == nullptr) return;
        const long long n = std::strtoll(v, nullptr, 10);
        if (n > 0) g_inject_countdown.store(n);
    });
}

bool injected_failure() {
    read_fault_inject_env();
    long long c = g_inject_countdown.load();
    while (c > 0) {
        if (g_inject_countdown.compare_exchange_weak(c, c - 1)) {
            if (c != 1) return false;
            note_text("injected launch failure");
            return true;
        }
    }
    return false;
}

struct DeviceTable {
    std::mutex mu;
    std::vector<DeviceInfo> devs;
};
DeviceTable &device_table() {
    static DeviceTable t;
    return t;
}

// Facts about the current device, gathered once per device.
gtg_status current_device(DeviceInfo *out) {
    int id = -1;
    cudaError_t e = cudaGetDevice(&id);
    if (e != cudaSuccess) {
        note_cuda_error(e);
        return GTG_ERR_DEVICE;
    }
    DeviceTable &t = device_table();
    std::lock_guard<std::mutex> lk(t.mu);
    for (const DeviceInfo &d : t.devs)
        if (d.id == id) {
            *out = d;
            return GTG_OK;
        }
    DeviceInfo d;
    d.id = id;
    if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, id)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, id)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, id)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, id)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.l2_bytes, cudaDevAttrL2CacheSize, id)) != cudaSuccess ||
        (e = cudaGetSymbolAddress(reinterpret_cast<void **>(&d.status), g_device_status)) != cudaSuccess) {
        note_cuda_error(e);
        return GTG_ERR_DEVICE;
    }
    t.devs.push_back(d);
    *out = d;
    return GTG_OK;
}

// Byte range [lo, hi) spanned by a rows x cols matrix with leading dimension ld.
struct Span {
    uintptr_t lo, hi;
};
Span span_of(const void *p, int64_t rows, int64_t cols, int64_t ld, int64_t elem) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    if (rows <= 0 || cols <= 0) return {lo, lo};
    const uint64_t n = static_cast<uint64_t>((rows - 1) * ld + cols) * static_cast<uint64_t>(elem);
    return {lo, lo + n};
}
bool overlaps(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi && a.lo != a.hi && b.lo != b.hi; }

gtg_status validate_gemm(const GemmArgs &g) {
    if (g.M < 0 || g.N < 0 || g.K < 0) return GTG_ERR_INVALID_VALUE;
    if (g.M > INT32_MAX || g.N > INT32_MAX || g.K > INT32_MAX) return GTG_ERR_INVALID_VALUE;
    if (g.lda < (g.K > 1 ? g.K : 1) || g.ldb < (g.N > 1 ? g.N : 1) || g.ldc < (g.N > 1 ? g.N : 1))
        return GTG_ERR_INVALID_VALUE;
    if (g.M == 0 || g.N == 0) return GTG_OK;  // nothing to write
    if (g.C == nullptr) return GTG_ERR_INVALID_VALUE;
    if (g.K > 0 && (g.A == nullptr || g.B == nullptr)) return GTG_ERR_INVALID_VALUE;
    const int64_t in_elem = (g.prec == GTG_PREC_BF16 || g.prec == GTG_PREC_F16) ? 2 : 4;
    if ((reinterpret_cast<uintptr_t>(g.A) % in_elem) || (reinterpret_cast<uintptr_t>(g.B) % in_elem) ||
        (reinterpret_cast<uintptr_t>(g.C) % 4))
        return GTG_ERR_MISALIGNED;
    const Span c = span_of(g.C, g.M, g.N, g.ldc, 4);
    if (g.K > 0 && (overlaps(c, span_of(g.A, g.M, g.K, g.lda, in_elem)) ||
                    overlaps(c, span_of(g.B, g.K, g.N, g.ldb, in_elem))))
        return GTG_ERR_ALIAS;
    if (g.act != GTG_ACT_NONE && g.act != GTG_ACT_RELU) return GTG_ERR_INVALID_VALUE;
    if (g.bias) {
        if (reinterpret_cast<uintptr_t>(g.bias) % 4) return GTG_ERR_MISALIGNED;
        if (overlaps(c, span_of(g.bias, 1, g.N, g.N, 4))) return GTG_ERR_ALIAS;
    }
    return GTG_OK;
}

// A strided batch: every item is a valid single product (checked on item 0;
// the others differ only by the strides), the outputs are pairwise apart,
// and no output overlaps any input.
gtg_status validate_batched(const GemmArgs &g) {
    if (g.batch < 0 || g.strideA < 0 || g.strideB < 0 || g.strideC < 0) return GTG_ERR_INVALID_VALUE;
    if (g.batch == 0 || g.M == 0 || g.N == 0) return GTG_OK;
    GemmArgs one = g;
    one.batch = 1;
    gtg_status st = validate_gemm(one);
    if (st != GTG_OK || g.batch == 1) return st;
    const int64_t in_elem = (g.prec == GTG_PREC_BF16 || g.prec == GTG_PREC_F16) ? 2 : 4;
    if (g.strideC < (g.M - 1) * g.ldc + g.N) return GTG_ERR_INVALID_VALUE;   // outputs would overlap
    auto whole = [&](const void *p, int64_t rows, int64_t cols, int64_t ld, int64_t stride, int64_t elem) {
        Span first = span_of(p, rows, cols, ld, elem);
        first.hi += static_cast<uint64_t>((g.batch - 1) * stride * elem);
        return first;
    };
    const Span c = whole(g.C, g.M, g.N, g.ldc, g.strideC, 4);
    if (g.K > 0 && (overlaps(c, whole(g.A, g.M, g.K, g.lda, g.strideA, in_elem)) ||
                    overlaps(c, whole(g.B, g.K, g.N, g.ldb, g.strideB, in_elem))))
        return GTG_ERR_ALIAS;
    if (g.bias && overlaps(c, span_of(g.bias, 1, g.N, g.N, 4))) return GTG_ERR_ALIAS;
    const int64_t last = (g.batch - 1) * g.strideC + (g.M - 1) * g.ldc + g.N;
    if (last > (int64_t{1} << 62)) return GTG_ERR_INVALID_VALUE;
    return GTG_OK;
}

gtg_status validate_gemv(const GemvArgs &g) {
    if (g.M < 0 || g.N < 0 || g.M > INT32_MAX || g.N > INT32_MAX) return GTG_ERR_INVALID_VALUE;
    if (g.batch < 1 || g.batch > 8) return GTG_ERR_INVALID_VALUE;
    if (g.lda < (g.N > 1 ? g.N : 1)) return GTG_ERR_INVALID_VALUE;
    if (g.batch > 1 && (g.ldx < g.N || g.ldy < g.M)) return GTG_ERR_INVALID_VALUE;
    if (g.M == 0) return GTG_OK;
    if (g.y == nullptr) return GTG_ERR_INVALID_VALUE;
    if (g.N > 0 && (g.A == nullptr || g.x == nullptr)) return GTG_ERR_INVALID_VALUE;
    if ((reinterpret_cast<uintptr_t>(g.A) % g.a_elem) || (reinterpret_cast<uintptr_t>(g.x) % 4) ||
        (reinterpret_cast<uintptr_t>(g.y) % 4))
        return GTG_ERR_MISALIGNED;
    const int64_t ldx = g.batch > 1 ? g.ldx : g.N, ldy = g.batch > 1 ? g.ldy : g.M;
    const Span y = span_of(g.y, g.batch, g.M, ldy, 4);
    if (g.N > 0 && (overlaps(y, span_of(g.A, g.M, g.N, g.lda, g.a_elem)) ||
                    overlaps(y, span_of(g.x, g.batch, g.N, ldx, 4))))
        return GTG_ERR_ALIAS;
    if (g.act != GTG_ACT_NONE && g.act != GTG_ACT_RELU) return GTG_ERR_INVALID_VALUE;
    if (g.bias) {
        if (reinterpret_cast<uintptr_t>(g.bias) % 4) return GTG_ERR_MISALIGNED;
        if (overlaps(y, span_of(g.bias, 1, g.M, g.M, 4))) return GTG_ERR_ALIAS;
    }
    return GTG_OK;
}

gtg_status plan_gemm_impl(const DeviceInfo &dev, const GemmArgs &g, gtg_plan *plan, bool may_repack = true) {
    std::memset(plan, 0, sizeof(*plan));
    if (g.M == 0 || g.N == 0) {
        plan->kernel = GTG_KERNEL_NONE;
        return GTG_OK;
    }
    if (g.K == 0) {
        plan->kernel = GTG_KERNEL_ZERO_FILL;
        return GTG_OK;
    }
    if (!(dev.cc_major == 10 && dev.cc_minor == 3)) return GTG_ERR_UNSUPPORTED;
    if (g.prec != GTG_PREC_F32 && !g_force_simt.load() && tc_supported(dev) &&
        (tc_eligible(g) || (may_repack && tc_eligible_repacked(g))))
        tc_plan(dev, g, plan);
    else
        simt_plan(dev, g, plan);
    return GTG_OK;
}

gtg_status run_gemm(const GemmArgs &g, cudaStream_t stream) {
    gtg_status st = g.batch == 1 ? validate_gemm(g) : validate_batched(g);
    if (st != GTG_OK) return st;
    if (g.M == 0 || g.N == 0 || g.batch == 0) return GTG_OK;
    if (injected_failure()) return GTG_ERR_LAUNCH;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != GTG_OK) return st;
    gtg_plan plan;
    if ((st = plan_gemm_impl(dev, g, &plan)) != GTG_OK) return st;
    cudaError_t e = cudaSuccess;
    switch (plan.kernel) {
        case GTG_KERNEL_ZERO_FILL:
            for (int64_t b = 0; b < g.batch && e == cudaSuccess; ++b) {
                float *Cb = g.C + b * g.strideC;
                e = (g.bias || g.act) ? epilogue_fill_launch(Cb, g.M, g.N, g.ldc, g.bias, 1, g.act, stream)
                                      : zero_fill_launch(Cb, g.M, g.N, g.ldc, stream);
            }
            break;
        case GTG_KERNEL_TCGEN05: e = tc_launch(dev, g, plan, stream); break;
        case GTG_KERNEL_SIMT: e = simt_launch(dev, g, plan, stream); break;
        default: break;
    }
    if (e != cudaSuccess) {
        note_cuda_error(e);
        return GTG_ERR_LAUNCH;
    }
    return GTG_OK;
}

}  // namespace

int debug_shrink_setting() { return g_debug_shrink.load(); }

}  // namespace gtg

using namespace gtg;

extern "C" {

gtg_status gemm_f32(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B,
                    int64_t ldb, float *C, int64_t ldc, cudaStream_t stream) {
    return run_gemm(GemmArgs{GTG_PREC_F32, M, N, K, A, lda, B, ldb, C, ldc}, stream);
}

gtg_status gemm_tf32(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B,
                     int64_t ldb, float *C, int64_t ldc, cudaStream_t stream) {
    return run_gemm(GemmArgs{GTG_PREC_TF32, M, N, K, A, lda, B, ldb, C, ldc}, stream);
}

gtg_status gemm_bf16(int64_t M, int64_t N, int64_t K, const gtg_bf16 *A, int64_t lda,
                     const gtg_bf16 *B, int64_t ldb, float *C, int64_t ldc, cudaStream_t stream) {
    return run_gemm(GemmArgs{GTG_PREC_BF16, M, N, K, A, lda, B, ldb, C, ldc}, stream);
}

static gtg_status run_gemv(const GemvArgs &g, cudaStream_t stream) {
    const int64_t M = g.M, N = g.N;
    const int batch = g.batch;
    gtg_status st = validate_gemv(g);
    if (st != GTG_OK || M == 0) return st;
    if (injected_failure()) return GTG_ERR_LAUNCH;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != GTG_OK) return st;
    if (!(dev.cc_major == 10 && dev.cc_minor == 3)) return GTG_ERR_UNSUPPORTED;
    cudaError_t e;
    if (N == 0) {
        // empty sums: every output is act(0 + bias) (zero without an epilogue)
        e = (g.bias || g.act) ? epilogue_fill_launch(g.y, batch, M, g.ldy, g.bias, 1, g.act, stream)
                              : zero_fill_launch(g.y, batch, M, g.ldy, stream);
    } else {
        gtg_plan plan;
        gemv_plan(dev, g, &plan);
        e = gemv_launch(dev, g, plan, stream);
    }
    if (e != cudaSuccess) {
        note_cuda_error(e);
        return GTG_ERR_LAUNCH;
    }
    return GTG_OK;
}

// The plan of gemm_tf32_noalloc: never a K split (split partial products
// would need a workspace) and never the CTA-pair kernel (the fixed-scratch
// launch runs the single-CTA tensor-core kernel), no repacked operands.
static gtg_status plan_noalloc_impl(const DeviceInfo &dev, const GemmArgs &g, gtg_plan *plan) {
    gtg_status st = plan_gemm_impl(dev, g, plan, false);
    if (st != GTG_OK) return st;
    // the tensor-core kernel reads the caller's A through TMA (16-byte base and
    // rows); gemm_tf32 would copy another layout, which needs pool memory
    const bool a_tma = (reinterpret_cast<uintptr_t>(g.A) & 15) == 0 && (g.lda * 4) % 16 == 0;
    if (plan->kernel == GTG_KERNEL_TCGEN05 && !a_tma) simt_plan(dev, g, plan);
    if (plan->kernel == GTG_KERNEL_TCGEN05) {
        tc_plan_unsplit_single(dev, g, plan);
    } else if (plan->kernel == GTG_KERNEL_SIMT && plan->splits > 1) {
        // one K range: the SIMT kernel then writes C directly
        plan->grid /= plan->splits;
        plan->splits = 1;
    }
    return GTG_OK;
}

gtg_status gemm_tf32_noalloc(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B,
                             int64_t ldb, float *C, int64_t ldc, cudaStream_t stream) {
    const GemmArgs g{GTG_PREC_TF32, M, N, K, A, lda, B, ldb, C, ldc};
    gtg_status st = validate_gemm(g);
    if (st != GTG_OK) return st;
    if (M == 0 || N == 0) return GTG_OK;
    if (tf32_bt_bytes(N, K) > tf32_fixed_scratch_bytes()) return GTG_ERR_SCRATCH_LIMIT;
    if (injected_failure()) return GTG_ERR_LAUNCH;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != GTG_OK) return st;
    gtg_plan plan;
    if ((st = plan_noalloc_impl(dev, g, &plan)) != GTG_OK) return st;
    cudaError_t e = cudaSuccess;
    switch (plan.kernel) {
        case GTG_KERNEL_ZERO_FILL: e = zero_fill_launch(g.C, g.M, g.N, g.ldc, stream); break;
        case GTG_KERNEL_TCGEN05: e = tc_launch_tf32_fixed_scratch(dev, g, plan, stream); break;
        case GTG_KERNEL_SIMT: e = simt_launch(dev, g, plan, stream); break;
        default: break;
    }
    if (e != cudaSuccess) {
        note_cuda_error(e);
        return GTG_ERR_LAUNCH;
    }
    return GTG_OK;
}

gtg_status gtg_plan_gemm_tf32_noalloc(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                                      const float *B, int64_t ldb, const float *C, int64_t ldc, gtg_plan *plan) {
    if (plan == nullptr) return GTG_ERR_INVALID_VALUE;
    const GemmArgs g{GTG_PREC_TF32, M, N, K, A, lda, B, ldb, const_cast<float *>(C), ldc};
    gtg_status st = validate_gemm(g);
    if (st != GTG_OK) return st;
    std::memset(plan, 0, sizeof(*plan));
    if (M == 0 || N == 0) return GTG_OK;
    if (tf32_bt_bytes(N, K) > tf32_fixed_scratch_bytes()) return GTG_ERR_SCRATCH_LIMIT;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != GTG_OK) return st;
    return plan_noalloc_impl(dev, g, plan);
}

gtg_status gemv_f32(int64_t M, int64_t N, const float *A, int64_t lda, const float *x, int64_t ldx,
                    float *y, int64_t ldy, int batch, cudaStream_t stream) {
    return run_gemv(GemvArgs{M, N, A, lda, x, batch > 1 ? ldx : N, y, batch > 1 ? ldy : M, batch}, stream);
}

gtg_status gemv_f32_ex(int64_t M, int64_t N, const float *A, int64_t lda, const float *x, int64_t ldx,
                       float *y, int64_t ldy, int batch, const gtg_epilogue *ep, cudaStream_t stream) {
    GemvArgs g{M, N, A, lda, x, batch > 1 ? ldx : N, y, batch > 1 ? ldy : M, batch};
    if (ep) {
        g.bias = ep->bias;
        g.act = ep->activation;
    }
    return run_gemv(g, stream);
}

gtg_status gemv_bf16(int64_t M, int64_t N, const gtg_bf16 *A, int64_t lda, const float *x, int64_t ldx,
                     float *y, int64_t ldy, int batch, cudaStream_t stream) {
    GemvArgs g{M, N, A, lda, x, batch > 1 ? ldx : N, y, batch > 1 ? ldy : M, batch};
    g.a_elem = 2;
    return run_gemv(g, stream);
}

gtg_status gemv_bf16_ex(int64_t M, int64_t N, const gtg_bf16 *A, int64_t lda, const float *x, int64_t ldx,
                        float *y, int64_t ldy, int batch, const gtg_epilogue *ep, cudaStream_t stream) {
    GemvArgs g{M, N, A, lda, x, batch > 1 ? ldx : N, y, batch > 1 ? ldy : M, batch};
    g.a_elem = 2;
    if (ep) {
        g.bias = ep->bias;
        g.act = ep->activation;
    }
    return run_gemv(g, stream);
}

// Testing hook: 0 chooses the convolution path, 1 always writes the patch
// matrix, 2 requires the implicit GEMM (GTG_ERR_UNSUPPORTED otherwise), 3 and
// 4 require it on single-CTA tiles or on CTA pairs.
static std::atomic<int> g_conv_mode{0};

static gtg_status validate_conv(ConvArgs &c) {
    if (c.prec < GTG_PREC_F32 || c.prec > GTG_PREC_F16) return GTG_ERR_INVALID_VALUE;
    c.elem = c.prec == GTG_PREC_BF16 || c.prec == GTG_PREC_F16 ? 2 : 4;
    if (c.N < 0 || c.H < 1 || c.W < 1 || c.C < 1 || c.CO < 0 || c.KH < 1 || c.KW < 1) return GTG_ERR_INVALID_VALUE;
    if (c.sh < 1 || c.sw < 1 || c.dh < 1 || c.dw < 1 || c.ph < 0 || c.pw < 0) return GTG_ERR_INVALID_VALUE;
    const int64_t lim = INT32_MAX;
    if (c.H > lim || c.W > lim || c.C > lim || c.CO > lim || c.KH > lim || c.KW > lim || c.sh > lim ||
        c.sw > lim || c.dh > lim || c.dw > lim || c.ph > lim || c.pw > lim || c.N > lim)
        return GTG_ERR_INVALID_VALUE;
    const int64_t span_h = c.H + 2 * c.ph - c.dh * (c.KH - 1) - 1, span_w = c.W + 2 * c.pw - c.dw * (c.KW - 1) - 1;
    if (span_h < 0 || span_w < 0) return GTG_ERR_INVALID_VALUE;   // the window does not fit the padded image
    c.OH = span_h / c.sh + 1;
    c.OW = span_w / c.sw + 1;
    // the product's sizes: M = N*OH*OW rows, K = KH*KW*C
    if (c.N * c.OH * c.OW > lim || c.KH * c.KW * c.C > lim) return GTG_ERR_INVALID_VALUE;
    if (c.act != GTG_ACT_NONE && c.act != GTG_ACT_RELU) return GTG_ERR_INVALID_VALUE;
    if (c.N == 0 || c.CO == 0) return GTG_OK;
    if (!c.X || !c.Wt || !c.Y) return GTG_ERR_INVALID_VALUE;
    if (reinterpret_cast<uintptr_t>(c.X) % c.elem || reinterpret_cast<uintptr_t>(c.Wt) % c.elem ||
        reinterpret_cast<uintptr_t>(c.Y) % 4 || (c.bias && reinterpret_cast<uintptr_t>(c.bias) % 4))
        return GTG_ERR_MISALIGNED;
    const Span y = span_of(c.Y, c.N * c.OH * c.OW, c.CO, c.CO, 4);
    if (overlaps(y, span_of(c.X, c.N * c.H * c.W, c.C, c.C, c.elem)) ||
        overlaps(y, span_of(c.Wt, c.KH * c.KW * c.C, c.CO, c.CO, c.elem)) ||
        (c.bias && overlaps(y, span_of(c.bias, 1, c.CO, c.CO, 4))))
        return GTG_ERR_ALIAS;
    return GTG_OK;
}

static GemmArgs with_epilogue(GemmArgs g, const gtg_epilogue *ep) {
    if (ep) {
        g.bias = ep->bias;
        g.act = ep->activation;
    }
    return g;
}

gtg_status gemm_f16(int64_t M, int64_t N, int64_t K, const gtg_f16 *A, int64_t lda, const gtg_f16 *B,
                    int64_t ldb, float *C, int64_t ldc, cudaStream_t stream) {
    return run_gemm(GemmArgs{GTG_PREC_F16, M, N, K, A, lda, B, ldb, C, ldc}, stream);
}

gtg_status gemm_f16_ex(int64_t M, int64_t N, int64_t K, const gtg_f16 *A, int64_t lda, const gtg_f16 *B,
                       int64_t ldb, float *C, int64_t ldc, const gtg_epilogue *ep, cudaStream_t stream) {
    return run_gemm(with_epilogue(GemmArgs{GTG_PREC_F16, M, N, K, A, lda, B, ldb, C, ldc}, ep), stream);
}

gtg_status gemm_strided_batched(int precision, int64_t M, int64_t N, int64_t K, const void *A, int64_t lda,
                                int64_t strideA, const void *B, int64_t ldb, int64_t strideB, float *C,
                                int64_t ldc, int64_t strideC, int64_t batch, const gtg_epilogue *ep,
                                cudaStream_t stream) {
    if (precision < GTG_PREC_F32 || precision > GTG_PREC_F16) return GTG_ERR_INVALID_VALUE;
    GemmArgs g = with_epilogue(GemmArgs{precision, M, N, K, A, lda, B, ldb, C, ldc}, ep);
    g.batch = batch;
    g.strideA = strideA;
    g.strideB = strideB;
    g.strideC = strideC;
    if (batch < 0) return GTG_ERR_INVALID_VALUE;
    return run_gemm(g, stream);
}

gtg_status gemm_f32_ex(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B,
                       int64_t ldb, float *C, int64_t ldc, const gtg_epilogue *ep, cudaStream_t stream) {
    return run_gemm(with_epilogue(GemmArgs{GTG_PREC_F32, M, N, K, A, lda, B, ldb, C, ldc}, ep), stream);
}

gtg_status gemm_tf32_ex(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B,
                        int64_t ldb, float *C, int64_t ldc, const gtg_epilogue *ep, cudaStream_t stream) {
    return run_gemm(with_epilogue(GemmArgs{GTG_PREC_TF32, M, N, K, A, lda, B, ldb, C, ldc}, ep), stream);
}

gtg_status gemm_bf16_ex(int64_t M, int64_t N, int64_t K, const gtg_bf16 *A, int64_t lda, const gtg_bf16 *B,
                        int64_t ldb, float *C, int64_t ldc, const gtg_epilogue *ep, cudaStream_t stream) {
    return run_gemm(with_epilogue(GemmArgs{GTG_PREC_BF16, M, N, K, A, lda, B, ldb, C, ldc}, ep), stream);
}

gtg_status gtg_ablation_gemm_f32(int variant, int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                                 const float *B, int64_t ldb, float *C, int64_t ldc, cudaStream_t stream) {
    if (variant < GTG_ABL_GEMM_NAIVE_16 || variant > GTG_ABL_GEMM_TILED_32) return GTG_ERR_INVALID_VALUE;
    const GemmArgs g{GTG_PREC_F32, M, N, K, A, lda, B, ldb, C, ldc};
    gtg_status st = validate_gemm(g);
    if (st != GTG_OK || M == 0 || N == 0) return st;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != GTG_OK) return st;
    if (!(dev.cc_major == 10 && dev.cc_minor == 3)) return GTG_ERR_UNSUPPORTED;
    if (grid_too_large(M, N, 16)) return GTG_ERR_UNSUPPORTED;
    const cudaError_t e = K == 0 ? zero_fill_launch(C, M, N, ldc, stream) : ablation_gemm_launch(variant, g, stream);
    if (e != cudaSuccess) {
        note_cuda_error(e);
        return GTG_ERR_LAUNCH;
    }
    return GTG_OK;
}

gtg_status gtg_ablation_gemv_f32(int variant, int64_t M, int64_t N, const float *A, int64_t lda, const float *x,
                                 float *y, cudaStream_t stream) {
    if (variant != GTG_ABL_GEMV_NAIVE && variant != GTG_ABL_GEMV_SHARED) return GTG_ERR_INVALID_VALUE;
    const GemvArgs g{M, N, A, lda, x, N, y, M, 1};
    gtg_status st = validate_gemv(g);
    if (st != GTG_OK || M == 0) return st;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != GTG_OK) return st;
    if (!(dev.cc_major == 10 && dev.cc_minor == 3)) return GTG_ERR_UNSUPPORTED;
    const cudaError_t e = N == 0 ? zero_fill_launch(y, 1, M, M, stream) : ablation_gemv_launch(variant, g, stream);
    if (e != cudaSuccess) {
        note_cuda_error(e);
        return GTG_ERR_LAUNCH;
    }
    return GTG_OK;
}

const char *gtg_status_string(gtg_status s) {
    switch (s) {
        case GTG_OK: return "success";
        case GTG_ERR_INVALID_VALUE: return "invalid value (size, leading dimension, null pointer or batch)";
        case GTG_ERR_MISALIGNED: return "pointer not aligned to its element size";
        case GTG_ERR_ALIAS: return "output overlaps an input";
        case GTG_ERR_UNSUPPORTED: return "unsupported device (needs sm_103a)";
        case GTG_ERR_LAUNCH: return "kernel launch failed";
        case GTG_ERR_TIMEOUT: return "a device pipeline wait exceeded its time limit";
        case GTG_ERR_DEVICE: return "CUDA runtime error";
        case GTG_ERR_SCRATCH_LIMIT:
            return "problem too large for the fixed scratch of gemm_tf32_noalloc (N * roundup(K, 4) * 4 > 16 MiB)";
        case GTG_ERR_BOUNDS:
            return "a kernel computed an address outside an operand and skipped the access (GTG_DEBUG build)";
        default: return "unknown status";
    }
}

gtg_status gemm_host(int precision, int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B,
                     int64_t ldb, float *C, int64_t ldc, const gtg_epilogue *ep) {
    if (precision < GTG_PREC_F32 || precision > GTG_PREC_F16) return GTG_ERR_INVALID_VALUE;
    GemmArgs g{precision, M, N, K, A, lda, B, ldb, C, ldc};
    if (ep) {
        g.bias = ep->bias;
        g.act = ep->activation;
    }
    gtg_status st = validate_gemm(g);
    if (st != GTG_OK || M == 0 || N == 0) return st;
    if (injected_failure()) return GTG_ERR_LAUNCH;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != GTG_OK) return st;
    if (!(dev.cc_major == 10 && dev.cc_minor == 3)) return GTG_ERR_UNSUPPORTED;
    cudaError_t e = cudaSuccess;
    st = gemm_host_pipeline(dev, g, run_gemm, &e);
    if (e != cudaSuccess) note_cuda_error(e);
    if (st != GTG_OK) return st;
    // the call has synchronised: report (and clear) what the kernels latched
    int v = 0;
    const int zero = 0;
    if ((e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int))) != cudaSuccess ||
        (e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int))) != cudaSuccess) {
        note_cuda_error(e);
        return GTG_ERR_DEVICE;
    }
    return v;
}

gtg_status gtg_pool_trim(void) {
    const cudaError_t e = ws_trim();
    if (e != cudaSuccess) {
        note_cuda_error(e);
        return GTG_ERR_DEVICE;
    }
    return GTG_OK;
}

gtg_status gtg_sync_status(cudaStream_t stream) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) {
        note_cuda_error(e);
        return GTG_ERR_DEVICE;
    }
    int v = 0;
    const int zero = 0;
    if ((e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int))) != cudaSuccess ||
        (e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int))) != cudaSuccess) {
        note_cuda_error(e);
        return GTG_ERR_DEVICE;
    }
    return v;
}

const char *gtg_last_cuda_error(void) { return t_cuda_error; }

gtg_status gtg_plan_gemm(int precision, int64_t M, int64_t N, int64_t K, const void *A, int64_t lda,
                         const void *B, int64_t ldb, const void *C, int64_t ldc, gtg_plan *plan) {
    if (plan == nullptr || precision < GTG_PREC_F32 || precision > GTG_PREC_F16) return GTG_ERR_INVALID_VALUE;
    const GemmArgs g{precision, M, N, K, A, lda, B, ldb, const_cast<float *>(static_cast<const float *>(C)), ldc};
    gtg_status st = validate_gemm(g);
    if (st != GTG_OK) return st;
    std::memset(plan, 0, sizeof(*plan));
    if (M == 0 || N == 0) return GTG_OK;   // GTG_KERNEL_NONE, as the call itself
    DeviceInfo dev;
    if ((st = current_device(&dev)) != GTG_OK) return st;
    return plan_gemm_impl(dev, g, plan);
}

static gtg_status plan_gemv_impl(const GemvArgs &g, gtg_plan *plan) {
    const int64_t M = g.M, N = g.N;
    if (plan == nullptr) return GTG_ERR_INVALID_VALUE;
    gtg_status st = validate_gemv(g);
    if (st != GTG_OK) return st;
    std::memset(plan, 0, sizeof(*plan));
    if (M == 0) return GTG_OK;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != GTG_OK) return st;
    if (N == 0) {
        plan->kernel = GTG_KERNEL_ZERO_FILL;
        return GTG_OK;
    }
    gemv_plan(dev, g, plan);
    return GTG_OK;
}

gtg_status conv2d_nhwc(int precision, int64_t N, int64_t H, int64_t W, int64_t C, int64_t CO, int64_t KH,
                       int64_t KW, int64_t stride_h, int64_t stride_w, int64_t pad_h, int64_t pad_w, int64_t dil_h,
                       int64_t dil_w, const void *X, const void *Wt, float *Y, const gtg_epilogue *ep,
                       cudaStream_t stream) {
    ConvArgs c;
    c.prec = precision;
    c.N = N; c.H = H; c.W = W; c.C = C; c.CO = CO; c.KH = KH; c.KW = KW;
    c.sh = stride_h; c.sw = stride_w; c.ph = pad_h; c.pw = pad_w; c.dh = dil_h; c.dw = dil_w;
    c.X = X; c.Wt = Wt; c.Y = Y;
    if (ep) {
        c.bias = ep->bias;
        c.act = ep->activation;
    }
    gtg_status st = validate_conv(c);
    if (st != GTG_OK || N == 0 || CO == 0) return st;
    if (injected_failure()) return GTG_ERR_LAUNCH;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != GTG_OK) return st;
    if (!(dev.cc_major == 10 && dev.cc_minor == 3)) return GTG_ERR_UNSUPPORTED;
    const int64_t M = N * c.OH * c.OW, K = KH * KW * C;
    // a 1x1 window at stride 1 without padding reads X itself as the patch matrix
    const bool direct = KH == 1 && KW == 1 && stride_h == 1 && stride_w == 1 && pad_h == 0 && pad_w == 0;
    const int mode = g_conv_mode.load();
    const bool implicit_only = mode >= 2;
    if ((implicit_only || (mode == 0 && !direct)) && tc_conv_eligible(dev, c)) {
        // implicit GEMM: the tensor-core kernel reads the patches from X itself
        const cudaError_t e = tc_conv_launch(dev, c, stream, mode == 3 ? 1 : (mode == 4 ? 2 : 0));
        if (e == cudaErrorNotSupported) return GTG_ERR_UNSUPPORTED;
        if (e != cudaSuccess) {
            note_cuda_error(e);
            return GTG_ERR_LAUNCH;
        }
        return GTG_OK;
    }
    if (implicit_only) return GTG_ERR_UNSUPPORTED;
    const void *A = X;
    int64_t lda = C;
    void *P = nullptr;
    if (!direct) {
        lda = (K + 7) / 8 * 8;   // 16-byte aligned rows for the tensor-memory-access path
        cudaError_t e = ws_alloc(&P, static_cast<size_t>(M * lda * c.elem), stream);
        if (e == cudaSuccess) e = im2col_launch(dev, c, P, lda, stream);
        if (e != cudaSuccess) {
            note_cuda_error(e);
            if (P) cudaFreeAsync(P, stream);
            return GTG_ERR_LAUNCH;
        }
        A = P;
    }
    GemmArgs g{precision, M, CO, K, A, lda, Wt, CO, Y, CO};
    g.bias = c.bias;
    g.act = c.act;
    st = run_gemm(g, stream);
    if (P) cudaFreeAsync(P, stream);   // stream-ordered: after the product has read it
    return st;
}

gtg_status gtg_plan_gemv(int64_t M, int64_t N, const float *A, int64_t lda, const float *x, int64_t ldx,
                         const float *y, int64_t ldy, int batch, gtg_plan *plan) {
    return plan_gemv_impl(GemvArgs{M, N, A, lda, x, batch > 1 ? ldx : N, const_cast<float *>(y),
                                   batch > 1 ? ldy : M, batch},
                          plan);
}

gtg_status gtg_plan_gemv_bf16(int64_t M, int64_t N, const gtg_bf16 *A, int64_t lda, const float *x, int64_t ldx,
                              const float *y, int64_t ldy, int batch, gtg_plan *plan) {
    GemvArgs g{M, N, A, lda, x, batch > 1 ? ldx : N, const_cast<float *>(y), batch > 1 ? ldy : M, batch};
    g.a_elem = 2;
    return plan_gemv_impl(g, plan);
}

void gtg_force_simt(int force) { g_force_simt.store(force ? 1 : 0); }

void gtg_set_wait_limit_ns(uint64_t ns) { tc_set_wait_limit_ns(ns); }

gtg_status gtg_test_drop_load(int slice) {
    if (!testing_enabled()) return GTG_ERR_UNSUPPORTED;
    tc_drop_next_load(slice);
    return GTG_OK;
}

gtg_status gtg_test_skip_vector_copy(int on) {
    if (!testing_enabled()) return GTG_ERR_UNSUPPORTED;
    gemv_skip_next_x(on);
    return GTG_OK;
}

gtg_status gtg_test_inject_launch_failure(int n) {
    if (!testing_enabled()) return GTG_ERR_UNSUPPORTED;
    read_fault_inject_env();   // so that the environment's value cannot overwrite this one later
    g_inject_countdown.store(n > 0 ? n : 0);
    return GTG_OK;
}

uint64_t gtg_test_workspace_allocations(void) { return ws_alloc_count(); }

gtg_status gtg_test_debug_shrink_extent(int elements) {
#ifdef GTG_DEBUG
    if (!testing_enabled()) return GTG_ERR_UNSUPPORTED;
    g_debug_shrink.store(elements > 0 ? elements : 0);
    return GTG_OK;
#else
    (void)elements;
    return GTG_ERR_UNSUPPORTED;
#endif
}

int gtg_debug_build(void) {
#ifdef GTG_DEBUG
    return 1;
#else
    return 0;
#endif
}

void gtg_gemv_force_path(int mode) { gemv_force_path(mode); }

void gtg_force_gemm_splits(int splits) { tc_force_splits(splits); }

void gtg_force_c_store(int mode) { tc_force_c_store(mode); }

void gtg_conv_force_path(int mode) { g_conv_mode.store(mode >= 1 && mode <= 4 ? mode : 0); }

gtg_status gtg_plan_conv2d(int precision, int64_t N, int64_t H, int64_t W, int64_t C, int64_t CO, int64_t KH,
                           int64_t KW, int64_t stride_h, int64_t stride_w, int64_t pad_h, int64_t pad_w,
                           int64_t dil_h, int64_t dil_w, const void *X, const void *Wt, const float *Y,
                           gtg_plan *plan) {
    if (plan == nullptr) return GTG_ERR_INVALID_VALUE;
    ConvArgs c;
    c.prec = precision;
    c.N = N; c.H = H; c.W = W; c.C = C; c.CO = CO; c.KH = KH; c.KW = KW;
    c.sh = stride_h; c.sw = stride_w; c.ph = pad_h; c.pw = pad_w; c.dh = dil_h; c.dw = dil_w;
    c.X = X; c.Wt = Wt; c.Y = const_cast<float *>(Y);
    gtg_status st = validate_conv(c);
    if (st != GTG_OK) return st;
    std::memset(plan, 0, sizeof(*plan));
    if (N == 0 || CO == 0) return GTG_OK;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != GTG_OK) return st;
    if (!(dev.cc_major == 10 && dev.cc_minor == 3)) return GTG_ERR_UNSUPPORTED;
    const bool direct = KH == 1 && KW == 1 && stride_h == 1 && stride_w == 1 && pad_h == 0 && pad_w == 0;
    const int mode = g_conv_mode.load();
    if ((mode >= 2 || (mode == 0 && !direct)) && tc_conv_eligible(dev, c))
        return tc_conv_plan(dev, c, mode == 3 ? 1 : (mode == 4 ? 2 : 0), plan) ? GTG_OK : GTG_ERR_UNSUPPORTED;
    if (mode >= 2) return GTG_ERR_UNSUPPORTED;
    // the explicit route: the plan of the product P x Wt (P's rows padded to 8 elements unless X is P)
    const int64_t M = N * c.OH * c.OW, K = KH * KW * C;
    const int64_t lda = direct ? C : (K + 7) / 8 * 8;
    // (the patch matrix comes from the pool: 256-byte aligned)
    const void *P = direct ? X : reinterpret_cast<const void *>(uintptr_t{1} << 40);
    const GemmArgs g{precision, M, CO, K, P, lda, Wt, CO, c.Y, CO};
    return plan_gemm_impl(dev, g, plan);
}

int gtg_version(void) { return 100; }

}  // extern "C"
