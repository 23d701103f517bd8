// Device workspaces: every temporary buffer of the library (split-K slabs,
// the TF32 path's B^T, the patch matrix of a convolution, the device copies
// of gemm_host) comes from a stream-ordered memory pool of the library's own,
// one per device, created on first use. The pool keeps up to kKeepBytes
// reserved across synchronisations, so that a call after a synchronisation
// reuses pages instead of mapping them again (a mapping can hold the host
// for most of a millisecond); gtg_pool_trim hands them back.
#include <atomic>
#include <mutex>

#include "internal.h"

namespace gtg {
namespace {

constexpr uint64_t kKeepBytes = 1ull << 30;
constexpr int kMaxDevices = 64;

struct Pools {
    std::mutex mu;
    cudaMemPool_t pool[kMaxDevices] = {};
};

Pools &pools() {
    static Pools p;
    return p;
}

cudaError_t device_pool(int device, cudaMemPool_t *out) {
    if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
    Pools &ps = pools();
    std::lock_guard<std::mutex> lk(ps.mu);
    if (ps.pool[device] == nullptr) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = device;
        cudaMemPool_t p;
        cudaError_t e = cudaMemPoolCreate(&p, &props);
        if (e != cudaSuccess) return e;
        uint64_t keep = kKeepBytes;
        if ((e = cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep)) != cudaSuccess) {
            cudaMemPoolDestroy(p);
            return e;
        }
        ps.pool[device] = p;
    }
    *out = ps.pool[device];
    return cudaSuccess;
}

}  // namespace

namespace {
std::atomic<uint64_t> g_ws_allocs{0};
}

uint64_t ws_alloc_count() { return g_ws_allocs.load(); }

cudaError_t ws_alloc(void **p, size_t bytes, cudaStream_t stream) {
    g_ws_allocs.fetch_add(1);
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    cudaMemPool_t pool;
    if (e == cudaSuccess) e = device_pool(device, &pool);
    if (e == cudaSuccess) e = cudaMallocFromPoolAsync(p, bytes, pool, stream);
    return e;
}

cudaError_t ws_trim() {
    Pools &ps = pools();
    std::lock_guard<std::mutex> lk(ps.mu);
    for (cudaMemPool_t p : ps.pool)
        if (p) {
            const cudaError_t e = cudaMemPoolTrimTo(p, 0);
            if (e != cudaSuccess) return e;
        }
    return cudaSuccess;
}

}  // namespace gtg
