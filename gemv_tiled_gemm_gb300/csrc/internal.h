// Internal interface between the C-ABI layer (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "gtg.h"

namespace gtg {

// Per-device facts the planners need (filled once per device by api.cu).
struct DeviceInfo {
    int id = -1;
    int sms = 0;                 // streaming multiprocessors
    int cc_major = 0, cc_minor = 0;
    int smem_optin = 0;          // max dynamic shared memory per block (bytes)
    int l2_bytes = 0;
    int *status = nullptr;       // device address of the library's status word
};

// One GEMM call after validation. Pointers are device pointers. The optional
// epilogue computes C = act(A * B + bias) with one bias per column of C.
struct GemmArgs {
    int prec;                    // GTG_PREC_*
    int64_t M, N, K;
    const void *A; int64_t lda;
    const void *B; int64_t ldb;
    float *C; int64_t ldc;
    const float *bias = nullptr; // N entries or null
    int act = 0;                 // GTG_ACT_*
    // strided batch: item b uses A + b*strideA, B + b*strideB, C + b*strideC (elements)
    int64_t batch = 1, strideA = 0, strideB = 0, strideC = 0;
};

// y_b = act(A * x_b + bias) with one bias per row of A. A holds FP32 values
// (a_elem 4) or BF16 bit patterns (a_elem 2); x and y are FP32.
struct GemvArgs {
    int64_t M, N;
    const void *A; int64_t lda;
    const float *x; int64_t ldx;
    float *y; int64_t ldy;
    int batch;
    const float *bias = nullptr; // M entries or null
    int act = 0;
    int a_elem = 4;              // bytes per element of A
};

// One convolutional layer after validation: X channels-last N x H x W x C,
// weights KH x KW x C x CO, Y channels-last N x OH x OW x CO (FP32).
struct ConvArgs {
    int prec;                    // GTG_PREC_*
    int elem;                    // bytes per element of X and the weights
    int64_t N, H, W, C, CO, KH, KW, sh, sw, ph, pw, dh, dw, OH, OW;
    const void *X;
    const void *Wt;
    float *Y;
    const float *bias = nullptr; // CO entries or null
    int act = 0;
};

// The epilogue applied to one FP32 result before it is stored.
__host__ __device__ __forceinline__ float apply_epilogue(float v, const float *bias, int index, int act) {
    if (bias) v += bias[index];
    if (act == GTG_ACT_RELU) v = v > 0.f ? v : 0.f;
    return v;
}

// GTG_DEBUG builds (libgtg_debug.so): the index-heavy kernels check every
// global address they compute, and every shared-memory index they write,
// against the extent of the operand or buffer it belongs to before using it.
// A failed check latches GTG_ERR_BOUNDS in the status word (read by
// gtg_sync_status) and the access is skipped: a load gives zero, a store is
// dropped. Release builds compile the checks away (they are constant true).
#ifdef GTG_DEBUG
__device__ __forceinline__ bool debug_in(const void *p, unsigned long long bytes, const void *lo, const void *hi,
                                         int *status) {
    const unsigned long long a = reinterpret_cast<unsigned long long>(p);
    if (a >= reinterpret_cast<unsigned long long>(lo) && a + bytes <= reinterpret_cast<unsigned long long>(hi))
        return true;
    atomicCAS(status, 0, static_cast<int>(GTG_ERR_BOUNDS));
    return false;
}
__device__ __forceinline__ unsigned dynamic_smem_bytes() {
    unsigned v;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(v));
    return v;
}
#define GTG_DEBUG_IN(p, bytes, lo, hi, status) ::gtg::debug_in((p), (bytes), (lo), (hi), (status))
#else
#define GTG_DEBUG_IN(p, bytes, lo, hi, status) true
#endif

// Elements by which GTG_DEBUG builds shrink the matrix extent the GEMV
// kernels check against (testing: makes the last loads fail their check
// without any access outside the real matrix); 0 in release builds.
int debug_shrink_setting();

// Time limit for any pipeline wait inside a kernel (nanoseconds).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// ---- tcgen05 tensor-core GEMM (gemm_tc.cu)
bool tc_supported(const DeviceInfo &dev);
bool tc_eligible(const GemmArgs &g);
// as tc_eligible, for a single product whose A (or 16-bit B) is first copied
// into 16-byte rows because its base or row stride does not suit TMA
bool tc_eligible_repacked(const GemmArgs &g);
void tc_plan(const DeviceInfo &dev, const GemmArgs &g, gtg_plan *plan);
cudaError_t tc_launch(const DeviceInfo &dev, const GemmArgs &g, const gtg_plan &plan,
                      cudaStream_t stream);

// testing hooks of the tensor-core kernels (gemm_tc.cu)
void tc_set_wait_limit_ns(unsigned long long ns);
void tc_drop_next_load(int slice);
void tc_force_splits(int splits);   // > 0: every eligible single product splits K that many ways
void tc_force_c_store(int mode);    // CTA-pair kernel's C stores: 0 auto, 1 direct, 2 tensor stores

// ---- TF32 GEMM whose B^T staging buffer is a fixed array in the library
// (gemm_tc.cu), for callers that cannot allocate device memory
size_t tf32_fixed_scratch_bytes();
size_t tf32_bt_bytes(int64_t N, int64_t K);
// the single-CTA tile width for a product computed in one K range (no
// workspace); replaces *plan (the fixed-scratch launch runs only that kernel)
void tc_plan_unsplit_single(const DeviceInfo &dev, const GemmArgs &g, gtg_plan *plan);
cudaError_t tc_launch_tf32_fixed_scratch(const DeviceInfo &dev, const GemmArgs &g, const gtg_plan &plan,
                                         cudaStream_t stream);

// ---- SIMT GEMM (gemm_simt.cu): FP32 or BF16 inputs, FP32 arithmetic
void simt_plan(const DeviceInfo &dev, const GemmArgs &g, gtg_plan *plan);
cudaError_t simt_launch(const DeviceInfo &dev, const GemmArgs &g, const gtg_plan &plan,
                        cudaStream_t stream);
cudaError_t zero_fill_launch(float *C, int64_t M, int64_t N, int64_t ldc, cudaStream_t stream);
// C = act(sum_{z < splits} ws[z] + bias), the slabs ws[z] (M x N, packed)
// added in order z = 0, 1, ... (results independent of scheduling)
cudaError_t split_reduce_launch(const float *ws, int splits, int64_t M, int64_t N, float *C, int64_t ldc,
                                const float *bias, int act, cudaStream_t stream);
// C[i][j] = act(bias[j] or bias[i]) -- the result of an empty product with an epilogue
cudaError_t epilogue_fill_launch(float *C, int64_t M, int64_t N, int64_t ldc, const float *bias, int per_column,
                                 int act, cudaStream_t stream);

// ---- the pages' kernel designs, for measurement (ablation.cu)
cudaError_t ablation_gemm_launch(int variant, const GemmArgs &g, cudaStream_t stream);
cudaError_t ablation_gemv_launch(int variant, const GemvArgs &g, cudaStream_t stream);
bool grid_too_large(int64_t M, int64_t N, int tile);

// ---- host operands (host.cu): the pipeline of gemm_host; `run` launches one
// block's product on a stream. Synchronous; on a CUDA error sets *cuda_error.
gtg_status gemm_host_pipeline(const DeviceInfo &dev, const GemmArgs &g, gtg_status (*run)(const GemmArgs &, cudaStream_t),
                              cudaError_t *cuda_error);

// ---- device workspaces (pool.cu): stream-ordered allocations from the
// library's own pool on the current device (release with cudaFreeAsync on a
// stream ordered after the last use); ws_trim returns the reserved pages.
cudaError_t ws_alloc(void **p, size_t bytes, cudaStream_t stream);
cudaError_t ws_trim();
uint64_t ws_alloc_count();   // ws_alloc calls so far (every device)

// ---- implicit-GEMM convolution on the tensor cores (gemm_tc.cu): A tiles
// loaded from X by TMA in im2col mode (16-bit, C % 64 == 0, small windows)
// choice: 0 any kernel, 1 single-CTA tiles only, 2 the CTA pair only
// (tc_conv_launch returns cudaErrorNotSupported, tc_conv_plan false, if
// `choice` rules out every kernel)
bool tc_conv_eligible(const DeviceInfo &dev, const ConvArgs &c);
cudaError_t tc_conv_launch(const DeviceInfo &dev, const ConvArgs &c, cudaStream_t stream, int choice);
bool tc_conv_plan(const DeviceInfo &dev, const ConvArgs &c, int choice, gtg_plan *plan);

// ---- im2col (im2col.cu): the patch matrix P (N*OH*OW x KH*KW*C, ldp >= K)
cudaError_t im2col_launch(const DeviceInfo &dev, const ConvArgs &c, void *P, int64_t ldp, cudaStream_t stream);

// Current bound of in-kernel waits (gtg_set_wait_limit_ns; gemm_tc.cu).
unsigned long long wait_limit_setting();
// The K slice whose load a tensor-core kernel leaves out once (gtg_test_drop_load), then -1.
int take_test_drop_slice();
// A 2-D tiled tensor map (128-byte swizzle, zero fill outside the tensor):
// `outer` rows of `inner` elements, `ld_elems` apart; boxes of box_inner x box_outer.
bool tma_map_2d(CUtensorMap *map, int prec, const void *base, uint64_t inner, uint64_t outer, uint64_t ld_elems,
                uint32_t box_inner, uint32_t box_outer);

// ---- batched GEMV of a BF16 matrix on the tensor cores (gemv_tc.cu), batch 3..8
// any_size: also below the size where the CUDA-core kernels are faster
bool gemv_tc_eligible(const DeviceInfo &dev, const GemvArgs &g, bool any_size);
void gemv_tc_plan(const DeviceInfo &dev, const GemvArgs &g, gtg_plan *plan);
cudaError_t gemv_tc_launch(const DeviceInfo &dev, const GemvArgs &g, cudaStream_t stream);

// ---- GEMV (gemv.cu)
// testing hook: the next GEMV launch that stages x by bulk copies announces
// them but issues none, so its wait runs out
void gemv_skip_next_x(int on);
int take_gemv_skip_x();
// testing / tuning hook for BF16 GEMVs of batch 3..8: 0 planner's choice,
// 1 CUDA-core kernels, 2 tensor cores whenever the layout allows
void gemv_force_path(int mode);
void gemv_plan(const DeviceInfo &dev, const GemvArgs &g, gtg_plan *plan);
cudaError_t gemv_launch(const DeviceInfo &dev, const GemvArgs &g, const gtg_plan &plan,
                        cudaStream_t stream);

}  // namespace gtg
