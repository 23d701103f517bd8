/*
 * gtg_testing.h -- testing and tuning hooks of libgtg.so.
 *
 * These calls are for test suites, benchmarks and tuning runs. An
 * application that only multiplies never needs them; they are kept out of
 * gtg.h so that it does not see them. The calls fall in three groups:
 *
 *  - Path switches (gtg_force_*, gtg_conv_force_path, gtg_gemv_force_path):
 *    they select among kernels that compute the same product within the same
 *    bounds. Process-wide, in effect for later calls.
 *  - Failure-path hooks (gtg_test_drop_load, gtg_test_skip_vector_copy,
 *    gtg_test_inject_launch_failure, gtg_test_debug_shrink_extent): they
 *    make a later call fail on purpose.
 *    They act only when the environment variable GTG_TESTING is "1" at the
 *    time of the hook call; otherwise they change nothing and return
 *    GTG_ERR_UNSUPPORTED. No hook faults, traps or hangs the GPU: a kernel
 *    that is made to wait for data that never comes gives up after its time
 *    limit and reports GTG_ERR_TIMEOUT through gtg_sync_status().
 *  - Probes (gtg_test_workspace_allocations, gtg_plan_gemm_tf32_noalloc,
 *    gtg_debug_build): read-only.
 *
 * The environment variable GTG_FAULT_INJECT=<n> (n >= 1), read once when the
 * library first dispatches a call, makes the n-th dispatched call after that
 * fail on the host with GTG_ERR_LAUNCH before anything is launched (see
 * gtg_test_inject_launch_failure). It needs no GTG_TESTING: setting it is
 * itself the opt-in.
 */
#ifndef GTG_TESTING_H
#define GTG_TESTING_H

#include "gtg.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * With splits > 0 every tensor-core GEMM of a single product (and every
 * implicit-GEMM convolution) that has at least 2 * splits K slices computes K
 * in `splits` ranges whose partial tiles are added in order by a second
 * kernel (workspace from the stream-ordered pool); 0 restores the planner's
 * own choice. Results stay within the same bounds.
 */
GTG_API void gtg_force_gemm_splits(int splits);

/*
 * How the CTA-pair tensor-core kernel (16-bit and TF32 inputs, 256 x 256
 * tiles) writes C: 0 (default) lets each call choose; 1 always stores each
 * thread's row of the tile straight to global memory; 2 goes through shared
 * memory and tensor stores (32 x 32 FP32 blocks) whenever C's layout allows
 * them (16-byte aligned base, ldc and batch stride multiples of 4 elements,
 * K not split). Other values act as 0. Results are identical in every mode.
 */
GTG_API void gtg_force_c_store(int mode);

/*
 * conv2d_nhwc: 0 (default) lets each call choose; 1 always writes the patch
 * matrix and multiplies it (im2col + GEMM); 2 requires the implicit GEMM,
 * whose tensor-core kernels load the patches straight from X with TMA in
 * im2col mode, and makes a call that cannot take it return
 * GTG_ERR_UNSUPPORTED; 3 and 4 require the implicit GEMM on single-CTA tiles
 * (128 x 64..256) or on CTA pairs (256 x 256) respectively, likewise. Other
 * values act as 0.
 */
GTG_API void gtg_conv_force_path(int mode);

/*
 * Which kernel conv2d_nhwc would run for these arguments under the current
 * gtg_conv_force_path mode (no launch, no device work apart from reading the
 * device's properties once): the implicit GEMM's tensor-core kernel (bm, bn,
 * cluster = 2 for CTA pairs, splits), or, for the im2col route, the plan of
 * the product of the patch matrix and Wt. Returns the status the call itself
 * would return before launching.
 */
GTG_API gtg_status gtg_plan_conv2d(int precision, int64_t N, int64_t H, int64_t W, int64_t C, int64_t CO,
                                   int64_t KH, int64_t KW, int64_t stride_h, int64_t stride_w, int64_t pad_h,
                                   int64_t pad_w, int64_t dil_h, int64_t dil_w, const void *X, const void *Wt,
                                   const float *Y, gtg_plan *plan);

/* Force the tensor-core GEMM paths onto the SIMT kernel (force = 1) or
 * restore the normal choice (force = 0). */
GTG_API void gtg_force_simt(int force);

/*
 * GEMV kernel choice. gemv_bf16 with batch 3..8: by default (mode 0) such a
 * call runs on the tensor cores (the vectors split into three BF16 pieces
 * each, see gemv_bf16) when the tensor memory accelerator can read the
 * matrix (16-byte aligned A, lda * 2 a multiple of 16), it has at least 2^25
 * elements and batch >= 6, else on the CUDA-core kernels. Mode 1 always takes
 * the CUDA-core kernels; mode 2 takes the tensor cores whenever the layout
 * allows, at any size. Mode 3 takes the CUDA-core kernels and, for one or two
 * vectors, the streaming kernel (one row per warp) instead of the ring kernel
 * (equal step ranges per warp) that mode 0 picks for FP32 rows and for BF16
 * rows at batch 1 from 2^25 elements. Mode 4 takes the CUDA-core kernels and,
 * at batch 8, stages the vectors one after another by bulk copies instead of
 * interleaved for packed FMAs (the same result, bit for bit). Other values
 * act as 0.
 */
GTG_API void gtg_gemv_force_path(int mode);

/*
 * Time limit of every pipeline wait inside the tensor-core GEMM kernels and
 * of the GEMV kernels' wait for their bulk-copied vectors, in nanoseconds
 * (0 restores the default of 2 s). A wait that runs out makes the kernel
 * stop, release its resources and latch GTG_ERR_TIMEOUT for
 * gtg_sync_status(). Applies to later launches.
 */
GTG_API void gtg_set_wait_limit_ns(uint64_t ns);

/*
 * The next tensor-core GEMM launch leaves out the load of K slice `slice`
 * (counted over the tiles of the first CTA or CTA pair), so the wait for it
 * can only run out. The call that launches it returns GTG_OK;
 * gtg_sync_status() then reports GTG_ERR_TIMEOUT and later calls work
 * normally. A negative value cancels a pending drop.
 * Returns GTG_OK, or GTG_ERR_UNSUPPORTED (nothing armed) without GTG_TESTING=1.
 */
GTG_API gtg_status gtg_test_drop_load(int slice);

/*
 * With on != 0, the next GEMV launch that stages its vectors by bulk copies
 * announces the copies to its mbarrier but issues none, so its bounded wait
 * can only run out; the call returns GTG_OK and gtg_sync_status() reports
 * GTG_ERR_TIMEOUT. 0 cancels.
 * Returns GTG_OK, or GTG_ERR_UNSUPPORTED (nothing armed) without GTG_TESTING=1.
 */
GTG_API gtg_status gtg_test_skip_vector_copy(int on);

/*
 * Host-side fault injection in the dispatcher: with n >= 1, the n-th call
 * dispatched from now on (counting every product call that passed argument
 * validation, including the per-region products inside gemm_host) returns
 * GTG_ERR_LAUNCH without launching anything, and gtg_last_cuda_error() reads
 * "injected launch failure". Later calls work normally. n = 0 cancels.
 * Returns GTG_OK, or GTG_ERR_UNSUPPORTED (nothing armed) without GTG_TESTING=1.
 */
GTG_API gtg_status gtg_test_inject_launch_failure(int n);

/* Number of device workspaces the library has taken from its memory pools
 * since the process started (every caller, every device). */
GTG_API uint64_t gtg_test_workspace_allocations(void);

/*
 * Which kernel gemm_tf32_noalloc would run for these arguments (no launch,
 * no device work apart from reading the device's properties once). Fills
 * *plan; returns the status the call itself would return before launching
 * (GTG_ERR_SCRATCH_LIMIT when B^T does not fit the fixed array).
 */
GTG_API gtg_status gtg_plan_gemm_tf32_noalloc(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                                              const float *B, int64_t ldb, const float *C, int64_t ldc,
                                              gtg_plan *plan);

/*
 * GTG_DEBUG builds only: the GEMV kernels check their matrix loads against
 * an extent `elements` shorter than the real one, so that the last loads of
 * a call fail their check (the access is skipped; nothing outside the real
 * matrix is touched) and GTG_ERR_BOUNDS is latched for gtg_sync_status(): a
 * test that the checks are live. 0 restores the real extent.
 * Returns GTG_OK; GTG_ERR_UNSUPPORTED in a release build or without
 * GTG_TESTING=1.
 */
GTG_API gtg_status gtg_test_debug_shrink_extent(int elements);

/* 1 if this library was built with GTG_DEBUG (kernels check the addresses
 * they compute and latch GTG_ERR_BOUNDS instead of making an access outside
 * an operand), else 0. */
GTG_API int gtg_debug_build(void);

#ifdef __cplusplus
}
#endif

#endif /* GTG_TESTING_H */
