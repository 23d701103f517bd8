/*
 * gtg -- dense matrix products on one NVIDIA GB300 (sm_103a).
 *
 * C ABI of libgtg.so. Every entry point is callable from C, C++, ctypes or
 * any FFI: plain pointers, 64-bit sizes and a CUDA stream handle.
 *
 * The operations are the two defined in "Matrix Operations" (Vulkan
 * ML-inference tutorial, sections "Matrix-Vector Multiplication" and
 * "Matrix-Matrix Multiplication (GEMM)"), also given in "CUDA Programming (6):
 * Shared Memory and Matrix Multiplication Optimization" (section 3) and "GPU
 * Matrix Multiplication: Tiling and Shared Memory" (section 1):
 *
 *     GEMM   C[i][j] = sum_{k<K} A[i][k] * B[k][j]     A: M x K, B: K x N, C: M x N
 *     GEMV   y[i]    = sum_{j<N} A[i][j] * x[j]        A: M x N, x: N,     y: M
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Layout: row-major. Element (r, c) of a matrix with leading dimension ld
 *    is at p[r * ld + c]. The pages index A[row*K + k], B[k*N + col] and
 *    C[row*N + col]; the leading dimensions generalise that to padded rows
 *    and require ld >= the row length.
 *  - Memory: every array pointer is a DEVICE pointer (cudaMalloc, or any
 *    memory the device can address) on the current device. The caller owns
 *    all buffers; the library never frees or keeps them after the call.
 *  - Output: C (or y) is overwritten, never read ("writeonly" in the pages'
 *    shaders): no alpha/beta scaling. K = 0 writes zeros (the empty sum).
 *  - Stream: work is enqueued on `stream` (0 = legacy default stream) and
 *    the call returns without waiting for it. Inputs must stay valid and
 *    unmodified, and outputs untouched, until the stream reaches that point.
 *  - Aliasing: C (or y) must not overlap A, B (or A, x): GTG_ERR_ALIAS.
 *  - Errors: a non-zero status means nothing was launched (except
 *    GTG_ERR_LAUNCH, reported when the launch itself failed). Device-side
 *    failures (a pipeline wait that ran out of time) are latched in a device
 *    status word and returned by gtg_sync_status().
 *  - Allocation: the calls never synchronise. Paths that need a temporary
 *    device buffer take it from the library's own stream-ordered memory
 *    pool on the current device (allocated on `stream`, returned with
 *    cudaFreeAsync on `stream` after use, so the host never waits): the TF32
 *    tensor-core path (B^T, see gemm_tf32), products that split K and add
 *    the partial products (splits * M * N * 4 bytes), the patch matrix of a
 *    convolution, and gemm_host's device copies. The pool is created on
 *    first use and keeps up to 1 GiB reserved between calls, so that a call
 *    after a synchronisation does not map its pages afresh; gtg_pool_trim
 *    returns them. gemv_f32 allocates nothing; gemm_tf32_noalloc never
 *    allocates. Per device the library otherwise keeps only host-side state
 *    (device properties and a table of kernel attributes).
 *  - Thread safety: calls may be made concurrently from several host
 *    threads; the host-side state is guarded by a mutex.
 *  - Testing: hooks for test suites and tuning (path switches, failure
 *    injection, wait limits) are declared in gtg_testing.h, not here.
 */
#ifndef GTG_H
#define GTG_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GTG_API __attribute__((visibility("default")))
#else
#define GTG_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as the CUDA runtime's cudaStream_t (a redeclaration is allowed). */
typedef struct CUstream_st *cudaStream_t;

/* A bfloat16 value stored as its 16-bit pattern (1 sign, 8 exponent, 7 mantissa). */
typedef uint16_t gtg_bf16;

typedef int gtg_status;
enum {
    GTG_OK = 0,
    GTG_ERR_INVALID_VALUE = 1, /* negative size, ld < row length, NULL with non-zero extent, batch out of range */
    GTG_ERR_MISALIGNED = 2,    /* a pointer not aligned to its element size */
    GTG_ERR_ALIAS = 3,         /* the output overlaps an input */
    GTG_ERR_UNSUPPORTED = 4,   /* no kernel for this device (not sm_103a / sm_100-class) */
    GTG_ERR_LAUNCH = 5,        /* the CUDA launch failed (cudaGetLastError text via gtg_last_cuda_error) */
    GTG_ERR_TIMEOUT = 6,       /* device side: a pipeline wait exceeded its time limit */
    GTG_ERR_DEVICE = 7,        /* a CUDA runtime call failed (no device, context error, ...) */
    GTG_ERR_SCRATCH_LIMIT = 8, /* gemm_tf32_noalloc: B^T would not fit its fixed 16 MiB scratch */
    GTG_ERR_BOUNDS = 9         /* device side, GTG_DEBUG builds only: a kernel computed an address
                                  outside one of its operands and skipped that access */
};

/*
 * gemm_f32 -- C = A*B in FP32 with exact-FP32 arithmetic: every product and
 * sum is an IEEE binary32 fused multiply-add on the CUDA cores
 * (register-blocked, shared-memory-tiled SIMT kernel; "CUDA Programming (6)",
 * section 3.2 tiling and 3.4 thread-level tiling; "Matrix Operations",
 * "Register Blocking"). Out-of-range tile elements are zero-padded and
 * out-of-range stores skipped, so any M, N, K >= 0 is accepted.
 *   M, N, K    sizes (>= 0)
 *   A          M x K, leading dimension lda >= max(K, 1)
 *   B          K x N, leading dimension ldb >= max(N, 1)
 *   C          M x N, leading dimension ldc >= max(N, 1), overwritten
 * Pointers must be 4-byte aligned. 16-byte alignment and ld % 4 == 0 enable
 * 128-bit loads; other layouts use a scalar-load variant with the same result.
 * When the output has too few tiles to keep every SM busy, K is split into
 * up to 16 ranges computed concurrently; their FP32 partial products go to a
 * pool buffer of splits * M * N * 4 bytes and are added in a fixed order
 * (results are the same run to run).
 */
GTG_API gtg_status gemm_f32(int64_t M, int64_t N, int64_t K,
                    const float *A, int64_t lda,
                    const float *B, int64_t ldb,
                    float *C, int64_t ldc,
                    cudaStream_t stream);

/*
 * gemm_tf32 -- C = A*B with FP32 storage, TF32 multiplication on the tensor
 * cores (tcgen05.mma kind::tf32) and FP32 accumulation in tensor memory
 * ("Matrix Operations", "Performance Considerations": tensor cores). Same
 * arguments and layouts as gemm_f32. Each product uses the operands rounded
 * to the nearest TF32 value (10 explicit mantissa bits, ties away from zero)
 * before the tensor core multiplies them: B as it is transposed, A in shared
 * memory between its load and the multiply. (The tensor core itself would
 * truncate, which can cost twice the error of rounding.)
 * The TF32 tensor-core MMA reads B only K-major, so the call first writes
 * B^T into a temporary buffer of 4 * N * roundup(K, 4) bytes. That buffer
 * comes from the library's stream-ordered workspace pool (allocated on
 * `stream`) and is returned to it (cudaFreeAsync on `stream`) after the
 * multiply, so it never blocks the host; if the pool cannot supply it the
 * call returns GTG_ERR_LAUNCH and launches nothing.
 * The tensor-core kernel reads A through TMA, which needs a 16-byte aligned
 * base and lda a multiple of 4; for other layouts A is first copied into
 * such rows in a second temporary from the same pool (4 * M * roundup(K, 4)
 * bytes, released the same way).
 */
GTG_API gtg_status gemm_tf32(int64_t M, int64_t N, int64_t K,
                     const float *A, int64_t lda,
                     const float *B, int64_t ldb,
                     float *C, int64_t ldc,
                     cudaStream_t stream);

/*
 * gemm_bf16 -- C = A*B with BF16 inputs, FP32 accumulation on the tensor
 * cores (tcgen05.mma kind::f16) and an FP32 output ("Matrix Operations",
 * "Performance Considerations": half-precision data types and tensor cores).
 * BF16 products are exact in FP32; only the accumulation rounds.
 *   A  M x K bf16, lda >= max(K, 1);  B  K x N bf16, ldb >= max(N, 1)
 *   C  M x N FP32, ldc >= max(N, 1), overwritten
 * Pointers must be 2-byte (A, B) and 4-byte (C) aligned. The tensor-core
 * kernels read A and B through TMA, which needs 16-byte aligned bases and
 * lda, ldb multiples of 8; an operand in another layout is first copied into
 * such rows in a temporary from the library's stream-ordered pool (released
 * on `stream` after the multiply; GTG_ERR_LAUNCH if the pool cannot supply
 * it).
 */
GTG_API gtg_status gemm_bf16(int64_t M, int64_t N, int64_t K,
                     const gtg_bf16 *A, int64_t lda,
                     const gtg_bf16 *B, int64_t ldb,
                     float *C, int64_t ldc,
                     cudaStream_t stream);

/* An IEEE binary16 value stored as its 16-bit pattern. */
typedef uint16_t gtg_f16;

/*
 * gemm_f16 -- C = A*B with FP16 inputs, FP32 accumulation on the tensor cores
 * (tcgen05.mma kind::f16) and an FP32 output ("Matrix Operations",
 * "Performance Considerations": half precision). FP16 products are exact in
 * FP32. Same arguments, alignment rules and fallback as gemm_bf16.
 */
GTG_API gtg_status gemm_f16(int64_t M, int64_t N, int64_t K,
                            const gtg_f16 *A, int64_t lda,
                            const gtg_f16 *B, int64_t ldb,
                            float *C, int64_t ldc,
                            cudaStream_t stream);

/*
 * gemv_f32 -- y_b = A*x_b for `batch` vectors at once, in FP32 ("Matrix
 * Operations", "Matrix-Vector Multiplication": the fully connected layer;
 * the vector is staged in shared memory once per thread block as in its
 * "Optimized Implementation with Shared Memory", in chunks when it is too
 * large, as in "Handling Large Vectors"). Every row of A is read once from
 * memory for all `batch` vectors.
 *   M, N   A is M x N (M rows, N columns), lda >= max(N, 1)
 *   x      batch vectors of N entries; vector b starts at x + b * ldx
 *          (ldx >= N; ignored when batch == 1)
 *   y      batch outputs of M entries; output b starts at y + b * ldy
 *          (ldy >= M; ignored when batch == 1), overwritten
 *   batch  1 <= batch <= 8
 * Pointers must be 4-byte aligned; a 16-byte aligned A with lda % 4 == 0
 * enables 128-bit row loads throughout. Other rows take their first 0-3
 * entries (up to a 16-byte boundary) by single loads and the rest by 128-bit
 * loads when the vectors and the rows' partial sums fit one CTA's shared
 * memory (N up to about 51200 / batch entries); beyond that the rows are
 * read one entry per load. The result is the same either way.
 */
GTG_API gtg_status gemv_f32(int64_t M, int64_t N,
                    const float *A, int64_t lda,
                    const float *x, int64_t ldx,
                    float *y, int64_t ldy,
                    int batch,
                    cudaStream_t stream);

/*
 * gemv_bf16 -- gemv_f32 with the matrix stored in BF16 (bit patterns, 2 bytes
 * per element); x, y and every multiply-add stay FP32. The matrix is the
 * traffic that bounds a matrix-vector product ("Matrix Operations",
 * "Matrix-Vector Multiplication", and its "Performance Considerations" on
 * half-precision storage), so halving its bytes halves the time; each BF16
 * value is widened to FP32 exactly before it is used, and the result differs
 * from gemv_f32 on the widened matrix only by the order of FP32 additions.
 * Batch 6..8 with a 16-byte aligned A, lda % 8 == 0 and M * N >= 2^25 runs
 * on the tensor cores: each FP32 vector entry is split into three BF16 pieces (x = x1 + x2
 * + x3 to within 2^-27 |x|), every product of a matrix element with a piece
 * is exact, and the tensor core accumulates in FP32, so the result meets the
 * same FP32 bound; it takes two temporaries from the workspace pool (the
 * pieces, 6 * batch * roundup(N, 8) bytes, and the partial sums of the row
 * tiles whose columns are shared between SMs).
 *   Arguments as gemv_f32; A must be 2-byte aligned (x and y 4-byte); a
 *   16-byte aligned A with lda % 8 == 0 enables 128-bit row loads. Other
 *   rows take their first 0-3 entries (up to an 8-byte boundary) by single
 *   loads and the rest by 64-bit loads when the vectors and the rows'
 *   partial sums fit one CTA's shared memory (N up to about 51200 / batch
 *   entries), else one entry per load.
 */
GTG_API gtg_status gemv_bf16(int64_t M, int64_t N,
                             const gtg_bf16 *A, int64_t lda,
                             const float *x, int64_t ldx,
                             float *y, int64_t ldy,
                             int batch,
                             cudaStream_t stream);

/*
 * gemm_tf32_noalloc -- the product of gemm_tf32, for callers that cannot
 * allocate device memory. The pages have no counterpart to this entry point;
 * it exists for users of this library.
 *
 * Who needs it: code that must not allocate once it is running. Examples: a
 * serving process whose own allocator has already reserved nearly all of the
 * GPU's memory for weights and caches, so a pool allocation would fail or
 * fragment that reservation; a driver or virtualisation set-up that offers no
 * stream-ordered memory pools; a latency-critical loop that forbids
 * allocation calls because their cost is unbounded. gemm_tf32 takes its B^T
 * staging buffer from the memory pool; this entry point uses instead a fixed
 * array of 16 MiB that is part of the library's device image.
 *
 * Arguments, layouts, result and accuracy are those of gemm_tf32; the caller
 * still provides A, B and C. The call makes no cudaMalloc, cudaMallocAsync,
 * cudaFree or other allocating call (on the SIMT path it multiplies without
 * splitting K).
 *
 * Limit: B^T takes N * roundup(K, 4) * 4 bytes, which must not exceed the
 * array's 16 MiB (16777216 bytes; K = N = 2048 just fits). A larger problem
 * returns GTG_ERR_SCRATCH_LIMIT and launches nothing.
 *
 * Sharing: there is one array per device; every device that loads the
 * library holds it until the process exits, and all calls on that device
 * share it. It keeps the last call's contents. A call overwrites every
 * element it reads before reading it, so nothing needs clearing, but two
 * calls whose GPU work overlaps (issued on streams not ordered with each
 * other, e.g. from different host threads) race on the array and can give
 * wrong results: order them, for instance on one stream.
 *
 * Set-up: the first call on a device, made with that device current, looks up
 * the array's device address (cudaGetSymbolAddress) and caches it. Make that
 * first call before any stream capture begins.
 */
GTG_API gtg_status gemm_tf32_noalloc(int64_t M, int64_t N, int64_t K,
                             const float *A, int64_t lda,
                             const float *B, int64_t ldb,
                             float *C, int64_t ldc,
                             cudaStream_t stream);

/*
 * Fully connected layers: the same products with an epilogue applied to each
 * FP32 result before it is stored ("Matrix Operations": fully connected
 * layers are matrix-vector products; activation functions add the
 * non-linearity):
 *
 *   GEMM  C[i][j] = act(sum_k A[i][k] B[k][j] + bias[j])   (a batch of inputs
 *                                                            in the rows of A)
 *   GEMV  y_b[i]  = act(sum_j A[i][j] x_b[j] + bias[i])     (one layer, W = A)
 *
 *   bias        device pointer to N (GEMM) or M (GEMV) FP32 values, 4-byte
 *               aligned, not overlapping the output; NULL for no bias
 *   activation  GTG_ACT_NONE (identity) or GTG_ACT_RELU (max(v, 0))
 *
 * The epilogue is fused into the kernels' stores: it adds no pass over C.
 * epilogue == NULL is the plain product. Other arguments and errors are
 * those of the corresponding call above; an unknown activation or a bias
 * overlapping the output returns GTG_ERR_INVALID_VALUE / GTG_ERR_ALIAS.
 * With K = 0 (or N = 0 for the GEMV) the outputs are act(bias).
 */
enum { GTG_ACT_NONE = 0, GTG_ACT_RELU = 1 };
typedef struct {
    const float *bias;
    int activation;
} gtg_epilogue;

GTG_API gtg_status gemm_f32_ex(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                               const float *B, int64_t ldb, float *C, int64_t ldc,
                               const gtg_epilogue *epilogue, cudaStream_t stream);
GTG_API gtg_status gemm_tf32_ex(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                                const float *B, int64_t ldb, float *C, int64_t ldc,
                                const gtg_epilogue *epilogue, cudaStream_t stream);
GTG_API gtg_status gemm_bf16_ex(int64_t M, int64_t N, int64_t K, const gtg_bf16 *A, int64_t lda,
                                const gtg_bf16 *B, int64_t ldb, float *C, int64_t ldc,
                                const gtg_epilogue *epilogue, cudaStream_t stream);
GTG_API gtg_status gemv_f32_ex(int64_t M, int64_t N, const float *A, int64_t lda,
                               const float *x, int64_t ldx, float *y, int64_t ldy, int batch,
                               const gtg_epilogue *epilogue, cudaStream_t stream);
GTG_API gtg_status gemm_f16_ex(int64_t M, int64_t N, int64_t K, const gtg_f16 *A, int64_t lda,
                               const gtg_f16 *B, int64_t ldb, float *C, int64_t ldc,
                               const gtg_epilogue *epilogue, cudaStream_t stream);
GTG_API gtg_status gemv_bf16_ex(int64_t M, int64_t N, const gtg_bf16 *A, int64_t lda,
                                const float *x, int64_t ldx, float *y, int64_t ldy, int batch,
                                const gtg_epilogue *epilogue, cudaStream_t stream);

/*
 * conv2d_nhwc -- a convolutional layer as one matrix product: the im2col
 * route that "GPU Matrix Multiplication: Tiling and Shared Memory" (closing
 * section) and "Matrix Operations" (introduction) name for convolutions.
 *
 *   Y[n][oh][ow][co] = act(bias[co] + sum_{kh, kw, ci}
 *       X[n][oh*stride_h - pad_h + kh*dil_h][ow*stride_w - pad_w + kw*dil_w][ci]
 *       * Wt[kh][kw][ci][co])
 *
 * with input positions outside the image contributing zero (zero padding).
 *   precision  GTG_PREC_F32, _TF32 (X, Wt FP32), _BF16 or _F16 (X, Wt 16-bit);
 *              arithmetic and accumulation as gemm_<precision>
 *   X          N x H x W x C, channels last, packed (device)
 *   Wt         KH x KW x C x CO, packed: read row-major it is the
 *              (KH*KW*C) x CO weight matrix (device)
 *   Y          N x OH x OW x CO, channels last, packed, FP32, overwritten;
 *              OH = (H + 2 pad_h - dil_h (KH - 1) - 1) / stride_h + 1 (floor),
 *              OW likewise
 *   epilogue   optional bias (CO values, one per output channel) and activation
 * 16-bit layers with C a multiple of 64 (16-byte aligned X and Wt, CO a
 * multiple of 8, window offsets below 256 and strides up to 8) run as an
 * implicit GEMM: the tensor-core kernel (single-CTA tiles of 128 x 64..256 or
 * CTA pairs with 256 x 256 tiles, whichever the planner estimates faster)
 * loads each tile of the patch matrix straight from X with a TMA im2col copy,
 * and no temporary is needed unless K is split. TF32 layers with C a multiple
 * of 32 (same window and stride limits, any alignment) take the same route
 * from a copy of X rounded to TF32 (a temporary of X's size from the pool)
 * and the rounded W^T (CO x K), as gemm_tf32 rounds its operands. Other layers write the patch
 * matrix P (N*OH*OW x KH*KW*C, rows padded to a multiple of 8 elements) into
 * a temporary from the device's stream-ordered memory pool, freed on the
 * stream after the product; a 1x1 window with stride 1 and no padding needs
 * none (X is P). Then Y = P * Wt through the GEMM kernels of
 * gemm_<precision>.
 * Errors: GTG_ERR_INVALID_VALUE for sizes < 1 (N, CO may be 0: nothing is
 * done), strides or dilations < 1, negative padding, a window larger than the
 * padded image, N*OH*OW or KH*KW*C above 2^31 - 1, an unknown precision or
 * activation; GTG_ERR_MISALIGNED for element-misaligned pointers;
 * GTG_ERR_ALIAS when Y overlaps X, Wt or the bias; GTG_ERR_LAUNCH when the
 * temporary cannot be allocated or a launch fails.
 */
GTG_API gtg_status conv2d_nhwc(int precision, int64_t N, int64_t H, int64_t W, int64_t C, int64_t CO,
                               int64_t KH, int64_t KW, int64_t stride_h, int64_t stride_w,
                               int64_t pad_h, int64_t pad_w, int64_t dil_h, int64_t dil_w,
                               const void *X, const void *Wt, float *Y,
                               const gtg_epilogue *epilogue, cudaStream_t stream);

/*
 * gemm_host -- C = act(A * B + bias) with A, B, C (and the bias) in HOST
 * memory: the end-to-end call for data that is not on the device yet.
 *   precision  GTG_PREC_F32, _TF32, _BF16 or _F16, as gemm_<precision>
 *   A, B, C    host pointers, row-major with leading dimensions as gemm_f32;
 *              A and B of the precision's storage type, C FP32
 *   epilogue   optional; its bias pointer is a host pointer (N floats)
 * A goes to the device in blocks of rows and B in panels of columns, in the
 * order that keeps the rows sent and the columns sent about equal (an output
 * block needs its rows of A and its columns of B, so this order makes the
 * most of C computable soonest); each region of C is multiplied as soon as
 * its pieces are in and copied back while later pieces are still coming in
 * (three streams of the library's own; A, B and C whole on the device for
 * the duration of the call, in buffers from the library's workspace pool,
 * see Allocation above). Page-locked (pinned) host memory lets the copies
 * run asynchronously and overlap; pageable memory works but serialises them.
 * Synchronous: returns once C holds the result, with the status
 * gtg_sync_status would give (GTG_ERR_TIMEOUT if a kernel gave up a wait).
 * Errors: as gemm_<precision> for the arguments; GTG_ERR_DEVICE when a
 * copy, allocation or synchronisation fails.
 */
GTG_API gtg_status gemm_host(int precision, int64_t M, int64_t N, int64_t K,
                             const void *A, int64_t lda, const void *B, int64_t ldb,
                             float *C, int64_t ldc, const gtg_epilogue *epilogue);

/*
 * gtg_pool_trim -- returns to the driver the device memory that the
 * library's workspace pools keep reserved between calls (on every device
 * used so far). Buffers still in use by queued work are not affected.
 * Errors: GTG_ERR_DEVICE if the driver refuses.
 */
GTG_API gtg_status gtg_pool_trim(void);

/*
 * gemm_strided_batched -- `batch` independent products in one call ("Matrix
 * Operations", "Performance Considerations": processing several matrix
 * multiplications in parallel):
 *
 *   C_b = act(A_b * B_b + bias),  A_b = A + b*strideA, B_b = B + b*strideB,
 *   C_b = C + b*strideC  (strides in elements, b = 0 .. batch-1)
 *
 *   precision  GTG_PREC_F32, _TF32, _BF16 or _F16 (A and B element type as in
 *              the single-matrix calls; C is FP32)
 *   batch      >= 0; strideA, strideB >= 0 (0 reuses one operand for every
 *              item); strideC must keep the outputs apart
 *              (strideC >= (M-1)*ldc + N when batch > 1)
 *   epilogue   as for gemm_*_ex (the same bias for every item), or NULL
 *
 * The tensor-core kernels walk the output tiles of all items in one launch
 * (their tensor maps get the batch as a third dimension). When strideA or,
 * for 16-bit inputs, strideB or a leading dimension is not a multiple of 16
 * bytes, the items of that operand (one copy if its stride is 0) are first
 * copied into aligned rows in a temporary from the pool. FP32 batches run
 * on the SIMT kernel, also in one launch over all items (at most 65535 items
 * per launch; larger batches take several). Errors as for the single calls;
 * no item is computed if the arguments of any item are invalid.
 */
GTG_API gtg_status gemm_strided_batched(int precision, int64_t M, int64_t N, int64_t K,
                                        const void *A, int64_t lda, int64_t strideA,
                                        const void *B, int64_t ldb, int64_t strideB,
                                        float *C, int64_t ldc, int64_t strideC,
                                        int64_t batch, const gtg_epilogue *epilogue,
                                        cudaStream_t stream);

/*
 * The pages' own kernel designs, kept for measurement against the kernels
 * above (they are not used by any other call). FP32, same products, same
 * argument conventions as gemm_f32 / gemv_f32 (batch 1):
 *
 *   GTG_ABL_GEMM_NAIVE_16 / _32  one thread per output of C, 16 x 16 or
 *        32 x 32 threads per block, operands read from global memory for
 *        every multiply-add ("Matrix Operations", GEMM "Naive
 *        Implementation"; "CUDA Programming (6)" section 3.1);
 *   GTG_ABL_GEMM_TILED_16 / _32  16 x 16 or 32 x 32 shared-memory tiles,
 *        zero-padded edges, two barriers per tile ("Tiled Implementation with
 *        Shared Memory"; section 3.2);
 *   GTG_ABL_GEMV_NAIVE   one thread per row, the vector read from global
 *        memory by every thread ("Matrix-Vector Multiplication", "Naive
 *        Implementation");
 *   GTG_ABL_GEMV_SHARED  the vector staged in shared memory in chunks of 256
 *        with a barrier on each side ("Optimized Implementation with Shared
 *        Memory", "Handling Large Vectors").
 *
 * An unknown variant returns GTG_ERR_INVALID_VALUE; a grid beyond the CUDA
 * limits (more than 65535 row blocks) returns GTG_ERR_UNSUPPORTED.
 */
enum { GTG_ABL_GEMM_NAIVE_16 = 0, GTG_ABL_GEMM_NAIVE_32 = 1, GTG_ABL_GEMM_TILED_16 = 2,
       GTG_ABL_GEMM_TILED_32 = 3 };
enum { GTG_ABL_GEMV_NAIVE = 0, GTG_ABL_GEMV_SHARED = 1 };

GTG_API gtg_status gtg_ablation_gemm_f32(int variant, int64_t M, int64_t N, int64_t K,
                                         const float *A, int64_t lda, const float *B, int64_t ldb,
                                         float *C, int64_t ldc, cudaStream_t stream);
GTG_API gtg_status gtg_ablation_gemv_f32(int variant, int64_t M, int64_t N, const float *A,
                                         int64_t lda, const float *x, float *y, cudaStream_t stream);

/* Static English text for a status code (never NULL). */
GTG_API const char *gtg_status_string(gtg_status status);

/*
 * Waits for `stream`, then returns and clears the device status word of the
 * current device: GTG_OK, or GTG_ERR_TIMEOUT if some kernel launched since
 * the last call gave up a pipeline wait (its output is then incomplete).
 * GTG_ERR_DEVICE if the synchronisation itself failed.
 */
GTG_API gtg_status gtg_sync_status(cudaStream_t stream);

/* Text of the last CUDA runtime error seen by the library on this thread. */
GTG_API const char *gtg_last_cuda_error(void);

/*
 * Which kernel a GEMM call with these arguments would run (no launch, no
 * device work). Fills *plan. `precision` is GTG_PREC_F32, _TF32 or _BF16.
 * Returns the same validation status the GEMM call itself would.
 */
enum { GTG_PREC_F32 = 0, GTG_PREC_TF32 = 1, GTG_PREC_BF16 = 2, GTG_PREC_F16 = 3 };
enum { GTG_KERNEL_NONE = 0, GTG_KERNEL_SIMT = 1, GTG_KERNEL_TCGEN05 = 2,
       GTG_KERNEL_ZERO_FILL = 3, GTG_KERNEL_GEMV = 4 };
typedef struct {
    int kernel;   /* GTG_KERNEL_* */
    int bm, bn, bk;
    int stages;   /* shared-memory pipeline depth */
    int grid;     /* thread blocks launched */
    int threads;  /* threads per block */
    int smem;     /* dynamic shared memory per block, bytes */
    int cluster;  /* thread blocks per cluster (1: no cluster launch) */
    int splits;   /* GEMM: slices of K computed apart (partial products added in
                     order by a second kernel; 1: none) */
} gtg_plan;

GTG_API gtg_status gtg_plan_gemm(int precision, int64_t M, int64_t N, int64_t K,
                         const void *A, int64_t lda,
                         const void *B, int64_t ldb,
                         const void *C, int64_t ldc,
                         gtg_plan *plan);

/* Same for gemv_f32 (bm = rows per warp task, bn = entries of each vector
 * staged per CTA, bk = 16-byte loads in flight per row, stages = staging
 * passes, cluster = CTAs sharing a block of rows, each with its own block of
 * columns). */
GTG_API gtg_status gtg_plan_gemv(int64_t M, int64_t N, const float *A, int64_t lda,
                         const float *x, int64_t ldx, const float *y, int64_t ldy,
                         int batch, gtg_plan *plan);

/* Same for gemv_bf16. */
GTG_API gtg_status gtg_plan_gemv_bf16(int64_t M, int64_t N, const gtg_bf16 *A, int64_t lda,
                              const float *x, int64_t ldx, const float *y, int64_t ldy,
                              int batch, gtg_plan *plan);

/* Version of this ABI (major * 10000 + minor * 100 + patch). */
GTG_API int gtg_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GTG_H */
