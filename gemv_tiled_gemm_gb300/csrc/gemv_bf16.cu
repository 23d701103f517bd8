// The BF16-matrix instantiations of the GEMV kernels (gemv_kernels.cuh):
// A holds BF16 bit patterns, x, y and every multiply-add are FP32.
#include "gemv_kernels.cuh"

namespace gtg {
namespace gemv {

void *kernel_for_bf16(int batch, int kind, bool vec) { return kernel_for<uint16_t>(batch, kind, vec); }

}  // namespace gemv
}  // namespace gtg
