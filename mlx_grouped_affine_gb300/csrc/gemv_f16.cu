// Decode path of quantized_matmul in fp16 (fp16 x, scales and biases; M <=
// 16): the kernels of gemv_impl.cuh with fp16 elements, in a translation unit
// of its own so that it compiles beside the bf16 one.
#include "gemv_impl.cuh"

namespace qmm {

cudaError_t launch_gemv_f16(const uint16_t *x, int64_t M, const PackedWeight &w, bool transpose,
                            void *y, bool y_f16, cudaStream_t stream) {
  return gemv_entry<ElemF16>(x, M, w, transpose, y, y_f16, stream);
}

}  // namespace qmm
