// Host-side interface between the C ABI (api.cpp) and the kernel files.
// Arguments reaching these launchers have already been validated.
#pragma once
#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace qmm {

// Bits of the device error word (read back by qmm_get_device_error).
constexpr unsigned kErrIndexBit = 1u;    // a qmm_rows index outside the table
constexpr unsigned kErrTimeoutBit = 2u;  // a bounded wait inside a kernel ran out

// Launch options of the calling host thread (qmm_set_launch_flags).
constexpr unsigned kLaunchPdl = 1u;
unsigned launch_flags();
// Polls a bounded wait of the calling host thread's kernels makes before it
// gives up (qmm_set_wait_limit; default kDefaultWaitLimit).
constexpr uint32_t kDefaultWaitLimit = 1u << 24;
uint32_t wait_limit();

// Element types, numbered as the C ABI's qmm_dtype.
constexpr int kTypeF32 = 0, kTypeBF16 = 1, kTypeF16 = 2;

struct PackedWeight {
  const uint32_t *w;       // [rows, cols*bits/32]
  const uint16_t *scales;  // [rows, cols/group] of sb_type (fp32 values when kTypeF32)
  const uint16_t *biases;  // [rows, cols/group] of sb_type
  int64_t rows, cols;
  int group, bits;
  int sb_type = kTypeBF16;
};

// The current device's error word (a static __device__ variable); its device
// address, looked up once per device.  nullptr if the lookup failed.
unsigned *device_error_word();
// Synchronize `stream`, read the word and clear it.
cudaError_t take_device_error(cudaStream_t stream, unsigned *bits);

// tensormap.cpp: a 2-D tiled tensor map over a row-major array of `outer`
// rows of `inner` elements, `row_bytes` apart; boxes of box_inner x
// box_outer elements, out-of-range elements read as zero.
cudaError_t encode_map_2d(CUtensorMap *map, CUtensorMapDataType type, const void *base,
                          uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                          uint32_t box_outer, CUtensorMapSwizzle swizzle);
int sm_count();

// Raise Kern's dynamic shared memory limit on the current device to at least
// `bytes`, calling the runtime only when this device's limit is lower.  The
// limit is remembered per kernel (the template argument is the kernel itself,
// so each kernel has its own record) and per device.  Safe from several host
// threads: a race repeats the (idempotent) call.
template <auto Kern>
inline cudaError_t ensure_smem_limit(size_t bytes) {
  constexpr int kMaxDevices = 64;
  static std::atomic<size_t> limit[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool known = dev >= 0 && dev < kMaxDevices;
  if (known && limit[dev].load(std::memory_order_acquire) >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e != cudaSuccess) return e;
  if (known) {
    size_t cur = limit[dev].load(std::memory_order_relaxed);
    while (cur < bytes && !limit[dev].compare_exchange_weak(cur, bytes, std::memory_order_release)) {
    }
  }
  return cudaSuccess;
}

// dequant.cu: out[r, :] = dequant(W[src(r), :]) for r < out_rows, where
// src(r) = idx[r] if idx is given (a rows gather) else r; out of out_type.
cudaError_t launch_dequantize(const PackedWeight &w, const uint32_t *idx,
                              int64_t out_rows, void *out, int out_type,
                              cudaStream_t stream);

// gemv.cu: decode path, M <= 16.
cudaError_t launch_gemv(const uint16_t *x, int64_t M, const PackedWeight &w,
                        bool transpose, void *y, bool y_bf16,
                        cudaStream_t stream);

// gemv_f16.cu: the same for fp16 x, scales and biases (y fp16 if y_f16).
cudaError_t launch_gemv_f16(const uint16_t *x, int64_t M, const PackedWeight &w,
                            bool transpose, void *y, bool y_f16, cudaStream_t stream);

// gemm_sm103.cu: tensor-core path for larger M.
cudaError_t launch_gemm(const uint16_t *x, int64_t M, const PackedWeight &w,
                        bool transpose, void *y, bool y_bf16,
                        cudaStream_t stream);

cudaError_t launch_gemm_f16(const uint16_t *x, int64_t M, const PackedWeight &w,
                            bool transpose, void *y, bool y_f16, cudaStream_t stream);

// gather_qmm: output batch b (of `batches`) is x[lhs[b]] (M x K, of
// x_batches) times weight batch rhs[b] (of w_batches, each shaped as w);
// lhs / rhs null means b itself.  `sorted` promises rhs is sorted.  Device
// indices out of range zero their batch and raise kErrIndexBit.
cudaError_t launch_gather(const uint16_t *x, int64_t x_batches, int64_t M, const PackedWeight &w,
                          int64_t w_batches, const uint32_t *lhs, const uint32_t *rhs,
                          int64_t batches, bool transpose, bool sorted, void *y, bool y_bf16,
                          cudaStream_t stream);

// gemm_sm103.cu: gather_qmm on the tensor cores for sorted weight-batch
// indices with one x row per batch and no lhs indices (W transposed).
// cudaErrorNotSupported (nothing launched) when the shape does not suit it.
cudaError_t launch_gemm_grouped(const uint16_t *x, int64_t batches, const PackedWeight &w,
                                int64_t w_batches, const uint32_t *rhs, void *y, bool y_bf16,
                                cudaStream_t stream);

// Fused decode GEMVs on a transposed W ([N, K], K a multiple of 128):
// y_gate = x . gate^T and y_up = x . up^T in one launch (M <= 16; the two
// weights share N, K, bits and group size); y = silu(gate) * up . w^T (+ resid,
// bf16 [M, N], when not null) with M <= 8.  cudaErrorNotSupported otherwise.
cudaError_t launch_gate_up(const uint16_t *x, int64_t M, const PackedWeight &gate,
                           const PackedWeight &up, void *y_gate, void *y_up, bool y_bf16,
                           cudaStream_t stream);
cudaError_t launch_silu_gate(const uint16_t *gate, const uint16_t *up, int64_t M,
                             const PackedWeight &w, const uint16_t *resid, void *y, bool y_bf16,
                             cudaStream_t stream);

// quantize: w [rows, cols] of w_type (cols a multiple of group) -> packed
// uint32 [rows, cols*bits/32], scales and biases [rows, cols/group] of w_type.
cudaError_t launch_quantize(const void *w, int w_type, int64_t rows, int64_t cols, int group,
                            int bits, uint32_t *packed, void *scales, void *biases,
                            cudaStream_t stream);

// mm_f32.cu: quantized_matmul computed in fp32 on the CUDA cores, for x,
// scales and biases that promote to fp32: x [M, K] of x_type, scales and
// biases of w.sb_type, y fp32 [M, N].
cudaError_t launch_mm_f32(const void *x, int x_type, int64_t M, const PackedWeight &w,
                          bool transpose, float *y, cudaStream_t stream);

// The variant of launch_gemm whose split-K partials go to `scratch` (the
// library's static array, see static_scratch) instead of a stream-ordered
// allocation.  *needed gets the partials' bytes; cudaErrorInvalidValue, with
// nothing launched, when they exceed static_scratch_bytes().
size_t static_scratch_bytes();
float *static_scratch();
cudaError_t launch_gemm_static_scratch(const uint16_t *x, int64_t M, const PackedWeight &w,
                                       bool transpose, void *y, bool y_bf16, float *scratch,
                                       cudaStream_t stream, size_t *needed);

}  // namespace qmm
