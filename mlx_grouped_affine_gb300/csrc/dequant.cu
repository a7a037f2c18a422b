// Standalone dequantize and the rows gather-dequant.
//
// out[r, :] = dequant(W[src(r), :]) with src(r) = r (nuvec_core quantized.rs,
// `dequantize`; spark_runtime weights/mlx_int8.rs, `dequantize_to`) or
// src(r) = idx[r] (maya2_mlx quant.py, `rows`: gather then dequantize, done
// here in one pass that reads only the gathered rows).
//
// HBM-bound: per 32 outputs a thread reads `bits` words of codes (32 codes
// always take exactly `bits` words, so every thread's codes start on a word
// boundary and load with the widest aligned vector loads) and writes 64 (bf16)
// or 128 (fp32) contiguous bytes; consecutive threads cover consecutive code
// groups, so a warp streams 2 or 4 KB of output.  Each element is fp32
// fma(scale, code, bias), scale * code + bias rounded once (rlx-moshi
// src/mlx_dequant.rs, `dequantize_affine`: scale * code + bias); for 16-bit
// scales the product is exact.  Scales and biases are bf16, fp16 or fp32
// (nuvec_core quantized.rs: they keep the quantized weights' dtype, and
// `dequantize` returns the scales' dtype); a 16-bit output is the
// round-to-nearest-even of the fp32 value.
#include "common.cuh"
#include "internal.h"

#include <mutex>
#include <type_traits>

namespace qmm {

// One error word per device, reached from the host through its address.
static __device__ unsigned g_device_error;

namespace {

constexpr int kThreads = 256;

// Element i of a scale or bias array of type t, in fp32 (exact).
__device__ __forceinline__ float load_sb(const uint16_t *p, int t, int64_t i) {
  if (t == kTypeF32) return __ldg(reinterpret_cast<const float *>(p) + i);
  const uint32_t h = __ldg(p + i);
  return t == kTypeF16 ? ElemF16::to_f32(h) : ElemBF16::to_f32(h);
}

// 32 bytes to global memory in one instruction (p 32-byte aligned).
__device__ __forceinline__ void st_global_256(void *p, const uint4 &a, const uint4 &b) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a.x),
               "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
               : "memory");
}

template <int BITS, int OUT, bool GATHER>
__global__ void __launch_bounds__(kThreads)
dequant_kernel(const uint32_t *__restrict__ w, const uint16_t *__restrict__ scales,
               const uint16_t *__restrict__ biases, int sb_type, const uint32_t *__restrict__ idx,
               int64_t row0, uint32_t groups_total, uint32_t groups_per_row, int64_t table_rows,
               int64_t cols, int group_shift, void *__restrict__ out, unsigned *err) {
  const int64_t words_per_row = (cols * BITS) >> 5;
  const int64_t sb_per_row = cols >> group_shift;
  const bool out32 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;
  for (uint32_t gid = blockIdx.x * kThreads + threadIdx.x; gid < groups_total;
       gid += gridDim.x * kThreads) {
    const uint32_t rl = gid / groups_per_row, j = gid - rl * groups_per_row;
    const int64_t r = row0 + rl;
    int64_t src = r;
    bool in_table = true;
    if (GATHER) {
      src = __ldg(idx + r);
      in_table = src < table_rows;
      if (!in_table && j == 0) atomicOr(err, kErrIndexBit);
    }
    float v[32];
    if (in_table) {
      uint32_t words[BITS];
      load_words<BITS>(w + src * words_per_row + static_cast<int64_t>(j) * BITS, words);
      const int64_t g = (static_cast<int64_t>(j) * 32) >> group_shift;
      const float s = load_sb(scales, sb_type, src * sb_per_row + g);
      const float b = load_sb(biases, sb_type, src * sb_per_row + g);
#pragma unroll
      for (int i = 0; i < 32; ++i)
        v[i] = __fmaf_rn(s, static_cast<float>(code_at<BITS>(words, i)), b);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0.0f;
    }
    const int64_t o = r * cols + static_cast<int64_t>(j) * 32;
    // The thread's 32 outputs are 64 (16-bit) or 128 (fp32) contiguous bytes:
    // 32-byte stores when the output is 32-byte aligned, else 16-byte ones.
    if constexpr (OUT != kTypeF32) {
      using E = typename std::conditional<OUT == kTypeF16, ElemF16, ElemBF16>::type;
      uint4 q4[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        q4[q] = make_uint4(E::pack2(v[8 * q], v[8 * q + 1]), E::pack2(v[8 * q + 2], v[8 * q + 3]),
                           E::pack2(v[8 * q + 4], v[8 * q + 5]), E::pack2(v[8 * q + 6], v[8 * q + 7]));
      uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + o);
      if (out32) {
        st_global_256(dst, q4[0], q4[1]);
        st_global_256(dst + 2, q4[2], q4[3]);
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) dst[q] = q4[q];
      }
    } else {
      float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(out) + o);
      if (out32) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          st_global_256(dst + 2 * q,
                        make_uint4(__float_as_uint(v[8 * q]), __float_as_uint(v[8 * q + 1]),
                                   __float_as_uint(v[8 * q + 2]), __float_as_uint(v[8 * q + 3])),
                        make_uint4(__float_as_uint(v[8 * q + 4]), __float_as_uint(v[8 * q + 5]),
                                   __float_as_uint(v[8 * q + 6]), __float_as_uint(v[8 * q + 7])));
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      }
    }
  }
}

template <int BITS, int OUT, bool GATHER>
cudaError_t launch_t(const PackedWeight &pw, const uint32_t *idx, int64_t out_rows,
                     void *out, cudaStream_t stream) {
  const int group_shift = pw.group == 32 ? 5 : pw.group == 64 ? 6 : 7;
  unsigned *err = device_error_word();
  if (!err) return cudaErrorInvalidSymbol;
  const int64_t gpr = pw.cols / 32;
  if (gpr >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
  // Batches of whole rows with fewer than 2^31 code groups each, so that the
  // kernel's index arithmetic stays in 32 bits.
  const int64_t rows_per_batch = ((int64_t(1) << 31) - 1) / gpr;
  const int max_blocks = 16 * sm_count();
  for (int64_t r0 = 0; r0 < out_rows; r0 += rows_per_batch) {
    const int64_t rows = out_rows - r0 < rows_per_batch ? out_rows - r0 : rows_per_batch;
    const uint32_t total = static_cast<uint32_t>(rows * gpr);
    const int64_t blocks = (static_cast<int64_t>(total) + kThreads - 1) / kThreads;
    const unsigned grid = static_cast<unsigned>(blocks < max_blocks ? blocks : max_blocks);
    dequant_kernel<BITS, OUT, GATHER><<<grid, kThreads, 0, stream>>>(
        pw.w, pw.scales, pw.biases, pw.sb_type, idx, r0, total, static_cast<uint32_t>(gpr), pw.rows,
        pw.cols, group_shift, out, err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <int BITS, bool GATHER>
cudaError_t launch_out(const PackedWeight &pw, const uint32_t *idx, int64_t out_rows, void *out,
                       int out_type, cudaStream_t stream) {
  switch (out_type) {
    case kTypeF32: return launch_t<BITS, kTypeF32, GATHER>(pw, idx, out_rows, out, stream);
    case kTypeBF16: return launch_t<BITS, kTypeBF16, GATHER>(pw, idx, out_rows, out, stream);
    case kTypeF16: return launch_t<BITS, kTypeF16, GATHER>(pw, idx, out_rows, out, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int BITS>
cudaError_t launch_bits(const PackedWeight &pw, const uint32_t *idx, int64_t out_rows,
                        void *out, int out_type, cudaStream_t stream) {
  return idx ? launch_out<BITS, true>(pw, idx, out_rows, out, out_type, stream)
             : launch_out<BITS, false>(pw, idx, out_rows, out, out_type, stream);
}

}  // namespace

cudaError_t launch_dequantize(const PackedWeight &pw, const uint32_t *idx, int64_t out_rows,
                              void *out, int out_type, cudaStream_t stream) {
  switch (pw.bits) {
    case 1: return launch_bits<1>(pw, idx, out_rows, out, out_type, stream);
    case 2: return launch_bits<2>(pw, idx, out_rows, out, out_type, stream);
    case 3: return launch_bits<3>(pw, idx, out_rows, out, out_type, stream);
    case 4: return launch_bits<4>(pw, idx, out_rows, out, out_type, stream);
    case 5: return launch_bits<5>(pw, idx, out_rows, out, out_type, stream);
    case 6: return launch_bits<6>(pw, idx, out_rows, out, out_type, stream);
    case 8: return launch_bits<8>(pw, idx, out_rows, out, out_type, stream);
    default: return cudaErrorInvalidValue;
  }
}

// ----------------------------------------------------------- error word ----

unsigned *device_error_word() {
  constexpr int kMaxDevices = 64;
  static unsigned *addr[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<unsigned *>(p);
  }
  return addr[dev];
}

cudaError_t take_device_error(cudaStream_t stream, unsigned *bits) {
  *bits = 0;
  unsigned *err = device_error_word();
  if (!err) return cudaErrorInvalidSymbol;
  cudaError_t e = cudaMemcpyAsync(bits, err, sizeof(unsigned), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(err, 0, sizeof(unsigned), stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  return e;
}

}  // namespace qmm
