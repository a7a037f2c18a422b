// Standalone dequantize and the rows gather-dequant.
//
// out[r, :] = dequant(W[src(r), :]) with src(r) = r (nuvec_core quantized.rs,
// `dequantize`; spark_runtime weights/mlx_int8.rs, `dequantize_to`) or
// src(r) = idx[r] (maya2_mlx quant.py, `rows`: gather then dequantize, done
// here in one pass that reads only the gathered rows).
//
// HBM-bound: per 8 outputs a thread reads `bits` bytes of codes and writes 16
// (bf16) or 32 (fp32) bytes, so the kernel is sized for coalesced 16-byte
// stores.  A block covers 2048 consecutive columns of one output row: thread t
// owns the 8-code chunk t, whose codes are the `bits` bytes at byte offset
// 8*bits*t/8 of the row, read through the one or two aligned words that hold
// them.  Each element is fp32 fma(scale, code, bias): the product of a bf16
// scale and a code below 2^8 is exact, so this rounds once, at the add
// (rlx-moshi src/mlx_dequant.rs, `dequantize_affine`: scale * code + bias).
#include "common.cuh"
#include "internal.h"

#include <mutex>

namespace qmm {

// One error word per device, reached from the host through its address.
static __device__ unsigned g_device_error;

namespace {

constexpr int kThreads = 256;
constexpr int kColsPerBlock = kThreads * 8;

template <int BITS>
__device__ __forceinline__ uint64_t load_chunk_window(const uint32_t *__restrict__ row,
                                                      int chunk) {
  // The chunk's codes start at bit 8*BITS*chunk of the row's stream.
  const int bit = 8 * BITS * chunk;
  const int word = bit >> 5, sh = bit & 31;
  uint32_t lo = __ldg(row + word);
  uint32_t hi = (sh + 8 * BITS > 32) ? __ldg(row + word + 1) : 0u;
  return ((static_cast<uint64_t>(hi) << 32) | lo) >> sh;
}

template <int BITS, bool OUT_BF16, bool GATHER>
__global__ void __launch_bounds__(kThreads)
dequant_kernel(const uint32_t *__restrict__ w, const uint16_t *__restrict__ scales,
               const uint16_t *__restrict__ biases, const uint32_t *__restrict__ idx,
               int64_t out_rows, int64_t table_rows, int64_t cols, int group_shift,
               int blocks_per_row, void *__restrict__ out, unsigned *err) {
  const int64_t words_per_row = (cols * BITS) >> 5;
  const int64_t groups = cols >> group_shift;
  const int chunks_per_row = static_cast<int>(cols >> 3);
  const int64_t total_blocks = out_rows * blocks_per_row;
  for (int64_t blk = blockIdx.x; blk < total_blocks; blk += gridDim.x) {
    const int64_t r = blk / blocks_per_row;
    const int chunk = static_cast<int>(blk - r * blocks_per_row) * kThreads + threadIdx.x;
    if (chunk >= chunks_per_row) continue;
    int64_t src = r;
    bool in_table = true;
    if (GATHER) {
      src = __ldg(idx + r);
      in_table = src < table_rows;
      if (!in_table && chunk == 0) atomicOr(err, kErrIndexBit);
    }
    float v[8];
    if (in_table) {
      const uint64_t win = load_chunk_window<BITS>(w + src * words_per_row, chunk);
      const int64_t g = (static_cast<int64_t>(chunk) * 8) >> group_shift;
      const float s = bf16_bits_to_f32(__ldg(scales + src * groups + g));
      const float b = bf16_bits_to_f32(__ldg(biases + src * groups + g));
      constexpr uint32_t mask = (1u << BITS) - 1u;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t code = static_cast<uint32_t>(win >> (j * BITS)) & mask;
        v[j] = __fmaf_rn(s, static_cast<float>(code), b);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = 0.0f;
    }
    const int64_t o = r * cols + static_cast<int64_t>(chunk) * 8;
    if (OUT_BF16) {
      uint4 p;
      p.x = pack_bf16x2(v[0], v[1]);
      p.y = pack_bf16x2(v[2], v[3]);
      p.z = pack_bf16x2(v[4], v[5]);
      p.w = pack_bf16x2(v[6], v[7]);
      *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + o) = p;
    } else {
      float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(out) + o);
      dst[0] = make_float4(v[0], v[1], v[2], v[3]);
      dst[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
  }
}

template <int BITS, bool OUT_BF16, bool GATHER>
cudaError_t launch_t(const PackedWeight &pw, const uint32_t *idx, int64_t out_rows,
                     void *out, cudaStream_t stream) {
  const int blocks_per_row = static_cast<int>((pw.cols + kColsPerBlock - 1) / kColsPerBlock);
  const int64_t total = out_rows * blocks_per_row;
  const unsigned grid = static_cast<unsigned>(total < (1ll << 30) ? total : (1ll << 30));
  const int group_shift = pw.group == 32 ? 5 : pw.group == 64 ? 6 : 7;
  unsigned *err = device_error_word();
  if (!err) return cudaErrorInvalidSymbol;
  dequant_kernel<BITS, OUT_BF16, GATHER><<<grid, kThreads, 0, stream>>>(
      pw.w, pw.scales, pw.biases, idx, out_rows, pw.rows, pw.cols, group_shift,
      blocks_per_row, out, err);
  return cudaGetLastError();
}

template <int BITS>
cudaError_t launch_bits(const PackedWeight &pw, const uint32_t *idx, int64_t out_rows,
                        void *out, bool out_bf16, cudaStream_t stream) {
  if (idx)
    return out_bf16 ? launch_t<BITS, true, true>(pw, idx, out_rows, out, stream)
                    : launch_t<BITS, false, true>(pw, idx, out_rows, out, stream);
  return out_bf16 ? launch_t<BITS, true, false>(pw, idx, out_rows, out, stream)
                  : launch_t<BITS, false, false>(pw, idx, out_rows, out, stream);
}

}  // namespace

cudaError_t launch_dequantize(const PackedWeight &pw, const uint32_t *idx, int64_t out_rows,
                              void *out, bool out_bf16, cudaStream_t stream) {
  switch (pw.bits) {
    case 1: return launch_bits<1>(pw, idx, out_rows, out, out_bf16, stream);
    case 2: return launch_bits<2>(pw, idx, out_rows, out, out_bf16, stream);
    case 3: return launch_bits<3>(pw, idx, out_rows, out, out_bf16, stream);
    case 4: return launch_bits<4>(pw, idx, out_rows, out, out_bf16, stream);
    case 5: return launch_bits<5>(pw, idx, out_rows, out, out_bf16, stream);
    case 6: return launch_bits<6>(pw, idx, out_rows, out, out_bf16, stream);
    case 8: return launch_bits<8>(pw, idx, out_rows, out, out_bf16, stream);
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
