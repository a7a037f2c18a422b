// quantize: bf16 w [rows, cols] -> packed codes, bf16 scales and biases.
//
// nuvec_core quantized.rs, module doc: a value w is stored as
// round((w - bias) / scale), clamped to [0, 2^bits - 1]; `dequantize` doc:
// bias = the group minimum.  The scale is the plain min-max one,
// (max - min) / (2^bits - 1) in fp32, stored as its round-to-nearest-even
// bf16; the codes come from the stored scale and bias, each step one IEEE fp32
// operation, rounding half to even.  A zero scale (a constant group) gives
// every code 0, so the group dequantizes to its value exactly.
//
// HBM-bound: one thread per group.  It reads its group twice (minimum and
// maximum, then the codes; the second read hits L1), assembles the group's
// bits*group_size/32 words in registers and writes them with the widest
// aligned stores.
#include "common.cuh"
#include "internal.h"

namespace qmm {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void unpack8(const uint4 &u, float (&v)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu);
    v[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
  }
}

template <int BITS, int G>
__global__ void __launch_bounds__(kThreads)
quantize_kernel(const uint16_t *__restrict__ w, uint32_t total, uint32_t groups_per_row,
                int64_t cols, uint32_t *__restrict__ packed, uint16_t *__restrict__ scales,
                uint16_t *__restrict__ biases) {
  constexpr int NW = G * BITS / 32;  // words per group
  constexpr uint32_t TOP = (1u << BITS) - 1u;
  const int64_t wpr = (cols * BITS) >> 5;
  for (uint32_t gid = blockIdx.x * kThreads + threadIdx.x; gid < total;
       gid += gridDim.x * kThreads) {
    const uint32_t r = gid / groups_per_row, j = gid - r * groups_per_row;
    const uint4 *src = reinterpret_cast<const uint4 *>(w + static_cast<int64_t>(r) * cols +
                                                       static_cast<int64_t>(j) * G);
    // Minimum and maximum, compared in the group's order.
    float lo = 0.0f, hi = 0.0f;
#pragma unroll
    for (int q = 0; q < G / 8; ++q) {
      float v[8];
      unpack8(__ldg(src + q), v);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (q == 0 && e == 0) {
          lo = hi = v[0];
        } else {
          if (v[e] < lo) lo = v[e];
          if (v[e] > hi) hi = v[e];
        }
      }
    }
    const uint16_t sb = f32_to_bf16_bits(__fdiv_rn(__fsub_rn(hi, lo), static_cast<float>(TOP)));
    const uint16_t bb = f32_to_bf16_bits(lo);  // exact: lo is a bf16 value
    const float s = bf16_bits_to_f32(sb), b = bf16_bits_to_f32(bb);
    uint32_t words[NW];
#pragma unroll
    for (int i = 0; i < NW; ++i) words[i] = 0u;
    if (s != 0.0f) {
#pragma unroll
      for (int q = 0; q < G / 8; ++q) {
        float v[8];
        unpack8(__ldg(src + q), v);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float qf = fminf(fmaxf(rintf(__fdiv_rn(__fsub_rn(v[e], b), s)), 0.0f),
                                 static_cast<float>(TOP));
          const uint32_t code = static_cast<uint32_t>(qf);
          const int bit = (8 * q + e) * BITS, wi = bit >> 5, sh = bit & 31;
          words[wi] |= code << sh;
          if (sh + BITS > 32) words[wi + 1] |= code >> (32 - sh);
        }
      }
    }
    uint32_t *dst = packed + static_cast<int64_t>(r) * wpr + static_cast<int64_t>(j) * NW;
    if (NW % 4 == 0 && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
#pragma unroll
      for (int i = 0; i < NW / 4; ++i)
        reinterpret_cast<uint4 *>(dst)[i] =
            make_uint4(words[4 * i], words[4 * i + 1], words[4 * i + 2], words[4 * i + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < NW; ++i) dst[i] = words[i];
    }
    const int64_t o = static_cast<int64_t>(r) * groups_per_row + j;
    scales[o] = sb;
    biases[o] = bb;
  }
}

template <int BITS, int G>
cudaError_t launch_g(const uint16_t *w, int64_t rows, int64_t cols, uint32_t *packed,
                     uint16_t *scales, uint16_t *biases, cudaStream_t stream) {
  const int64_t gpr = cols / G;
  if (gpr >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
  // Batches of whole rows with fewer than 2^31 groups each (32-bit indices).
  const int64_t rows_per_batch = ((int64_t(1) << 31) - 1) / gpr;
  const int max_blocks = 16 * sm_count();
  for (int64_t r0 = 0; r0 < rows; r0 += rows_per_batch) {
    const int64_t nr = rows - r0 < rows_per_batch ? rows - r0 : rows_per_batch;
    const uint32_t total = static_cast<uint32_t>(nr * gpr);
    const int64_t blocks = (static_cast<int64_t>(total) + kThreads - 1) / kThreads;
    const unsigned grid = static_cast<unsigned>(blocks < max_blocks ? blocks : max_blocks);
    const int64_t wpr = (cols * BITS) / 32;
    quantize_kernel<BITS, G><<<grid, kThreads, 0, stream>>>(
        w + r0 * cols, total, static_cast<uint32_t>(gpr), cols, packed + r0 * wpr,
        scales + r0 * gpr, biases + r0 * gpr);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <int BITS>
cudaError_t launch_bits(const uint16_t *w, int64_t rows, int64_t cols, int group,
                        uint32_t *packed, uint16_t *scales, uint16_t *biases, cudaStream_t stream) {
  switch (group) {
    case 32: return launch_g<BITS, 32>(w, rows, cols, packed, scales, biases, stream);
    case 64: return launch_g<BITS, 64>(w, rows, cols, packed, scales, biases, stream);
    case 128: return launch_g<BITS, 128>(w, rows, cols, packed, scales, biases, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_quantize(const uint16_t *w, int64_t rows, int64_t cols, int group, int bits,
                            uint32_t *packed, uint16_t *scales, uint16_t *biases,
                            cudaStream_t stream) {
  switch (bits) {
    case 1: return launch_bits<1>(w, rows, cols, group, packed, scales, biases, stream);
    case 2: return launch_bits<2>(w, rows, cols, group, packed, scales, biases, stream);
    case 3: return launch_bits<3>(w, rows, cols, group, packed, scales, biases, stream);
    case 4: return launch_bits<4>(w, rows, cols, group, packed, scales, biases, stream);
    case 5: return launch_bits<5>(w, rows, cols, group, packed, scales, biases, stream);
    case 6: return launch_bits<6>(w, rows, cols, group, packed, scales, biases, stream);
    case 8: return launch_bits<8>(w, rows, cols, group, packed, scales, biases, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qmm
