// quantize: w [rows, cols] (bf16, fp16 or fp32) -> packed codes, scales and
// biases in w's type (nuvec_core quantized.rs, `quantize` doc).
//
// nuvec_core quantized.rs, module doc: a value w is stored as
// round((w - bias) / scale), clamped to [0, 2^bits - 1]; `dequantize` doc:
// bias = the group minimum.  The scale is the plain min-max one,
// (max - min) / (2^bits - 1) in fp32, stored in w's type (rounded to nearest
// even for the 16-bit types); the bias is the minimum, exactly; the codes
// come from the stored scale and bias, each step one IEEE fp32 operation,
// rounding half to even.  A zero scale (a constant group) gives
// every code 0, so the group dequantizes to its value exactly.
//
// One thread per group.  It reads its group twice (minimum and
// maximum, then the codes; the second read hits L1), assembles the group's
// bits*group_size/32 words in registers and writes them with the widest
// aligned stores.
#include "common.cuh"
#include "internal.h"

#include <type_traits>

namespace qmm {
namespace {

constexpr int kThreads = 256;

// rint(RN((w - bias) / scale)) -- the code before clamping -- given d = w - bias,
// the scale s and r = RN(1/s), without a division for almost every element.
// q = RN(d * r) is within 2^-23 |d/s| of d/s (two roundings of 2^-24 each), and
// RN(d/s) within 2^-24 |d/s| of it, so the two are less than |q| 2^-21 apart.
// Unless q lies within |q| 2^-20 of the half-integer between its neighbours,
// both round to the same integer; those few elements, and every element of a
// group whose reciprocal is not finite (the comparison is false for NaN),
// take the correctly rounded division.
// Codes stay below 2^9, so for |q| < 512 the margin |q| 2^-20 is below 2^-11
// and a fixed one serves: q - n is exact (n is q's nearest integer), and
// |q - n| < 1/2 - 2^-11 keeps q more than 2^-11 from the half-integer between
// n and its neighbour on q's side.
__device__ __forceinline__ float rint_quotient(float d, float s, float r) {
  const float q = __fmul_rn(d, r);
  const float n = rintf(q);
  if (fabsf(q - n) < 0.5f - 0x1p-11f && fabsf(q) < 512.0f) return n;
  return rintf(__fdiv_rn(d, s));
}

// Elements 8q .. 8q+7 of a group of type WT, in fp32 (exact).
template <int WT>
__device__ __forceinline__ void load8(const void *group, int q, float (&v)[8]) {
  if constexpr (WT == kTypeF32) {
    const float4 *p = reinterpret_cast<const float4 *>(group) + 2 * q;
    const float4 a = __ldg(p), b = __ldg(p + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
    using E = typename std::conditional<WT == kTypeF16, ElemF16, ElemBF16>::type;
    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(group) + q);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = E::to_f32(w[i] & 0xFFFFu);
      v[2 * i + 1] = E::to_f32(w[i] >> 16);
    }
  }
}

// Store v as element o of a WT array (16-bit types rounded to nearest even)
// and return the stored value in fp32.
template <int WT>
__device__ __forceinline__ float store_value(void *p, int64_t o, float v) {
  if constexpr (WT == kTypeF32) {
    static_cast<float *>(p)[o] = v;
    return v;
  } else {
    using E = typename std::conditional<WT == kTypeF16, ElemF16, ElemBF16>::type;
    const uint16_t h = E::from_f32(v);
    static_cast<uint16_t *>(p)[o] = h;
    return E::to_f32(h);
  }
}

template <int BITS, int G, int WT>
__global__ void __launch_bounds__(kThreads)
quantize_kernel(const void *__restrict__ w, uint32_t total, uint32_t groups_per_row,
                int64_t cols, uint32_t *__restrict__ packed, void *__restrict__ scales,
                void *__restrict__ biases) {
  constexpr int ESZ = WT == kTypeF32 ? 4 : 2;
  constexpr int NW = G * BITS / 32;  // words per group
  constexpr uint32_t TOP = (1u << BITS) - 1u;
  const int64_t wpr = (cols * BITS) >> 5;
  for (uint32_t gid = blockIdx.x * kThreads + threadIdx.x; gid < total;
       gid += gridDim.x * kThreads) {
    const uint32_t r = gid / groups_per_row, j = gid - r * groups_per_row;
    const void *src = static_cast<const char *>(w) +
                      (static_cast<int64_t>(r) * cols + static_cast<int64_t>(j) * G) * ESZ;
    // Minimum and maximum as compared in the group's order (a value replaces
    // the running one only when strictly smaller / larger): the first element
    // that attains each.  fminf / fmaxf skip NaNs the same way, except a NaN
    // first element, which the ordered comparison keeps; and they may return
    // either zero when both signs occur, so a zero extremum is taken again as
    // the first zero of the group.
    float lo = 0.0f, hi = 0.0f, first = 0.0f;
#pragma unroll
    for (int q = 0; q < G / 8; ++q) {
      float v[8];
      load8<WT>(src, q, v);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (q == 0 && e == 0) {
          lo = hi = first = v[0];
        } else {
          lo = fminf(lo, v[e]);
          hi = fmaxf(hi, v[e]);
        }
      }
    }
    if (first != first) {
      lo = hi = first;
    } else if (lo == 0.0f || hi == 0.0f) {
      float z = 0.0f;
      for (int q = 0; q < G / 8; ++q) {
        float v[8];
        load8<WT>(src, q, v);
        bool found = false;
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (!found && v[e] == 0.0f) { z = v[e]; found = true; }
        if (found) break;
      }
      if (lo == 0.0f) lo = z;
      if (hi == 0.0f) hi = z;
    }
    const int64_t o = static_cast<int64_t>(r) * groups_per_row + j;
    const float s = store_value<WT>(scales, o, __fdiv_rn(__fsub_rn(hi, lo), static_cast<float>(TOP)));
    const float b = store_value<WT>(biases, o, lo);  // exact: lo is a value of w
    uint32_t words[NW];
#pragma unroll
    for (int i = 0; i < NW; ++i) words[i] = 0u;
    if (s != 0.0f) {
      const float rs = __frcp_rn(s);
#pragma unroll
      for (int q = 0; q < G / 8; ++q) {
        float v[8];
        load8<WT>(src, q, v);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float qf = fminf(fmaxf(rint_quotient(__fsub_rn(v[e], b), s, rs), 0.0f),
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
  }
}

template <int BITS, int G, int WT>
cudaError_t launch_g(const void *w, int64_t rows, int64_t cols, uint32_t *packed, void *scales,
                     void *biases, cudaStream_t stream) {
  constexpr int ESZ = WT == kTypeF32 ? 4 : 2;
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
    quantize_kernel<BITS, G, WT><<<grid, kThreads, 0, stream>>>(
        static_cast<const char *>(w) + r0 * cols * ESZ, total, static_cast<uint32_t>(gpr), cols,
        packed + r0 * wpr, static_cast<char *>(scales) + r0 * gpr * ESZ,
        static_cast<char *>(biases) + r0 * gpr * ESZ);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <int BITS, int WT>
cudaError_t launch_wt(const void *w, int64_t rows, int64_t cols, int group, uint32_t *packed,
                      void *scales, void *biases, cudaStream_t stream) {
  switch (group) {
    case 32: return launch_g<BITS, 32, WT>(w, rows, cols, packed, scales, biases, stream);
    case 64: return launch_g<BITS, 64, WT>(w, rows, cols, packed, scales, biases, stream);
    case 128: return launch_g<BITS, 128, WT>(w, rows, cols, packed, scales, biases, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int BITS>
cudaError_t launch_bits(const void *w, int w_type, int64_t rows, int64_t cols, int group,
                        uint32_t *packed, void *scales, void *biases, cudaStream_t stream) {
  switch (w_type) {
    case kTypeF32: return launch_wt<BITS, kTypeF32>(w, rows, cols, group, packed, scales, biases, stream);
    case kTypeBF16: return launch_wt<BITS, kTypeBF16>(w, rows, cols, group, packed, scales, biases, stream);
    case kTypeF16: return launch_wt<BITS, kTypeF16>(w, rows, cols, group, packed, scales, biases, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_quantize(const void *w, int w_type, int64_t rows, int64_t cols, int group,
                            int bits, uint32_t *packed, void *scales, void *biases,
                            cudaStream_t stream) {
  switch (bits) {
    case 1: return launch_bits<1>(w, w_type, rows, cols, group, packed, scales, biases, stream);
    case 2: return launch_bits<2>(w, w_type, rows, cols, group, packed, scales, biases, stream);
    case 3: return launch_bits<3>(w, w_type, rows, cols, group, packed, scales, biases, stream);
    case 4: return launch_bits<4>(w, w_type, rows, cols, group, packed, scales, biases, stream);
    case 5: return launch_bits<5>(w, w_type, rows, cols, group, packed, scales, biases, stream);
    case 6: return launch_bits<6>(w, w_type, rows, cols, group, packed, scales, biases, stream);
    case 8: return launch_bits<8>(w, w_type, rows, cols, group, packed, scales, biases, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qmm
