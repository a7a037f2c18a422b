// Device helpers shared by the kernels: bf16 bit patterns, the packed-code
// window reader and small PTX wrappers.  Format (nuvec_core quantized.rs,
// module doc): a row is a little-endian bit stream of `bits`-bit codes in
// uint32 words, code j at stream bits [j*bits, (j+1)*bits).
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace qmm {

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h) {
  return __uint_as_float(h << 16);  // exact widening
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));  // round to nearest even
}

// Two fp32 -> one bf16x2 register (lo in bits 0..15), each rounded to
// nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// ---------------------------------------------------------------- PTX ----

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// (a & b) | c in one instruction.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// bf16x2 a - b and a*b + c, each lane rounded once to nearest even.
__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bf16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------ mbarriers ----

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count));
}

// One bounded poll: while the phase is incomplete the thread may be
// suspended for at most kSuspendNs, so a few million polls take at most a
// few seconds.
constexpr uint32_t kSuspendNs = 256;
__device__ __forceinline__ bool mbar_try_wait(uint64_t *b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity), "n"(kSuspendNs)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)),
               "r"(bytes)
               : "memory");
}

// Global -> this block's shared memory, `bytes` a multiple of 16, both
// addresses 16-byte aligned; completion is counted on `bar` in bytes.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ------------------------------------------------- 16-bit element types ----
//
// The tensor-core paths dequantize to, and multiply in, one 16-bit type: bf16
// (the pages' scales) or IEEE fp16 (fp16 scales with fp16 x).  Values travel
// as bit patterns; pairs as one 32-bit register (low half first).  kMagic2 is
// a pair of a power of two P whose mantissa has room for any code: OR-ing a
// code c into each half gives P + c exactly, and subtracting P leaves c
// (P = 128 for bf16's 7 fraction bits, codes below 2^7; 1024 for fp16's 10,
// codes below 2^10, which covers 8-bit codes too).
struct ElemBF16 {
  static constexpr bool kF16 = false;
  static constexpr uint32_t kMagic2 = 0x43004300u;  // (128.0, 128.0)
  __device__ static __forceinline__ float to_f32(uint32_t h) { return bf16_bits_to_f32(h); }
  __device__ static __forceinline__ uint16_t from_f32(float f) { return f32_to_bf16_bits(f); }
  __device__ static __forceinline__ uint32_t pack2(float lo, float hi) { return pack_bf16x2(lo, hi); }
  __device__ static __forceinline__ uint32_t sub2(uint32_t a, uint32_t b) { return bf16x2_sub(a, b); }
  __device__ static __forceinline__ uint32_t fma2(uint32_t a, uint32_t b, uint32_t c) {
    return bf16x2_fma(a, b, c);
  }
};

struct ElemF16 {
  static constexpr bool kF16 = true;
  static constexpr uint32_t kMagic2 = 0x64006400u;  // (1024.0, 1024.0)
  __device__ static __forceinline__ float to_f32(uint32_t h) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
  }
  __device__ static __forceinline__ uint16_t from_f32(float f) {
    return __half_as_ushort(__float2half_rn(f));  // round to nearest even
  }
  __device__ static __forceinline__ uint32_t pack2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
  }
  __device__ static __forceinline__ uint32_t sub2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  }
  __device__ static __forceinline__ uint32_t fma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
  }
};

// ----------------------------------------------------- register dequant ----


// Code j (0 <= j < n) of a little-endian bit stream held in words v[].
template <int BITS>
__device__ __forceinline__ uint32_t code_at(const uint32_t *v, int j) {
  const int bit = j * BITS, word = bit >> 5, sh = bit & 31;
  constexpr uint32_t mask = (1u << BITS) - 1u;
  if (sh + BITS <= 32) return (v[word] >> sh) & mask;
  return __funnelshift_r(v[word], v[word + 1], sh) & mask;
}

// Codes j and j+1 (j even) of a little-endian bit stream held in words v[],
// as code j in bits [0, BITS) and code j+1 in bits [16, 16 + BITS), the rest
// zero: one (funnel) shift brings the pair's 2*BITS bits to the bottom, a
// copy shifted by 16 - BITS carries the second code into the high half, and
// one select-and-mask keeps each half's code.
template <int BITS>
__device__ __forceinline__ uint32_t pair_at(const uint32_t *v, int j) {
  const int bit = j * BITS, word = bit >> 5, sh = bit & 31;
  const uint32_t y = sh + 2 * BITS <= 32 ? v[word] >> sh : __funnelshift_r(v[word], v[word + 1], sh);
  constexpr uint32_t lo = (1u << BITS) - 1u, hi = lo << 16;
  // low half from y, high half from the shifted copy, then the two code fields
  return ((y & lo) | ((y << (16 - BITS)) & hi));
}

// Dequantize the 2*NP codes held in v[] (bit stream, LSB first) to NP
// natural pairs of E (code 2i in the low half, 2i+1 in the high half), each
// RN(s*c + b).  s2, b2 are (s, s) and (b, b) as E pairs; sf, bf the same in
// fp32 (8-bit codes in bf16 go through fp32: 255 does not fit bf16's magic).
template <int BITS, int NP, typename E = ElemBF16>
__device__ __forceinline__ void dequant_pairs(const uint32_t *v, uint32_t s2, uint32_t b2,
                                              float sf, float bf, uint32_t *out) {
  if constexpr (BITS == 4) {
#pragma unroll
    for (int q = 0; q < NP / 4; ++q) {
      const uint32_t w = v[q], w4 = w >> 4;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        // byte i of w holds codes 8q+2i (low nibble) and 8q+2i+1 (high nibble)
        const uint32_t t = prmt(w, w4, 0x0400u | (i << 8) | i);
        const uint32_t c = E::sub2(and_or(t, 0x000F000Fu, E::kMagic2), E::kMagic2);
        out[4 * q + i] = E::fma2(c, s2, b2);
      }
    }
  } else if constexpr (BITS == 8 && E::kF16) {
#pragma unroll
    for (int q = 0; q < NP / 2; ++q) {
      const uint32_t w = v[q];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        // bytes 2i, 2i+1 into the low bytes of the halves, over the magic
        const uint32_t t = prmt(w, 0u, 0x4040u | (2 * i) | ((2 * i + 1) << 8)) | E::kMagic2;
        out[2 * q + i] = E::fma2(E::sub2(t, E::kMagic2), s2, b2);
      }
    }
  } else if constexpr (BITS == 8) {
#pragma unroll
    for (int q = 0; q < NP / 2; ++q) {
      const uint32_t w = v[q];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        // fp32 2^23 + byte, exact; minus 2^23 gives the code exactly.
        const float c0 = __uint_as_float(prmt(w, 0x4B000000u, 0x7650u | (2 * i))) - 8388608.0f;
        const float c1 = __uint_as_float(prmt(w, 0x4B000000u, 0x7650u | (2 * i + 1))) - 8388608.0f;
        out[2 * q + i] = E::pack2(__fmaf_rn(sf, c0, bf), __fmaf_rn(sf, c1, bf));
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      const uint32_t p = pair_at<BITS>(v, 2 * i) | E::kMagic2;
      out[i] = E::fma2(E::sub2(p, E::kMagic2), s2, b2);
    }
  }
}

// Natural code pairs of a run of 32 codes held in v[] (bits words), pair p =
// codes (2p, 2p+1), each half RN(scale * code + bias), in two forms.
//
// Fast form: a bf16 bit pattern P <= 0xFF is worth exactly P * 2^-133
// (subnormal below 0x80; exponent field 1 above, whose implicit one is bit 7
// of P).  A code c at bit o (o + bits <= 8) of an otherwise clear half reads
// as c * 2^(o-133), so one bf16x2 FMA with the multiplier s * 2^(133-o) and
// addend b gives RN(s*c + b): the product is exact and the FMA rounds once.
// The multiplier is s with 133 - o added to its exponent field, exact while
// that stays below 255: taken when the scale is a normal number below 2^-5.
// Exact form, for any scale: the code OR-ed into the mantissa of 128.0,
// minus 128 exactly, then the FMA; 8-bit codes through fp32.
// Multiplier slots of the fast form: slot k serves the pairs whose codes sit
// at bit offsets (fast_lo(k), fast_hi(k)) of their halves.
template <int BITS>
__host__ __device__ constexpr int fast_slots() {
  return BITS == 1 ? 4 : BITS == 2 ? 2 : 1;
}
template <int BITS>
__host__ __device__ constexpr int fast_lo(int k) {
  return BITS == 1 ? 2 * k : BITS == 2 ? 4 * k : 0;
}
template <int BITS>
__host__ __device__ constexpr int fast_hi(int k) {
  return BITS == 1 ? 2 * k + 1 : BITS == 2 ? 4 * k + 2 : BITS == 4 ? 4 : 0;
}

// Whether the bf16 scale h is a normal number of magnitude below 2^-5.
__device__ __forceinline__ bool fast_scale(uint32_t h) {
  return ((h >> 7) & 0xFFu) - 1u < 121u;
}

// (s * 2^(133 - lo), s * 2^(133 - hi)) for every slot, from the scale bits h.
template <int BITS>
__device__ __forceinline__ void fast_muls(uint32_t h, uint32_t (&m)[fast_slots<BITS>()]) {
#pragma unroll
  for (int k = 0; k < fast_slots<BITS>(); ++k)
    m[k] = h * 0x00010001u + ((static_cast<uint32_t>(133 - fast_lo<BITS>(k)) << 7) |
                              (static_cast<uint32_t>(133 - fast_hi<BITS>(k)) << 23));
}

template <int BITS>
__device__ __forceinline__ uint32_t pair_fast(const uint32_t *v, int p,
                                              const uint32_t (&m)[fast_slots<BITS>()],
                                              uint32_t b2) {
  if constexpr (BITS == 8) {
    // bytes 2i, 2i+1 of word p/2 into the low bytes of the halves
    const uint32_t i = p & 1;
    return bf16x2_fma(prmt(v[p >> 1], 0u, 0x4040u | (2 * i) | ((2 * i + 1) << 8)), m[0], b2);
  } else if constexpr (BITS == 4) {
    // byte j of word p/4 holds the pair as its two nibbles
    const uint32_t j = p & 3;
    const uint32_t t = prmt(v[p >> 2], 0u, 0x4040u | j | (j << 8)) & 0x00F0000Fu;
    return bf16x2_fma(t, m[0], b2);
  } else if constexpr (BITS == 2) {
    // byte j of word p/8 holds pairs 2j, 2j+1 of the word at bits 0..3, 4..7
    const uint32_t j = (p >> 1) & 3, k = p & 1;
    const uint32_t t = prmt(v[p >> 3], 0u, 0x4040u | j | (j << 8)) & (0x000C0003u << (4 * k));
    return bf16x2_fma(t, m[k], b2);
  } else if constexpr (BITS == 1) {
    // byte j of word p/16 holds pairs 4j .. 4j+3 of the word at bits 2k, 2k+1
    const uint32_t j = (p >> 2) & 3, k = p & 3;
    const uint32_t t = prmt(v[p >> 4], 0u, 0x4040u | j | (j << 8)) & (0x00020001u << (2 * k));
    return bf16x2_fma(t, m[k], b2);
  } else {
    const uint32_t t = pair_at<BITS>(v, 2 * p);
    return bf16x2_fma(t, m[0], b2);
  }
}

template <int BITS, typename E = ElemBF16>
__device__ __forceinline__ uint32_t pair_exact(const uint32_t *v, int p, uint32_t s2, uint32_t b2,
                                               float sf, float bf) {
  if constexpr (BITS == 8 && E::kF16) {
    // bytes 2i, 2i+1 of word p/2 into the low bytes of the halves
    const uint32_t i = p & 1;
    const uint32_t q = prmt(v[p >> 1], 0u, 0x4040u | (2 * i) | ((2 * i + 1) << 8)) | E::kMagic2;
    return E::fma2(E::sub2(q, E::kMagic2), s2, b2);
  } else if constexpr (BITS == 8) {
    // fp32 2^23 + byte, exact; minus 2^23 gives the code exactly.
    const uint32_t w = v[p >> 1], i = p & 1;
    const float c0 = __uint_as_float(prmt(w, 0x4B000000u, 0x7650u | (2 * i))) - 8388608.0f;
    const float c1 = __uint_as_float(prmt(w, 0x4B000000u, 0x7650u | (2 * i + 1))) - 8388608.0f;
    return E::pack2(__fmaf_rn(sf, c0, bf), __fmaf_rn(sf, c1, bf));
  } else if constexpr (BITS == 4) {
    // byte j of w and of w >> 4 hold codes 2j and 2j+1 in their low nibbles
    const uint32_t w = v[p >> 2], j = p & 3;
    const uint32_t q = and_or(prmt(w, w >> 4, 0x0400u | j | (j << 8)), 0x000F000Fu, E::kMagic2);
    return E::fma2(E::sub2(q, E::kMagic2), s2, b2);
  } else {
    const uint32_t q = pair_at<BITS>(v, 2 * p) | E::kMagic2;
    return E::fma2(E::sub2(q, E::kMagic2), s2, b2);
  }
}

// Load n words from p (4-byte aligned, and 8/16-byte aligned when the width
// allows it) as wide as the alignment lets us.
template <int BITS>
__device__ __forceinline__ void load_words(const uint32_t *__restrict__ p, uint32_t *v) {
  if constexpr (BITS % 4 == 0) {
#pragma unroll
    for (int i = 0; i < BITS / 4; ++i) {
      const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p) + i);
      v[4 * i] = u.x; v[4 * i + 1] = u.y; v[4 * i + 2] = u.z; v[4 * i + 3] = u.w;
    }
  } else if constexpr (BITS % 2 == 0) {
#pragma unroll
    for (int i = 0; i < BITS / 2; ++i) {
      const uint2 u = __ldg(reinterpret_cast<const uint2 *>(p) + i);
      v[2 * i] = u.x; v[2 * i + 1] = u.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < BITS; ++i) v[i] = __ldg(p + i);
  }
}

// (h, h): a 16-bit pattern in both halves of a pair.
__device__ __forceinline__ uint32_t bcast2(uint16_t h) {
  return static_cast<uint32_t>(h) * 0x00010001u;
}

}  // namespace qmm
