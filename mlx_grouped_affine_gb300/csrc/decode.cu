// The decode kernel of quantized_matmul for a transposed W with K a multiple
// of 128 and M <= 16 (nuvec_core quantized.rs, `quantized_matmul`;
// spark_runtime weights/mlx_int8.rs, `gemv`), in bf16 and fp16.  It lives in
// a translation unit of its own so that it compiles beside the other decode
// kernels (gemv_impl.cuh), whose helpers it shares.
#include "gemv_impl.cuh"

#include <algorithm>

namespace qmm {
namespace {

// ------------------------------------------------------------------------
// The decode kernel: transpose = true, K a multiple of 128, M <= 16.
//
// Where the time goes at M <= 16 is instruction issue after the dependency
// wait, and on the integer (ALU) pipe in particular: every weight needs its
// code moved into place before the bf16x2 FMA that dequantizes it.  This
// kernel is laid out to keep that work small and evenly spread, and to keep
// the launch chain busy:
//
//  * Word-local pairs.  For widths whose codes never cross a word (1, 2, 4
//    and 8 bits), pair j of a word of n = 32/bits codes is (c_j, c_{j+n/2}):
//    code j sits in the low half-word and code j + n/2 sixteen bits higher,
//    so one mask (and one byte permute per half of the word) lifts both into
//    a bf16x2 register at the same bit offset o.  At 4 bits a word costs one
//    permute and four masks for its four pairs (four permutes and four masks
//    on natural pairs).  The contraction index is permuted to match: x is
//    staged in shared memory with each word's values in the same pair order,
//    so the MMA's B operand is read as it lies.  Widths whose codes cross
//    words (3, 5, 6 bits) keep natural pairs and natural x.
//  * Dequantization is the fast form (the code at bit o of a half reads as
//    c * 2^(o-133); one bf16x2 FMA with s * 2^(133-o) and b rounds s*c + b
//    once) when every scale of a warp's chunk is a normal number below 2^-5,
//    else the exact form (code OR-ed into the mantissa of a power of two,
//    subtracted, then the FMA).  fp16 takes the exact form.
//  * One block per SM and kernel: the grid has about as many blocks as the
//    GPU has SMs, each taking one or two 16-row tiles, and a block's shared
//    memory is sized so that at most two fit an SM.  With programmatic
//    dependent launch the next kernel's blocks then land one per SM beside
//    the running ones (never piled several to an SM), stream their weight
//    chunks (one TMA box each, issued at kernel start) and stage their scales
//    and biases in shared memory before griddepcontrol.wait; after the wait
//    the block stages x once, in pair order, and its 16 warps run their
//    chunks.
//  * K is split across the warps of a tile (contiguous chunk ranges) and,
//    when the tiles are fewer than the SMs or K is long, across the blocks of
//    a cluster; partials are reduced through shared and distributed shared
//    memory.  No global scratch.

constexpr int kDecWarps = 16;
constexpr int kDecMaxTiles = 2;     // 16-row tiles per block
constexpr int kDecMaxChunks = 64;   // 128-code chunks per tile and block: 8192 codes

// Whether a width's codes are paired inside a word (see above).
template <int BITS>
__host__ __device__ constexpr bool word_pairs() {
  return BITS == 1 || BITS == 2 || BITS == 4 || BITS == 8;
}

// Fast-form multiplier slots: slot k serves the pairs at bit offset
// dec_off(k) of their halves.
template <int BITS>
__host__ __device__ constexpr int dec_slots() {
  return BITS == 8 ? 1 : BITS == 4 ? 2 : word_pairs<BITS>() ? 4 : 1;
}
template <int BITS>
__host__ __device__ constexpr int dec_off(int k) {
  return BITS == 4 ? 4 * k : BITS == 2 ? 2 * k : BITS == 1 ? k : 0;
}

// (s * 2^(133 - dec_off(k)), same) for each slot, from the bf16 scale bits h
// (a normal number below 2^-5: the exponent field stays below 255).
template <int BITS>
__device__ __forceinline__ void dec_muls(uint32_t h, uint32_t (&m)[dec_slots<BITS>()]) {
#pragma unroll
  for (int k = 0; k < dec_slots<BITS>(); ++k)
    m[k] = h * 0x00010001u + static_cast<uint32_t>(133 - dec_off<BITS>(k)) * 0x00800080u;
}

// Pairs are made in sub-blocks of at most 8 (a 1-bit word's 16 pairs in two)
// to bound the registers they occupy.
template <int BITS>
__host__ __device__ constexpr int dec_subs() { return BITS == 1 ? 2 : 1; }

// Sub-block SUB of the n/2 word-local pairs of word w, fast form: out[j] =
// (RN(s c_p + b), RN(s c_{p+n/2} + b)) for pair p = SUB * n / (2 * subs) + j.
template <int BITS, int SUB = 0>
__device__ __forceinline__ void word_pairs_fast(uint32_t w, const uint32_t (&m)[dec_slots<BITS>()],
                                                uint32_t b2, uint32_t *out) {
  if constexpr (BITS == 8) {
    out[0] = bf16x2_fma(prmt(w, 0u, 0x4240u), m[0], b2);  // bytes 0, 2: (c0, c2)
    out[1] = bf16x2_fma(prmt(w, 0u, 0x4341u), m[0], b2);  // bytes 1, 3: (c1, c3)
  } else if constexpr (BITS == 4) {
    const uint32_t u = prmt(w, 0u, 0x4341u);              // bytes 1, 3 to 0, 2
    out[0] = bf16x2_fma(w & 0x000F000Fu, m[0], b2);       // (c0, c4) at bit 0
    out[1] = bf16x2_fma(w & 0x00F000F0u, m[1], b2);       // (c1, c5) at bit 4
    out[2] = bf16x2_fma(u & 0x000F000Fu, m[0], b2);       // (c2, c6)
    out[3] = bf16x2_fma(u & 0x00F000F0u, m[1], b2);       // (c3, c7)
  } else if constexpr (BITS == 2) {
    const uint32_t u = prmt(w, 0u, 0x4341u);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      out[j] = bf16x2_fma(w & (0x00030003u << (2 * j)), m[j], b2);      // (c_j, c_{8+j})
      out[4 + j] = bf16x2_fma(u & (0x00030003u << (2 * j)), m[j], b2);  // (c_{4+j}, c_{12+j})
    }
  } else if constexpr (BITS == 1) {
    // bytes SUB, SUB + 2 into 0, 2: codes 8 SUB .. 8 SUB + 7 and 16 + the same
    const uint32_t u = prmt(w, 0u, SUB ? 0x4341u : 0x4240u);
    const uint32_t v = u >> 4;  // the masks drop what crosses halves
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      out[j] = bf16x2_fma(u & (0x00010001u << j), m[j], b2);      // (c_{8S+j}, c_{16+8S+j})
      out[4 + j] = bf16x2_fma(v & (0x00010001u << j), m[j], b2);  // (c_{8S+4+j}, c_{20+8S+j})
    }
  }
}

// The same pairs in the exact form (any scale).
template <int BITS, typename E, int SUB = 0>
__device__ __forceinline__ void word_pairs_exact(uint32_t w, uint32_t s2, uint32_t b2, float sf,
                                                 float bf, uint32_t *out) {
  if constexpr (BITS == 8 && !E::kF16) {
    // fp32 2^23 + byte, exact; minus 2^23 gives the code exactly.
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float c0 = __uint_as_float(prmt(w, 0x4B000000u, 0x7650u | j)) - 8388608.0f;
      const float c1 = __uint_as_float(prmt(w, 0x4B000000u, 0x7650u | (j + 2))) - 8388608.0f;
      out[j] = E::pack2(__fmaf_rn(sf, c0, bf), __fmaf_rn(sf, c1, bf));
    }
  } else if constexpr (BITS == 8) {
    out[0] = E::fma2(E::sub2(prmt(w, 0u, 0x4240u) | E::kMagic2, E::kMagic2), s2, b2);
    out[1] = E::fma2(E::sub2(prmt(w, 0u, 0x4341u) | E::kMagic2, E::kMagic2), s2, b2);
  } else {
    constexpr int n = 32 / BITS, per = n / 2 / dec_subs<BITS>();
    constexpr uint32_t mask = ((1u << BITS) - 1u) * 0x00010001u;
#pragma unroll
    for (int j = 0; j < per; ++j) {
      // code p at bit BITS*p of the low half, code p + n/2 at the same bit of the high half
      const uint32_t q = and_or(w >> (BITS * (SUB * per + j)), mask, E::kMagic2);
      out[j] = E::fma2(E::sub2(q, E::kMagic2), s2, b2);
    }
  }
}

// x[8t .. 8t+n) of one word in pair order, from natural bf16x2 registers
// r[i] = (x_2i, x_2i+1): o[2i] = (x_i... ) -- pair j = (x_j, x_{j+n/2}).
template <int BITS>
__device__ __forceinline__ void x_to_pairs(const uint32_t *r, uint32_t *o) {
  constexpr int n = 32 / BITS, q = n / 4;  // n/2 registers per word
#pragma unroll
  for (int i = 0; i < q; ++i) {
    o[2 * i] = prmt(r[i], r[i + q], 0x5410u);      // (x_2i, x_{2i+n/2})
    o[2 * i + 1] = prmt(r[i], r[i + q], 0x7632u);  // (x_2i+1, x_{2i+1+n/2})
  }
}

struct DecLayout {
  int kr;         // codes per block along K (multiple of 128)
  int tiles;      // 16-row tiles of W
  int nblk;       // blocks along N: block b takes tiles [tiles*b/nblk, tiles*(b+1)/nblk)
  int box_bytes;  // one chunk box (16 rows)
  int x_off, xpitch;      // staged x rows: M rows, xpitch bytes apart
  int sb_off, gblk, sbp;  // staged scales, then biases: [32][sbp] each, gblk used
  int red_off, bar_off;
  uint32_t spin_limit;
};

// At most two blocks an SM: 512 threads of at most 64 registers, and the
// launcher pads shared memory so that a third never fits.
template <typename E, int BITS, int NT, bool OUT_BF16>
__global__ void __launch_bounds__(32 * kDecWarps, 2)
gemv_decode_kernel(const __grid_constant__ CUtensorMap wmap, GemvArgs a, DecLayout L,
                   unsigned *err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar_off);
  float *red = reinterpret_cast<float *>(smem + L.red_off);
  uint16_t *ss = reinterpret_cast<uint16_t *>(smem + L.sb_off);
  uint16_t *bs = ss + 16 * kDecMaxTiles * L.sbp;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  uint32_t crank = 0, csize = 1;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(crank));
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(csize));
  const int tb0 = static_cast<int>(static_cast<int64_t>(L.tiles) * blockIdx.x / L.nblk);
  const int ntile = static_cast<int>(static_cast<int64_t>(L.tiles) * (blockIdx.x + 1) / L.nblk) - tb0;
  const int r0 = tb0 * 16;  // first weight row of the block
  const int k0 = static_cast<int>(crank) * L.kr;
  const int ncodes = max(0, min(a.K, k0 + L.kr) - k0);
  const int nchunks = ncodes >> 7;
  const int nboxes = ntile * nchunks;

  if (threadIdx.x == 0) {
    for (int i = 0; i < nboxes; ++i) mbar_init(&bars[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (warp == 0) {
    // Box i = tile i / nchunks, chunk i % nchunks.
    for (int i = lane; i < nboxes; i += 32) {
      const int j = i / nchunks, c = i - j * nchunks;
      mbar_expect_tx(&bars[i], L.box_bytes);
      const int xw = ((k0 + (c << 7)) * BITS) >> 5;  // word coordinate
      asm volatile(
          "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
          " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem + i * L.box_bytes)),
          "l"(&wmap), "r"(xw), "r"(r0 + 16 * j), "r"(smem_u32(&bars[i]))
          : "memory");
    }
  }
  griddep_launch_dependents();

  // Scales and biases of the block's rows and K range into shared memory
  // (weights: read before the dependency wait).  Rows past N repeat row N-1.
  // Every load of a thread is issued before its first store, so the staging
  // costs one memory latency.
  {
    const int groups = a.K >> a.group_shift, gb0 = k0 >> a.group_shift;
    const int gn = min(L.gblk, groups - gb0), nrows = 16 * ntile;
    if (groups % 8 == 0 && gb0 % 8 == 0 && L.gblk % 8 == 0 && gn == L.gblk) {
      const int vpr = L.gblk / 8, total = 2 * nrows * vpr;  // 16-byte vectors
      for (int i0 = 0; i0 < total; i0 += 2 * blockDim.x) {
        uint4 v[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int i = i0 + j * blockDim.x + threadIdx.x;
          if (i < total) {
            const int arr = i / (nrows * vpr), r = (i / vpr) % nrows, q = i % vpr;
            const int64_t row = min(r0 + r, a.N - 1);
            const uint16_t *src = (arr ? a.biases : a.scales) + row * groups + gb0 + 8 * q;
            v[j] = __ldg(reinterpret_cast<const uint4 *>(src));
          }
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int i = i0 + j * blockDim.x + threadIdx.x;
          if (i < total) {
            const int arr = i / (nrows * vpr), r = (i / vpr) % nrows, q = i % vpr;
            *reinterpret_cast<uint4 *>((arr ? bs : ss) + r * L.sbp + 8 * q) = v[j];
          }
        }
      }
    } else {
      const int total = nrows * L.gblk;
      for (int i0 = 0; i0 < total; i0 += 4 * blockDim.x) {
        uint16_t sv[4], bv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int i = i0 + j * blockDim.x + threadIdx.x;
          const int r = i / L.gblk, q = i - r * L.gblk;
          sv[j] = bv[j] = 0;
          if (i < total && q < gn) {
            const int64_t row = min(r0 + r, a.N - 1);
            sv[j] = __ldg(a.scales + row * groups + gb0 + q);
            bv[j] = __ldg(a.biases + row * groups + gb0 + q);
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int i = i0 + j * blockDim.x + threadIdx.x;
          const int r = i / L.gblk, q = i - r * L.gblk;
          if (i < total) {
            ss[r * L.sbp + q] = sv[j];
            bs[r * L.sbp + q] = bv[j];
          }
        }
      }
    }
  }

  // This warp's tile and chunks: with two tiles, warps 0-7 take the first
  // and 8-15 the second, 8 K ranges each; with one, 16 K ranges.
  const int wpt = kDecWarps / ntile;  // warps per tile
  const int wt = warp / wpt, wr = warp - wt * wpt;
  const int cpw = (nchunks + wpt - 1) / wpt;
  const int c_begin = min(nchunks, wr * cpw), c_end = min(nchunks, c_begin + cpw);

  // x may be written by the previous kernel in the stream.
  griddep_wait();

  // Stage the block's x columns [k0, k0 + 128*nchunks) of every row, with
  // each word's values in pair order: units of U values (one word, or two
  // 4-value words at 8 bits) are loaded, permuted in registers and stored;
  // each thread issues up to four 16-byte loads before its first store.
  {
    constexpr int U = word_pairs<BITS>() ? (32 / BITS > 8 ? 32 / BITS : 8) : 8;
    constexpr int LPU = U / 8, UPB = 4 / LPU;  // loads per unit, units per batch
    const int per_row = (nchunks << 7) / U, total = a.M * per_row;
    for (int i0 = 0; i0 < total; i0 += blockDim.x * UPB) {
      uint32_t r[UPB][U / 2];
#pragma unroll
      for (int b = 0; b < UPB; ++b) {
        const int i = i0 + blockDim.x * b + threadIdx.x;
        if (i < total) {
          const int m = i / per_row, u = i - m * per_row;
          const uint4 *src = reinterpret_cast<const uint4 *>(a.x + static_cast<int64_t>(m) * a.K + k0 + u * U);
#pragma unroll
          for (int l = 0; l < LPU; ++l) {
            const uint4 v = __ldg(src + l);
            r[b][4 * l] = v.x; r[b][4 * l + 1] = v.y; r[b][4 * l + 2] = v.z; r[b][4 * l + 3] = v.w;
          }
        }
      }
#pragma unroll
      for (int b = 0; b < UPB; ++b) {
        const int i = i0 + blockDim.x * b + threadIdx.x;
        if (i < total) {
          const int m = i / per_row, u = i - m * per_row;
          uint32_t o[U / 2];
          if constexpr (word_pairs<BITS>()) {
            constexpr int n = 32 / BITS;
#pragma unroll
            for (int wd = 0; wd < U / n; ++wd) x_to_pairs<BITS>(r[b] + wd * (n / 2), o + wd * (n / 2));
          } else {
#pragma unroll
            for (int k = 0; k < U / 2; ++k) o[k] = r[b][k];
          }
          uint4 *dst = reinterpret_cast<uint4 *>(smem + L.x_off + m * L.xpitch + u * U * 2);
#pragma unroll
          for (int l = 0; l < LPU; ++l) dst[l] = make_uint4(o[4 * l], o[4 * l + 1], o[4 * l + 2], o[4 * l + 3]);
        }
      }
    }
  }
  __syncthreads();  // x and the scales and biases are in place

  float acc[2][NT][4];
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[h][nt][i] = 0.0f;

  // x rows this lane reads as its B column (rows past M repeat row 0; their
  // outputs are never stored).
  int xrow[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) xrow[nt] = (g + 8 * nt < a.M) ? g + 8 * nt : 0;

  bool ok = true;
  constexpr int kRowBytes = 16 * BITS;
  const uint16_t *ssw = ss + wt * 16 * L.sbp, *bsw = bs + wt * 16 * L.sbp;
  for (int c = c_begin; c < c_end; ++c) {
    // The lane's x pairs of this chunk: values [32t, 32t + 32) of the chunk's
    // 128, read per word (or per MMA) as they are used.
    const uint8_t *xc[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) xc[nt] = smem + L.x_off + xrow[nt] * L.xpitch + ((c << 7) + 32 * t) * 2;
    const int gi = ((c << 7) + 32 * t) >> a.group_shift;
    const uint32_t hs0 = ssw[g * L.sbp + gi], hb0 = bsw[g * L.sbp + gi];
    const uint32_t hs1 = ssw[(g + 8) * L.sbp + gi], hb1 = bsw[(g + 8) * L.sbp + gi];
    const int bi = wt * nchunks + c;
    uint32_t spins = 0;
    while (!mbar_try_wait(&bars[bi], 0)) {
      if (++spins >= L.spin_limit) {
        if (lane == 0) atomicOr(err, kErrTimeoutBit);
        ok = false;
        break;
      }
    }
    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
    const uint8_t *box = smem + bi * L.box_bytes;
    uint32_t v0[BITS], v1[BITS];
    if constexpr (BITS == 8) {
      // 128-byte swizzle: the lane's 32 bytes are 16-byte units 2t, 2t+1.
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint4 u0 = *reinterpret_cast<const uint4 *>(box + g * 128 + (((2 * t + i) ^ g) << 4));
        const uint4 u1 = *reinterpret_cast<const uint4 *>(box + (g + 8) * 128 + (((2 * t + i) ^ g) << 4));
        v0[4 * i] = u0.x; v0[4 * i + 1] = u0.y; v0[4 * i + 2] = u0.z; v0[4 * i + 3] = u0.w;
        v1[4 * i] = u1.x; v1[4 * i + 1] = u1.y; v1[4 * i + 2] = u1.z; v1[4 * i + 3] = u1.w;
      }
    } else {
      lds_words<BITS>(box + g * kRowBytes + t * 4 * BITS, v0);
      lds_words<BITS>(box + (g + 8) * kRowBytes + t * 4 * BITS, v1);
    }
    const uint32_t b0 = bcast2(static_cast<uint16_t>(hb0)), b1 = bcast2(static_cast<uint16_t>(hb1));
    bool fast = false;
    if constexpr (!E::kF16) fast = __all_sync(0xffffffffu, fast_scale(hs0) && fast_scale(hs1));
    if constexpr (word_pairs<BITS>()) {
      constexpr int n = 32 / BITS, np = n / 2, per = np / dec_subs<BITS>();  // pairs per sub-block
      // MMAs over sub-block S of word q: pairs q*np + S*per .. + per, x read
      // as per/2 pairs of registers (per * 4 bytes).
      auto mmas = [&](const uint32_t *p0, const uint32_t *p1, int q, int S) {
        const int r0m = q * (np / 2) + S * (per / 2);  // first MMA of the sub-block
        uint32_t xr[NT][per];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint8_t *xp = xc[nt] + (q * np + S * per) * 4;
          if constexpr (per >= 4) {
#pragma unroll
            for (int i = 0; i < per / 4; ++i) {
              const uint4 u = reinterpret_cast<const uint4 *>(xp)[i];
              xr[nt][4 * i] = u.x; xr[nt][4 * i + 1] = u.y; xr[nt][4 * i + 2] = u.z; xr[nt][4 * i + 3] = u.w;
            }
          } else {
            const uint2 u = *reinterpret_cast<const uint2 *>(xp);
            xr[nt][0] = u.x; xr[nt][1] = u.y;
          }
        }
#pragma unroll
        for (int i = 0; i < per / 2; ++i) {
          const int r = r0m + i;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mma_16816<E>(acc[r & 1][nt], p0[2 * i], p1[2 * i], p0[2 * i + 1], p1[2 * i + 1],
                         xr[nt][2 * i], xr[nt][2 * i + 1]);
        }
      };
      if (fast) {
        uint32_t m0[dec_slots<BITS>()], m1[dec_slots<BITS>()];
        dec_muls<BITS>(hs0, m0);
        dec_muls<BITS>(hs1, m1);
#pragma unroll
        for (int q = 0; q < BITS; ++q) {
          {
            uint32_t p0[per], p1[per];
            word_pairs_fast<BITS, 0>(v0[q], m0, b0, p0);
            word_pairs_fast<BITS, 0>(v1[q], m1, b1, p1);
            mmas(p0, p1, q, 0);
          }
          if constexpr (dec_subs<BITS>() > 1) {
            uint32_t p0[per], p1[per];
            word_pairs_fast<BITS, 1>(v0[q], m0, b0, p0);
            word_pairs_fast<BITS, 1>(v1[q], m1, b1, p1);
            mmas(p0, p1, q, 1);
          }
        }
      } else {
        const uint32_t s0 = bcast2(static_cast<uint16_t>(hs0)), s1 = bcast2(static_cast<uint16_t>(hs1));
        const float fs0 = E::to_f32(hs0), fb0 = E::to_f32(hb0);
        const float fs1 = E::to_f32(hs1), fb1 = E::to_f32(hb1);
#pragma unroll
        for (int q = 0; q < BITS; ++q) {
          {
            uint32_t p0[per], p1[per];
            word_pairs_exact<BITS, E, 0>(v0[q], s0, b0, fs0, fb0, p0);
            word_pairs_exact<BITS, E, 0>(v1[q], s1, b1, fs1, fb1, p1);
            mmas(p0, p1, q, 0);
          }
          if constexpr (dec_subs<BITS>() > 1) {
            uint32_t p0[per], p1[per];
            word_pairs_exact<BITS, E, 1>(v0[q], s0, b0, fs0, fb0, p0);
            word_pairs_exact<BITS, E, 1>(v1[q], s1, b1, fs1, fb1, p1);
            mmas(p0, p1, q, 1);
          }
        }
      }
    } else {
      // 3, 5, 6 bits: natural pairs (2p, 2p+1) of the lane's 32 codes; MMA r
      // contracts codes 4r .. 4r+3, whose x is 8 bytes.
      auto xpair = [&](int nt, int r, uint32_t &lo, uint32_t &hi) {
        const uint2 u = *reinterpret_cast<const uint2 *>(xc[nt] + r * 8);
        lo = u.x;
        hi = u.y;
      };
      if (fast) {
        uint32_t m0[fast_slots<BITS>()], m1[fast_slots<BITS>()];
        fast_muls<BITS>(hs0, m0);
        fast_muls<BITS>(hs1, m1);
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const uint32_t a0 = pair_fast<BITS>(v0, 2 * r, m0, b0), a2 = pair_fast<BITS>(v0, 2 * r + 1, m0, b0);
          const uint32_t a1 = pair_fast<BITS>(v1, 2 * r, m1, b1), a3 = pair_fast<BITS>(v1, 2 * r + 1, m1, b1);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            uint32_t xlo, xhi;
            xpair(nt, r, xlo, xhi);
            mma_16816<E>(acc[r & 1][nt], a0, a1, a2, a3, xlo, xhi);
          }
        }
      } else {
        const uint32_t s0 = bcast2(static_cast<uint16_t>(hs0)), s1 = bcast2(static_cast<uint16_t>(hs1));
        const float fs0 = E::to_f32(hs0), fb0 = E::to_f32(hb0);
        const float fs1 = E::to_f32(hs1), fb1 = E::to_f32(hb1);
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const uint32_t a0 = pair_exact<BITS, E>(v0, 2 * r, s0, b0, fs0, fb0);
          const uint32_t a2 = pair_exact<BITS, E>(v0, 2 * r + 1, s0, b0, fs0, fb0);
          const uint32_t a1 = pair_exact<BITS, E>(v1, 2 * r, s1, b1, fs1, fb1);
          const uint32_t a3 = pair_exact<BITS, E>(v1, 2 * r + 1, s1, b1, fs1, fb1);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            uint32_t xlo, xhi;
            xpair(nt, r, xlo, xhi);
            mma_16816<E>(acc[r & 1][nt], a0, a1, a2, a3, xlo, xhi);
          }
        }
      }
    }
  }

  float flat[NT * 4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) flat[nt * 4 + i] = acc[0][nt][i] + acc[1][nt][i];
  // The warps of a tile hold partials of the same outputs: sum them through
  // shared memory (the tile's first warp), then across the cluster's K split
  // through distributed shared memory (the rank-0 block), and store.
  constexpr int ACC = NT * 4;
#pragma unroll
  for (int i = 0; i < ACC; ++i) red[(warp * ACC + i) * 32 + lane] = flat[i];
  __syncthreads();
  const bool lead = wr == 0;
  float sum[ACC];
#pragma unroll
  for (int i = 0; i < ACC; ++i) sum[i] = 0.0f;
  if (lead) {
    for (int w = warp; w < warp + wpt; ++w)
#pragma unroll
      for (int i = 0; i < ACC; ++i) sum[i] += red[(w * ACC + i) * 32 + lane];
  }
  if (csize > 1) {
    __syncthreads();  // every read of red is done
    if (lead) {
#pragma unroll
      for (int i = 0; i < ACC; ++i) red[(wt * ACC + i) * 32 + lane] = sum[i];
    }
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (crank == 0 && lead) {
      const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(red));
      for (uint32_t r = 1; r < csize; ++r) {
        uint32_t remote;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(base), "r"(r));
#pragma unroll
        for (int i = 0; i < ACC; ++i) {
          float v;
          asm volatile("ld.shared::cluster.f32 %0, [%1];"
                       : "=f"(v) : "r"(remote + static_cast<uint32_t>(((wt * ACC + i) * 32 + lane) * 4)));
          sum[i] += v;
        }
      }
    }
    // Peers keep their shared memory alive until the leader has read it.
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  }
  if (lead && crank == 0) {
    const int n0 = r0 + 16 * wt;
#pragma unroll
    for (int i = 0; i < ACC; ++i) {
      const int nt = i >> 2, e = i & 3;
      const int n = n0 + g + 8 * (e >> 1), m = 8 * nt + 2 * t + (e & 1);
      if (m < a.M && n < a.N) {
        const int64_t o = static_cast<int64_t>(m) * a.N + n;
        if (OUT_BF16) static_cast<uint16_t *>(a.y)[o] = E::from_f32(sum[i]);
        else static_cast<float *>(a.y)[o] = sum[i];
      }
    }
  }
  if (!ok) {
    // A wait ran out: before the block exits, wait (bounded) for this warp's
    // copies still in flight into its shared memory.
    for (int c = c_begin; c < c_end; ++c)
      for (uint32_t q = 0; q < kDefaultWaitLimit; ++q)
        if (mbar_try_wait(&bars[wt * nchunks + c], 0)) break;
  }
}

// The decode launch: grid (blocks of one or two 16-row tiles, K split), 512
// threads, cluster over the K split.  cudaErrorNotSupported when the layout
// does not fit.
template <typename E, int BITS, int NT, bool OUT_BF16>
cudaError_t launch_decode(const GemvArgs &a, bool pdl, cudaStream_t stream) {
  const int sms = sm_count();
  const int tiles = (a.N + 15) / 16;
  // As many blocks as SMs (one or two tiles each); more when two tiles a
  // block cannot cover the weight.
  const int nblk = max((tiles + kDecMaxTiles - 1) / kDecMaxTiles, min(tiles, sms));
  const int box_bytes = 16 * 16 * BITS;
  const int G = 1 << a.group_shift;
  auto kr_of = [&](int c) { return ((a.K / c + 127) / 128) * 128; };
  auto layout_of = [&](int c) {
    DecLayout L{};
    L.kr = kr_of(c);
    L.tiles = tiles;
    L.nblk = nblk;
    L.box_bytes = box_bytes;
    const int nch = L.kr / 128;
    L.x_off = kDecMaxTiles * nch * box_bytes;
    L.xpitch = a.M > 1 ? L.kr * 2 + 16 : L.kr * 2;
    L.sb_off = L.x_off + a.M * L.xpitch;
    L.gblk = (L.kr + G - 1) / G;
    L.sbp = (L.gblk + 7) / 8 * 8 + 8;  // rows 16 bytes apart in banks
    L.red_off = (L.sb_off + 2 * 16 * kDecMaxTiles * L.sbp * 2 + 15) & ~15;
    L.bar_off = L.red_off + kDecWarps * NT * 4 * 32 * 4;
    L.spin_limit = a.spin_limit;
    return L;
  };
  auto smem_of = [&](const DecLayout &L) {
    return static_cast<size_t>(L.bar_off) + 8 * kDecMaxTiles * (L.kr / 128) + 1024;
  };
  // Split K over a cluster while blocks are short of the SMs, or a block's
  // K range is longer than kDecMaxChunks chunks or its shared memory would
  // keep two blocks from fitting an SM.
  int C = 1;
  while (C < 8 && kr_of(2 * C) >= 128 &&
         (nblk * 2 * C <= sms || kr_of(C) > 128 * kDecMaxChunks || smem_of(layout_of(C)) > 110 * 1024))
    C *= 2;
  const DecLayout L = layout_of(C);
  // Never let a third block fit an SM (228 KB of shared memory, 1 KB of it
  // reserved per block): two blocks of consecutive kernels then share each SM.
  const size_t smem = std::max(smem_of(L), static_cast<size_t>(77 * 1024));
  if (L.kr > 128 * kDecMaxChunks || smem > 220 * 1024) return cudaErrorNotSupported;
  CUtensorMap wmap;
  cudaError_t e = encode_map_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.w,
                                static_cast<uint64_t>(a.K) * BITS / 32, static_cast<uint64_t>(a.N),
                                static_cast<uint64_t>(a.K) * BITS / 8, 4 * BITS, 16,
                                BITS == 8 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  unsigned *err = device_error_word();
  if (!err) return cudaErrorInvalidSymbol;
  auto kern = gemv_decode_kernel<E, BITS, NT, OUT_BF16>;
  e = ensure_smem_limit<gemv_decode_kernel<E, BITS, NT, OUT_BF16>>(smem);
  if (e != cudaSuccess) return e;
  return launch_ex(kern, dim3(static_cast<unsigned>(nblk), C, 1), dim3(32 * kDecWarps), smem, C,
                   pdl, stream, wmap, a, L, err);
}

template <typename E, int BITS>
cudaError_t decode_bits(const GemvArgs &a, bool y_16, bool pdl, cudaStream_t stream) {
  if (a.M <= 8)
    return y_16 ? launch_decode<E, BITS, 1, true>(a, pdl, stream)
                : launch_decode<E, BITS, 1, false>(a, pdl, stream);
  return y_16 ? launch_decode<E, BITS, 2, true>(a, pdl, stream)
              : launch_decode<E, BITS, 2, false>(a, pdl, stream);
}

template <typename E>
cudaError_t decode_entry(const GemvArgs &a, int bits, bool y_16, bool pdl, cudaStream_t stream) {
  switch (bits) {
    case 1: return decode_bits<E, 1>(a, y_16, pdl, stream);
    case 2: return decode_bits<E, 2>(a, y_16, pdl, stream);
    case 3: return decode_bits<E, 3>(a, y_16, pdl, stream);
    case 4: return decode_bits<E, 4>(a, y_16, pdl, stream);
    case 5: return decode_bits<E, 5>(a, y_16, pdl, stream);
    case 6: return decode_bits<E, 6>(a, y_16, pdl, stream);
    case 8: return decode_bits<E, 8>(a, y_16, pdl, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode(const uint16_t *x, int64_t M, const PackedWeight &w, void *y, bool y_16,
                          bool f16, bool pdl, cudaStream_t stream) {
  if (M < 1 || M > 16 || w.cols % 128 != 0) return cudaErrorNotSupported;
  GemvArgs a;
  a.x = x;
  a.w = w.w;
  a.scales = w.scales;
  a.biases = w.biases;
  a.y = y;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(w.rows);
  a.K = static_cast<int>(w.cols);
  a.group_shift = w.group == 32 ? 5 : w.group == 64 ? 6 : 7;
  a.parts = 1;
  a.resid = nullptr;
  a.spin_limit = wait_limit();
  return f16 ? decode_entry<ElemF16>(a, w.bits, y_16, pdl, stream)
             : decode_entry<ElemBF16>(a, w.bits, y_16, pdl, stream);
}

}  // namespace qmm
