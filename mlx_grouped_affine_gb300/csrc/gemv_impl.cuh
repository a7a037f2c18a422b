// Decode path of quantized_matmul (M <= 16): kernels and launchers,
// templated on the 16-bit element type; included by gemv.cu (bf16 plain and
// fused), gemv_gather.cu (bf16 gather_qmm) and gemv_f16.cu (fp16), which
// compile in parallel.
//
// y = x . dequant(W)^T (transpose) or x . dequant(W) (nuvec_core
// quantized.rs, `quantized_matmul`; spark_runtime weights/mlx_int8.rs,
// `gemv`).  The kernel streams the packed weight once from HBM; everything
// else serves that stream:
//
//  * Each weight is dequantized in registers to the element type (bf16, or
//    fp16 for fp16 scales and x) with one rounding, w = RN(scale * code +
//    bias), from exact codes: a code c becomes (P + c) by OR-ing it into the
//    mantissa of a power of two P (128 in bf16, 1024 in fp16), and P is then
//    subtracted exactly.  8-bit codes in bf16 go through fp32.
//  * The products x * w and their fp32 sums run on the tensor pipe
//    (mma.sync m16n8k16, bf16 or fp16 in, fp32 accumulate) with the dequantized
//    weights as the A operand straight from registers: at M <= 16 the FMA
//    pipe would otherwise be the bottleneck, and no shared-memory round trip
//    is needed.  x rows beyond M are zero.
//  * K is split across the warps of a block (partials reduced through shared
//    memory) and, when the weight has few rows, across the blocks of a thread
//    block cluster (partials reduced through distributed shared memory).  No
//    global scratch memory is used.
//
// Fragment layout of m16n8k16 (g = lane / 4, t = lane % 4):
//   A 16x16: {a0a1} row g, k 2t..2t+1; {a2a3} row g+8, same k;
//            {a4a5} row g, k 2t+8..; {a6a7} row g+8, k 2t+8..
//   B 16x8:  {b0b1} k 2t..2t+1, col g; {b2b3} k 2t+8.., col g
//   D 16x8:  d0,d1 row g, cols 2t, 2t+1; d2,d3 row g+8, cols 2t, 2t+1
// The contraction index may be permuted freely as long as A and B agree.
#pragma once
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace qmm {
namespace {

// Eight words from p (32-byte aligned, read-only for the kernel's lifetime)
// with one 256-bit load.
__device__ __forceinline__ void ldg_v8(const void *p, uint32_t *v) {
  asm volatile("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                 "=r"(v[6]), "=r"(v[7])
               : "l"(p));
}

// d += A B on the tensor pipe, A and B of E (bf16 or fp16), fp32 accumulate.
template <typename E>
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (E::kF16)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

struct GemvArgs {
  const uint16_t *x;
  const uint32_t *w;
  const uint16_t *scales, *biases;
  void *y;
  int M, N, K;
  int group_shift;
  int parts;  // K parts = cluster size * warps per block
  const uint16_t *resid;  // bf16 [M, N] added to y before it is stored, or null
  uint32_t spin_limit = kDefaultWaitLimit;  // polls of a bounded wait
};

// Fused decode GEMVs (spark_runtime weights/mlx_int8.rs, `gemv_gate_up`,
// `gemv_silu_gate`, `gemv_silu_gate_resid`).
//   kFuseDual: blockIdx.z = 1 computes a second weight (scales2, biases2,
//     through the second tensor map) on the same x into y2.
//   kFuseSilu: x[m, k] = RN_bf16(silu(gate[m, k]) * up[m, k]) in fp32,
//     formed in shared memory by the warp that multiplies it, chunk by chunk.
constexpr int kFuseNone = 0, kFuseDual = 1, kFuseSilu = 2;
struct FuseArgs {
  const uint16_t *scales2, *biases2;
  void *y2;
  const uint16_t *gate, *up;   // bf16 [M, K]
};

// gather_qmm (nuvec_core quantized.rs, `gather_qmm`): output batch b is
// x[lhs[b]] times weight batch rhs[b].  blockIdx.z (+ z0) is the output
// batch, or -- sorted -- the weight batch whose run of tokens the block walks.
struct GatherArgs {
  const uint32_t *lhs, *rhs;       // device [batches], or null: batch b itself
  int x_batches, w_batches, batches;
  int z0;                          // first batch (or weight batch) of this launch
  int sorted;                      // runs of equal, sorted rhs; M == 1 and lhs null
  int64_t x_bstride, y_bstride;    // elements between batches of x and of y
  int64_t w_bstride, sb_bstride;   // words between weight batches; elements between scale batches
  int64_t x_off, y_off;            // elements: the 16-row slice of a batch this launch covers
};

// First position in the sorted v[0, n) whose value is >= key.
__device__ __forceinline__ int lower_bound_u32(const uint32_t *v, int n, uint32_t key) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(v + mid) < key) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// Zero outputs y[m, n] for m < rows, n in [n0, n0 + cols) (clipped to N): the
// part of an output batch a block owns, when its index is out of range.
__device__ __forceinline__ void zero_y_tile(void *y, bool out_bf16, int rows, int N, int n0, int cols) {
  for (int i = threadIdx.x; i < rows * cols; i += blockDim.x) {
    const int m = i / cols, n = n0 + (i - m * cols);
    if (n >= N) continue;
    const int64_t o = static_cast<int64_t>(m) * N + n;
    if (out_bf16) static_cast<uint16_t *>(y)[o] = 0;
    else static_cast<float *>(y)[o] = 0.0f;
  }
}

// Unsorted gather for the kernels that read W with plain loads: point `a` at
// the block's batches.  False (after zeroing the block's outputs and raising
// the index bit) when an index is out of range.
template <bool OUT_BF16>
__device__ __forceinline__ bool gather_point(GemvArgs &a, const GatherArgs &g, int n0, int cols,
                                             unsigned *err) {
  const int z = g.z0 + static_cast<int>(blockIdx.z);
  const uint32_t wb = g.rhs ? __ldg(g.rhs + z) : static_cast<uint32_t>(z);
  const uint32_t xb = g.lhs ? __ldg(g.lhs + z) : static_cast<uint32_t>(z);
  a.y = static_cast<char *>(a.y) + (z * g.y_bstride + g.y_off) * (OUT_BF16 ? 2 : 4);
  if (wb >= static_cast<uint32_t>(g.w_batches) || xb >= static_cast<uint32_t>(g.x_batches)) {
    zero_y_tile(a.y, OUT_BF16, a.M, a.N, n0, cols);
    if (threadIdx.x == 0) atomicOr(err, kErrIndexBit);
    return false;
  }
  a.x += xb * g.x_bstride + g.x_off;
  a.w += wb * g.w_bstride;
  a.scales += wb * g.sb_bstride;
  a.biases += wb * g.sb_bstride;
  return true;
}

// ------------------------------------------------------------------------
// Cross-warp and cross-block reduction of ACC fp32 values per lane, then the
// store.  Every warp of every block in the cluster holds a partial of the
// same output tile with the same lane -> (m, n) mapping.
template <typename E, int ACC, typename MapFn>
__device__ __forceinline__ void reduce_and_store(float (&acc)[ACC], float *red, int warps,
                                                 int cluster, const GemvArgs &a, bool out_bf16,
                                                 MapFn map) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int i = 0; i < ACC; ++i) red[(warp * ACC + i) * 32 + lane] = acc[i];
  __syncthreads();
  float sum[ACC];
  if (warp == 0) {
#pragma unroll
    for (int i = 0; i < ACC; ++i) {
      float s = 0.0f;
      for (int w = 0; w < warps; ++w) s += red[(w * ACC + i) * 32 + lane];
      sum[i] = s;
    }
  }
  if (cluster > 1) {
    // Block partials go to the first warp-slot of `red`; the leader block adds
    // its peers' through distributed shared memory.
    __syncthreads();
    if (warp == 0) {
#pragma unroll
      for (int i = 0; i < ACC; ++i) red[i * 32 + lane] = sum[i];
    }
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    uint32_t rank;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
    if (rank == 0 && warp == 0) {
      const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(red));
      for (int r = 1; r < cluster; ++r) {
        uint32_t remote;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(base), "r"(r));
#pragma unroll
        for (int i = 0; i < ACC; ++i) {
          float v;
          asm volatile("ld.shared::cluster.f32 %0, [%1];"
                       : "=f"(v) : "r"(remote + static_cast<uint32_t>((i * 32 + lane) * 4)));
          sum[i] += v;
        }
      }
    }
    // Peers keep their shared memory alive until the leader has read it.
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (rank != 0) return;
  }
  if (warp != 0) return;
#pragma unroll
  for (int i = 0; i < ACC; ++i) {
    int m, n;
    map(lane, i, m, n);
    if (m < a.M && n < a.N) {
      const int64_t o = static_cast<int64_t>(m) * a.N + n;
      const float v = a.resid ? sum[i] + E::to_f32(a.resid[o]) : sum[i];
      if (out_bf16) static_cast<uint16_t *>(a.y)[o] = E::from_f32(v);
      else static_cast<float *>(a.y)[o] = v;
    }
  }
}

// ------------------------------------------------------------------------
// transpose = true: W stored [N, K].  A warp owns a 16-row tile and a range of
// 128-code chunks of K.  In a chunk, lane (g, t) holds codes [32t, 32t+32) of
// rows g and g+8: `BITS` words per row, loaded with the widest aligned loads.
// Its 16 natural pairs per row feed 8 MMAs; MMA r contracts logical k
// (2t, 2t+1) with physical codes 32t+4r, +1 and logical (2t+8, 2t+9) with
// 32t+4r+2, +3, so the matching x values are the two words of x at
// k = 32t + 4r: lane (g, t) reads x[m][32t .. 32t+32) with four 16-byte loads.
template <typename E, int BITS, int NT, bool OUT_BF16, bool GATHER>
__global__ void __launch_bounds__(512)
gemv_t_kernel(GemvArgs a, GatherArgs ga, unsigned *err) {
  extern __shared__ float red[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, warps = blockDim.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  uint32_t crank = 0, csize = 1;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(crank));
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(csize));
  const int n0 = blockIdx.x * 16;
  if constexpr (GATHER) {
    if (!gather_point<OUT_BF16>(a, ga, n0, 16, err)) return;
  }
  const int part = static_cast<int>(crank) * warps + warp;
  const int nchunks = (a.K + 127) >> 7;
  const int c_begin = static_cast<int>(static_cast<int64_t>(nchunks) * part / a.parts);
  const int c_end = static_cast<int>(static_cast<int64_t>(nchunks) * (part + 1) / a.parts);

  const int64_t wpr = (static_cast<int64_t>(a.K) * BITS) >> 5;
  const int groups = a.K >> a.group_shift;
  const int row0 = n0 + g, row1 = n0 + g + 8;
  const bool ok0 = row0 < a.N, ok1 = row1 < a.N;
  const uint32_t *w0 = a.w + static_cast<int64_t>(ok0 ? row0 : 0) * wpr;
  const uint32_t *w1 = a.w + static_cast<int64_t>(ok1 ? row1 : 0) * wpr;

  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[nt][i] = 0.0f;

  for (int c = c_begin; c < c_end; ++c) {
    const int k = (c << 7) + 32 * t;  // first code of this lane's 32
    const bool kin = k < a.K;
    uint32_t v0[BITS], v1[BITS];
#pragma unroll
    for (int i = 0; i < BITS; ++i) { v0[i] = 0u; v1[i] = 0u; }
    uint16_t s0 = 0, b0 = 0, s1 = 0, b1 = 0;
    if (kin && ok0) {
      load_words<BITS>(w0 + (k >> 5) * BITS, v0);
      s0 = __ldg(a.scales + static_cast<int64_t>(row0) * groups + (k >> a.group_shift));
      b0 = __ldg(a.biases + static_cast<int64_t>(row0) * groups + (k >> a.group_shift));
    }
    if (kin && ok1) {
      load_words<BITS>(w1 + (k >> 5) * BITS, v1);
      s1 = __ldg(a.scales + static_cast<int64_t>(row1) * groups + (k >> a.group_shift));
      b1 = __ldg(a.biases + static_cast<int64_t>(row1) * groups + (k >> a.group_shift));
    }
    uint32_t xv[NT][16];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int m = g + 8 * nt;
      if (kin && m < a.M) {
        const uint4 *xp = reinterpret_cast<const uint4 *>(a.x + static_cast<int64_t>(m) * a.K + k);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 u = __ldg(xp + i);
          xv[nt][4 * i] = u.x; xv[nt][4 * i + 1] = u.y; xv[nt][4 * i + 2] = u.z; xv[nt][4 * i + 3] = u.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) xv[nt][i] = 0u;
      }
    }
    uint32_t p0[16], p1[16];
    dequant_pairs<BITS, 16, E>(v0, bcast2(s0), bcast2(b0), E::to_f32(s0), E::to_f32(b0), p0);
    dequant_pairs<BITS, 16, E>(v1, bcast2(s1), bcast2(b1), E::to_f32(s1), E::to_f32(b1), p1);
    if (!kin) {
#pragma unroll
      for (int i = 0; i < 16; ++i) { p0[i] = 0u; p1[i] = 0u; }
    }
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        mma_16816<E>(acc[nt], p0[2 * r], p1[2 * r], p0[2 * r + 1], p1[2 * r + 1],
                     xv[nt][2 * r], xv[nt][2 * r + 1]);
  }

  float flat[NT * 4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) flat[nt * 4 + i] = acc[nt][i];
  reduce_and_store<E, NT * 4>(flat, red, warps, static_cast<int>(csize), a, OUT_BF16,
                           [&](int ln, int i, int &m, int &n) {
                             const int gg = ln >> 2, tt = ln & 3, nt = i >> 2, e = i & 3;
                             n = n0 + gg + 8 * (e >> 1);
                             m = 8 * nt + 2 * tt + (e & 1);
                           });
}

// ------------------------------------------------------------------------
// transpose = false: W stored [K, N], packed and grouped along N.  A warp owns
// a 32-column tile of y and a range of 16-row steps of K.  In a step, lane
// (g, t) reads the 8 codes [8t, 8t+8) of the tile from stored rows k0+g and
// k0+8+g (one 8-code chunk each) and dequantizes them to 4 natural pairs
// along N.  Pair j of lane (g, t) is element (g, t) of an 8x8 bf16 block Q_j
// whose rows are k and whose column 2t+e is n = 8t + 2j + e; movmatrix.trans
// turns Q_j into the B fragment of n8-tile j, whose column c is
// n = 8(c/2) + 2j + (c%2).  x is the A operand (natural pairs along K).
template <typename E, int BITS, bool OUT_BF16, bool GATHER>
__global__ void __launch_bounds__(512)
gemv_n_kernel(GemvArgs a, GatherArgs ga, unsigned *err) {
  extern __shared__ float red[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, warps = blockDim.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  uint32_t crank = 0, csize = 1;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(crank));
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(csize));
  const int n0 = blockIdx.x * 32;
  if constexpr (GATHER) {
    if (!gather_point<OUT_BF16>(a, ga, n0, 32, err)) return;
  }
  const int part = static_cast<int>(crank) * warps + warp;
  const int nsteps = (a.K + 15) >> 4;  // K (the stored row count) may be any size
  const int s_begin = static_cast<int>(static_cast<int64_t>(nsteps) * part / a.parts);
  const int s_end = static_cast<int>(static_cast<int64_t>(nsteps) * (part + 1) / a.parts);

  const int64_t wpr = (static_cast<int64_t>(a.N) * BITS) >> 5;
  const int groups = a.N >> a.group_shift;
  const int nc = n0 + 8 * t;          // first column of this lane's chunk
  const bool nok = nc < a.N;
  const int gcol = nc >> a.group_shift;
  // The chunk's codes start at bit 8*BITS*(nc/8) of a stored row.
  const int cbit = BITS * nc, cword = cbit >> 5, csh = cbit & 31;
  constexpr bool kTwoWords = (BITS == 8) || (BITS == 3) || (BITS == 5) || (BITS == 6);

  float acc[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[j][i] = 0.0f;

  for (int s = s_begin; s < s_end; ++s) {
    const int k0 = s << 4;
    uint32_t bfrag[4][2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int krow = k0 + 8 * h + g;
      uint32_t win[2] = {0u, 0u};
      uint16_t sv = 0, bv = 0;
      if (nok && krow < a.K) {
        const uint32_t *rp = a.w + static_cast<int64_t>(krow) * wpr + cword;
        const uint32_t lo = __ldg(rp);
        uint32_t hi = 0u;
        if (kTwoWords && (csh + 8 * BITS > 32)) hi = __ldg(rp + 1);
        win[0] = csh ? __funnelshift_r(lo, hi, csh) : lo;
        win[1] = csh ? (hi >> csh) : hi;
        sv = __ldg(a.scales + static_cast<int64_t>(krow) * groups + gcol);
        bv = __ldg(a.biases + static_cast<int64_t>(krow) * groups + gcol);
      }
      uint32_t pr[4];
      dequant_pairs<BITS, 4, E>(win, bcast2(sv), bcast2(bv), E::to_f32(sv), E::to_f32(bv), pr);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t tr;
        asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(tr) : "r"(pr[j]));
        bfrag[j][h] = tr;
      }
    }
    // A = x rows g and g+8 (zero beyond M and K), natural pairs along K.  x
    // rows need not be 4-byte aligned here (K may be odd): 16-bit loads.
    uint32_t xa[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int m = g + 8 * (q & 1), kk = k0 + 2 * t + 8 * (q >> 1);
      uint32_t lo = 0u, hi = 0u;
      if (m < a.M) {
        const uint16_t *xr = a.x + static_cast<int64_t>(m) * a.K;
        if (kk < a.K) lo = __ldg(xr + kk);
        if (kk + 1 < a.K) hi = __ldg(xr + kk + 1);
      }
      xa[q] = lo | (hi << 16);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      mma_16816<E>(acc[j], xa[0], xa[1], xa[2], xa[3], bfrag[j][0], bfrag[j][1]);
  }

  float flat[16];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) flat[j * 4 + i] = acc[j][i];
  reduce_and_store<E, 16>(flat, red, warps, static_cast<int>(csize), a, OUT_BF16,
                       [&](int ln, int i, int &m, int &n) {
                         const int gg = ln >> 2, tt = ln & 3, j = i >> 2, e = i & 3;
                         m = gg + 8 * (e >> 1);
                         n = n0 + 8 * tt + 2 * j + (e & 1);
                       });
}

// ------------------------------------------------------------------------
// Shared by the transposed decode kernels.
//
// Code pairs.  Every width is paired naturally: pair p of a lane's 32 codes
// is (2p, 2p+1), so x is used as it lies.  Each pair becomes one bf16x2
// register, each half RN(s*c + b), in one of two forms.
//
// Fast form.  A bf16 bit pattern P <= 0xFF has the value P * 2^-133 exactly:
// below 0x80 it is a subnormal, above it the exponent field is 1 and its
// implicit leading one is worth exactly bit 7 of P.  So a code c sitting at
// bit o (o + bits <= 8) of an otherwise clear 16-bit half reads as
// c * 2^(o-133), and one bf16x2 FMA against the multiplier s * 2^(133-o)
// with addend b yields RN(s*c + b): the product is exactly s*c and the FMA
// rounds once.  The multiplier is s with 133 - o added to its exponent
// field, which is exact while the exponent stays below 255; the fast form is
// used when every scale of the warp's chunk is a normal number below 2^-5.
// Per pair this costs one byte permute (the pair's byte, or two bytes at
// 8 bits, into both halves), one mask (none at 8 bits) and the FMA.
//
// Exact form, for any scale: the code OR-ed into the mantissa of 128.0 gives
// bf16 (128 + c), 128 is subtracted exactly, then the same FMA; 8-bit codes
// go through fp32.
//
// Warps take 128-code chunks in turn; lane (g, t) handles codes
// [32t, 32t+32) of rows g and g+8, i.e. 16 pairs per row, and MMA r
// contracts pairs 2r and 2r+1 with the two x words at the same positions.
// (pair_fast / pair_exact and the multiplier helpers live in common.cuh.)

template <int BITS>
__device__ __forceinline__ void lds_words(const uint8_t *p, uint32_t *v) {
  if constexpr (BITS % 4 == 0) {
#pragma unroll
    for (int i = 0; i < BITS / 4; ++i) {
      const uint4 u = reinterpret_cast<const uint4 *>(p)[i];
      v[4 * i] = u.x; v[4 * i + 1] = u.y; v[4 * i + 2] = u.z; v[4 * i + 3] = u.w;
    }
  } else if constexpr (BITS % 2 == 0) {
#pragma unroll
    for (int i = 0; i < BITS / 2; ++i) {
      const uint2 u = reinterpret_cast<const uint2 *>(p)[i];
      v[2 * i] = u.x; v[2 * i + 1] = u.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < BITS; ++i) v[i] = reinterpret_cast<const uint32_t *>(p)[i];
  }
}

// ------------------------------------------------------------------------
// transpose = true, chunk-pipelined through the tensor-memory-access unit.
// Used when K is a multiple of 128.
//
// Every 128-code chunk of the block's 16-row tile is one 2-D TMA box (16 rows
// x 16*BITS bytes) with its own mbarrier; one thread issues all of them at
// kernel start, so the weight is in flight at once, and a warp waits only for
// the chunks it computes -- compute overlaps the stream instead of starting
// after it.  A box lands densely (row pitch 16*BITS bytes), which keeps the
// reads of lanes (g, t) in distinct banks for every width but 8 bits; 8-bit
// boxes use the 128-byte swizzle (16-byte unit q of row r at q ^ (r % 8)).
// The weight copies and the scale/bias loads come before griddepcontrol.wait;
// x, which the previous kernel may write, is read after it; 8 MMAs per chunk.

// Two values of silu(g) * u, g / (1 + e^-g) * u in fp32, as one pair of E
// (each rounded to nearest even).
template <typename E>
__device__ __forceinline__ uint32_t silu_mul2(uint32_t g2, uint32_t u2) {
  float r[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float gf = E::to_f32((g2 >> (16 * h)) & 0xFFFFu);
    const float uf = E::to_f32((u2 >> (16 * h)) & 0xFFFFu);
    r[h] = __fdividef(gf, 1.0f + __expf(-gf)) * uf;
  }
  return E::pack2(r[0], r[1]);
}

struct TmaLayout {
  int kr;           // codes per block (multiple of 128)
  int box_bytes;    // shared bytes of one chunk box
  int x_off;        // offset of the x rows formed in shared memory (silu fusion)
  int xpitch;       // their pitch, bytes
  int red_off;      // offset of the reduction buffer
  int bar_off;      // offset of the chunk mbarriers
  int x32;          // x starts on a 32-byte boundary: 256-bit x loads
};

// Warps per block: 16 for one n8 tile of x rows; 8 for two (twice the
// registers), so that two blocks fit on an SM either way.
template <int NT>
__host__ __device__ constexpr int tma_warps() { return NT == 1 ? 16 : 8; }
constexpr int kTmaMaxChunksPerWarp = 4;

// (A minimum of 0 blocks leaves the register budget to the compiler, as with
// no minimum given; the gather and fused instantiations are held to two
// blocks per SM.)
// W: warps per block (the default for NT, or 8 for one n8 tile: blocks of
// 16K registers, four an SM, for weights with many row tiles).  X32: one n8
// tile reads x with 32-byte loads (the launcher takes it at 2 <= M <= 8 when
// x is 32-byte aligned; two tiles decide at run time from L.x32).
template <typename E, int BITS, int NT, bool OUT_BF16, bool GATHER, int FUSE, int W = tma_warps<NT>(),
          bool X32 = false>
__global__ void __launch_bounds__(32 * W, W < tma_warps<NT>() ? 4 : (GATHER || FUSE ? 2 : 0))
gemv_t_tma_kernel(const __grid_constant__ CUtensorMap wmap, GemvArgs a, TmaLayout L,
                  unsigned *err, GatherArgs ga, const __grid_constant__ CUtensorMap wmap2,
                  FuseArgs fa) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar_off);
  float *red = reinterpret_cast<float *>(smem + L.red_off);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  uint32_t crank = 0, csize = 1;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(crank));
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(csize));
  const int n0 = blockIdx.x * 16;
  const int k0 = static_cast<int>(crank) * L.kr;
  const int ncodes = max(0, min(a.K, k0 + L.kr) - k0);
  const int nchunks = ncodes >> 7;
  // The block's weight rows start at wrow0 (its weight batch's first row in
  // the tensor map); it computes `rows` rows of x from xbase into ybase.
  const CUtensorMap *map = &wmap;
  if constexpr (FUSE == kFuseDual) {
    if (blockIdx.z == 1) {
      map = &wmap2;
      a.scales = fa.scales2;
      a.biases = fa.biases2;
      a.y = fa.y2;
    }
  }
  int wrow0 = 0, rows = a.M;
  const uint16_t *xbase = a.x;
  char *ybase = static_cast<char *>(a.y);
  if constexpr (GATHER) {
    constexpr int ysz = OUT_BF16 ? 2 : 4;
    const int z = ga.z0 + static_cast<int>(blockIdx.z);
    uint32_t wb;
    if (ga.sorted) {
      // Weight batch z walks its run [lo, hi) of the sorted rhs (one x row per
      // batch); z == w_batches takes the indices past the weights.
      const int lo = lower_bound_u32(ga.rhs, ga.batches, static_cast<uint32_t>(z));
      const int hi = z < ga.w_batches ? lower_bound_u32(ga.rhs, ga.batches, static_cast<uint32_t>(z + 1))
                                      : ga.batches;
      if (hi <= lo) return;
      ybase += static_cast<int64_t>(lo) * a.N * ysz;
      if (z >= ga.w_batches) {
        if (crank == 0) zero_y_tile(ybase, OUT_BF16, hi - lo, a.N, n0, 16);
        if (threadIdx.x == 0) atomicOr(err, kErrIndexBit);
        return;
      }
      wb = static_cast<uint32_t>(z);
      rows = hi - lo;
      xbase = a.x + static_cast<int64_t>(lo) * a.K;
    } else {
      wb = ga.rhs ? __ldg(ga.rhs + z) : static_cast<uint32_t>(z);
      const uint32_t xb = ga.lhs ? __ldg(ga.lhs + z) : static_cast<uint32_t>(z);
      ybase += z * ga.y_bstride * ysz;
      if (wb >= static_cast<uint32_t>(ga.w_batches) || xb >= static_cast<uint32_t>(ga.x_batches)) {
        if (crank == 0) zero_y_tile(ybase, OUT_BF16, a.M, a.N, n0, 16);
        if (threadIdx.x == 0) atomicOr(err, kErrIndexBit);
        return;
      }
      xbase = a.x + xb * ga.x_bstride;
    }
    wrow0 = static_cast<int>(wb) * a.N;
  }

  if (warp == 0) {
    for (int c = lane; c < nchunks; c += 32) mbar_init(&bars[c], 1);  // one per chunk
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (warp == 0) {
    // Lane c issues chunk c's box (and c + 32, ...).
    for (int c = lane; c < nchunks; c += 32) {
      mbar_expect_tx(&bars[c], L.box_bytes);
      const int xw = ((k0 + (c << 7)) * BITS) >> 5;  // word coordinate
      asm volatile(
          "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
          " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem + c * L.box_bytes)),
          "l"(map), "r"(xw), "r"(wrow0 + n0), "r"(smem_u32(&bars[c]))
          : "memory");
    }
  }
  griddep_launch_dependents();

  const int groups = a.K >> a.group_shift;
  const int row0 = wrow0 + min(n0 + g, a.N - 1), row1 = wrow0 + min(n0 + g + 8, a.N - 1);
  const uint16_t *s0p = a.scales + static_cast<int64_t>(row0) * groups;
  const uint16_t *b0p = a.biases + static_cast<int64_t>(row0) * groups;
  const uint16_t *s1p = a.scales + static_cast<int64_t>(row1) * groups;
  const uint16_t *b1p = a.biases + static_cast<int64_t>(row1) * groups;
  auto load_sb = [&](int c, uint16_t (&sv)[4]) {
    const int gi = (k0 + (c << 7) + 32 * t) >> a.group_shift;
    sv[0] = __ldg(s0p + gi); sv[1] = __ldg(b0p + gi);
    sv[2] = __ldg(s1p + gi); sv[3] = __ldg(b1p + gi);
  };
  // Scales and biases of every chunk this warp will compute, before the
  // wait: they are weights too, and their HBM latency then overlaps the
  // previous kernel instead of the chunk loop.
  constexpr int kW = W;
  uint16_t sv[kTmaMaxChunksPerWarp][4];
#pragma unroll
  for (int j = 0; j < kTmaMaxChunksPerWarp; ++j) {
    sv[j][0] = sv[j][1] = sv[j][2] = sv[j][3] = 0;
    if (warp + j * kW < nchunks) load_sb(warp + j * kW, sv[j]);
  }

  // x may be written by the previous kernel in the stream.  Each lane reads
  // its own 32 x values per chunk (L2-resident: every block reads the same x),
  // natural pairs like the weights.
  griddep_wait();
  bool ok = true;
  // One pass computes mrows <= 8 * NT rows of x, from xc, into yc.
  auto pass = [&](const uint16_t *xc, void *yc, int mrows) {
    GemvArgs ac = a;
    ac.x = xc;
    ac.y = yc;
    ac.M = mrows;
    // Lanes whose x row is beyond M keep zero fragments throughout.
    auto load_x_nt = [&](int c, int nt, uint32_t (&xt)[16]) {
      const int m = g + 8 * nt;
      if (m < ac.M) {
        if constexpr (FUSE == kFuseSilu) {
          const uint4 *xp =
              reinterpret_cast<const uint4 *>(smem + L.x_off + m * L.xpitch + ((c << 7) + 32 * t) * 2);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint4 u = xp[i];
            xt[4 * i] = u.x; xt[4 * i + 1] = u.y; xt[4 * i + 2] = u.z; xt[4 * i + 3] = u.w;
          }
        } else if ((NT == 1 && X32) || (NT == 2 && L.x32)) {
          // Two 32-byte loads: each fills whole sectors, half the requests
          // of 16-byte loads (at M > 8 the x reads set the L1's pace).  One
          // n8 tile takes them only by its template flag: the branch alone
          // costs 1 % at M = 1.
          const uint16_t *xp = ac.x + static_cast<int64_t>(m) * a.K + k0 + (c << 7) + 32 * t;
          ldg_v8(xp, &xt[0]);
          ldg_v8(xp + 16, &xt[8]);
        } else {
          const uint4 *xp =
              reinterpret_cast<const uint4 *>(ac.x + static_cast<int64_t>(m) * a.K + k0 + (c << 7) + 32 * t);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint4 u = __ldg(xp + i);
            xt[4 * i] = u.x; xt[4 * i + 1] = u.y; xt[4 * i + 2] = u.z; xt[4 * i + 3] = u.w;
          }
        }
      }
    };
    auto load_x = [&](int c, uint32_t (&xv)[NT][16]) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) load_x_nt(c, nt, xv[nt]);
    };
    // silu fusion: before a warp reads chunk c's x, its 32 lanes form that
    // chunk's x = RN_bf16(silu(gate) * up) (fp32) in shared memory, 4 values
    // a lane per row; the chunks are the warp's own, so a warp barrier is all
    // the ordering it needs.
    auto stage_silu = [&](int c) {
      if constexpr (FUSE == kFuseSilu) {
        for (int m = 0; m < ac.M; ++m) {
          const int kk = (c << 7) + 4 * lane;
          const int64_t off = static_cast<int64_t>(m) * a.K + k0 + kk;
          const uint2 gv = __ldg(reinterpret_cast<const uint2 *>(fa.gate + off));
          const uint2 uv = __ldg(reinterpret_cast<const uint2 *>(fa.up + off));
          *reinterpret_cast<uint2 *>(smem + L.x_off + m * L.xpitch + kk * 2) =
              make_uint2(silu_mul2<E>(gv.x, uv.x), silu_mul2<E>(gv.y, uv.y));
        }
        __syncwarp();
      }
    };
    uint32_t xv[NT][16];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 16; ++i) xv[nt][i] = 0u;

    // Two accumulator sets (even and odd MMA steps) keep the MMA chain short.
    float acc[2][NT][4];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[h][nt][i] = 0.0f;

    constexpr int kRowBytes = 16 * BITS;  // one row of a chunk box
    // Two n8 tiles of x (M > 8): the next chunk's x is loaded while this one
    // computes -- a tile's registers are reloaded as soon as its MMAs have
    // read them, so the chunk's pairs are dequantized up front.  The MMAs
    // then run tile by tile; each accumulator sees the same steps in the
    // same order as below.  (Not for 8-bit gathers, which would spill.)
    constexpr bool kPrefetchX = NT == 2 && FUSE != kFuseSilu && !(GATHER && BITS == 8);
    if constexpr (kPrefetchX) {
      if (warp < nchunks) load_x(warp, xv);
    }
#pragma unroll
    for (int j = 0; j < kTmaMaxChunksPerWarp; ++j) {
      const int c = warp + j * kW;
      if (!ok || c >= nchunks) break;
      const uint16_t *cur = sv[j];
      if constexpr (!kPrefetchX) {
        stage_silu(c);
        load_x(c, xv);
      }
      uint32_t spins = 0;
      while (!mbar_try_wait(&bars[c], 0)) {
        if (++spins >= a.spin_limit) {
          if (lane == 0) atomicOr(err, kErrTimeoutBit);
          ok = false;
          break;
        }
      }
      if (!ok) break;
      const uint8_t *box = smem + c * L.box_bytes;
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
      const uint32_t b0 = bcast2(cur[1]), b1 = bcast2(cur[3]);
      // The fast form is bf16's (fp16 has no room for its multipliers).
      bool fast = false;
      if constexpr (!E::kF16) fast = __all_sync(0xffffffffu, fast_scale(cur[0]) && fast_scale(cur[2]));
      if constexpr (kPrefetchX) {
        uint32_t p0[16], p1[16];
        if (fast) {
          uint32_t m0[fast_slots<BITS>()], m1[fast_slots<BITS>()];
          fast_muls<BITS>(cur[0], m0);
          fast_muls<BITS>(cur[2], m1);
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            p0[q] = pair_fast<BITS>(v0, q, m0, b0);
            p1[q] = pair_fast<BITS>(v1, q, m1, b1);
          }
        } else {
          const uint32_t s0 = bcast2(cur[0]), s1 = bcast2(cur[2]);
          const float fs0 = E::to_f32(cur[0]), fb0 = E::to_f32(cur[1]);
          const float fs1 = E::to_f32(cur[2]), fb1 = E::to_f32(cur[3]);
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            p0[q] = pair_exact<BITS, E>(v0, q, s0, b0, fs0, fb0);
            p1[q] = pair_exact<BITS, E>(v1, q, s1, b1, fs1, fb1);
          }
        }
        const int cn = c + kW;
        const bool more = j + 1 < kTmaMaxChunksPerWarp && cn < nchunks;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
          for (int r = 0; r < 8; ++r)
            mma_16816<E>(acc[r & 1][nt], p0[2 * r], p1[2 * r], p0[2 * r + 1], p1[2 * r + 1],
                         xv[nt][2 * r], xv[nt][2 * r + 1]);
          if (more) load_x_nt(cn, nt, xv[nt]);
        }
      } else if (fast) {
        uint32_t m0[fast_slots<BITS>()], m1[fast_slots<BITS>()];
        fast_muls<BITS>(cur[0], m0);
        fast_muls<BITS>(cur[2], m1);
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const uint32_t a0 = pair_fast<BITS>(v0, 2 * r, m0, b0), a2 = pair_fast<BITS>(v0, 2 * r + 1, m0, b0);
          const uint32_t a1 = pair_fast<BITS>(v1, 2 * r, m1, b1), a3 = pair_fast<BITS>(v1, 2 * r + 1, m1, b1);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mma_16816<E>(acc[r & 1][nt], a0, a1, a2, a3, xv[nt][2 * r], xv[nt][2 * r + 1]);
        }
      } else {
        const uint32_t s0 = bcast2(cur[0]), s1 = bcast2(cur[2]);
        const float fs0 = E::to_f32(cur[0]), fb0 = E::to_f32(cur[1]);
        const float fs1 = E::to_f32(cur[2]), fb1 = E::to_f32(cur[3]);
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const uint32_t a0 = pair_exact<BITS, E>(v0, 2 * r, s0, b0, fs0, fb0);
          const uint32_t a2 = pair_exact<BITS, E>(v0, 2 * r + 1, s0, b0, fs0, fb0);
          const uint32_t a1 = pair_exact<BITS, E>(v1, 2 * r, s1, b1, fs1, fb1);
          const uint32_t a3 = pair_exact<BITS, E>(v1, 2 * r + 1, s1, b1, fs1, fb1);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mma_16816<E>(acc[r & 1][nt], a0, a1, a2, a3, xv[nt][2 * r], xv[nt][2 * r + 1]);
        }
      }
    }

    float flat[NT * 4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) flat[nt * 4 + i] = acc[0][nt][i] + acc[1][nt][i];
    reduce_and_store<E, NT * 4>(flat, red, W, static_cast<int>(csize), ac, OUT_BF16,
                             [&](int ln, int i, int &m, int &n) {
                               const int gg = ln >> 2, tt = ln & 3, nt = i >> 2, e = i & 3;
                               n = n0 + gg + 8 * (e >> 1);
                               m = 8 * nt + 2 * tt + (e & 1);
                             });
  };
  if constexpr (GATHER) {
    for (int mc = 0; mc < rows; mc += 8 * NT) {
      if (mc > 0) __syncthreads();  // the previous pass's reduction has read `red`
      pass(xbase + static_cast<int64_t>(mc) * a.K,
           ybase + static_cast<int64_t>(mc) * a.N * (OUT_BF16 ? 2 : 4), min(8 * NT, rows - mc));
    }
  } else {
    pass(xbase, ybase, rows);
  }
  if (!ok) {
    // A wait ran out: before the block exits, wait (bounded) for the copies
    // still in flight into its shared memory.
    for (int j = 0; j < kTmaMaxChunksPerWarp; ++j) {
      const int c = warp + j * kW;
      if (c >= nchunks) break;
      for (uint32_t s = 0; s < kDefaultWaitLimit; ++s)
        if (mbar_try_wait(&bars[c], 0)) break;
    }
  }
}

// ------------------------------------------------------------------------

struct Shape {
  int warps, cluster;
};

// Split K over `warps` warps per block and `cluster` blocks so that about
// 4096 warps stream the weight (enough loads in flight to cover HBM latency
// on 152 SMs), without giving a warp less than one K step.
Shape pick_shape(int64_t tiles, int64_t ksteps) {
  int64_t split = (4096 + tiles - 1) / tiles;
  if (split > ksteps) split = ksteps;
  int p = 1;
  while (p * 2 <= split && p < 128) p *= 2;
  Shape s;
  s.warps = p < 16 ? (p < 4 ? 4 : p) : 16;
  s.cluster = p > 16 ? p / 16 : 1;
  if (s.cluster > 8) s.cluster = 8;
  return s;
}

template <typename Kern, typename... Args>
cudaError_t launch_ex(Kern kern, dim3 grid, dim3 block, size_t smem, int cluster, bool pdl,
                      cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  // A cluster of one is the default; naming it costs about 0.1 us a launch.
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 1;
    attr[n].val.clusterDim.y = cluster;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// The z extent of a launch: 1, or the batches of a gather (output batches,
// or weight batches + 1 when sorted), with the arguments its kernels read.
struct Batches {
  GatherArgs g{};
  int64_t count = 1;
};

// Launches over z in pieces the grid's z dimension can hold.
template <typename Launch>
cudaError_t over_z(const Batches &b, Launch launch) {
  constexpr int64_t kMaxZ = 65535;
  GatherArgs g = b.g;
  for (int64_t z0 = 0; z0 < b.count; z0 += kMaxZ) {
    g.z0 = static_cast<int>(z0);
    const cudaError_t e = launch(g, static_cast<unsigned>(b.count - z0 < kMaxZ ? b.count - z0 : kMaxZ));
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <typename E, int BITS, int NT, bool OUT_BF16, bool GATHER>
cudaError_t launch_t(const GemvArgs &a0, const Batches &b, cudaStream_t stream) {
  GemvArgs a = a0;
  const int64_t tiles = (a.N + 15) / 16;
  Shape s = pick_shape(tiles, (a.K + 127) / 128);
  a.parts = s.warps * s.cluster;
  const size_t smem = sizeof(float) * s.warps * NT * 4 * 32;
  unsigned *err = device_error_word();
  if (!err) return cudaErrorInvalidSymbol;
  return over_z(b, [&](const GatherArgs &g, unsigned nz) {
    return launch_ex(gemv_t_kernel<E, BITS, NT, OUT_BF16, GATHER>,
                     dim3(static_cast<unsigned>(tiles), s.cluster, nz), dim3(32 * s.warps), smem,
                     s.cluster, false, stream, a, g, err);
  });
}

// Whether x starts on a 32-byte boundary (the decode's 32-byte x loads).
inline bool x_aligned32(const void *x) { return (reinterpret_cast<uintptr_t>(x) & 31u) == 0; }

template <typename E, int BITS, int NT, bool OUT_BF16, bool GATHER, int FUSE = kFuseNone,
          int W = tma_warps<NT>(), bool X32 = false>
cudaError_t launch_t_tma(const GemvArgs &a, bool pdl, const Batches &b, cudaStream_t stream,
                         const FuseArgs &f = FuseArgs{}, const uint32_t *w2 = nullptr) {
  const int64_t tiles = (a.N + 15) / 16;
  const int box_bytes = 16 * 16 * BITS;
  auto kr_of = [&](int c) { return ((a.K / c + 127) / 128) * 128; };
  auto smem_of = [&](int c) {
    const int kr = kr_of(c);
    return (kr / 128) * (box_bytes + 8) + W * NT * 4 * 32 * 4 + 2048;
  };
  // Split K over a cluster only when the weight has too few 16-row tiles to
  // give every SM work, or one block's share would not fit.
  int C = 1;
  const int max_kr = 128 * kTmaMaxChunksPerWarp * W;
  while (C < 8 && kr_of(2 * C) >= 128 &&
         (tiles * C < 240 || smem_of(C) > 100 * 1024 || kr_of(C) > max_kr))
    C *= 2;
  if (smem_of(C) > 200 * 1024 || kr_of(C) > max_kr) return cudaErrorNotSupported;
  TmaLayout L;
  L.kr = kr_of(C);
  L.box_bytes = box_bytes;
  const int nch = L.kr / 128;
  // x is read from global memory by each lane, or (silu) from the rows the
  // warps form in shared memory.
  L.x_off = nch * box_bytes;
  L.xpitch = FUSE == kFuseSilu ? L.kr * 2 + 16 : 0;
  L.red_off = L.x_off + a.M * L.xpitch;
  L.bar_off = L.red_off + W * NT * 4 * 32 * 4;
  // Row and batch offsets of x are multiples of K (a multiple of 128), so the
  // base decides the alignment of every lane's 32 values.
  L.x32 = x_aligned32(a.x);
  if (X32 && !L.x32) return cudaErrorInvalidValue;
  const size_t smem = L.bar_off + 8 * nch + 1024;  // + slack for the 1024-byte base
  if (smem > 220 * 1024) return cudaErrorNotSupported;
  // The tensor map spans every weight batch: batch e's row n is row e*N + n.
  const uint64_t map_rows = static_cast<uint64_t>(a.N) * (GATHER ? b.g.w_batches : 1);
  if (map_rows >= (uint64_t(1) << 31)) return cudaErrorNotSupported;
  CUtensorMap wmap;
  cudaError_t e = encode_map_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.w,
                                static_cast<uint64_t>(a.K) * BITS / 32, map_rows,
                                static_cast<uint64_t>(a.K) * BITS / 8, 4 * BITS, 16,
                                BITS == 8 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  CUtensorMap wmap2 = wmap;
  if (FUSE == kFuseDual) {
    e = encode_map_2d(&wmap2, CU_TENSOR_MAP_DATA_TYPE_UINT32, w2, static_cast<uint64_t>(a.K) * BITS / 32,
                      map_rows, static_cast<uint64_t>(a.K) * BITS / 8, 4 * BITS, 16,
                      BITS == 8 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
  }
  unsigned *err = device_error_word();
  if (!err) return cudaErrorInvalidSymbol;
  auto kern = gemv_t_tma_kernel<E, BITS, NT, OUT_BF16, GATHER, FUSE, W, X32>;
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  return over_z(b, [&](const GatherArgs &g, unsigned nz) {
    return launch_ex(kern, dim3(static_cast<unsigned>(tiles), C, nz), dim3(32 * W),
                     smem, C, pdl, stream, wmap, a, L, err, g, wmap2, f);
  });
}

template <typename E, int BITS, bool OUT_BF16, bool GATHER>
cudaError_t launch_n(const GemvArgs &a0, const Batches &b, cudaStream_t stream) {
  GemvArgs a = a0;
  const int64_t tiles = (a.N + 31) / 32;
  Shape s = pick_shape(tiles, (a.K + 15) / 16);
  a.parts = s.warps * s.cluster;
  const size_t smem = sizeof(float) * s.warps * 16 * 32;
  unsigned *err = device_error_word();
  if (!err) return cudaErrorInvalidSymbol;
  return over_z(b, [&](const GatherArgs &g, unsigned nz) {
    return launch_ex(gemv_n_kernel<E, BITS, OUT_BF16, GATHER>,
                     dim3(static_cast<unsigned>(tiles), s.cluster, nz), dim3(32 * s.warps), smem,
                     s.cluster, false, stream, a, g, err);
  });
}

// The plain decode GEMV in element type E: the TMA kernel for a transposed W
// with K a multiple of 128 (when its layout fits), else the plain-load
// kernels.  y_16 stores y in E, else fp32.
template <typename E, int BITS>
cudaError_t launch_bits(const GemvArgs &a, bool transpose, bool y_16, bool pdl,
                        cudaStream_t stream) {
  const Batches one;
  if (transpose && a.K % 128 == 0) {
    cudaError_t e;
    // More row tiles than two 16-warp blocks an SM hold: 8-warp blocks (four an
    // SM), so that twice the tiles stream at once (measured at M = 1: [14336,
    // 4096] 4-bit 13.1 -> 10.8 us, [11008, 4096] 3-bit 12.9 -> 11.6 us).  6 and
    // 8 bits keep 16 warps (6-bit 14.0 -> 14.6 us, 8-bit [14336, 4096] 15.2 ->
    // 18.4 us), as do one-wave shapes ([4096, 4096] 4.24 us against 4.83).
    // At 2 <= M <= 8, 32-byte x loads when x allows them (M = 8 [4096, 4096]
    // 4-bit 5.22 -> 4.61 us).
    const bool wide = a.M > 1 && x_aligned32(a.x);
    bool many = false;
    if constexpr (BITS < 6) many = a.M <= 8 && (a.N + 15) / 16 > 2 * sm_count();
    if (many) {
      if constexpr (BITS < 6) {
        if (wide)
          e = y_16 ? launch_t_tma<E, BITS, 1, true, false, kFuseNone, 8, true>(a, pdl, one, stream)
                   : launch_t_tma<E, BITS, 1, false, false, kFuseNone, 8, true>(a, pdl, one, stream);
        else
          e = y_16 ? launch_t_tma<E, BITS, 1, true, false, kFuseNone, 8>(a, pdl, one, stream)
                   : launch_t_tma<E, BITS, 1, false, false, kFuseNone, 8>(a, pdl, one, stream);
      }
    } else if (a.M <= 8) {
      if (wide)
        e = y_16 ? launch_t_tma<E, BITS, 1, true, false, kFuseNone, tma_warps<1>(), true>(a, pdl, one, stream)
                 : launch_t_tma<E, BITS, 1, false, false, kFuseNone, tma_warps<1>(), true>(a, pdl, one, stream);
      else
        e = y_16 ? launch_t_tma<E, BITS, 1, true, false>(a, pdl, one, stream)
                 : launch_t_tma<E, BITS, 1, false, false>(a, pdl, one, stream);
    } else
      e = y_16 ? launch_t_tma<E, BITS, 2, true, false>(a, pdl, one, stream)
               : launch_t_tma<E, BITS, 2, false, false>(a, pdl, one, stream);
    if (e != cudaErrorNotSupported) return e;
  }
  if (transpose) {
    if (a.M <= 8)
      return y_16 ? launch_t<E, BITS, 1, true, false>(a, one, stream)
                  : launch_t<E, BITS, 1, false, false>(a, one, stream);
    return y_16 ? launch_t<E, BITS, 2, true, false>(a, one, stream)
                : launch_t<E, BITS, 2, false, false>(a, one, stream);
  }
  return y_16 ? launch_n<E, BITS, true, false>(a, one, stream)
              : launch_n<E, BITS, false, false>(a, one, stream);
}

// The decode GEMV entry for element type E (x, scales, biases and a 16-bit y
// all of E).
template <typename E>
cudaError_t gemv_entry(const uint16_t *x, int64_t M, const PackedWeight &w, bool transpose,
                       void *y, bool y_16, cudaStream_t stream) {
  GemvArgs a;
  a.x = x;
  a.w = w.w;
  a.scales = w.scales;
  a.biases = w.biases;
  a.y = y;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(transpose ? w.rows : w.cols);
  a.K = static_cast<int>(transpose ? w.cols : w.rows);
  a.group_shift = w.group == 32 ? 5 : w.group == 64 ? 6 : 7;
  a.parts = 1;
  a.resid = nullptr;
  a.spin_limit = wait_limit();
  const bool pdl = (launch_flags() & kLaunchPdl) != 0;
  switch (w.bits) {
    case 1: return launch_bits<E, 1>(a, transpose, y_16, pdl, stream);
    case 2: return launch_bits<E, 2>(a, transpose, y_16, pdl, stream);
    case 3: return launch_bits<E, 3>(a, transpose, y_16, pdl, stream);
    case 4: return launch_bits<E, 4>(a, transpose, y_16, pdl, stream);
    case 5: return launch_bits<E, 5>(a, transpose, y_16, pdl, stream);
    case 6: return launch_bits<E, 6>(a, transpose, y_16, pdl, stream);
    case 8: return launch_bits<E, 8>(a, transpose, y_16, pdl, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace
}  // namespace qmm
