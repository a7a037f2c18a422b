// quantized_matmul in fp32: x, scales and biases that promote to fp32
// (nuvec_core quantized.rs, `quantized_matmul`: x, scales and biases are
// promoted to one floating-point type, and the product is taken in it).
//
// The tensor cores have no fp32 form (their fp32-input form, tf32, keeps 10
// fraction bits), so this path runs on the CUDA cores with fp32 FMAs: every
// weight is dequantized exactly as the standalone dequantize does it, fp32
// fma(scale, code, bias), x is widened exactly from its type, and the sums
// are fp32.
//
// Tiled: a block owns a BM x BN tile of y and walks K in steps of BK = 32.
// Per step the block's 256 threads dequantize the BK x BN weight tile into
// shared memory (Ws[k][n]) and stage the BM x BK x tile transposed (Xs[k][m]),
// then each thread accumulates a TM x TN micro-tile from them.  The codes, the
// scales and biases and the x values of the next PF steps are in flight in a
// register ring while the current step computes (PF = 6 for the small-M tile,
// whose steps are short, 1 for the 128 x 128 tile).  An octet of 8 codes is what a
// thread dequantizes at a time: its 8*bits bits sit in one 64-bit window of
// two consecutive words of the stored row.
//
// When the tiles are too few to fill the GPU (small M or N), K is split over
// grid z; each slice writes fp32 partials to a stream-ordered workspace and
// a second kernel adds them in slice order, so results repeat bit for bit.
// At M <= 16 with W stored [N, K] a GEMV form (mm_f32_gemv_kernel, below)
// replaces the tiles.
#include "common.cuh"
#include "internal.h"

namespace qmm {
namespace {

constexpr int kThreads = 256;
constexpr int BK = 32;

// Element i of an array of type t, in fp32 (exact).
__device__ __forceinline__ float load_elem(const void *p, int t, int64_t i) {
  if (t == kTypeF32) return __ldg(static_cast<const float *>(p) + i);
  const uint32_t h = __ldg(static_cast<const uint16_t *>(p) + i);
  return t == kTypeF16 ? ElemF16::to_f32(h) : ElemBF16::to_f32(h);
}

// Elements i .. i+3 of an array of type t (i a multiple of 4, 16-byte
// aligned rows), in fp32.
__device__ __forceinline__ float4 load4(const void *p, int t, int64_t i) {
  if (t == kTypeF32) return __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(p) + i));
  const uint2 u = __ldg(reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(p) + i));
  if (t == kTypeF16)
    return make_float4(ElemF16::to_f32(u.x & 0xFFFFu), ElemF16::to_f32(u.x >> 16),
                       ElemF16::to_f32(u.y & 0xFFFFu), ElemF16::to_f32(u.y >> 16));
  return make_float4(ElemBF16::to_f32(u.x & 0xFFFFu), ElemBF16::to_f32(u.x >> 16),
                     ElemBF16::to_f32(u.y & 0xFFFFu), ElemBF16::to_f32(u.y >> 16));
}

struct MmArgs {
  const void *x;
  int x_type;
  const uint32_t *w;
  const uint16_t *scales, *biases;  // of sb_type (fp32 values when kTypeF32)
  int sb_type;
  float *y;  // [M, N], or the partials [gridDim.z, M, N]
  int M, N, K, group_shift;
  int steps_per_split;  // k-steps per z slice
};

// The codes of one octet with their scale and bias; s = b = 0 outside W.
struct Octet {
  uint32_t lo, hi, sh;
  float s, b;
};

template <int BITS, bool TRANS>
__device__ __forceinline__ Octet fetch_octet(const MmArgs &a, int row, int col) {
  Octet o{0u, 0u, 0u, 0.0f, 0.0f};
  const int rows = TRANS ? a.N : a.K, cols = TRANS ? a.K : a.N;
  if (row < rows && col < cols) {
    const int64_t wpr = (static_cast<int64_t>(cols) * BITS) >> 5;
    const int64_t bit = static_cast<int64_t>(col) * BITS;
    const uint32_t *rp = a.w + static_cast<int64_t>(row) * wpr + (bit >> 5);
    o.sh = static_cast<uint32_t>(bit & 31);
    o.lo = __ldg(rp);
    // The octet ends inside the row (cols is a multiple of 32), so a second
    // word it needs is a word of the row.
    if (o.sh + 8 * BITS > 32) o.hi = __ldg(rp + 1);
    const int64_t g = static_cast<int64_t>(row) * (cols >> a.group_shift) + (col >> a.group_shift);
    o.s = load_elem(a.scales, a.sb_type, g);
    o.b = load_elem(a.biases, a.sb_type, g);
  }
  return o;
}

template <int BITS>
__device__ __forceinline__ void dequant_octet(const Octet &o, float (&v)[8]) {
  const uint64_t win = (static_cast<uint64_t>(o.hi) << 32 | o.lo) >> o.sh;
  constexpr uint32_t mask = (1u << BITS) - 1u;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    v[i] = __fmaf_rn(o.s, static_cast<float>(static_cast<uint32_t>(win >> (BITS * i)) & mask), o.b);
}

template <int BITS, int BM, int BN, int PF, bool TRANS>
__global__ void __launch_bounds__(kThreads) mm_f32_kernel(MmArgs a) {
  constexpr int TM = BM / 16, TN = BN / 16;      // micro-tile of a thread (16 x 16 threads)
  constexpr int XPITCH = BM + 4;                  // Xs rows stay 16-byte aligned
  constexpr int XPER = BM * BK / kThreads;        // x values a thread stages per step
  constexpr int OCT = BN * BK / (8 * kThreads);   // octets a thread dequantizes per step
  static_assert(TN == 4 || TN == 8, "micro-tile width");
  static_assert(TM == 1 || TM % 4 == 0, "micro-tile height");
  __shared__ __align__(16) float Xs[BK][XPITCH];
  __shared__ __align__(16) float Ws[BK][BN];
  const int t = threadIdx.x, tm = t / 16, tn = t % 16;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int nk = (a.K + BK - 1) / BK;
  const int kb0 = blockIdx.z * a.steps_per_split;
  const int kb1 = min(nk, kb0 + a.steps_per_split);

  // Octet j of thread t: stored row and column of its first code, and where
  // its 8 weights go in Ws.
  auto octet_place = [&](int kb, int j, int &row, int &col, int &wk, int &wn) {
    const int o = t + kThreads * j;
    if (TRANS) {  // W [N, K]: 4 octets per row of the step
      const int r = o % BN, q = o / BN;
      row = n0 + r;
      col = kb * BK + 8 * q;
      wk = 8 * q;
      wn = r;
    } else {  // W [K, N]: BN / 8 octets per stored row
      const int kr = o / (BN / 8), h = o % (BN / 8);
      row = kb * BK + kr;
      col = n0 + 8 * h;
      wk = kr;
      wn = 8 * h;
    }
  };
  // Ring stage p holds step kb0 + PF*i + p for the i-th turn of the loop.
  Octet oct[PF][OCT];
  float xr[PF][XPER];
  auto fetch = [&](int kb, Octet (&oc)[OCT], float (&xv)[XPER]) {
#pragma unroll
    for (int j = 0; j < OCT; ++j) {
      int row, col, wk, wn;
      octet_place(kb, j, row, col, wk, wn);
      oc[j] = fetch_octet<BITS, TRANS>(a, row, col);
    }
#pragma unroll
    for (int j = 0; j < XPER; ++j) {
      const int e = t + kThreads * j, m = e / BK, k = e % BK;
      const int gm = m0 + m, gk = kb * BK + k;
      xv[j] = (gm < a.M && gk < a.K) ? load_elem(a.x, a.x_type, static_cast<int64_t>(gm) * a.K + gk)
                                     : 0.0f;
    }
  };

  float acc[TM][TN];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) acc[i][j] = 0.0f;

#pragma unroll
  for (int p = 0; p < PF; ++p)
    if (kb0 + p < kb1) fetch(kb0 + p, oct[p], xr[p]);
  for (int kbase = kb0; kbase < kb1; kbase += PF) {
#pragma unroll
    for (int p = 0; p < PF; ++p) {
      const int kb = kbase + p;
      if (kb >= kb1) break;
      __syncthreads();  // the previous step's reads of Xs and Ws are done
#pragma unroll
      for (int j = 0; j < OCT; ++j) {
        int row, col, wk, wn;
        octet_place(kb, j, row, col, wk, wn);
        float v[8];
        dequant_octet<BITS>(oct[p][j], v);
        if (TRANS) {
#pragma unroll
          for (int i = 0; i < 8; ++i) Ws[wk + i][wn] = v[i];
        } else {
          *reinterpret_cast<float4 *>(&Ws[wk][wn]) = make_float4(v[0], v[1], v[2], v[3]);
          *reinterpret_cast<float4 *>(&Ws[wk][wn + 4]) = make_float4(v[4], v[5], v[6], v[7]);
        }
      }
#pragma unroll
      for (int j = 0; j < XPER; ++j) {
        const int e = t + kThreads * j;
        Xs[e % BK][e / BK] = xr[p][j];
      }
      __syncthreads();
      if (kb + PF < kb1) fetch(kb + PF, oct[p], xr[p]);  // in flight while PF steps compute
#pragma unroll 4
      for (int k = 0; k < BK; ++k) {
        float av[TM], bv[TN];
        if constexpr (TM == 1) {
          av[0] = Xs[k][tm];
        } else {
#pragma unroll
          for (int i = 0; i < TM; i += 4) {
            const float4 u = *reinterpret_cast<const float4 *>(&Xs[k][tm * TM + i]);
            av[i] = u.x; av[i + 1] = u.y; av[i + 2] = u.z; av[i + 3] = u.w;
          }
        }
#pragma unroll
        for (int j = 0; j < TN; j += 4) {
          const float4 u = *reinterpret_cast<const float4 *>(&Ws[k][tn * TN + j]);
          bv[j] = u.x; bv[j + 1] = u.y; bv[j + 2] = u.z; bv[j + 3] = u.w;
        }
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
          for (int j = 0; j < TN; ++j) acc[i][j] = __fmaf_rn(av[i], bv[j], acc[i][j]);
      }
    }
  }

  float *out = a.y + static_cast<int64_t>(blockIdx.z) * a.M * a.N;
#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int m = m0 + tm * TM + i;
    if (m >= a.M) break;
#pragma unroll
    for (int j = 0; j < TN; ++j) {
      const int n = n0 + tn * TN + j;
      if (n < a.N) out[static_cast<int64_t>(m) * a.N + n] = acc[i][j];
    }
  }
}

// Decode form (M <= 16, W stored [N, K]): no shared-memory round trip for the
// weights.  A block owns 32 rows of W and a K slice of at most kGemvSteps steps
// of 64 codes; thread (r, q) = (t / 8, t % 8) takes octet q of every step of
// row r (the 8 threads of a row read its 64 codes of a step as consecutive
// words), issues all of its octets' loads at once, then dequantizes each
// octet and multiplies it into MT accumulators against x, which the block
// stages in shared memory once (MT x slice, fp32).  The 8 partial sums of a
// row meet by warp shuffles.  At M = 16 the x reads from shared memory bound
// the kernel, so x is laid out for conflict-free reads (see the staging).
constexpr int kGemvSteps = 8;  // 64-code steps per block at most (512 codes)

template <int BITS, int MT>
__global__ void __launch_bounds__(kThreads) mm_f32_gemv_kernel(MmArgs a) {
  constexpr int KS = 64 * kGemvSteps;
  __shared__ __align__(16) float xs[MT][KS];
  const int t = threadIdx.x, r = t >> 3, q = t & 7;
  const int n = blockIdx.x * 32 + r;
  const int kb0 = blockIdx.z * a.steps_per_split;  // first 64-code step
  const int nsteps = min(a.steps_per_split, (a.K + 63) / 64 - kb0);
  Octet oct[kGemvSteps];
#pragma unroll
  for (int i = 0; i < kGemvSteps; ++i) {
    oct[i] = Octet{0u, 0u, 0u, 0.0f, 0.0f};
    if (i < nsteps) oct[i] = fetch_octet<BITS, true>(a, n, (kb0 + i) * 64 + 8 * q);
  }
  // x rows of the slice, widened exactly (zero beyond M and K), four values
  // a load; every load is issued before the first store.
  const int k0 = kb0 * 64;
  constexpr int NV = MT * KS / 4, NJ = (NV + kThreads - 1) / kThreads;
  float4 xv[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int e = 4 * (t + kThreads * j), m = e / KS, k = e - m * KS;
    xv[j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (e < MT * KS && m < a.M && k < nsteps * 64 && k0 + k < a.K)
      xv[j] = load4(a.x, a.x_type, static_cast<int64_t>(m) * a.K + k0 + k);
  }
  // Within each 64-value step, value 8q + 4h + j (octet q, half h) sits at
  // 32h + 4q + j: the 8 threads of a row then read 128 contiguous bytes per
  // half, one shared-memory wavefront without bank conflicts.
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int e = 4 * (t + kThreads * j);
    if (e < MT * KS) {
      const int k = e % KS, rem = k & 63;
      const int pos = (k & ~63) + 32 * ((rem >> 2) & 1) + 4 * (rem >> 3);
      *reinterpret_cast<float4 *>(&xs[e / KS][pos]) = xv[j];
    }
  }
  __syncthreads();
  float acc[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) acc[m] = 0.0f;
#pragma unroll
  for (int i = 0; i < kGemvSteps; ++i) {
    if (i < nsteps) {
      float v[8];
      dequant_octet<BITS>(oct[i], v);
      const int kk = 64 * i + 4 * q;  // the octet's two halves, permuted as staged
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const float4 x0 = *reinterpret_cast<const float4 *>(&xs[m][kk]);
        const float4 x1 = *reinterpret_cast<const float4 *>(&xs[m][kk + 32]);
        float s = acc[m];
        s = __fmaf_rn(v[0], x0.x, s); s = __fmaf_rn(v[1], x0.y, s);
        s = __fmaf_rn(v[2], x0.z, s); s = __fmaf_rn(v[3], x0.w, s);
        s = __fmaf_rn(v[4], x1.x, s); s = __fmaf_rn(v[5], x1.y, s);
        s = __fmaf_rn(v[6], x1.z, s); s = __fmaf_rn(v[7], x1.w, s);
        acc[m] = s;
      }
    }
  }
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    float s = acc[m];
    s += __shfl_xor_sync(0xffffffffu, s, 4);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    acc[m] = s;
  }
  if (q == 0 && n < a.N) {
    float *out = a.y + static_cast<int64_t>(blockIdx.z) * a.M * a.N;
#pragma unroll
    for (int m = 0; m < MT; ++m)
      if (m < a.M) out[static_cast<int64_t>(m) * a.N + n] = acc[m];
  }
}

// y = the sum of the `splits` partial slices, in slice order.
__global__ void __launch_bounds__(256)
mm_f32_finalize(const float *__restrict__ ws, int splits, int64_t mn, float *__restrict__ y) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < mn; i += stride) {
    float acc = ws[i];
    for (int s = 1; s < splits; ++s) acc += ws[s * mn + i];
    y[i] = acc;
  }
}

// Launch kern over grid (gx, gy, splits) with a.steps_per_split steps a
// slice; partials through a stream-ordered workspace when splits > 1.
template <typename Kern>
cudaError_t launch_split(Kern kern, MmArgs a, unsigned gx, unsigned gy, int nk, int splits,
                         cudaStream_t stream) {
  a.steps_per_split = (nk + splits - 1) / splits;
  splits = (nk + a.steps_per_split - 1) / a.steps_per_split;
  float *y = a.y;
  float *ws = nullptr;
  const int64_t mn = static_cast<int64_t>(a.M) * a.N;
  if (splits > 1) {
    void *p = nullptr;
    if (cudaMallocAsync(&p, static_cast<size_t>(splits) * mn * sizeof(float), stream) != cudaSuccess) {
      cudaGetLastError();
      return cudaErrorMemoryAllocation;
    }
    ws = static_cast<float *>(p);
    a.y = ws;
  }
  kern<<<dim3(gx, gy, splits), kThreads, 0, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (ws) {
    if (e == cudaSuccess) {
      int64_t blocks = (mn + 255) / 256;
      if (blocks > 4 * sm_count()) blocks = 4 * sm_count();
      mm_f32_finalize<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(ws, splits, mn, y);
      e = cudaGetLastError();
    }
    const cudaError_t fe = cudaFreeAsync(ws, stream);
    if (e == cudaSuccess) e = fe;
  }
  return e;
}

template <int BITS, int BM, int BN, int PF, bool TRANS>
cudaError_t launch_cfg(const MmArgs &a, cudaStream_t stream) {
  const int64_t mt = (a.M + BM - 1) / BM, nt = (a.N + BN - 1) / BN;
  if (mt > 65535) return cudaErrorInvalidValue;
  const int nk = (a.K + BK - 1) / BK;
  // Split K until the blocks cover the SMs four times, keeping at least PF
  // (and 4) steps a slice.
  const int64_t want = 4 * static_cast<int64_t>(sm_count());
  const int min_steps = PF > 4 ? PF : 4;
  int splits = 1;
  if (mt * nt < want) {
    splits = static_cast<int>((want + mt * nt - 1) / (mt * nt));
    if (splits > nk / min_steps) splits = nk / min_steps;
    if (splits > 64) splits = 64;
    if (splits < 1) splits = 1;
  }
  cudaError_t e = launch_split(mm_f32_kernel<BITS, BM, BN, PF, TRANS>, a, static_cast<unsigned>(nt),
                               static_cast<unsigned>(mt), nk, splits, stream);
  if (e == cudaErrorMemoryAllocation && splits > 1)  // no workspace: one slice
    e = launch_split(mm_f32_kernel<BITS, BM, BN, PF, TRANS>, a, static_cast<unsigned>(nt),
                     static_cast<unsigned>(mt), nk, 1, stream);
  return e;
}

// The decode form: slices of at most kGemvSteps 64-code steps, so K is always
// split when it exceeds 512 (the workspace is then required).
template <int BITS, int MT>
cudaError_t launch_gemv_cfg(const MmArgs &a, cudaStream_t stream) {
  const int nk = (a.K + 63) / 64;
  const int splits = (nk + kGemvSteps - 1) / kGemvSteps;
  return launch_split(mm_f32_gemv_kernel<BITS, MT>, a, static_cast<unsigned>((a.N + 31) / 32), 1u,
                      nk, splits, stream);
}

template <int BITS>
cudaError_t launch_bits(const MmArgs &a, bool transpose, cudaStream_t stream) {
  if (a.M <= 16 && transpose) {
    const cudaError_t e = a.M == 1   ? launch_gemv_cfg<BITS, 1>(a, stream)
                          : a.M <= 4 ? launch_gemv_cfg<BITS, 4>(a, stream)
                          : a.M <= 8 ? launch_gemv_cfg<BITS, 8>(a, stream)
                                     : launch_gemv_cfg<BITS, 16>(a, stream);
    // Without the slices' workspace the tiled form runs K unsplit.
    if (e != cudaErrorMemoryAllocation) return e;
    return launch_cfg<BITS, 16, 128, 6, true>(a, stream);
  }
  if (a.M <= 16) return launch_cfg<BITS, 16, 128, 6, false>(a, stream);
  return transpose ? launch_cfg<BITS, 128, 128, 1, true>(a, stream)
                   : launch_cfg<BITS, 128, 128, 1, false>(a, stream);
}

}  // namespace

cudaError_t launch_mm_f32(const void *x, int x_type, int64_t M, const PackedWeight &w,
                          bool transpose, float *y, cudaStream_t stream) {
  MmArgs a;
  a.x = x;
  a.x_type = x_type;
  a.w = w.w;
  a.scales = w.scales;
  a.biases = w.biases;
  a.sb_type = w.sb_type;
  a.y = y;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(transpose ? w.rows : w.cols);
  a.K = static_cast<int>(transpose ? w.cols : w.rows);
  a.group_shift = w.group == 32 ? 5 : w.group == 64 ? 6 : 7;
  a.steps_per_split = 0;
  switch (w.bits) {
    case 1: return launch_bits<1>(a, transpose, stream);
    case 2: return launch_bits<2>(a, transpose, stream);
    case 3: return launch_bits<3>(a, transpose, stream);
    case 4: return launch_bits<4>(a, transpose, stream);
    case 5: return launch_bits<5>(a, transpose, stream);
    case 6: return launch_bits<6>(a, transpose, stream);
    case 8: return launch_bits<8>(a, transpose, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qmm
