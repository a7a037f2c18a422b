// Decode path of quantized_matmul for weights with many 16-row tiles:
// transposed W [N, K] of 1- to 3-bit codes, M <= 8, bf16 x / scales / biases,
// K a multiple of 128 up to 4096 (nuvec_core quantized.rs, `quantized_matmul`; spark_runtime
// weights/mlx_int8.rs, `gemv`, x shared across rows).
//
// The one-wave decode kernel gives each block one 16-row tile and streams it
// in at kernel start; with more tiles than two blocks an SM can hold, its
// later waves each pay the full HBM latency before they compute.  Here a
// block stays resident and walks tiles b, b + grid, ...: a producer warp
// keeps the next tiles in flight by TMA, each tile whole (its 16 rows of
// packed codes as row-long boxes, so every row is read as one contiguous run,
// then the rows' scales and biases) into one of a few tile slots, while the
// 16 consumer warps dequantize and multiply the tile that has landed.
//
//   warps 0-15  consumers: warp w takes 128-code chunks w, w + 16, ... of
//               each tile; lane (g, t) handles codes [32t, 32t+32) of rows g
//               and g+8 (16 pairs a row, RN_bf16(s*c + b) each), mma.sync
//               m16n8k16 against x in natural pairs; per tile the warps'
//               partials are added in warp order by one warp and stored
//   warp 16     producer: per tile, the code boxes ([16 rows x up to 2 KiB])
//               and the scale and bias boxes ([16 x K/G]) into the next slot
//
// The weights and scales stream before griddepcontrol.wait; x is read after
// it.  Every wait is bounded; after one runs out the block's waits all fail
// at once, the warps finish their tiles without waiting (the output is then
// undefined) and the producer waits for its copies in flight.
#include "gemv_impl.cuh"

namespace qmm {
namespace {

constexpr int kStWarps = 16;                          // consumer warps
constexpr int kStThreads = 32 * (kStWarps + 1);       // + the producer warp
constexpr int kStMaxSlots = 8;                        // tile slots
constexpr int kStChunks = 2;                          // 128-code chunks a warp takes per tile (K <= 4096)
constexpr size_t kStSmemBudget = 220 * 1024;          // one block an SM

struct StreamArgs {
  const uint16_t *x;
  void *y;
  int M, N, K;
  int group_shift;
  int tiles;       // 16-row tiles of W
  int nch;         // 128-code chunks of a row
  int slots;       // tile slots
  int slot_bytes;  // one slot: codes, then scales, then biases
  int box_bytes;   // bytes of a row in one code box (a code box is 16 rows of it)
  int nbox;        // code boxes per tile
  int sb_off;      // offset of the scales in a slot (the biases follow, sb_bytes on)
  int sb_bytes;    // 16 rows x K/G x 2 bytes
  int red_off, bar_off;
  uint32_t spin_limit;
};

struct StreamBars {
  uint64_t full[kStMaxSlots], empty[kStMaxSlots];
  int abort;
};

// Bounded wait of one warp (warp-uniform result); false once any wait of the
// block has run out.
__device__ __forceinline__ bool st_wait(uint64_t *b, uint32_t parity, StreamBars *bars,
                                        uint32_t limit, unsigned *err) {
  volatile int *abort = &bars->abort;
  uint32_t spins = 0;
  while (true) {
    if (__all_sync(0xffffffffu, mbar_try_wait(b, parity))) return true;
    if (__any_sync(0xffffffffu, *abort != 0)) return false;
    if (++spins >= limit) {
      if ((threadIdx.x & 31) == 0) {
        *abort = 1;
        atomicOr(err, kErrTimeoutBit);
      }
      __syncwarp();
      return false;
    }
  }
}

__device__ __forceinline__ void st_tma(uint32_t dst, const CUtensorMap *map, int x, int y,
                                       uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

template <int BITS, bool OUT_BF16>
__global__ void __launch_bounds__(kStThreads, 1)
gemv_stream_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap smap,
                   const __grid_constant__ CUtensorMap bmap, StreamArgs a, unsigned *err) {
  using E = ElemBF16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  StreamBars *bars = reinterpret_cast<StreamBars *>(smem + a.bar_off);
  float *red = reinterpret_cast<float *>(smem + a.red_off);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    for (int i = 0; i < a.slots; ++i) {
      mbar_init(&bars->full[i], 1);
      mbar_init(&bars->empty[i], kStWarps);
    }
    bars->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  griddep_launch_dependents();

  if (warp == kStWarps) {
    // Producer.  The weights do not depend on the previous kernel.
    int slot = 0, issued = 0;
    uint32_t ph = 0;
    for (int tile = blockIdx.x; tile < a.tiles; tile += gridDim.x) {
      if (!st_wait(&bars->empty[slot], ph ^ 1u, bars, a.spin_limit, err)) break;
      if (lane == 0) {
        const uint32_t dst = smem_u32(smem + slot * a.slot_bytes);
        mbar_expect_tx(&bars->full[slot], 16 * a.box_bytes * a.nbox + 2 * a.sb_bytes);
        for (int j = 0; j < a.nbox; ++j)
          st_tma(dst + j * 16 * a.box_bytes, &wmap, j * (a.box_bytes / 8), tile * 16, &bars->full[slot]);
        st_tma(dst + a.sb_off, &smap, 0, tile * 16, &bars->full[slot]);
        st_tma(dst + a.sb_off + a.sb_bytes, &bmap, 0, tile * 16, &bars->full[slot]);
      }
      ++issued;
      if (++slot == a.slots) { slot = 0; ph ^= 1u; }
    }
    // After a stop: wait (bounded) for the copies still in flight, the last
    // tile issued into each slot (tile loads n = 0 .. issued-1 went to slot
    // n % slots).
    if (bars->abort) {
      for (int i = 0; i < a.slots && i < issued; ++i) {
        const int n = issued - 1 - ((issued - 1 - i) % a.slots);
        const uint32_t p = static_cast<uint32_t>(n / a.slots) & 1u;
        for (uint32_t s = 0; s < kDefaultWaitLimit; ++s)
          if (__all_sync(0xffffffffu, mbar_try_wait(&bars->full[i], p))) break;
      }
    }
    return;
  }

  // Consumers.  x may be written by the previous kernel in the stream.  A
  // warp's chunks are the same in every tile, so its x fragments are read
  // once (lanes whose x row is past M keep zeros).
  griddep_wait();
  const int g = lane >> 2, t = lane & 3;
  const int groups = a.K >> a.group_shift;
  uint32_t xr[kStChunks][16];
#pragma unroll
  for (int j = 0; j < kStChunks; ++j) {
    const int c = warp + kStWarps * j;
#pragma unroll
    for (int i = 0; i < 16; ++i) xr[j][i] = 0u;
    if (g < a.M && c < a.nch) {
      const uint4 *xp = reinterpret_cast<const uint4 *>(a.x + static_cast<int64_t>(g) * a.K + (c << 7) + 32 * t);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 u = __ldg(xp + i);
        xr[j][4 * i] = u.x; xr[j][4 * i + 1] = u.y; xr[j][4 * i + 2] = u.z; xr[j][4 * i + 3] = u.w;
      }
    }
  }
  int slot = 0;
  uint32_t ph = 0;
  for (int tile = blockIdx.x, it = 0; tile < a.tiles; tile += gridDim.x, ++it) {
    st_wait(&bars->full[slot], ph, bars, a.spin_limit, err);
    const uint8_t *sl = smem + slot * a.slot_bytes;
    const uint16_t *ss = reinterpret_cast<const uint16_t *>(sl + a.sb_off);
    const uint16_t *bs = ss + a.sb_bytes / 2;
    float acc[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
#pragma unroll
    for (int j = 0; j < kStChunks; ++j) {
      const int c = warp + kStWarps * j;
      if (c >= a.nch) break;
      const uint32_t (&xv)[16] = xr[j];
      const int gi = ((c << 7) + 32 * t) >> a.group_shift;
      const uint32_t s0 = ss[g * groups + gi], b0h = bs[g * groups + gi];
      const uint32_t s1 = ss[(g + 8) * groups + gi], b1h = bs[(g + 8) * groups + gi];
      // Chunk c of a row: bytes [16*bits*c, 16*bits*(c+1)), inside code box jb.
      const int cb = c * 16 * BITS;
      const int jb = cb / a.box_bytes, o = cb - jb * a.box_bytes;
      const uint8_t *r0 = sl + jb * 16 * a.box_bytes + g * a.box_bytes + o + t * 4 * BITS;
      uint32_t v0[BITS], v1[BITS];
      lds_words<BITS>(r0, v0);
      lds_words<BITS>(r0 + 8 * a.box_bytes, v1);
      const uint32_t b0 = bcast2(b0h), b1 = bcast2(b1h);
      const bool fast = __all_sync(0xffffffffu, fast_scale(s0) && fast_scale(s1));
      if (fast) {
        uint32_t m0[fast_slots<BITS>()], m1[fast_slots<BITS>()];
        fast_muls<BITS>(s0, m0);
        fast_muls<BITS>(s1, m1);
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const uint32_t a0 = pair_fast<BITS>(v0, 2 * r, m0, b0), a2 = pair_fast<BITS>(v0, 2 * r + 1, m0, b0);
          const uint32_t a1 = pair_fast<BITS>(v1, 2 * r, m1, b1), a3 = pair_fast<BITS>(v1, 2 * r + 1, m1, b1);
          mma_16816<E>(acc[r & 1], a0, a1, a2, a3, xv[2 * r], xv[2 * r + 1]);
        }
      } else {
        const uint32_t s0p = bcast2(s0), s1p = bcast2(s1);
        const float fs0 = E::to_f32(s0), fb0 = E::to_f32(b0h);
        const float fs1 = E::to_f32(s1), fb1 = E::to_f32(b1h);
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const uint32_t a0 = pair_exact<BITS, E>(v0, 2 * r, s0p, b0, fs0, fb0);
          const uint32_t a2 = pair_exact<BITS, E>(v0, 2 * r + 1, s0p, b0, fs0, fb0);
          const uint32_t a1 = pair_exact<BITS, E>(v1, 2 * r, s1p, b1, fs1, fb1);
          const uint32_t a3 = pair_exact<BITS, E>(v1, 2 * r + 1, s1p, b1, fs1, fb1);
          mma_16816<E>(acc[r & 1], a0, a1, a2, a3, xv[2 * r], xv[2 * r + 1]);
        }
      }
    }
    // Every word and scale this warp needs from the slot has been read.
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->empty[slot]);
    if (++slot == a.slots) { slot = 0; ph ^= 1u; }
    // The tile's partials: red[it % 2][warp][i][lane]; after the consumers'
    // barrier, warp (it % 16) adds them in warp order and stores y.
    float *rt = red + (it & 1) * (kStWarps * 4 * 32);
#pragma unroll
    for (int i = 0; i < 4; ++i) rt[(warp * 4 + i) * 32 + lane] = acc[0][i] + acc[1][i];
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kStWarps) : "memory");
    if (warp == (it & (kStWarps - 1))) {
      const int n0 = tile * 16;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float s = 0.0f;
        for (int w = 0; w < kStWarps; ++w) s += rt[(w * 4 + i) * 32 + lane];
        const int n = n0 + g + 8 * (i >> 1), m = 2 * t + (i & 1);
        if (m < a.M && n < a.N) {
          const int64_t o = static_cast<int64_t>(m) * a.N + n;
          if (OUT_BF16) static_cast<uint16_t *>(a.y)[o] = f32_to_bf16_bits(s);
          else static_cast<float *>(a.y)[o] = s;
        }
      }
    }
  }
}

template <int BITS, bool OUT_BF16>
cudaError_t launch_stream(const uint16_t *x, int M, const PackedWeight &w, void *y, bool pdl,
                          cudaStream_t stream) {
  StreamArgs a{};
  a.x = x;
  a.y = y;
  a.M = M;
  a.N = static_cast<int>(w.rows);
  a.K = static_cast<int>(w.cols);
  a.group_shift = w.group == 32 ? 5 : w.group == 64 ? 6 : 7;
  a.tiles = (a.N + 15) / 16;
  a.nch = a.K / 128;
  if (a.nch > kStWarps * kStChunks) return cudaErrorNotSupported;
  // Code boxes of at most 256 8-byte elements (2 KiB) of a row; a chunk
  // (16*bits bytes) never straddles two of them.
  const int row_bytes = a.K / 8 * BITS;
  a.box_bytes = row_bytes <= 2048 ? row_bytes : 2048;
  if (row_bytes % a.box_bytes != 0 || a.box_bytes % (16 * BITS) != 0) return cudaErrorNotSupported;
  a.nbox = row_bytes / a.box_bytes;
  const int groups = a.K >> a.group_shift;
  a.sb_bytes = 16 * groups * 2;
  a.sb_off = 16 * row_bytes;
  a.slot_bytes = (a.sb_off + 2 * a.sb_bytes + 127) & ~127;
  const size_t fixed = 2 * kStWarps * 4 * 32 * 4 + sizeof(StreamBars) + 1024 + 64;
  int slots = static_cast<int>((kStSmemBudget - fixed) / a.slot_bytes);
  if (slots > kStMaxSlots) slots = kStMaxSlots;
  if (slots < 2) return cudaErrorNotSupported;
  a.slots = slots;
  a.red_off = slots * a.slot_bytes;
  a.bar_off = (a.red_off + 2 * kStWarps * 4 * 32 * 4 + 15) & ~15;
  a.spin_limit = wait_limit();
  const size_t smem = static_cast<size_t>(a.bar_off) + sizeof(StreamBars) + 1024;
  CUtensorMap wmap, smap, bmap;
  cudaError_t e = encode_map_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT64, w.w, row_bytes / 8, a.N,
                                row_bytes, a.box_bytes / 8, 16, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return cudaErrorNotSupported;
  e = encode_map_2d(&smap, CU_TENSOR_MAP_DATA_TYPE_UINT16, w.scales, groups, a.N, groups * 2, groups,
                    16, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return cudaErrorNotSupported;
  e = encode_map_2d(&bmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, w.biases, groups, a.N, groups * 2, groups,
                    16, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return cudaErrorNotSupported;
  unsigned *err = device_error_word();
  if (!err) return cudaErrorInvalidSymbol;
  e = ensure_smem_limit<gemv_stream_kernel<BITS, OUT_BF16>>(smem);
  if (e != cudaSuccess) return e;
  const int grid = a.tiles < sm_count() ? a.tiles : sm_count();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kStThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemv_stream_kernel<BITS, OUT_BF16>, wmap, smap, bmap, a, err);
}

}  // namespace

cudaError_t launch_gemv_stream(const uint16_t *x, int64_t M, const PackedWeight &w, void *y,
                               bool y_bf16, bool pdl, cudaStream_t stream) {
  if (M < 1 || M > 8 || w.cols % 128 != 0 || w.sb_type != kTypeBF16 || w.rows >= (int64_t(1) << 31))
    return cudaErrorNotSupported;
  const int64_t groups = w.cols / w.group;
  // TMA: 16-byte aligned arrays, scale rows of whole 16-byte units, one box
  // across a row of scales.
  if (groups % 8 != 0 || groups > 256 || (reinterpret_cast<uintptr_t>(x) & 15u) != 0 ||
      (reinterpret_cast<uintptr_t>(w.w) & 15u) != 0 ||
      (reinterpret_cast<uintptr_t>(w.scales) & 15u) != 0 ||
      (reinterpret_cast<uintptr_t>(w.biases) & 15u) != 0)
    return cudaErrorNotSupported;
  const int Mi = static_cast<int>(M);
  switch (w.bits) {
    case 1: return y_bf16 ? launch_stream<1, true>(x, Mi, w, y, pdl, stream) : launch_stream<1, false>(x, Mi, w, y, pdl, stream);
    case 2: return y_bf16 ? launch_stream<2, true>(x, Mi, w, y, pdl, stream) : launch_stream<2, false>(x, Mi, w, y, pdl, stream);
    case 3: return y_bf16 ? launch_stream<3, true>(x, Mi, w, y, pdl, stream) : launch_stream<3, false>(x, Mi, w, y, pdl, stream);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace qmm
