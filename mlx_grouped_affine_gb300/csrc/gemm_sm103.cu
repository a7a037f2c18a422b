// Prefill path of quantized_matmul (M > 16) on the sm_103a tensor cores.
//
// y = x . dequant(W)^T (nuvec_core quantized.rs, `quantized_matmul`;
// spark_runtime weights/mlx_int8.rs, `gemm`, whose naive kernel this
// replaces).  The dequantized weight is never written to global memory: each
// 256-row x 64-code tile of W is dequantized straight into shared memory,
// where the tensor cores read it.
//
// The element type E of x and of the dequantized weight is bf16, or fp16 for
// fp16 x, scales and biases (kind::f16 takes either, the same for A and B).
// One persistent block per SM walks output tiles of 256 x-rows by 256
// weight-rows.  Each dequantized W tile feeds two 128-row MMAs (the two x
// halves), which halves the dequantization work per tensor-core flop
// compared with a 128-row tile.  Its warps specialise:
//   warp 0      TMA: x tiles [256 x 64] of E into a 128-byte-swizzled ring
//   warp 1      allocates tensor memory and issues tcgen05.mma (one lane):
//               D[2 x 128 x 256] fp32 in TMEM (all 512 columns)
//   warps 2-5   epilogue: tcgen05.ld of the accumulators, convert, store y
//               (32-byte stores where the rows allow), or fp32 split-K partials
//   warps 6-21  dequantize: packed W -> E (one rounding per weight,
//               RN(scale * code + bias)), 32 codes a thread per stage, written
//               in the same 128-byte swizzle the MMA descriptor expects, then
//               fence.proxy.async and arrive; the packed codes of the next two
//               stages are kept in flight
// Stage hand-off uses mbarriers; every wait is bounded, and a wait that runs
// out sets the device error word, makes every role stop, and the block still
// waits for its own copies and MMAs and frees its tensor memory.
//
// Units are (output tile, K range) pairs: split-K when the tiles are too few
// for the SMs, and in grouped mode (gather_qmm over sorted expert runs) the
// row tiles come from a plan made on the device (see launch_gemm_grouped).
//
// Shared-memory tiles are K-major with the 128-byte swizzle: row r of a tile
// is 128 bytes (64 16-bit values) at r*128, and its 16-byte chunk c sits at chunk
// position c ^ (r % 8).  The UMMA descriptor gives stride 1024 bytes between
// 8-row groups; a 16-wide K step inside the 64-wide atom advances the start
// address by 32 bytes.
#include "common.cuh"
#include "internal.h"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

namespace qmm {
namespace {

constexpr int UM = 128;   // rows of one MMA (x rows)
constexpr int BM = 2 * UM; // x rows per tile: two MMAs share each dequantized W tile
constexpr int BN = 256;   // weight rows per tile (MMA N)
constexpr int BK = 64;    // codes per stage: one 128-byte swizzle atom of bf16
// Separate rings for the x tiles and the dequantized W tiles.  Measured on
// the 2048 x 14336 x 4096 and 128 x 4096 x 14336 cases: two or three W
// stages run as fast as four (the dequant warps, not the ring, set the
// pace), and the shared memory left to L1 serves their loads.
constexpr int SA = 2;  // x stages
constexpr int SB = 3;  // W stages
constexpr int kEpiWarps = 4;
constexpr int kDeqWarps = 16;  // one 32-code item of a stage per thread
constexpr int kLoadAhead = 2;  // stages of packed codes in flight per dequant thread
static_assert(32 * kDeqWarps == BN * BK / 32, "one item per dequant thread");
// TMA-fed dequant (W stored [N, K] at an even width whose rows and groups
// TMA can address): warp 2 + kEpiWarps + kDeqWarps stages each k-block's
// packed codes [BN rows x 64 codes] and, every kSbWin groups, a window of
// the tile rows' scales and biases in shared memory; the dequant warps read
// their items there instead of from global memory (per-thread global loads
// of 16-32 bytes from 16 rows a warp cost L1 a wavefront per row).
constexpr int kSbWin = 8;                               // groups per scale/bias window
constexpr int SS = 2;                                   // scale/bias window slots
constexpr uint32_t SB_WIN_BYTES = 2 * BN * kSbWin * 2;  // scales [BN][8], then biases
constexpr int kMaxPStages = 4;
template <int BITS>
__host__ __device__ constexpr uint32_t p_bytes() { return BN * 8 * BITS; }  // one k-block of codes
template <int BITS>
__host__ __device__ constexpr int p_stages() {
  return 49152 / p_bytes<BITS>() < kMaxPStages ? 49152 / p_bytes<BITS>() : kMaxPStages;
}
template <bool WTMA>
__host__ __device__ constexpr int gemm_threads() {
  return 32 * (2 + kEpiWarps + kDeqWarps + (WTMA ? 1 : 0));
}
constexpr uint32_t A_BYTES = BM * BK * 2;
constexpr uint32_t A_HALF = UM * BK * 2;
constexpr uint32_t B_BYTES = BN * BK * 2;
constexpr uint32_t TMEM_COLS = 2 * BN;  // accumulators of the two x halves
constexpr uint32_t kSpinLimit = 1u << 24;

struct Barriers {
  uint64_t full_a[SA], empty_a[SA], full_b[SB], empty_b[SB];
  uint64_t full_p[kMaxPStages], empty_p[kMaxPStages], full_s[SS], empty_s[SS];
  uint64_t tmem_full, tmem_empty, mma_done;
  uint32_t tmem_base;
  int abort;
};

// Shared memory: x ring, dequantized W ring, [packed code ring, scale/bias
// windows,] barriers; + 1024 for aligning the base.
template <int BITS, bool WTMA>
constexpr size_t smem_bytes() {
  return SA * A_BYTES + SB * B_BYTES +
         (WTMA ? p_stages<BITS>() * p_bytes<BITS>() + SS * SB_WIN_BYTES : 0) + sizeof(Barriers) + 1024;
}

struct GemmArgs {
  const uint32_t *w;
  const uint16_t *scales, *biases;
  void *y;
  int M, N, K;
  int group_shift;
  int m_tiles, n_tiles;
  int splits;   // K ranges per output tile (split-K when > 1)
  float *ws;    // split-K partials: slice s at ws + s * M * N, fp32 [M, N]
  unsigned *err;
  // Grouped mode (gather_qmm over sorted expert runs) when plan is not null:
  // plan[0] = the row tiles in use, then per row tile i (expert, first row,
  // end row) at plan[1 + 3i]; expert e's weights sit w_bstride words and
  // sb_bstride scale elements after expert e - 1's.  m_tiles is then read
  // from the plan on the device.
  const int *plan = nullptr;
  int64_t w_bstride = 0, sb_bstride = 0;
  int w_batches = 1;  // weight batches the arrays hold (host side: tensor map extents)
  uint32_t spin_limit = kDefaultWaitLimit;  // polls of a bounded wait before it gives up
};

// The rows [row0, row_end) of x and y one row tile covers, and its weight batch.
struct RowTile {
  int row0, row_end, expert;
};

__device__ __forceinline__ RowTile row_tile(const GemmArgs &a, int mi) {
  if (!a.plan) return RowTile{mi * BM, min(a.M, mi * BM + BM), 0};
  const int *p = a.plan + 1 + 3 * mi;
  return RowTile{__ldg(p + 1), __ldg(p + 2), __ldg(p)};
}

// A unit of work: one output tile over one K range (k-blocks [kb0, kb1)).
struct Unit {
  int tile, split, kb0, kb1;
};

// (splits <= 32 and nk < 2^26 keep the products in 32 bits.)
__device__ __forceinline__ Unit unit_of(const GemmArgs &a, int u, int nk) {
  Unit r;
  const unsigned sp = static_cast<unsigned>(a.splits);
  r.tile = static_cast<int>(static_cast<unsigned>(u) / sp);
  r.split = u - r.tile * a.splits;
  r.kb0 = static_cast<int>(static_cast<unsigned>(r.split) * static_cast<unsigned>(nk) / sp);
  r.kb1 = static_cast<int>(static_cast<unsigned>(r.split + 1) * static_cast<unsigned>(nk) / sp);
  return r;
}

// ------------------------------------------------------------- PTX glue ----

// Whole-warp bounded wait for the phase of parity `parity` to complete.
// Warp-uniform result: false if this wait ran out (the error word is set) or
// another role already gave up.
__device__ __noinline__ bool wait_warp(uint64_t *b, uint32_t parity, volatile int *abort,
                                       unsigned *err, uint32_t limit) {
  uint32_t spins = 0;
  while (true) {
    const bool done = mbar_try_wait(b, parity);
    if (__all_sync(0xffffffffu, done)) return true;
    if ((++spins & 255u) == 0 || spins >= limit) {
      int stop = *abort;
      if (!stop && spins >= limit) {
        stop = 1;
        *abort = 1;
        atomicOr(err, kErrTimeoutBit);
      }
      if (__any_sync(0xffffffffu, stop)) return false;
    }
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

// K-major, 128-byte swizzle, 8-row groups 1024 bytes apart (tcgen05 smem
// matrix descriptor: start>>4 [0,14), LBO>>4 [16,30), SBO>>4 [32,46),
// version 1 [46,48), swizzle mode [61,64) with 2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
  uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, A and B both bf16
// (format 1 in bits 7-9 and 10-12) or both fp16 (format 0), both K-major,
// N = BN, M = UM (each of the tile's two MMAs).
template <typename E>
__host__ __device__ constexpr uint32_t idesc_kmajor() {
  return (1u << 4) | (E::kF16 ? 0u : (1u << 7) | (1u << 10)) |
         (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(UM >> 4) << 24);
}

// The same with B (the dequantized weight) MN-major: bit 16 = transpose B.
template <typename E>
__host__ __device__ constexpr uint32_t idesc_bmn() { return idesc_kmajor<E>() | (1u << 16); }

// MN-major, 128-byte swizzle: atoms of 64 N-elements x 8 K-rows; LBO = 8192
// bytes between atoms along N, SBO = 1024 bytes between atoms along K.
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t saddr) {
  uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(8192 >> 4) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

template <uint32_t IDESC>
__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(IDESC), "r"(acc));
}

__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 bytes to global memory in one instruction (p 32-byte aligned).
__device__ __forceinline__ void st_global_256(void *p, const uint4 &a, const uint4 &b) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a.x),
               "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
               : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, const uint32_t (&v)[4]) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v[0]), "r"(v[1]),
               "r"(v[2]), "r"(v[3])
               : "memory");
}

// ---------------------------------------------------------------- roles ----

// Dequant side: 32 consecutive codes of one stored row (`bits` words) with
// their group's scale and bias (s | b << 16).  32 codes never straddle a
// group (group_size >= 32) and start on a word boundary.  `live` is false
// past the block's last stage.
template <int BITS>
struct ItemLoad {
  uint32_t v[BITS];
  uint32_t sb;
  bool live;
};

// The item a dequant thread owns in a stage, and the shared-memory byte
// offsets of its four 16-byte chunks (8 dequantized weights each).
//  TRANS: the W tile is K-major (as the x tile): 256 weight rows of 128 bytes;
//    thread (r, h) takes codes [32h, 32h+32) of the stage in row r, chunks
//    4h .. 4h+3 of the row, at chunk position c ^ (r % 8).
//  !TRANS: the W tile is MN-major: a chunk is 8 consecutive n of one k row.
//    Swizzle atoms of 64 n x 8 k (1024 bytes) sit at ((n/64) * 8 + k/8) *
//    1024; inside an atom, k row kw is at kw * 128 and n chunk j at position
//    j ^ kw.  Thread (k row kr, segment q) takes n [32q, 32q+32), chunks
//    4q .. 4q+3; the 8 lanes of a quarter warp take 8 consecutive k rows, so
//    their stores land in 8 distinct bank groups.
template <bool TRANS>
__device__ __forceinline__ void item_place(int dt, int tile_n0, int kb, int &row, int &col,
                                           uint32_t (&off)[4]) {
  if (TRANS) {
    const int r = dt >> 1, h = dt & 1;
    row = tile_n0 + r;
    col = kb * BK + 32 * h;
#pragma unroll
    for (int j = 0; j < 4; ++j) off[j] = r * 128 + (((4 * h + j) ^ (r & 7)) << 4);
  } else {
    const int kr = (dt >> 6) * 8 + (dt & 7), q = (dt >> 3) & 7, kw = kr & 7;
    row = kb * BK + kr;
    col = tile_n0 + 32 * q;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int jn = 4 * q + j;
      off[j] = ((jn >> 3) * 8 + (kr >> 3)) * 1024 + kw * 128 + (((jn & 7) ^ kw) << 4);
    }
  }
}

// One item's 32 codes (v, `bits` words) dequantized with scale bits hs and
// bias bits hb into the four 16-byte chunks of the W tile at base + off[j].
// The fast form is bf16's (fp16 has no room for its multipliers); a warp
// takes it when every lane's scale allows it.
template <typename E, int BITS>
__device__ __forceinline__ void dequant_store(const uint32_t (&v)[BITS], uint32_t hs, uint32_t hb,
                                              uint32_t base, const uint32_t (&off)[4]) {
  const uint32_t b2 = hb * 0x00010001u;
  bool fast = false;
  if constexpr (!E::kF16) fast = __all_sync(0xffffffffu, fast_scale(hs));
  if (fast) {
    uint32_t m[fast_slots<BITS>()];
    fast_muls<BITS>(hs, m);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = pair_fast<BITS>(v, 4 * j + i, m, b2);
      st_shared_v4(base + off[j], o);
    }
  } else {
    const uint32_t s2 = hs * 0x00010001u;
    const float sf = E::to_f32(hs), bf = E::to_f32(hb);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = pair_exact<BITS, E>(v, 4 * j + i, s2, b2, sf, bf);
      st_shared_v4(base + off[j], o);
    }
  }
}

// A dequant thread's item across the stages of its block: the unit and
// k-block it loads next, with the pointers of its codes and of its row's (or
// column's) scales and biases.  Moving to the next k-block is a pointer step;
// the unit's geometry is worked out once, when the thread moves to it.
template <int BITS, bool TRANS>
struct ItemCursor {
  const uint32_t *w;       // codes of the item at k-block kb
  const uint16_t *s, *b;   // TRANS: the row's scales / biases; else the item's, at kb
  int unit, kb, kb1;
  int kpos;                // TRANS: first code of the item at kb; else its k row
  bool in;                 // the item's weight row (TRANS) / column (else) exists
  bool vec;                // the codes allow vector loads
};

template <int BITS, bool TRANS>
__device__ __forceinline__ void cursor_unit(const GemmArgs &a, int nk, int dt,
                                            ItemCursor<BITS, TRANS> &c) {
  const Unit un = unit_of(a, c.unit, nk);
  c.kb = un.kb0;
  c.kb1 = un.kb1;
  const int n0 = (un.tile / a.m_tiles) * BN;
  const int expert = a.plan ? row_tile(a, un.tile % a.m_tiles).expert : 0;
  const uint32_t *wb = a.w + expert * a.w_bstride;
  const uint16_t *sb = a.scales + expert * a.sb_bstride, *bb = a.biases + expert * a.sb_bstride;
  if (TRANS) {
    const int row = n0 + (dt >> 1), h = dt & 1;
    const int64_t wpr = (static_cast<int64_t>(a.K) * BITS) >> 5;
    const int64_t gpr = a.K >> a.group_shift;
    c.in = row < a.N;
    c.kpos = c.kb * BK + 32 * h;
    c.w = wb + row * wpr + (c.kpos >> 5) * BITS;
    c.s = sb + row * gpr;
    c.b = bb + row * gpr;
  } else {
    const int kr = (dt >> 6) * 8 + (dt & 7), col = n0 + 32 * ((dt >> 3) & 7);
    const int64_t wpr = (static_cast<int64_t>(a.N) * BITS) >> 5;
    const int64_t gpr = a.N >> a.group_shift;
    c.in = col < a.N;
    c.kpos = c.kb * BK + kr;
    c.w = wb + c.kpos * wpr + (col >> 5) * BITS;
    c.s = sb + c.kpos * gpr + (col >> a.group_shift);
    c.b = bb + c.kpos * gpr + (col >> a.group_shift);
  }
  constexpr int kAlign = BITS % 4 == 0 ? 16 : BITS % 2 == 0 ? 8 : 4;  // bytes
  c.vec = (reinterpret_cast<uintptr_t>(c.w) & (kAlign - 1)) == 0;
}

// Load the item at the cursor's k-block into `it` and step the cursor.
// Items outside W (rows or columns past its edge, codes past K) read as zero.
template <int BITS, bool TRANS>
__device__ __forceinline__ void cursor_load(const GemmArgs &a, int nk, int dt, int num_units,
                                            ItemCursor<BITS, TRANS> &c, ItemLoad<BITS> &it) {
#pragma unroll
  for (int i = 0; i < BITS; ++i) it.v[i] = 0u;
  it.sb = 0u;
  it.live = c.unit < num_units;
  if (!it.live) return;
  if (c.in && c.kpos < a.K) {
    if (c.vec) {
      load_words<BITS>(c.w, it.v);
    } else {
#pragma unroll
      for (int i = 0; i < BITS; ++i) it.v[i] = __ldg(c.w + i);
    }
    const int g = TRANS ? (c.kpos >> a.group_shift) : 0;
    it.sb = __ldg(c.s + g) | (static_cast<uint32_t>(__ldg(c.b + g)) << 16);
  }
  if (++c.kb == c.kb1) {
    c.unit += gridDim.x;
    if (c.unit < num_units) cursor_unit<BITS, TRANS>(a, nk, dt, c);
  } else if (TRANS) {
    c.kpos += BK;
    c.w += 2 * BITS;
  } else {
    const int64_t wpr = (static_cast<int64_t>(a.N) * BITS) >> 5;
    const int64_t gpr = a.N >> a.group_shift;
    c.kpos += BK;
    c.w += BK * wpr;
    c.s += BK * gpr;
    c.b += BK * gpr;
  }
}

template <typename E, int BITS, bool TRANS>
__device__ void dequant_role(const GemmArgs &a, uint8_t *sB, Barriers *bars, int nk) {
  const int dt = threadIdx.x - 32 * (2 + kEpiWarps);  // 0 .. 32 * kDeqWarps - 1
  const int num_units = a.m_tiles * a.n_tiles * a.splits;
  volatile int *abort = &bars->abort;
  // Stages are consumed in order (unit, kb); the codes of the next kLoadAhead
  // stages are always in flight in register buffers while one is dequantized.
  ItemCursor<BITS, TRANS> c;
  c.unit = blockIdx.x;
  if (c.unit < num_units) cursor_unit<BITS, TRANS>(a, nk, dt, c);
  ItemLoad<BITS> buf[kLoadAhead];
#pragma unroll
  for (int i = 0; i < kLoadAhead; ++i) cursor_load<BITS, TRANS>(a, nk, dt, num_units, c, buf[i]);
  int s = 0;
  uint32_t ph = 0;
  uint32_t off[4];
  {
    int row, col;
    item_place<TRANS>(dt, 0, 0, row, col, off);
  }
  // One stage out of `buf`, which is then refilled; false when done or stopped.
  auto step = [&](ItemLoad<BITS> &buf) -> bool {
    const ItemLoad<BITS> cur = buf;
    if (!cur.live) return false;
    cursor_load<BITS, TRANS>(a, nk, dt, num_units, c, buf);
    if (!wait_warp(&bars->empty_b[s], ph ^ 1u, abort, a.err, a.spin_limit)) return false;
    const uint32_t base = smem_u32(sB + s * B_BYTES);
    dequant_store<E, BITS>(cur.v, cur.sb & 0xFFFFu, cur.sb >> 16, base, off);
    // Each thread makes its stores visible to the tensor cores, then one
    // arrival per warp.
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if ((dt & 31) == 0) mbar_arrive(&bars->full_b[s]);
    if (++s == SB) { s = 0; ph ^= 1u; }
    return true;
  };
  for (bool more = true; more;) {
#pragma unroll
    for (int i = 0; i < kLoadAhead; ++i)
      if (more) more = step(buf[i]);
  }
}

// TMA-fed dequant, producer (one warp, lane 0 issues): for every k-block of
// the block's units, the packed codes of the tile's BN rows (a [BN x 2*bits]
// word box) into the next code slot, and at each new window of kSbWin groups
// the rows' scales and biases ([BN x 8] boxes) into the next window slot.
// Weight batch e's row n is row e*N + n of the maps.
template <int BITS>
__device__ void w_tma_role(const CUtensorMap *wmap, const CUtensorMap *smap,
                           const CUtensorMap *bmap, const GemmArgs &a, uint8_t *sP, uint8_t *sS,
                           Barriers *bars, int nk) {
  constexpr int SP = p_stages<BITS>();
  const int lane = threadIdx.x & 31;
  const int num_units = a.m_tiles * a.n_tiles * a.splits;
  volatile int *abort = &bars->abort;
  int ps = 0, ss = 0;
  uint32_t pph = 0, sph = 0;
  // Parity of the last load issued into each slot, for the drain after a stop.
  int pend_p[SP], pend_s[SS];
#pragma unroll
  for (int i = 0; i < SP; ++i) pend_p[i] = -1;
#pragma unroll
  for (int i = 0; i < SS; ++i) pend_s[i] = -1;
  bool ok = true;
  for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
    const Unit un = unit_of(a, u, nk);
    const int expert = a.plan ? row_tile(a, un.tile % a.m_tiles).expert : 0;
    const int row0 = expert * a.N + (un.tile / a.m_tiles) * BN;
    int win = -1;
    for (int kb = un.kb0; kb < un.kb1; ++kb) {
      const int w = (kb * BK) >> (a.group_shift + 3);
      if (w != win) {
        if (!wait_warp(&bars->empty_s[ss], sph ^ 1u, abort, a.err, a.spin_limit)) { ok = false; break; }
        if (lane == 0) {
          const uint32_t dst = smem_u32(sS + ss * SB_WIN_BYTES);
          mbar_expect_tx(&bars->full_s[ss], SB_WIN_BYTES);
          tma_load_2d(dst, smap, w * kSbWin, row0, &bars->full_s[ss]);
          tma_load_2d(dst + SB_WIN_BYTES / 2, bmap, w * kSbWin, row0, &bars->full_s[ss]);
        }
        __syncwarp();
        pend_s[ss] = static_cast<int>(sph);
        win = w;
        if (++ss == SS) { ss = 0; sph ^= 1u; }
      }
      if (!wait_warp(&bars->empty_p[ps], pph ^ 1u, abort, a.err, a.spin_limit)) { ok = false; break; }
      if (lane == 0) {
        mbar_expect_tx(&bars->full_p[ps], p_bytes<BITS>());
        tma_load_2d(smem_u32(sP + ps * p_bytes<BITS>()), wmap, kb * 2 * BITS, row0, &bars->full_p[ps]);
      }
      __syncwarp();
      pend_p[ps] = static_cast<int>(pph);
      if (++ps == SP) { ps = 0; pph ^= 1u; }
    }
  }
  if (!ok) {
    // Stopped early: wait (bounded) for the copies still in flight.
#pragma unroll
    for (int i = 0; i < SP; ++i) {
      if (pend_p[i] < 0) continue;
      for (uint32_t spin = 0; spin < kSpinLimit; ++spin)
        if (__all_sync(0xffffffffu, mbar_try_wait(&bars->full_p[i], pend_p[i]))) break;
    }
#pragma unroll
    for (int i = 0; i < SS; ++i) {
      if (pend_s[i] < 0) continue;
      for (uint32_t spin = 0; spin < kSpinLimit; ++spin)
        if (__all_sync(0xffffffffu, mbar_try_wait(&bars->full_s[i], pend_s[i]))) break;
    }
  }
}

// TMA-fed dequant, consumers: the same items as dequant_role (thread (r, h)
// takes codes [32h, 32h+32) of tile row r), read from the staged codes and
// scale/bias window; a code slot is released as soon as its words are in
// registers, a window when the unit moves past it.  Rows and codes outside W
// arrive as zeros (codes 0, scale and bias 0: weight 0).
template <typename E, int BITS>
__device__ void dequant_role_tma(const GemmArgs &a, uint8_t *sB, const uint8_t *sP,
                                 const uint8_t *sS, Barriers *bars, int nk) {
  constexpr int SP = p_stages<BITS>();
  const int dt = threadIdx.x - 32 * (2 + kEpiWarps);  // 0 .. 32 * kDeqWarps - 1
  const int lane = dt & 31, r = dt >> 1, h = dt & 1;
  const int num_units = a.m_tiles * a.n_tiles * a.splits;
  volatile int *abort = &bars->abort;
  uint32_t off[4];
  {
    int row, col;
    item_place<true>(dt, 0, 0, row, col, off);
  }
  // This thread's words inside a code slot and its row inside a window.
  const uint32_t p_off = r * (8 * BITS) + h * (4 * BITS);
  const uint32_t s_off = r * (2 * kSbWin);
  int ps = 0, ss = 0, s = 0;
  uint32_t pph = 0, sph = 0, ph = 0;
  bool ok = true;
  for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
    const Unit un = unit_of(a, u, nk);
    int win = -1, cur = 0;
    for (int kb = un.kb0; kb < un.kb1; ++kb) {
      const int w = (kb * BK) >> (a.group_shift + 3);
      if (w != win) {
        if (win >= 0) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->empty_s[cur]);
        }
        if (!wait_warp(&bars->full_s[ss], sph, abort, a.err, a.spin_limit)) { ok = false; break; }
        cur = ss;
        win = w;
        if (++ss == SS) { ss = 0; sph ^= 1u; }
      }
      if (!wait_warp(&bars->full_p[ps], pph, abort, a.err, a.spin_limit)) { ok = false; break; }
      uint32_t v[BITS];
      const uint32_t pa = smem_u32(sP + ps * p_bytes<BITS>()) + p_off;
      if constexpr (BITS % 4 == 0) {
#pragma unroll
        for (int i = 0; i < BITS / 4; ++i)
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(v[4 * i]), "=r"(v[4 * i + 1]), "=r"(v[4 * i + 2]), "=r"(v[4 * i + 3])
                       : "r"(pa + 16 * i));
      } else {
#pragma unroll
        for (int i = 0; i < BITS / 2; ++i)
          asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v[2 * i]), "=r"(v[2 * i + 1]) : "r"(pa + 8 * i));
      }
      const int g = ((kb * BK + 32 * h) >> a.group_shift) & (kSbWin - 1);
      const uint32_t sa = smem_u32(sS + cur * SB_WIN_BYTES) + s_off + 2 * g;
      uint32_t hs, hb;
      asm volatile("ld.shared.u16 %0, [%1];" : "=r"(hs) : "r"(sa));
      asm volatile("ld.shared.u16 %0, [%1];" : "=r"(hb) : "r"(sa + SB_WIN_BYTES / 2));
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->empty_p[ps]);
      if (++ps == SP) { ps = 0; pph ^= 1u; }
      if (!wait_warp(&bars->empty_b[s], ph ^ 1u, abort, a.err, a.spin_limit)) { ok = false; break; }
      dequant_store<E, BITS>(v, hs, hb, smem_u32(sB + s * B_BYTES), off);
      // Each thread makes its stores visible to the tensor cores, then one
      // arrival per warp.
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->full_b[s]);
      if (++s == SB) { s = 0; ph ^= 1u; }
    }
    if (ok && win >= 0) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->empty_s[cur]);
    }
  }
}

__device__ void tma_role(const CUtensorMap *tmap, const GemmArgs &a, uint8_t *sA, Barriers *bars,
                         int nk) {
  const int lane = threadIdx.x & 31;
  const int num_units = a.m_tiles * a.n_tiles * a.splits;
  volatile int *abort = &bars->abort;
  int s = 0;
  uint32_t ph = 0;
  // Parity of the last load issued into each stage that has not been seen to
  // land, so that a role that stops early can wait for its copies.
  int pending[SA];
  for (int i = 0; i < SA; ++i) pending[i] = -1;
  bool ok = true;
  for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
    const Unit un = unit_of(a, u, nk);
    const int m0 = row_tile(a, un.tile % a.m_tiles).row0;
    for (int kb = un.kb0; kb < un.kb1; ++kb) {
      if (!wait_warp(&bars->empty_a[s], ph ^ 1u, abort, a.err, a.spin_limit)) { ok = false; break; }
      if (lane == 0) {
        mbar_expect_tx(&bars->full_a[s], A_BYTES);
        tma_load_2d(smem_u32(sA + s * A_BYTES), tmap, kb * BK, m0, &bars->full_a[s]);
      }
      __syncwarp();
      pending[s] = static_cast<int>(ph);
      if (++s == SA) { s = 0; ph ^= 1u; }
    }
  }
  if (!ok) {
    // Stopped early: wait (bounded) for the copies still in flight.
    for (int i = 0; i < SA; ++i) {
      if (pending[i] < 0) continue;
      for (uint32_t spin = 0; spin < kSpinLimit; ++spin)
        if (__all_sync(0xffffffffu, mbar_try_wait(&bars->full_a[i], pending[i]))) break;
    }
  }
}

template <typename E, bool TRANS>
__device__ void mma_role(const GemmArgs &a, uint8_t *sA, uint8_t *sB, Barriers *bars, int nk,
                         uint32_t tmem) {
  constexpr uint32_t idesc = TRANS ? idesc_kmajor<E>() : idesc_bmn<E>();
  // Start-address step of one 16-wide K slice: 32 bytes inside a K-major row,
  // two 8-row K atoms (2048 bytes) in the MN-major tile; in units of 16 bytes.
  constexpr uint64_t b_step = TRANS ? 2 : 128;
  const int lane = threadIdx.x & 31;
  const int num_units = a.m_tiles * a.n_tiles * a.splits;
  volatile int *abort = &bars->abort;
  int sa = 0, sb = 0, it = 0;
  uint32_t pha = 0, phb = 0;
  bool ok = true;
  for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x, ++it) {
    const Unit un = unit_of(a, u, nk);
    // The epilogue must have drained the accumulators of the previous unit.
    if (!wait_warp(&bars->tmem_empty, (it & 1) ^ 1u, abort, a.err, a.spin_limit)) break;
    tc_fence_after();
    // The second 128-row half only when this tile has x rows there.
    const RowTile rt = row_tile(a, un.tile % a.m_tiles);
    const bool two = rt.row0 + UM < rt.row_end;
    for (int kb = un.kb0; kb < un.kb1; ++kb) {
      if (!wait_warp(&bars->full_a[sa], pha, abort, a.err, a.spin_limit) ||
          !wait_warp(&bars->full_b[sb], phb, abort, a.err, a.spin_limit)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (lane == 0) {
        const uint64_t da0 = sw128_kmajor_desc(smem_u32(sA + sa * A_BYTES));
        const uint64_t da1 = sw128_kmajor_desc(smem_u32(sA + sa * A_BYTES + A_HALF));
        const uint32_t bs = smem_u32(sB + sb * B_BYTES);
        const uint64_t db = TRANS ? sw128_kmajor_desc(bs) : sw128_mnmajor_desc(bs);
#pragma unroll
        for (int j = 0; j < BK / 16; ++j) {
          const uint32_t accumulate = (kb != un.kb0 || j != 0) ? 1u : 0u;
          umma<idesc>(tmem, da0 + 2 * j, db + b_step * j, accumulate);
          if (two) umma<idesc>(tmem + BN, da1 + 2 * j, db + b_step * j, accumulate);
        }
        umma_commit(&bars->empty_a[sa]);
        umma_commit(&bars->empty_b[sb]);
      }
      __syncwarp();
      if (++sa == SA) { sa = 0; pha ^= 1u; }
      if (++sb == SB) { sb = 0; phb ^= 1u; }
    }
    if (!ok) break;
    if (lane == 0) umma_commit(&bars->tmem_full);
    __syncwarp();
  }
  // Retire every MMA this thread issued before the block frees TMEM.
  if (lane == 0) umma_commit(&bars->mma_done);
  __syncwarp();
  for (uint32_t spin = 0; spin < kSpinLimit; ++spin)
    if (__all_sync(0xffffffffu, mbar_try_wait(&bars->mma_done, 0))) break;
}

template <typename E, bool OUT_BF16>
__device__ void epilogue_role(const GemmArgs &a, Barriers *bars, uint32_t tmem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3;  // TMEM lane quarter this warp may access
  const int num_units = a.m_tiles * a.n_tiles * a.splits;
  volatile int *abort = &bars->abort;
  const bool vec = OUT_BF16 ? (a.N % 8 == 0) : (a.N % 4 == 0);
  const bool vec_ws = a.N % 4 == 0;
  // 32-byte stores: rows of y (and of the partials) 32-byte aligned.
  const bool y32 = (OUT_BF16 ? (a.N % 16 == 0) : (a.N % 8 == 0)) &&
                   (reinterpret_cast<uintptr_t>(a.y) & 31u) == 0;
  const bool ws32 = a.N % 8 == 0 && (reinterpret_cast<uintptr_t>(a.ws) & 31u) == 0;
  int it = 0;
  for (int u = blockIdx.x; u < num_units; u += gridDim.x, ++it) {
    if (!wait_warp(&bars->tmem_full, it & 1, abort, a.err, a.spin_limit)) return;
    tc_fence_after();
    const int tile = u / a.splits, split = u - tile * a.splits;
    const int n0 = (tile / a.m_tiles) * BN;
    const RowTile rt = row_tile(a, tile % a.m_tiles);
#pragma unroll 1
    for (int hc = 0; hc < 2 * (BN / 32); ++hc) {
      const int half = hc / (BN / 32), cc = hc % (BN / 32);
      const int m = rt.row0 + UM * half + 32 * q + lane;
      if (half == 1 && rt.row0 + UM >= rt.row_end) break;  // no second half
      uint32_t r[32];
      tmem_ld32(tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(half * BN + 32 * cc), r);
      const int n = n0 + 32 * cc;
      if (m >= rt.row_end || n >= a.N) continue;
      const int64_t o = static_cast<int64_t>(m) * a.N + n;
      if (a.splits > 1) {
        // A partial of a split tile: fp32 into this split's slice.
        float *wp = a.ws + static_cast<int64_t>(split) * a.M * a.N + o;
        if (ws32 && n + 32 <= a.N) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            st_global_256(wp + 8 * j, make_uint4(r[8 * j], r[8 * j + 1], r[8 * j + 2], r[8 * j + 3]),
                          make_uint4(r[8 * j + 4], r[8 * j + 5], r[8 * j + 6], r[8 * j + 7]));
        } else if (vec_ws && n + 32 <= a.N) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            reinterpret_cast<float4 *>(wp)[j] =
                make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                            __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (n + j < a.N) wp[j] = __uint_as_float(r[j]);
        }
      } else if (OUT_BF16) {
        uint16_t *yp = static_cast<uint16_t *>(a.y) + o;
        if (vec && n + 32 <= a.N) {
          uint4 p[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            p[j].x = E::pack2(__uint_as_float(r[8 * j + 0]), __uint_as_float(r[8 * j + 1]));
            p[j].y = E::pack2(__uint_as_float(r[8 * j + 2]), __uint_as_float(r[8 * j + 3]));
            p[j].z = E::pack2(__uint_as_float(r[8 * j + 4]), __uint_as_float(r[8 * j + 5]));
            p[j].w = E::pack2(__uint_as_float(r[8 * j + 6]), __uint_as_float(r[8 * j + 7]));
          }
          if (y32) {
            st_global_256(yp, p[0], p[1]);
            st_global_256(yp + 16, p[2], p[3]);
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) reinterpret_cast<uint4 *>(yp)[j] = p[j];
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (n + j < a.N) yp[j] = E::from_f32(__uint_as_float(r[j]));
        }
      } else {
        float *yp = static_cast<float *>(a.y) + o;
        if (y32 && n + 32 <= a.N) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            st_global_256(yp + 8 * j, make_uint4(r[8 * j], r[8 * j + 1], r[8 * j + 2], r[8 * j + 3]),
                          make_uint4(r[8 * j + 4], r[8 * j + 5], r[8 * j + 6], r[8 * j + 7]));
        } else if (vec && n + 32 <= a.N) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            reinterpret_cast<float4 *>(yp)[j] =
                make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                            __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (n + j < a.N) yp[j] = __uint_as_float(r[j]);
        }
      }
    }
    tc_fence_before();
    mbar_arrive(&bars->tmem_empty);
  }
}

// WTMA: the TMA-fed dequant (maps of the packed codes, scales and biases in
// tmap_w / tmap_s / tmap_b); otherwise those three maps are unused.
template <typename E, int BITS, bool OUT_BF16, bool TRANS, bool WTMA>
__global__ void __launch_bounds__(gemm_threads<WTMA>(), 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
            const __grid_constant__ CUtensorMap tmap_s, const __grid_constant__ CUtensorMap tmap_b,
            GemmArgs a) {
  // Grouped mode: the row tiles in use, as the plan kernel counted them.
  if (a.plan) a.m_tiles = __ldg(a.plan);
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + SA * A_BYTES;
  uint8_t *sP = sB + SB * B_BYTES;
  uint8_t *sS = sP + (WTMA ? p_stages<BITS>() * p_bytes<BITS>() : 0);
  Barriers *bars = reinterpret_cast<Barriers *>(sS + (WTMA ? SS * SB_WIN_BYTES : 0));
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    for (int i = 0; i < SA; ++i) {
      mbar_init(&bars->full_a[i], 1);
      mbar_init(&bars->empty_a[i], 1);
    }
    for (int i = 0; i < SB; ++i) {
      mbar_init(&bars->full_b[i], kDeqWarps);
      mbar_init(&bars->empty_b[i], 1);
    }
    for (int i = 0; i < kMaxPStages; ++i) {
      mbar_init(&bars->full_p[i], 1);
      mbar_init(&bars->empty_p[i], kDeqWarps);
    }
    for (int i = 0; i < SS; ++i) {
      mbar_init(&bars->full_s[i], 1);
      mbar_init(&bars->empty_s[i], kDeqWarps);
    }
    mbar_init(&bars->tmem_full, 1);
    mbar_init(&bars->tmem_empty, 32 * kEpiWarps);
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmap_x) : "memory");
    if (WTMA) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(&tmap_w) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(&tmap_s) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(&tmap_b) : "memory");
    }
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&bars->tmem_base)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const int nk = (a.K + BK - 1) / BK;

  if (warp == 0) tma_role(&tmap_x, a, sA, bars, nk);
  else if (warp == 1) mma_role<E, TRANS>(a, sA, sB, bars, nk, tmem);
  else if (warp < 2 + kEpiWarps) epilogue_role<E, OUT_BF16>(a, bars, tmem);
  else if (warp < 2 + kEpiWarps + kDeqWarps) {
    if constexpr (WTMA) dequant_role_tma<E, BITS>(a, sB, sP, sS, bars, nk);
    else dequant_role<E, BITS, TRANS>(a, sB, bars, nk);
  } else if constexpr (WTMA) {
    w_tma_role<BITS>(&tmap_w, &tmap_s, &tmap_b, a, sP, sS, bars, nk);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(TMEM_COLS));
  }
}

// Split-K: y = the sum of the `splits` fp32 partial slices, added in slice
// order (deterministic), converted to the output type.  Four outputs a thread
// with 16-byte loads when the slices are 16-byte aligned.
template <typename E, bool OUT_BF16>
__global__ void __launch_bounds__(256)
splitk_finalize(const float *__restrict__ ws, int splits, int64_t mn, void *__restrict__ y,
                const unsigned *err) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  // A bounded wait of the GEMM ran out (here or in an earlier call whose
  // error has not been read): its partials are incomplete, so y is NaN
  // rather than a plausible wrong sum.
  if (*reinterpret_cast<const volatile unsigned *>(err) & kErrTimeoutBit) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < mn; i += stride) {
      if (OUT_BF16) static_cast<uint16_t *>(y)[i] = E::kF16 ? 0x7E00u : 0x7FC0u;
      else static_cast<float *>(y)[i] = __int_as_float(0x7FC00000);
    }
    return;
  }
  if (mn % 4 == 0) {
    for (int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 4; i < mn;
         i += stride * 4) {
      float4 acc = *reinterpret_cast<const float4 *>(ws + i);
      for (int sl = 1; sl < splits; ++sl) {
        const float4 v = *reinterpret_cast<const float4 *>(ws + sl * mn + i);
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      }
      if (OUT_BF16) {
        uint2 o;
        o.x = E::pack2(acc.x, acc.y);
        o.y = E::pack2(acc.z, acc.w);
        *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(y) + i) = o;
      } else {
        *reinterpret_cast<float4 *>(static_cast<float *>(y) + i) = acc;
      }
    }
  } else {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < mn; i += stride) {
      float acc = ws[i];
      for (int sl = 1; sl < splits; ++sl) acc += ws[sl * mn + i];
      if (OUT_BF16) static_cast<uint16_t *>(y)[i] = E::from_f32(acc);
      else static_cast<float *>(y)[i] = acc;
    }
  }
}

// ----------------------------------------------------------------- host ----

// One persistent block per SM.  With fewer output tiles than SMs, each tile's
// K range is split so that the units fill the SMs (at least two k-blocks a
// unit); the partials then need splits * M * N fp32 of workspace, never more
// than one 256 x 256 tile per SM.
int choose_splits(int tiles, int nk, int sms) {
  if (tiles * 2 > sms) return 1;
  int s = sms / tiles;
  if (s > nk / 2) s = nk / 2;
  if (s > 32) s = 32;
  return s < 1 ? 1 : s;
}

size_t splitk_bytes(const GemmArgs &a) {
  return static_cast<size_t>(a.splits) * a.M * a.N * sizeof(float);
}

template <typename E, int BITS, bool OUT_BF16, bool TRANS>
cudaError_t launch_t(const uint16_t *x, const GemmArgs &a, cudaStream_t stream) {
  // TMA rows of x must start on 16-byte boundaries.
  if ((static_cast<int64_t>(a.K) * 2) % 16 != 0) return cudaErrorNotSupported;
  CUtensorMap map;
  cudaError_t me = encode_map_2d(&map, E::kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                               : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, a.K, a.M,
                                 static_cast<uint64_t>(a.K) * 2, BK, BM,
                                 CU_TENSOR_MAP_SWIZZLE_128B);
  if (me != cudaSuccess) return me;
  const int units = a.m_tiles * a.n_tiles * a.splits;
  const int grid = units < sm_count() ? units : sm_count();
  cudaError_t e = cudaErrorNotSupported;
  // The TMA-fed dequant where TMA can address W's rows, its k-blocks' words
  // and its scale/bias windows (16-byte boxes and strides).
  if constexpr (TRANS && BITS % 2 == 0) {
    const uint64_t rows = static_cast<uint64_t>(a.N) * a.w_batches;
    const int64_t groups = a.K >> a.group_shift;
    if ((static_cast<int64_t>(a.K) * BITS) % 128 == 0 && groups % kSbWin == 0 &&
        rows < (uint64_t(1) << 31) && (reinterpret_cast<uintptr_t>(a.w) & 15u) == 0 &&
        (reinterpret_cast<uintptr_t>(a.scales) & 15u) == 0 &&
        (reinterpret_cast<uintptr_t>(a.biases) & 15u) == 0) {
      CUtensorMap wm, sm, bm;
      const uint64_t wpr = static_cast<uint64_t>(a.K) * BITS / 32;
      if (encode_map_2d(&wm, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.w, wpr, rows, wpr * 4, 2 * BITS, BN,
                        CU_TENSOR_MAP_SWIZZLE_NONE) == cudaSuccess &&
          encode_map_2d(&sm, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.scales, groups, rows, groups * 2,
                        kSbWin, BN, CU_TENSOR_MAP_SWIZZLE_NONE) == cudaSuccess &&
          encode_map_2d(&bm, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.biases, groups, rows, groups * 2,
                        kSbWin, BN, CU_TENSOR_MAP_SWIZZLE_NONE) == cudaSuccess) {
        constexpr size_t smem = smem_bytes<BITS, true>();
        const cudaError_t ae = ensure_smem_limit<gemm_kernel<E, BITS, OUT_BF16, TRANS, true>>(smem);
        if (ae != cudaSuccess) return ae;
        gemm_kernel<E, BITS, OUT_BF16, TRANS, true><<<grid, gemm_threads<true>(), smem, stream>>>(
            map, wm, sm, bm, a);
        e = cudaGetLastError();
      }
    }
  }
  if (e == cudaErrorNotSupported) {
    constexpr size_t smem = smem_bytes<BITS, false>();
    const cudaError_t ae = ensure_smem_limit<gemm_kernel<E, BITS, OUT_BF16, TRANS, false>>(smem);
    if (ae != cudaSuccess) return ae;
    gemm_kernel<E, BITS, OUT_BF16, TRANS, false><<<grid, gemm_threads<false>(), smem, stream>>>(
        map, map, map, map, a);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess || a.splits == 1) return e;
  const int64_t mn = static_cast<int64_t>(a.M) * a.N;
  int64_t blocks = (mn / 4 + 255) / 256;
  if (blocks > 4 * sm_count()) blocks = 4 * sm_count();
  if (blocks < 1) blocks = 1;
  splitk_finalize<E, OUT_BF16><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a.ws, a.splits, mn, a.y, a.err);
  return cudaGetLastError();
}

template <typename E, int BITS>
cudaError_t launch_bits(const uint16_t *x, const GemmArgs &a, bool transpose, bool y_16,
                        cudaStream_t stream) {
  if (transpose)
    return y_16 ? launch_t<E, BITS, true, true>(x, a, stream) : launch_t<E, BITS, false, true>(x, a, stream);
  return y_16 ? launch_t<E, BITS, true, false>(x, a, stream) : launch_t<E, BITS, false, false>(x, a, stream);
}

template <typename E>
cudaError_t launch_any_bits(const uint16_t *x, const GemmArgs &a, int bits, bool transpose,
                            bool y_16, cudaStream_t stream) {
  switch (bits) {
    case 1: return launch_bits<E, 1>(x, a, transpose, y_16, stream);
    case 2: return launch_bits<E, 2>(x, a, transpose, y_16, stream);
    case 3: return launch_bits<E, 3>(x, a, transpose, y_16, stream);
    case 4: return launch_bits<E, 4>(x, a, transpose, y_16, stream);
    case 5: return launch_bits<E, 5>(x, a, transpose, y_16, stream);
    case 6: return launch_bits<E, 6>(x, a, transpose, y_16, stream);
    case 8: return launch_bits<E, 8>(x, a, transpose, y_16, stream);
    default: return cudaErrorInvalidValue;
  }
}

// x rows that TMA cannot address (K not a multiple of 8, possible when W is
// stored [K, N]): the decode kernel over 16-row slices of x instead.
template <typename E>
cudaError_t gemv_slices(const uint16_t *x, int64_t M, const PackedWeight &w, bool transpose,
                        int64_t N, int64_t K, void *y, bool y_16, cudaStream_t stream) {
  const size_t ysz = y_16 ? 2 : 4;
  for (int64_t m0 = 0; m0 < M; m0 += 16) {
    const int64_t rows = M - m0 < 16 ? M - m0 : 16;
    const uint16_t *xs = x + m0 * K;
    void *ys = static_cast<char *>(y) + m0 * N * static_cast<int64_t>(ysz);
    const cudaError_t e = E::kF16 ? launch_gemv_f16(xs, rows, w, transpose, ys, y_16, stream)
                                  : launch_gemv(xs, rows, w, transpose, ys, y_16, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <typename E>
cudaError_t gemm_entry(const uint16_t *x, int64_t M, const PackedWeight &w, bool transpose,
                       void *y, bool y_bf16, cudaStream_t stream) {
  GemmArgs a;
  a.w = w.w;
  a.scales = w.scales;
  a.biases = w.biases;
  a.y = y;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(transpose ? w.rows : w.cols);
  a.K = static_cast<int>(transpose ? w.cols : w.rows);
  a.group_shift = w.group == 32 ? 5 : w.group == 64 ? 6 : 7;
  a.m_tiles = (a.M + BM - 1) / BM;
  a.n_tiles = (a.N + BN - 1) / BN;
  a.err = device_error_word();
  a.spin_limit = wait_limit();
  if (!a.err) return cudaErrorInvalidSymbol;
  a.splits = choose_splits(a.m_tiles * a.n_tiles, (a.K + BK - 1) / BK, sm_count());
  a.ws = nullptr;
  if (a.splits > 1) {
    // Stream-ordered: the workspace belongs to this call on this stream
    // (a graph captures it as allocation and free nodes).  Without one the
    // call runs unsplit.
    void *p = nullptr;
    if (cudaMallocAsync(&p, splitk_bytes(a), stream) == cudaSuccess) {
      a.ws = static_cast<float *>(p);
    } else {
      cudaGetLastError();
      a.splits = 1;
    }
  }
  cudaError_t e = launch_any_bits<E>(x, a, w.bits, transpose, y_bf16, stream);
  if (a.ws) {
    const cudaError_t fe = cudaFreeAsync(a.ws, stream);
    if (e == cudaSuccess) e = fe;
  }
  if (e != cudaErrorNotSupported) return e;
  return gemv_slices<E>(x, M, w, transpose, a.N, a.K, y, y_bf16, stream);
}

}  // namespace

cudaError_t launch_gemm(const uint16_t *x, int64_t M, const PackedWeight &w, bool transpose,
                        void *y, bool y_bf16, cudaStream_t stream) {
  return gemm_entry<ElemBF16>(x, M, w, transpose, y, y_bf16, stream);
}

cudaError_t launch_gemm_f16(const uint16_t *x, int64_t M, const PackedWeight &w, bool transpose,
                            void *y, bool y_f16, cudaStream_t stream) {
  return gemm_entry<ElemF16>(x, M, w, transpose, y, y_f16, stream);
}

// ------------------------------------------------- grouped (MoE) mode ----
// gather_qmm with sorted weight-batch indices, one x row per batch and no
// lhs indices (nuvec_core quantized.rs, `gather_qmm` and `sorted_offsets`:
// sorted indices let each expert's weights be walked once): batch b is x row
// b times expert rhs[b], so expert e's batches are one run of consecutive x
// and y rows.  A one-block plan kernel finds the runs (binary search in the
// sorted indices), cuts them into row tiles of BM and writes the plan; the
// GEMM then walks (row tile, column tile) units of every expert.  Indices past
// the last expert zero their y rows and raise the index bit.
namespace {

__device__ __forceinline__ int lower_bound_rhs(const uint32_t *v, int n, uint32_t key) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(v + mid) < key) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

constexpr int kPlanThreads = 256;

// Dynamic shared memory: 2 * w_batches ints (row tiles of each expert, then
// its first plan entry).  The entries never exceed cap (1 + 3 * cap ints of
// plan), whatever the indices hold: unsorted indices give wrong runs, never
// writes outside the plan.
__global__ void __launch_bounds__(kPlanThreads)
group_plan_kernel(const uint32_t *rhs, int batches, int w_batches, int cap, int *plan, void *y,
                  int N, int ysz, unsigned *err) {
  extern __shared__ int sp[];
  int *count = sp, *first = sp + w_batches;
  const int t = threadIdx.x;
  for (int e = t; e < w_batches; e += kPlanThreads) {
    const int l = lower_bound_rhs(rhs, batches, static_cast<uint32_t>(e));
    const int h = lower_bound_rhs(rhs, batches, static_cast<uint32_t>(e) + 1u);
    count[e] = h > l ? (h - l + BM - 1) / BM : 0;
  }
  __syncthreads();
  if (t == 0) {
    int total = 0;
    for (int e = 0; e < w_batches; ++e) {
      const int n = min(count[e], cap - total);
      count[e] = n;
      first[e] = total;
      total += n;
    }
    plan[0] = total;
  }
  __syncthreads();
  for (int e = t; e < w_batches; e += kPlanThreads) {
    const int l = lower_bound_rhs(rhs, batches, static_cast<uint32_t>(e));
    const int h = lower_bound_rhs(rhs, batches, static_cast<uint32_t>(e) + 1u);
    for (int j = 0; j < count[e]; ++j) {
      const int i = first[e] + j, r0 = l + j * BM;
      plan[1 + 3 * i] = e;
      plan[2 + 3 * i] = r0;
      plan[3 + 3 * i] = min(h, r0 + BM);
    }
  }
  // Batches whose index is past the last expert: zero rows, index bit.
  const int tail = lower_bound_rhs(rhs, batches, static_cast<uint32_t>(w_batches));
  if (tail < batches) {
    const int64_t n0 = static_cast<int64_t>(tail) * N, n1 = static_cast<int64_t>(batches) * N;
    for (int64_t i = n0 + t; i < n1; i += kPlanThreads) {
      if (ysz == 2) static_cast<uint16_t *>(y)[i] = 0;
      else static_cast<float *>(y)[i] = 0.0f;
    }
    if (t == 0) atomicOr(err, kErrIndexBit);
  }
}

}  // namespace

cudaError_t launch_gemm_grouped(const uint16_t *x, int64_t batches, const PackedWeight &w,
                                int64_t w_batches, const uint32_t *rhs, void *y, bool y_bf16,
                                cudaStream_t stream) {
  if (w_batches > 4096 || batches >= (int64_t(1) << 30) || (w.cols * 2) % 16 != 0)
    return cudaErrorNotSupported;
  GemmArgs a;
  a.w = w.w;
  a.scales = w.scales;
  a.biases = w.biases;
  a.y = y;
  a.M = static_cast<int>(batches);
  a.N = static_cast<int>(w.rows);
  a.K = static_cast<int>(w.cols);
  a.group_shift = w.group == 32 ? 5 : w.group == 64 ? 6 : 7;
  // An upper bound of the row tiles (the grid's size); the kernel reads the
  // actual count from the plan.
  a.m_tiles = static_cast<int>((batches + BM - 1) / BM + w_batches);
  a.n_tiles = (a.N + BN - 1) / BN;
  a.splits = 1;
  a.ws = nullptr;
  a.err = device_error_word();
  a.spin_limit = wait_limit();
  if (!a.err) return cudaErrorInvalidSymbol;
  a.w_bstride = w.rows * ((w.cols * w.bits) / 32);
  a.sb_bstride = w.rows * (w.cols / w.group);
  a.w_batches = static_cast<int>(w_batches);
  void *p = nullptr;
  cudaError_t e = cudaMallocAsync(&p, sizeof(int) * (1 + 3 * static_cast<size_t>(a.m_tiles)), stream);
  if (e != cudaSuccess) {  // no plan buffer: the caller takes the decode kernels instead
    cudaGetLastError();
    return cudaErrorNotSupported;
  }
  int *plan = static_cast<int *>(p);
  const size_t plan_smem = 2 * sizeof(int) * static_cast<size_t>(w_batches);
  group_plan_kernel<<<1, kPlanThreads, plan_smem, stream>>>(
      rhs, static_cast<int>(batches), static_cast<int>(w_batches), a.m_tiles, plan, y, a.N,
      y_bf16 ? 2 : 4, a.err);
  e = cudaGetLastError();
  if (e == cudaSuccess) {
    a.plan = plan;
    e = launch_any_bits<ElemBF16>(x, a, w.bits, true, y_bf16, stream);
  }
  const cudaError_t fe = cudaFreeAsync(plan, stream);
  return e != cudaSuccess ? e : fe;
}

// ------------------------------------------- static-scratch variant ----
// For callers that cannot allocate device memory at call time: the same
// kernels as launch_gemm, with the split-K partials in a fixed array of
// kStaticScratchBytes that every device loading this library holds until
// the process exits.  All calls on a device share it.
namespace {
constexpr size_t kStaticScratchFloats = size_t(6) << 20;  // 24 MiB of fp32
static __device__ __align__(256) float g_static_scratch[kStaticScratchFloats];
}  // namespace

size_t static_scratch_bytes() { return kStaticScratchFloats * sizeof(float); }

// The array's device address on the current device, looked up once per
// device (with that device current); nullptr if the lookup fails.
float *static_scratch() {
  constexpr int kMaxDevices = 64;
  static float *addr[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    float *p = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_static_scratch) != cudaSuccess)
      return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

cudaError_t launch_gemm_static_scratch(const uint16_t *x, int64_t M, const PackedWeight &w,
                                       bool transpose, void *y, bool y_bf16, float *scratch,
                                       cudaStream_t stream, size_t *needed) {
  GemmArgs a;
  a.w = w.w;
  a.scales = w.scales;
  a.biases = w.biases;
  a.y = y;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(transpose ? w.rows : w.cols);
  a.K = static_cast<int>(transpose ? w.cols : w.rows);
  a.group_shift = w.group == 32 ? 5 : w.group == 64 ? 6 : 7;
  a.m_tiles = (a.M + BM - 1) / BM;
  a.n_tiles = (a.N + BN - 1) / BN;
  a.err = device_error_word();
  a.spin_limit = wait_limit();
  if (!a.err) return cudaErrorInvalidSymbol;
  // Same split as launch_gemm; x rows TMA cannot address take the decode
  // kernel below and need no partials.
  const bool tma_rows = (static_cast<int64_t>(a.K) * 2) % 16 == 0;
  a.splits = tma_rows ? choose_splits(a.m_tiles * a.n_tiles, (a.K + BK - 1) / BK, sm_count()) : 1;
  // Fewer splits when the partials of the usual split do not fit the array
  // (none when not even two do): the same kernels, a shorter split.
  const size_t slice = static_cast<size_t>(a.M) * a.N * sizeof(float);
  if (a.splits > 1 && splitk_bytes(a) > static_scratch_bytes()) {
    const size_t fit = static_scratch_bytes() / slice;
    a.splits = fit >= 2 ? static_cast<int>(fit) : 1;
  }
  *needed = a.splits > 1 ? splitk_bytes(a) : 0;
  if (*needed > static_scratch_bytes()) return cudaErrorInvalidValue;
  a.ws = a.splits > 1 ? scratch : nullptr;
  const cudaError_t e = launch_any_bits<ElemBF16>(x, a, w.bits, transpose, y_bf16, stream);
  if (e != cudaErrorNotSupported) return e;
  return gemv_slices<ElemBF16>(x, M, w, transpose, a.N, a.K, y, y_bf16, stream);
}

}  // namespace qmm
