// gather_qmm on the decode kernels of gemv_impl.cuh (bf16), in a translation
// unit of its own so that it compiles beside gemv.cu.
#include "gemv_impl.cuh"

namespace qmm {
namespace {

// gather_qmm.  Transposed W with K a multiple of 128 takes the TMA kernel,
// which walks each block's x rows in passes of 8 * NT (so any M); sorted
// batches (one x row each, lhs absent) let a block stream one weight tile
// for its whole run.  Otherwise the plain-load kernels, over 16-row slices
// of each batch.  No programmatic dependent launch: the indices may come
// from the previous kernel.
template <int BITS>
cudaError_t launch_gather_bits(const GemvArgs &a0, const Batches &b0, bool transpose, bool y_bf16,
                               bool sorted, cudaStream_t stream) {
  if (transpose && a0.K % 128 == 0) {
    cudaError_t e;
    if (sorted) {
      Batches bs = b0;
      bs.g.sorted = 1;
      bs.count = b0.g.w_batches + 1;
      if (BITS < 6 && ((a0.N + 15) / 16) * bs.count > 2 * sm_count())
        e = y_bf16 ? launch_t_tma<ElemBF16, BITS, 1, true, true, kFuseNone, 8>(a0, false, bs, stream)
                   : launch_t_tma<ElemBF16, BITS, 1, false, true, kFuseNone, 8>(a0, false, bs, stream);
      else
        e = y_bf16 ? launch_t_tma<ElemBF16, BITS, 1, true, true>(a0, false, bs, stream)
                   : launch_t_tma<ElemBF16, BITS, 1, false, true>(a0, false, bs, stream);
    } else if (a0.M <= 8 && BITS < 6 && ((a0.N + 15) / 16) * b0.count > 2 * sm_count()) {
      e = y_bf16 ? launch_t_tma<ElemBF16, BITS, 1, true, true, kFuseNone, 8>(a0, false, b0, stream)
                 : launch_t_tma<ElemBF16, BITS, 1, false, true, kFuseNone, 8>(a0, false, b0, stream);
    } else if (a0.M <= 8) {
      e = y_bf16 ? launch_t_tma<ElemBF16, BITS, 1, true, true>(a0, false, b0, stream)
                 : launch_t_tma<ElemBF16, BITS, 1, false, true>(a0, false, b0, stream);
    } else {
      e = y_bf16 ? launch_t_tma<ElemBF16, BITS, 2, true, true>(a0, false, b0, stream)
                 : launch_t_tma<ElemBF16, BITS, 2, false, true>(a0, false, b0, stream);
    }
    if (e != cudaErrorNotSupported) return e;
  }
  for (int64_t m0 = 0; m0 < a0.M; m0 += 16) {
    GemvArgs a = a0;
    a.M = static_cast<int>(a0.M - m0 < 16 ? a0.M - m0 : 16);
    Batches b = b0;
    b.g.x_off = m0 * a0.K;
    b.g.y_off = m0 * a0.N;
    cudaError_t e;
    if (transpose) {
      if (a.M <= 8)
        e = y_bf16 ? launch_t<ElemBF16, BITS, 1, true, true>(a, b, stream)
                   : launch_t<ElemBF16, BITS, 1, false, true>(a, b, stream);
      else
        e = y_bf16 ? launch_t<ElemBF16, BITS, 2, true, true>(a, b, stream)
                   : launch_t<ElemBF16, BITS, 2, false, true>(a, b, stream);
    } else {
      e = y_bf16 ? launch_n<ElemBF16, BITS, true, true>(a, b, stream)
                 : launch_n<ElemBF16, BITS, false, true>(a, b, stream);
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_gather(const uint16_t *x, int64_t x_batches, int64_t M, const PackedWeight &w,
                          int64_t w_batches, const uint32_t *lhs, const uint32_t *rhs,
                          int64_t batches, bool transpose, bool sorted, void *y, bool y_bf16,
                          cudaStream_t stream) {
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
  Batches b;
  b.g.lhs = lhs;
  b.g.rhs = rhs;
  b.g.x_batches = static_cast<int>(x_batches);
  b.g.w_batches = static_cast<int>(w_batches);
  b.g.batches = static_cast<int>(batches);
  b.g.sorted = 0;
  b.g.x_bstride = M * a.K;
  b.g.y_bstride = M * a.N;
  b.g.w_bstride = w.rows * ((w.cols * w.bits) / 32);
  b.g.sb_bstride = w.rows * (w.cols / w.group);
  b.g.x_off = b.g.y_off = 0;
  b.count = batches;
  // One weight tile streamed per run: batches sorted by weight batch, one x
  // row each, x batches in order.
  const bool by_runs = sorted && M == 1 && !lhs && rhs;
  // Long runs (prefill-sized: 32 or more batches per weight batch on
  // average) go to the tensor cores, one GEMM per run.
  if (by_runs && transpose && batches >= 32 * w_batches) {
    const cudaError_t e = launch_gemm_grouped(x, batches, w, w_batches, rhs, y, y_bf16, stream);
    if (e != cudaErrorNotSupported) return e;
  }
  switch (w.bits) {
    case 1: return launch_gather_bits<1>(a, b, transpose, y_bf16, by_runs, stream);
    case 2: return launch_gather_bits<2>(a, b, transpose, y_bf16, by_runs, stream);
    case 3: return launch_gather_bits<3>(a, b, transpose, y_bf16, by_runs, stream);
    case 4: return launch_gather_bits<4>(a, b, transpose, y_bf16, by_runs, stream);
    case 5: return launch_gather_bits<5>(a, b, transpose, y_bf16, by_runs, stream);
    case 6: return launch_gather_bits<6>(a, b, transpose, y_bf16, by_runs, stream);
    case 8: return launch_gather_bits<8>(a, b, transpose, y_bf16, by_runs, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qmm
