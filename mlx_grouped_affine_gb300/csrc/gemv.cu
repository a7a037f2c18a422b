// Decode path of quantized_matmul in bf16 (M <= 16) and the fused decode
// GEMVs.  The kernels are in gemv_impl.cuh; gather_qmm's instantiations
// compile beside these in gemv_gather.cu.
#include "gemv_impl.cuh"

namespace qmm {
namespace {

// The fused decode GEMVs: transposed W, K a multiple of 128; dual for
// M <= 16, silu for M <= 8.
template <int BITS>
cudaError_t launch_fused_bits(const GemvArgs &a, int fuse, const FuseArgs &f, const uint32_t *w2,
                              bool y_bf16, bool pdl, cudaStream_t stream) {
  if (fuse == kFuseDual) {
    Batches two;
    two.count = 2;
    // Both weights' row tiles together more than two 16-warp blocks an SM hold:
    // 8-warp blocks, as for the plain decode GEMV.
    if (BITS < 6 && a.M <= 8 && 2 * ((a.N + 15) / 16) > 2 * sm_count())
      return y_bf16 ? launch_t_tma<ElemBF16, BITS, 1, true, false, kFuseDual, 8>(a, pdl, two, stream, f, w2)
                    : launch_t_tma<ElemBF16, BITS, 1, false, false, kFuseDual, 8>(a, pdl, two, stream, f, w2);
    if (a.M <= 8)
      return y_bf16 ? launch_t_tma<ElemBF16, BITS, 1, true, false, kFuseDual>(a, pdl, two, stream, f, w2)
                    : launch_t_tma<ElemBF16, BITS, 1, false, false, kFuseDual>(a, pdl, two, stream, f, w2);
    return y_bf16 ? launch_t_tma<ElemBF16, BITS, 2, true, false, kFuseDual>(a, pdl, two, stream, f, w2)
                  : launch_t_tma<ElemBF16, BITS, 2, false, false, kFuseDual>(a, pdl, two, stream, f, w2);
  }
  const Batches one;
  return y_bf16 ? launch_t_tma<ElemBF16, BITS, 1, true, false, kFuseSilu>(a, pdl, one, stream, f)
                : launch_t_tma<ElemBF16, BITS, 1, false, false, kFuseSilu>(a, pdl, one, stream, f);
}

cudaError_t launch_fused(const GemvArgs &a, int bits, int fuse, const FuseArgs &f,
                         const uint32_t *w2, bool y_bf16, cudaStream_t stream) {
  const bool pdl = (launch_flags() & kLaunchPdl) != 0;
  switch (bits) {
    case 1: return launch_fused_bits<1>(a, fuse, f, w2, y_bf16, pdl, stream);
    case 2: return launch_fused_bits<2>(a, fuse, f, w2, y_bf16, pdl, stream);
    case 3: return launch_fused_bits<3>(a, fuse, f, w2, y_bf16, pdl, stream);
    case 4: return launch_fused_bits<4>(a, fuse, f, w2, y_bf16, pdl, stream);
    case 5: return launch_fused_bits<5>(a, fuse, f, w2, y_bf16, pdl, stream);
    case 6: return launch_fused_bits<6>(a, fuse, f, w2, y_bf16, pdl, stream);
    case 8: return launch_fused_bits<8>(a, fuse, f, w2, y_bf16, pdl, stream);
    default: return cudaErrorInvalidValue;
  }
}

GemvArgs transposed_args(const uint16_t *x, int64_t M, const PackedWeight &w, void *y) {
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
  return a;
}

}  // namespace

cudaError_t launch_gate_up(const uint16_t *x, int64_t M, const PackedWeight &gate,
                           const PackedWeight &up, void *y_gate, void *y_up, bool y_bf16,
                           cudaStream_t stream) {
  if (gate.cols % 128 != 0 || M > 16) return cudaErrorNotSupported;
  GemvArgs a = transposed_args(x, M, gate, y_gate);
  FuseArgs f{up.scales, up.biases, y_up, nullptr, nullptr};
  return launch_fused(a, gate.bits, kFuseDual, f, up.w, y_bf16, stream);
}

cudaError_t launch_silu_gate(const uint16_t *gate, const uint16_t *up, int64_t M,
                             const PackedWeight &w, const uint16_t *resid, void *y, bool y_bf16,
                             cudaStream_t stream) {
  if (w.cols % 128 != 0 || M > 8) return cudaErrorNotSupported;
  GemvArgs a = transposed_args(nullptr, M, w, y);
  a.resid = resid;
  FuseArgs f{nullptr, nullptr, nullptr, gate, up};
  return launch_fused(a, w.bits, kFuseSilu, f, nullptr, y_bf16, stream);
}

cudaError_t launch_gemv(const uint16_t *x, int64_t M, const PackedWeight &w, bool transpose,
                        void *y, bool y_bf16, cudaStream_t stream) {
  return gemv_entry<ElemBF16>(x, M, w, transpose, y, y_bf16, stream);
}

}  // namespace qmm
