// Down-projection x·[W^DQ | W^DKV | W^KR] (MlaPrologV2 README: c^Q, c^KV and k^R formulas).
#include "gemm_launch.cuh"

namespace mlap {

// Full quant: int8 W^DQ and W^DKV|W^KR expanded to f16 by the converter warps (exact).  Decode
// orientation: the converters expand the int8 token_x tiles too (WQ = 3), so the activation is
// an input of the call; otherwise the activation is the f16-widened token_x.
static cudaError_t launch_down_int8(const GemmLaunch& L, const DownParams& p) {
  if (L.swap) {
    switch (L.bn) {
      case 16: return launch_gemm_t<16, 3, 1>(L, EpiDown<true, 128, 16>{p});
      case 32: return launch_gemm_t<32, 3, 1>(L, EpiDown<true, 128, 32>{p});
      case 64: return launch_gemm_t<64, 3, 1>(L, EpiDown<true, 128, 32>{p});
      case 128: return launch_gemm_t<128, 3, 1>(L, EpiDown<true, 128, 32>{p});
      case 256: return launch_gemm_t<256, 3, 1>(L, EpiDown<true, 128, 32>{p});
      default: return cudaErrorInvalidValue;
    }
  }
  if (L.bn != 192) return cudaErrorInvalidValue;
  return launch_gemm_t<192, 2>(L, EpiDown<false, 192, 32>{p});
}

cudaError_t launch_down(const GemmLaunch& L, const DownParams& p) {
  if (L.a_int8) return launch_down_int8(L, p);
  if (L.swap) {
    if (L.mt == 2 && L.bn > 128) return cudaErrorInvalidValue;   // two accumulators must fit TMEM
    switch (L.bn) {
      case 16: return L.mt == 2 ? launch_gemm_t<16, 0, 2, 1>(L, EpiDown<true, 256, 16>{p})
                           : launch_gemm_t<16, 0, 1, 1>(L, EpiDown<true, 128, 16>{p});
      case 32: return L.mt == 2 ? launch_gemm_t<32, 0, 2, 1>(L, EpiDown<true, 256, 32>{p})
                           : launch_gemm_t<32, 0, 1, 1>(L, EpiDown<true, 128, 32>{p});
      case 64: return L.mt == 2 ? launch_gemm_t<64, 0, 2, 1>(L, EpiDown<true, 256, 32>{p})
                           : launch_gemm_t<64, 0, 1, 1>(L, EpiDown<true, 128, 32>{p});
      case 128: return L.mt == 2 ? launch_gemm_t<128, 0, 2, 1>(L, EpiDown<true, 256, 32>{p})
                           : launch_gemm_t<128, 0, 1, 1>(L, EpiDown<true, 128, 32>{p});
      case 256: return launch_gemm_t<256, 0, 1, 1>(L, EpiDown<true, 128, 32>{p});
      default: return cudaErrorInvalidValue;
    }
  }
  if (L.bn == 256) {
    if (L.cg == 2) return launch_gemm_t<256, 0, 1, 0, 2>(L, EpiDown<false, 256, 32>{p});
    return launch_gemm_t<256>(L, EpiDown<false, 256, 32>{p});
  }
  if (L.bn != 192) return cudaErrorInvalidValue;
  return launch_gemm_t<192>(L, EpiDown<false, 192, 32>{p});
}

}  // namespace mlap
