// Up-projection c^Q·[W^UQ | W^QR] with fused q^C rounding and query RoPE (MlaPrologV2 README:
// q^C and q^R formulas; RoPE of aclnnQkvRmsNormRopeCache "Formulas" (3)).
#include "gemm_launch.cuh"

namespace mlap {

cudaError_t launch_up(const GemmLaunch& L, const UpParams& p, bool int8) {
  if (int8) return cudaErrorNotSupported;
  if (L.swap) {
    switch (L.bn) {
      case 16: return launch_gemm_t<16>(L, EpiUp<true, false, 16>{p});
      case 32: return launch_gemm_t<32>(L, EpiUp<true, false, 32>{p});
      case 64: return launch_gemm_t<64>(L, EpiUp<true, false, 32>{p});
      case 128: return launch_gemm_t<128>(L, EpiUp<true, false, 32>{p});
      case 256: return launch_gemm_t<256>(L, EpiUp<true, false, 32>{p});
      default: return cudaErrorInvalidValue;
    }
  }
  if (L.bn != 256) return cudaErrorInvalidValue;
  return launch_gemm_t<256>(L, EpiUp<false, false, 32>{p});
}

}  // namespace mlap
