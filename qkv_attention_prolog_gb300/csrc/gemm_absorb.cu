// Per-head absorb q^N = q^C·W^UK (MlaPrologV2 README: q^N formula), batched over heads.
#include "gemm_launch.cuh"

namespace mlap {

cudaError_t launch_absorb(const GemmLaunch& L, const AbsorbParams& p) {
  if (L.swap) {
    if (L.mt == 2 && L.bn > 128) return cudaErrorInvalidValue;   // two accumulators must fit TMEM
    switch (L.bn) {
      case 16: return L.mt == 2 ? launch_gemm_t<16, 0, 2, 1>(L, EpiAbsorb<true, 16>{p})
                           : launch_gemm_t<16, 0, 1, 1>(L, EpiAbsorb<true, 16>{p});
      case 32: return L.mt == 2 ? launch_gemm_t<32, 0, 2, 1>(L, EpiAbsorb<true, 32>{p})
                           : launch_gemm_t<32, 0, 1, 1>(L, EpiAbsorb<true, 32>{p});
      case 64: return L.mt == 2 ? launch_gemm_t<64, 0, 2, 1>(L, EpiAbsorb<true, 32>{p})
                           : launch_gemm_t<64, 0, 1, 1>(L, EpiAbsorb<true, 32>{p});
      case 128: return L.mt == 2 ? launch_gemm_t<128, 0, 2, 1>(L, EpiAbsorb<true, 32>{p})
                           : launch_gemm_t<128, 0, 1, 1>(L, EpiAbsorb<true, 32>{p});
      case 256: return launch_gemm_t<256, 0, 1, 1>(L, EpiAbsorb<true, 32>{p});
      default: return cudaErrorInvalidValue;
    }
  }
  if (L.bn != 256) return cudaErrorInvalidValue;
  if (L.rr) return launch_gemm_t<256>(L, EpiAbsorb<false, 32, true>{p});
  return launch_gemm_t<256>(L, EpiAbsorb<false, 64>{p});   // whole 128-byte lines per store
}

}  // namespace mlap
