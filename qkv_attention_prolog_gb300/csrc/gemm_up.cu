// Up-projection c^Q·[W^UQ | W^QR] with fused q^C rounding and query RoPE (MlaPrologV2 README:
// q^C and q^R formulas; RoPE of aclnnQkvRmsNormRopeCache "Formulas" (3)), for a bf16 weight or an
// int8 weight with per-channel dequant (the partial-quant scenario).
#include "gemm_launch.cuh"

namespace mlap {

template <bool INT8>
static cudaError_t launch_up_t(const GemmLaunch& L, const UpParams& p) {
  constexpr int WA = INT8 ? 1 : 0;   // int8 weight as operand A (decode orientation)
  constexpr int WB = INT8 ? 2 : 0;   // int8 weight as operand B (prefill orientation)
  constexpr int AL = INT8 ? 0 : 1;   // bf16 weight: activation through the cp.async loaders
  if (L.swap) {
    if (L.mt == 2 && L.bn > 128) return cudaErrorInvalidValue;   // two accumulators must fit TMEM
    switch (L.bn) {
      case 16: return L.mt == 2 ? launch_gemm_t<16, WA, 2, AL>(L, EpiUp<true, INT8, 16>{p})
                           : launch_gemm_t<16, WA, 1, AL>(L, EpiUp<true, INT8, 16>{p});
      case 32: return L.mt == 2 ? launch_gemm_t<32, WA, 2, AL>(L, EpiUp<true, INT8, 32>{p})
                           : launch_gemm_t<32, WA, 1, AL>(L, EpiUp<true, INT8, 32>{p});
      case 64: return L.mt == 2 ? launch_gemm_t<64, WA, 2, AL>(L, EpiUp<true, INT8, 32>{p})
                           : launch_gemm_t<64, WA, 1, AL>(L, EpiUp<true, INT8, 32>{p});
      case 128: return L.mt == 2 ? launch_gemm_t<128, WA, 2, AL>(L, EpiUp<true, INT8, 32>{p})
                           : launch_gemm_t<128, WA, 1, AL>(L, EpiUp<true, INT8, 32>{p});
      case 256: return launch_gemm_t<256, WA, 1, AL>(L, EpiUp<true, INT8, 32>{p});
      default: return cudaErrorInvalidValue;
    }
  }
  if (L.bn != 256) return cudaErrorInvalidValue;
  if constexpr (!INT8) {
    if (L.rr) return launch_gemm_t<256>(L, EpiUp<false, false, 32, true>{p});
    if (L.cg == 2) return launch_gemm_t<256, 0, 1, 0, 2>(L, EpiUp<false, false, 32>{p});
  }
  return launch_gemm_t<256, WB>(L, EpiUp<false, INT8, 32>{p});
}

cudaError_t launch_up(const GemmLaunch& L, const UpParams& p, bool int8) {
  return int8 ? launch_up_t<true>(L, p) : launch_up_t<false>(L, p);
}

}  // namespace mlap
