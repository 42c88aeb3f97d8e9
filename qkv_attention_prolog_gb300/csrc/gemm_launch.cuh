// Host-side launcher for one instantiation of umma_gemm_kernel.
#pragma once
#include "internal.h"

namespace mlap {

template <int BN, int WQ = 0, int MT = 1, int ALD = 0, int CG = 1, class Epi>
cudaError_t launch_gemm_t(const GemmLaunch& L, const Epi& epi) {
  auto kern = umma_gemm_kernel<BN, Epi, WQ, MT, ALD, CG>;
  constexpr int kSmem = GemmCfg<BN, WQ, MT, ALD, CG>::SMEM_BYTES;
  // The dynamic shared memory opt-in is a per-device function attribute; setting it on every
  // launch costs little next to the launch itself and stays correct across devices.
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  if (CG == 2 && (L.grid % 2) != 0) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(L.grid));
  cfg.blockDim = dim3(GemmCfg<BN, WQ, MT, ALD, CG>::THREADS);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (L.pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (CG == 2) {   // CTA pairs: clusters of two along x
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 2;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, L.a0, L.a1, L.b0, L.b1, L.o0, L.o1, L.geo, epi, L.err);
}

}  // namespace mlap
