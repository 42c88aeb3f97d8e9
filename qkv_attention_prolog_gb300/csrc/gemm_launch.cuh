// Host-side launcher for one instantiation of umma_gemm_kernel.
#pragma once
#include "internal.h"

namespace mlap {

template <int BN, int WQ = 0, int MT = 1, int ALD = 0, class Epi>
cudaError_t launch_gemm_t(const GemmLaunch& L, const Epi& epi) {
  auto kern = umma_gemm_kernel<BN, Epi, WQ, MT, ALD>;
  constexpr int kSmem = GemmCfg<BN, WQ, MT, ALD>::SMEM_BYTES;
  // The dynamic shared memory opt-in is a per-device function attribute; setting it on every
  // launch costs little next to the launch itself and stays correct across devices.
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(L.grid));
  cfg.blockDim = dim3(GemmCfg<BN, WQ, MT, ALD>::THREADS);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = L.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, L.a0, L.a1, L.b0, L.b1, L.o0, L.o1, L.geo, epi, L.err);
}

}  // namespace mlap
