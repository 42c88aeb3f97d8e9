// Execution stamps: %globaltimer readings a kernel writes, when the caller asks for them, so that
// the time of each kernel inside a pipelined call (kernels overlapping through programmatic
// dependent launch) can be read back without events between the launches.  Layout of the
// caller's buffer (MLAP_STAMP_KERNELS slots of MLAP_STAMP_BLOCK 64-bit words, zeroed before the
// call): word 0 of slot k holds the bitwise complement of the earliest CTA start (a max of the
// complements is a min), word 1 the latest CTA end, and words 4 + 4c .. 4 + 4c + 3 the four
// stamps of CTA c < MLAP_STAMP_CTAS: start, dependency resolved, main work done, end.
#pragma once
#include <cstdint>

#include "mlaprolog.h"
#include "ptx.cuh"

namespace mlap {

enum : int { kStampStart = 0, kStampDep = 1, kStampMain = 2, kStampEnd = 3 };

__device__ __forceinline__ void stamp(uint64_t* s, int k, int what) {
  if (s == nullptr) return;
  const uint64_t t = globaltimer_ns();
  unsigned long long* b = reinterpret_cast<unsigned long long*>(s) +
                          static_cast<size_t>(k) * MLAP_STAMP_BLOCK;
  if (what == kStampStart) atomicMax(b, ~static_cast<unsigned long long>(t));
  if (what == kStampEnd) atomicMax(b + 1, static_cast<unsigned long long>(t));
  if (blockIdx.x < MLAP_STAMP_CTAS) b[4 + 4 * blockIdx.x + what] = t;
}

}  // namespace mlap
