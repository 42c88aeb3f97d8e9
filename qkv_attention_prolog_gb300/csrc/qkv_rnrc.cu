// QkvRmsNormRopeCache (aclnnQkvRmsNormRopeCache, "Formulas" (1)-(4) and "Other restrictions"):
//
//   q, k, v = SplitVD(qkv)                  heads [0,Nq) | [Nq, Nq+Nk) | [Nq+Nk, Nq+Nk+Nv)
//   y       = x / sqrt(mean(x^2) + eps) * gamma                      per q / k head, along D
//   y_embed = y * cos + cat(-y2, y1) * sin                           half-and-half, d = D
//   q_out   = y_embed(q);  k_cache[i] = Quant(y_embed(k));  v_cache[i] = Quant(v)
//   Quant   = identity, or value / scale rounded half to even and saturated to int8
//
// A pure HBM stream: every token's qkv row is read once and its outputs written once.  Sixteen
// lanes own one head row of D = 128 elements (16 bytes each); the RmsNorm sum is a 16-lane
// shuffle reduction and each RoPE partner (j, j + 64) sits 8 lanes away.  Each half-warp keeps
// two rows in flight.
#include "internal.h"

namespace mlap {

namespace {

constexpr int kD = 128;
constexpr int kThreads = 256;

template <bool BF16>
struct Elem;
template <>
struct Elem<false> {
  using T = __half;
  static __device__ __forceinline__ float to_f(T v) { return __half2float(v); }
  static __device__ __forceinline__ T from_f(float v) { return __float2half_rn(v); }
};
template <>
struct Elem<true> {
  using T = __nv_bfloat16;
  static __device__ __forceinline__ float to_f(T v) { return __bfloat162float(v); }
  static __device__ __forceinline__ T from_f(float v) { return __float2bfloat16_rn(v); }
};

template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4& raw, float (&x)[8]) {
  using E = Elem<BF16>;
  const typename E::T* e = reinterpret_cast<const typename E::T*>(&raw);
#pragma unroll
  for (int i = 0; i < 8; ++i) x[i] = E::to_f(e[i]);
}

template <bool BF16>
__device__ __forceinline__ uint4 pack8(const float (&x)[8]) {
  using E = Elem<BF16>;
  uint4 raw;
  typename E::T* e = reinterpret_cast<typename E::T*>(&raw);
#pragma unroll
  for (int i = 0; i < 8; ++i) e[i] = E::from_f(x[i]);
  return raw;
}

__device__ __forceinline__ uint2 quant8(const float (&x)[8], const float* scale) {
  const float4 s0 = reinterpret_cast<const float4*>(scale)[0];
  const float4 s1 = reinterpret_cast<const float4*>(scale)[1];
  const float sc[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
  uint2 out;
  int8_t* o = reinterpret_cast<int8_t*>(&out);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    int q = __float2int_rn(__fdiv_rn(x[i], sc[i]));
    q = q < -128 ? -128 : (q > 127 ? 127 : q);
    o[i] = static_cast<int8_t>(q);
  }
  return out;
}

template <bool BF16, bool QUANT>
__global__ void __launch_bounds__(kThreads) qkv_rnrc_kernel(const QkvParams p) {
  using E = Elem<BF16>;
  using T = typename E::T;
  grid_launch_dependents();
  grid_dependency_wait();
  const int Nh = p.Nq + p.Nk + p.Nv;
  const int64_t rows = static_cast<int64_t>(p.T) * Nh;
  const int hl = threadIdx.x & 15;                                  // lane within the half-warp
  const unsigned mask = 0xffffu << (threadIdx.x & 16);              // this half-warp's lanes
  const int64_t hw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 4;
  const int64_t nhw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 4;
  const int j0 = hl * 8;                                            // first element of this lane

  for (int64_t base = hw; base < rows; base += 2 * nhw) {
    uint4 raw[2];
    int64_t r[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      r[u] = base + u * nhw;
      if (r[u] < rows)
        raw[u] = reinterpret_cast<const uint4*>(static_cast<const T*>(p.qkv) + r[u] * kD)[hl];
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (r[u] >= rows) break;                                      // uniform in the half-warp
      const int t = static_cast<int>(r[u] / Nh);
      const int h = static_cast<int>(r[u] % Nh);
      float x[8];
      unpack8<BF16>(raw[u], x);
      const int64_t idx = p.index[t];
      const bool store = idx >= 0 && idx < p.slots;
      if (h < p.Nq + p.Nk) {
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) ss += x[i] * x[i];
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) ss += __shfl_xor_sync(mask, ss, o);
        const float rinv = 1.0f / sqrtf(ss / static_cast<float>(kD) + p.eps);
        const bool is_q = h < p.Nq;
        float g[8], c[8], s[8];
        unpack8<BF16>(reinterpret_cast<const uint4*>(is_q ? p.gamma_q : p.gamma_k)[hl], g);
        unpack8<BF16>(reinterpret_cast<const uint4*>(static_cast<const T*>(p.cos) +
                                                     static_cast<size_t>(t) * kD)[hl], c);
        unpack8<BF16>(reinterpret_cast<const uint4*>(static_cast<const T*>(p.sin) +
                                                     static_cast<size_t>(t) * kD)[hl], s);
        float y[8], e[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) y[i] = x[i] * rinv * g[i];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float partner = __shfl_xor_sync(mask, y[i], 8);    // element j +- 64
          e[i] = y[i] * c[i] + (hl < 8 ? -partner : partner) * s[i];
        }
        if (is_q) {
          reinterpret_cast<uint4*>(static_cast<T*>(p.q_out) +
                                   (static_cast<size_t>(t) * p.Nq + h) * kD)[hl] = pack8<BF16>(e);
        } else if (store) {
          const int hk = h - p.Nq;
          const size_t off = (static_cast<size_t>(idx) * p.Nk + hk) * kD;
          if (QUANT)
            reinterpret_cast<uint2*>(static_cast<int8_t*>(p.k_cache) + off)[hl] =
                quant8(e, p.k_scale + hk * kD + j0);
          else
            reinterpret_cast<uint4*>(static_cast<T*>(p.k_cache) + off)[hl] = pack8<BF16>(e);
        }
      } else if (store) {
        const int hv = h - p.Nq - p.Nk;
        const size_t off = (static_cast<size_t>(idx) * p.Nv + hv) * kD;
        if (QUANT)
          reinterpret_cast<uint2*>(static_cast<int8_t*>(p.v_cache) + off)[hl] =
              quant8(x, p.v_scale + hv * kD + j0);
        else
          reinterpret_cast<uint4*>(static_cast<T*>(p.v_cache) + off)[hl] = raw[u];
      }
      if (h == 0 && hl == 0 && idx != -1 && !store && p.slots > 0) atomicOr(p.err, kErrIndexRange);
    }
  }
}

}  // namespace

cudaError_t launch_qkv_rnrc(const QkvParams& p, cudaStream_t stream, int sm_count) {
  const int64_t rows = static_cast<int64_t>(p.T) * (p.Nq + p.Nk + p.Nv);
  const int64_t half_warps_needed = (rows + 1) / 2;
  int64_t blocks = (half_warps_needed * 16 + kThreads - 1) / kThreads;
  const int64_t cap = static_cast<int64_t>(sm_count) * (2048 / kThreads);   // one full wave
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const bool quant = p.k_scale != nullptr;
  if (p.bf16) {
    return quant ? cudaLaunchKernelEx(&cfg, qkv_rnrc_kernel<true, true>, p)
                 : cudaLaunchKernelEx(&cfg, qkv_rnrc_kernel<true, false>, p);
  }
  return quant ? cudaLaunchKernelEx(&cfg, qkv_rnrc_kernel<false, true>, p)
               : cudaLaunchKernelEx(&cfg, qkv_rnrc_kernel<false, false>, p);
}

}  // namespace mlap
