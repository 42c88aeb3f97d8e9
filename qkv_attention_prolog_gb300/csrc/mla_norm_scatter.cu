// RmsNorm / RoPE / quant / paged-scatter step of the MLA prolog, and the weight prepack kernel.
//
// norm_rope_scatter_kernel, one CTA per token t:
//   h        = sum over K-splits s (in order) of part[s][t][:]            (down-projection result)
//   c^Q      = RmsNorm(h[0:Hcq]; gamma_cq, eps_cq) rounded to bf16          (MlaPrologV2 README,
//              c^Q = RmsNorm(x·W^DQ); RmsNorm公式: eps added to the mean inside the root)
//   partial quant: s = c^Q * smooth_scales_cq; scale_t = max|s| / 127; code = rne(s / scale_t)
//              clamped to [-127, 127], all in fp32 (reading of the smooth_scales_cq parameter)
//   c^KV     = RmsNorm(h[Hcq:Hcq+Hckv]; gamma_ckv, eps_ckv)  -> kv_cache[cache_index[t]]
//   k^R      = RoPE(h[Hcq+Hckv:]; cos[t], sin[t])             -> kr_cache[cache_index[t]]
//              (half-and-half rule of aclnnQkvRmsNormRopeCache "Formulas" (3))
//   int8 caches: rne(value / quant_scale[j]) saturated to [-128, 127] ("Formulas" (4) division).
//   cache_index = -1 skips the token; other values outside [0, slots) are skipped and latched.
// With Nkv = 1 and a dense (BlockNum, BlockSize, 1, H) cache, slot i is row i of the cache.
#include "internal.h"

namespace mlap {

namespace {

constexpr int kNormThreads = 256;
constexpr int kMaxSplits = 16;   // upper bound on the down-projection's K splits

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float r = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) r += red[i];   // fixed order: deterministic
  return r;
}

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float r = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) r = fmaxf(r, red[i]);
  return r;
}

__device__ __forceinline__ int8_t quant_i8(float v, float scale, int lo, int hi) {
  int q = __float2int_rn(__fdiv_rn(v, scale));
  q = q < lo ? lo : (q > hi ? hi : q);
  return static_cast<int8_t>(q);
}

__global__ void __launch_bounds__(kNormThreads)
    norm_rope_scatter_kernel(const FinalizeParams p) {
  extern __shared__ float h[];
  __shared__ float red[32];
  const int t = blockIdx.x;
  grid_launch_dependents();
  grid_dependency_wait();

  // h = sum of the K-split partials, in split order.  All splits of a column are loaded before
  // the first add so up to kMaxSplits loads per thread are in flight.
  const size_t split_stride = static_cast<size_t>(p.T) * p.Ntot;
  const float* src = p.part + static_cast<size_t>(t) * p.Ntot;
  const bool vec = (p.Ntot % 4) == 0;                     // rows then start 16-byte aligned
  const int ncols = vec ? p.Ntot / 4 : p.Ntot;
  for (int c = threadIdx.x; c < ncols; c += blockDim.x) {
    if (vec) {
      float4 v[kMaxSplits];
#pragma unroll
      for (int s = 0; s < kMaxSplits; ++s)
        if (s < p.splits) v[s] = __ldg(reinterpret_cast<const float4*>(src + s * split_stride) + c);
      float4 a = v[0];
#pragma unroll
      for (int s = 1; s < kMaxSplits; ++s)
        if (s < p.splits) {
          a.x += v[s].x;
          a.y += v[s].y;
          a.z += v[s].z;
          a.w += v[s].w;
        }
      reinterpret_cast<float4*>(h)[c] = a;
    } else {
      float v[kMaxSplits];
#pragma unroll
      for (int s = 0; s < kMaxSplits; ++s)
        if (s < p.splits) v[s] = __ldg(src + s * split_stride + c);
      float a = v[0];
#pragma unroll
      for (int s = 1; s < kMaxSplits; ++s)
        if (s < p.splits) a += v[s];
      h[c] = a;
    }
  }
  __syncthreads();

  // ---- c^Q
  float ss = 0.f;
  for (int f = threadIdx.x; f < p.Hcq; f += blockDim.x) ss += h[f] * h[f];
  ss = block_sum(ss, red);
  const float rq = 1.0f / sqrtf(ss / static_cast<float>(p.Hcq) + p.eps_cq);
  __nv_bfloat16* cq = p.cq_out + static_cast<size_t>(t) * p.Hcq;
  if (p.smooth == nullptr) {
    for (int f = threadIdx.x; f < p.Hcq; f += blockDim.x)
      cq[f] = __float2bfloat16_rn(h[f] * rq * __bfloat162float(p.gamma_cq[f]));
  } else {
    float amax = 0.f;
    for (int f = threadIdx.x; f < p.Hcq; f += blockDim.x) {
      const float c = __bfloat162float(
          __float2bfloat16_rn(h[f] * rq * __bfloat162float(p.gamma_cq[f])));
      amax = fmaxf(amax, fabsf(__fmul_rn(c, p.smooth[f])));
    }
    amax = block_max(amax, red);
    const float scale = __fdiv_rn(amax, 127.0f);
    for (int f = threadIdx.x; f < p.Hcq; f += blockDim.x) {
      const float c = __bfloat162float(
          __float2bfloat16_rn(h[f] * rq * __bfloat162float(p.gamma_cq[f])));
      const float s = __fmul_rn(c, p.smooth[f]);
      const int code = scale > 0.f ? quant_i8(s, scale, -127, 127) : 0;
      cq[f] = __float2bfloat16_rn(static_cast<float>(code));   // exact: |code| <= 127
    }
    if (threadIdx.x == 0) p.scale_t[t] = scale;
  }

  // ---- c^KV
  const float* hkv = h + p.Hcq;
  float sk = 0.f;
  for (int f = threadIdx.x; f < p.Hckv; f += blockDim.x) sk += hkv[f] * hkv[f];
  sk = block_sum(sk, red);
  const float rkv = 1.0f / sqrtf(sk / static_cast<float>(p.Hckv) + p.eps_ckv);

  if (p.slots <= 0) return;                 // empty caches: outputs only
  const int64_t idx = p.cache_index[t];
  if (idx < 0 || idx >= p.slots) {
    if (idx != -1 && threadIdx.x == 0) atomicOr(p.err, kErrIndexRange);
    return;
  }
  for (int f = threadIdx.x; f < p.Hckv; f += blockDim.x) {
    const float v = hkv[f] * rkv * __bfloat162float(p.gamma_ckv[f]);
    if (p.kv_int8)
      static_cast<int8_t*>(p.kv_cache)[idx * p.Hckv + f] = quant_i8(v, p.qs_ckv[f], -128, 127);
    else
      static_cast<__nv_bfloat16*>(p.kv_cache)[idx * p.Hckv + f] = __float2bfloat16_rn(v);
  }
  // ---- k^R
  const float* hkr = h + p.Hcq + p.Hckv;
  const int half = p.Dr >> 1;
  for (int j = threadIdx.x; j < p.Dr; j += blockDim.x) {
    const float y = hkr[j];
    const float partner = j < half ? -hkr[j + half] : hkr[j - half];
    const float c = __bfloat162float(p.cos[static_cast<size_t>(t) * p.Dr + j]);
    const float s = __bfloat162float(p.sin[static_cast<size_t>(t) * p.Dr + j]);
    const float v = y * c + partner * s;
    if (p.kr_int8)
      static_cast<int8_t*>(p.kr_cache)[idx * p.Dr + j] = quant_i8(v, p.qs_ckr[j], -128, 127);
    else
      static_cast<__nv_bfloat16*>(p.kr_cache)[idx * p.Dr + j] = __float2bfloat16_rn(v);
  }
}

// dst[b][i][k] = src[b][k][perm(i)], 32x32 tiles through shared memory.
template <typename E>
__global__ void prepack_kernel(const PrepackParams p) {
  __shared__ E tile[32][33];
  const int b = blockIdx.z;
  const int i0 = blockIdx.x * 32, k0 = blockIdx.y * 32;
  const E* src = static_cast<const E*>(p.src) + static_cast<size_t>(b) * p.K * p.C;
  E* dst = static_cast<E*>(p.dst) + static_cast<size_t>(b) * p.R * p.K;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8 threads
  const int i = i0 + tx;
  int col = -1;
  if (i < p.R) {
    if (p.perm == kPermIdentity) {
      col = i;
    } else {
      const int nd = p.N * p.D;
      if (i < nd) {
        col = (i / p.D) * (p.D + p.Dr) + (i % p.D);
      } else {
        const int r = i - nd, n = r / p.Dr, q = r % p.Dr;
        col = n * (p.D + p.Dr) + p.D + (q >> 1) + (q & 1) * (p.Dr >> 1);
      }
    }
  }
  for (int kk = ty; kk < 32; kk += 8) {
    const int k = k0 + kk;
    if (col >= 0 && k < p.K) tile[kk][tx] = src[static_cast<size_t>(k) * p.C + col];
  }
  __syncthreads();
  for (int ii = ty; ii < 32; ii += 8) {
    const int io = i0 + ii, k = k0 + tx;
    if (io < p.R && k < p.K) dst[static_cast<size_t>(io) * p.K + k] = tile[tx][ii];
  }
}

}  // namespace

cudaError_t launch_finalize(const FinalizeParams& p, cudaStream_t stream, bool pdl) {
  const size_t smem = static_cast<size_t>(p.Ntot) * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(norm_rope_scatter_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.T));
  cfg.blockDim = dim3(kNormThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, norm_rope_scatter_kernel, p);
}

cudaError_t launch_prepack(const PrepackParams& p, cudaStream_t stream) {
  dim3 grid((p.R + 31) / 32, (p.K + 31) / 32, p.batches);
  if (grid.y > 65535u || grid.z > 65535u) return cudaErrorInvalidValue;
  if (p.elem_bytes == 2)
    prepack_kernel<uint16_t><<<grid, 256, 0, stream>>>(p);
  else if (p.elem_bytes == 1)
    prepack_kernel<uint8_t><<<grid, 256, 0, stream>>>(p);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace mlap
