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
//   full quant: h *= dequant_scale_x[t] * dequant_scale_w[column] after the split sum (the int8
//   products are exact), and the two helper kernels below (token_x widening beyond 256 tokens,
//   int8 query).
// rms_norm_quant_kernel: the optional input RmsNormQuant that runs ahead of the down-projection.
// With Nkv = 1 and a dense (BlockNum, BlockSize, 1, H) cache, slot i is row i of the cache.
#include "internal.h"

namespace mlap {

namespace {

constexpr int kMaxSplits = 16;   // upper bound on the down-projection's K splits

// Block reductions (every thread gets the result).  The buffer may be written again by a later
// reduction only with kReuse, which adds the barrier that lets every thread read it first.
template <int NT, bool kReuse = false>
__device__ __forceinline__ float2 block_sum2(float2 v, float2* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
    v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = v;
  __syncthreads();
  float2 r = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < NT / 32; ++i) {            // fixed order: deterministic
    r.x += red[i].x;
    r.y += red[i].y;
  }
  if (kReuse) __syncthreads();
  return r;
}

template <int NT, bool kReuse = false>
__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = v;
  __syncthreads();
  float r = 0.f;
#pragma unroll
  for (int i = 0; i < NT / 32; ++i) r = fmaxf(r, red[i]);
  if (kReuse) __syncthreads();
  return r;
}

__device__ __forceinline__ int8_t quant_i8(float v, float scale, int lo, int hi) {
  int q = __float2int_rn(__fdiv_rn(v, scale));
  q = q < lo ? lo : (q > hi ? hi : q);
  return static_cast<int8_t>(q);
}

__device__ __forceinline__ void load8_bf16(const __nv_bfloat16* p, float* out) {
  const uint4 r = __ldg(reinterpret_cast<const uint4*>(p));
  const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&r);
#pragma unroll
  for (int i = 0; i < 8; ++i) out[i] = __bfloat162float(e[i]);
}

__device__ __forceinline__ void store8_bf16(__nv_bfloat16* p, const float* v) {
  uint4 r;
  __nv_bfloat162* e = reinterpret_cast<__nv_bfloat162*>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) e[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
  *reinterpret_cast<uint4*>(p) = r;
}

// One CTA per token, or with PARTS two: CTA 2t the c^Q columns of token t, CTA 2t+1 its c^KV and
// k^R columns (the two norms are independent), so that the c^Q the next kernel waits for comes
// from a CTA with less than three quarters of the work.  MAXS bounds the K splits (1: prefill, no
// split), NT is the thread count: with splits every thread issues the loads of all splits of its
// columns at once (one round of latency), without them the kernel stays small enough for many
// CTAs per SM.
template <int MAXS, int NT, bool PARTS = false>
__global__ void __launch_bounds__(NT) norm_rope_scatter_kernel(const FinalizeParams p) {
  extern __shared__ float h[];
  __shared__ float2 red[NT / 32];                  // the sums of squares (each buffer is used
  __shared__ float redm[NT / 32];                  // once: no barrier after its reduction)
  const int t = PARTS ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const bool do_q = !PARTS || (blockIdx.x & 1) == 0;
  const bool do_kv = !PARTS || (blockIdx.x & 1) == 1;
  const int c0 = do_q ? 0 : p.Hcq;                 // this CTA's columns [c0, c1) of Ntot
  const int c1 = do_kv ? p.Ntot : p.Hcq;
  if (threadIdx.x == 0) stamp(p.stamps, MLAP_STAMP_NORM, kStampStart);
  grid_launch_dependents();
  // Decode (PARTS): the call's inputs this thread needs after the reduction (its gamma slice,
  // the token's RoPE tables and cache index) are read before the wait on the down-projection,
  // so the latency chain after it holds only the partials
  // With partial or full quant also its scale slices: smooth_scales_cq or quant_scale_ckv (8
  // columns, the gamma slice's), quant_scale_ckr (one column) and the full-quant dequant scales
  // (its columns of the split sum, kPreCols at most).
  constexpr int kPreCols = 8;
  uint4 g_pre = make_uint4(0, 0, 0, 0);
  float4 s_pre[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
  float qkr_pre = 0.f, dsx_pre = 0.f, dw_pre[kPreCols];
  __nv_bfloat16 cos_pre = __float2bfloat16(0.f), sin_pre = __float2bfloat16(0.f);
  int64_t idx_pre = -1;
  const int f8 = threadIdx.x * 8;
  if constexpr (PARTS) {
    if (do_q && p.Hcq <= NT * 8 && f8 < p.Hcq) {
      g_pre = __ldg(reinterpret_cast<const uint4*>(p.gamma_cq) + threadIdx.x);
      if (p.smooth != nullptr) {
        s_pre[0] = __ldg(reinterpret_cast<const float4*>(p.smooth + f8));
        s_pre[1] = __ldg(reinterpret_cast<const float4*>(p.smooth + f8) + 1);
      }
    }
    if (do_kv) {
      if (p.Hckv <= NT * 8 && f8 < p.Hckv) {
        g_pre = __ldg(reinterpret_cast<const uint4*>(p.gamma_ckv) + threadIdx.x);
        if (p.kv_int8 && p.slots > 0) {
          s_pre[0] = __ldg(reinterpret_cast<const float4*>(p.qs_ckv + f8));
          s_pre[1] = __ldg(reinterpret_cast<const float4*>(p.qs_ckv + f8) + 1);
        }
      }
      if (threadIdx.x < p.Dr) {
        cos_pre = p.cos[static_cast<size_t>(t) * p.Dr + threadIdx.x];
        sin_pre = p.sin[static_cast<size_t>(t) * p.Dr + threadIdx.x];
        if (p.kr_int8 && p.slots > 0) qkr_pre = __ldg(p.qs_ckr + threadIdx.x);
      }
      if (p.slots > 0) idx_pre = p.cache_index[t];
    }
    if (p.dsx != nullptr) {
      dsx_pre = __ldg(p.dsx + t);
#pragma unroll
      for (int i = 0; i < kPreCols; ++i) {
        const int c = c0 + static_cast<int>(threadIdx.x) + i * NT;
        dw_pre[i] = c < c1 ? __ldg(c < p.Hcq ? p.dsw_q + c : p.dsw_kv + (c - p.Hcq)) : 0.f;
      }
    }
  }
  grid_dependency_wait();
  if (threadIdx.x == 0) stamp(p.stamps, MLAP_STAMP_NORM, kStampDep);
  // the CTA's last stamp, at each of its (CTA-uniform) exits
  auto finish = [&]() {
    if (p.stamps != nullptr) {
      __syncthreads();
      if (threadIdx.x == 0) stamp(p.stamps, MLAP_STAMP_NORM, kStampEnd);
    }
  };

  // h = sum of the K-split partials, in split order.  Without the full-quant dequant the sums of
  // squares are taken from the registers here (a float4 column lies in one part: Hcq and Hckv
  // are multiples of 8), so no barrier and no pass over h precede the reduction.
  const size_t split_stride = static_cast<size_t>(p.T) * p.Ntot;
  const float* src = p.part + static_cast<size_t>(t) * p.Ntot;
  const bool reg_ss = (p.Ntot % 4) == 0 && p.dsx == nullptr;
  float2 ssr = make_float2(0.f, 0.f);
  auto add_ss = [&](int c, const float4& x) {   // column c (float4 units) of the row
    const float q = x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
    if (4 * c < p.Hcq) ssr.x += q;
    else if (4 * c < p.Hcq + p.Hckv) ssr.y += q;
  };
  if ((p.Ntot % 4) == 0) {                       // rows start 16-byte aligned (Hcq % 8 == 0)
    // with at most 8 splits, two columns per thread and round, all their split loads issued
    // before the sums (one L2 round trip where the c^Q CTA's 384 float4 columns take two per
    // thread; with 16 splits the second column's loads would not fit the registers)
    constexpr int kCols = MAXS <= 8 ? 2 : 1;
    const int ncols = c1 / 4;
    for (int c = c0 / 4 + threadIdx.x; c < ncols; c += kCols * NT) {
      const int c2 = kCols == 2 ? c + NT : ncols;
      float4 v[MAXS], w[MAXS];
#pragma unroll
      for (int s = 0; s < MAXS; ++s)
        if (s < p.splits) {
          v[s] = __ldg(reinterpret_cast<const float4*>(src + s * split_stride) + c);
          if (c2 < ncols) w[s] = __ldg(reinterpret_cast<const float4*>(src + s * split_stride) + c2);
        }
      float4 a = v[0];
#pragma unroll
      for (int s = 1; s < MAXS; ++s)
        if (s < p.splits) {
          a.x += v[s].x;
          a.y += v[s].y;
          a.z += v[s].z;
          a.w += v[s].w;
        }
      reinterpret_cast<float4*>(h)[c] = a;
      add_ss(c, a);
      if (c2 < ncols) {
        float4 b = w[0];
#pragma unroll
        for (int s = 1; s < MAXS; ++s)
          if (s < p.splits) {
            b.x += w[s].x;
            b.y += w[s].y;
            b.z += w[s].z;
            b.w += w[s].w;
          }
        reinterpret_cast<float4*>(h)[c2] = b;
        add_ss(c2, b);
      }
    }
  } else {
    for (int c = c0 + threadIdx.x; c < c1; c += NT) {
      float v[MAXS];
#pragma unroll
      for (int s = 0; s < MAXS; ++s)
        if (s < p.splits) v[s] = __ldg(src + s * split_stride + c);
      float a = v[0];
#pragma unroll
      for (int s = 1; s < MAXS; ++s)
        if (s < p.splits) a += v[s];
      h[c] = a;
    }
  }
  if (threadIdx.x == 0) stamp(p.stamps, MLAP_STAMP_NORM, kStampMain);
  if (!reg_ss) __syncthreads();
  if (p.dsx != nullptr) {   // full quant: dequant the exact integer products per token and column
    if (PARTS && c1 - c0 <= kPreCols * NT) {
#pragma unroll
      for (int i = 0; i < kPreCols; ++i) {
        const int c = c0 + static_cast<int>(threadIdx.x) + i * NT;
        if (c < c1) h[c] *= dsx_pre * dw_pre[i];
      }
    } else {
      const float sx = p.dsx[t];
      for (int c = c0 + threadIdx.x; c < c1; c += NT)
        h[c] *= sx * (c < p.Hcq ? p.dsw_q[c] : p.dsw_kv[c - p.Hcq]);
    }
    __syncthreads();
  }

  // sums of squares of the c^Q and c^KV parts, one reduction
  const float* hkv = h + p.Hcq;
  float2 ss = ssr;
  if (!reg_ss) {
    ss = make_float2(0.f, 0.f);
    if (do_q)
      for (int f = threadIdx.x; f < p.Hcq; f += NT) ss.x += h[f] * h[f];
    if (do_kv)
      for (int f = threadIdx.x; f < p.Hckv; f += NT) ss.y += hkv[f] * hkv[f];
  }
  ss = block_sum2<NT>(ss, red);                 // (its barrier also orders h before the reads)
  const float rq = 1.0f / sqrtf(ss.x / static_cast<float>(p.Hcq) + p.eps_cq);
  const float rkv = 1.0f / sqrtf(ss.y / static_cast<float>(p.Hckv) + p.eps_ckv);

  // ---- c^Q (Hcq % 8 == 0): bf16, or int8 codes held exactly in f16
  __nv_bfloat16* cq = p.cq_out + static_cast<size_t>(t) * p.Hcq;
  if (!do_q) {
    // (the c^KV / k^R CTA of a token)
  } else if (p.smooth == nullptr) {
    for (int f = threadIdx.x * 8; f < p.Hcq; f += NT * 8) {
      float g[8], v[8];
      if (PARTS && p.Hcq <= NT * 8) {
        const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&g_pre);
#pragma unroll
        for (int i = 0; i < 8; ++i) g[i] = __bfloat162float(e[i]);
      } else {
        load8_bf16(p.gamma_cq + f, g);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = h[f + i] * rq * g[i];
      store8_bf16(cq + f, v);
    }
  } else {
    // eight columns per thread (gamma and smooth_scales_cq read before the wait when they fit)
    float amax = 0.f;
    for (int f = f8; f < p.Hcq; f += NT * 8) {
      float g[8], sm[8];
      if (PARTS && p.Hcq <= NT * 8) {
        const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&g_pre);
#pragma unroll
        for (int i = 0; i < 8; ++i) g[i] = __bfloat162float(e[i]);
        const float* ps = reinterpret_cast<const float*>(s_pre);
#pragma unroll
        for (int i = 0; i < 8; ++i) sm[i] = ps[i];
      } else {
        load8_bf16(p.gamma_cq + f, g);
#pragma unroll
        for (int i = 0; i < 8; ++i) sm[i] = __ldg(p.smooth + f + i);
      }
      float4* h4 = reinterpret_cast<float4*>(h + f);
      float v[8];
      *reinterpret_cast<float4*>(v) = h4[0];
      *reinterpret_cast<float4*>(v + 4) = h4[1];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float c = __bfloat162float(__float2bfloat16_rn(v[i] * rq * g[i]));
        v[i] = __fmul_rn(c, sm[i]);
        amax = fmaxf(amax, fabsf(v[i]));
      }
      h4[0] = *reinterpret_cast<const float4*>(v);   // own columns only: no race
      h4[1] = *reinterpret_cast<const float4*>(v + 4);
    }
    amax = block_max<NT>(amax, redm);
    const float scale = __fdiv_rn(amax, 127.0f);
    for (int f = f8; f < p.Hcq; f += NT * 8) {
      const float4* h4 = reinterpret_cast<const float4*>(h + f);
      float v[8];
      *reinterpret_cast<float4*>(v) = h4[0];
      *reinterpret_cast<float4*>(v + 4) = h4[1];
      // f16, the operand type of the int8-weight MMAs (exact: |code| <= 127)
      uint4 r;
      __half* e = reinterpret_cast<__half*>(&r);
#pragma unroll
      for (int i = 0; i < 8; ++i) e[i] = __int2half_rn(scale > 0.f ? quant_i8(v[i], scale, -127, 127) : 0);
      *reinterpret_cast<uint4*>(reinterpret_cast<__half*>(cq) + f) = r;
    }
    if (threadIdx.x == 0) p.scale_t[t] = scale;
  }

  if (!do_kv || p.slots <= 0) {             // empty caches: outputs only
    finish();
    return;
  }
  const int64_t idx = PARTS ? idx_pre : p.cache_index[t];
  if (idx < 0 || idx >= p.slots) {
    if (idx != -1 && threadIdx.x == 0) atomicOr(p.err, kErrIndexRange);
    finish();
    return;
  }
  // ---- c^KV (Hckv % 8 == 0)
  for (int f = threadIdx.x * 8; f < p.Hckv; f += NT * 8) {
    float g[8], v[8];
    if (PARTS && p.Hckv <= NT * 8) {
      const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&g_pre);
#pragma unroll
      for (int i = 0; i < 8; ++i) g[i] = __bfloat162float(e[i]);
    } else {
      load8_bf16(p.gamma_ckv + f, g);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = hkv[f + i] * rkv * g[i];
    if (p.kv_int8) {
      uint2 q;
      int8_t* qb = reinterpret_cast<int8_t*>(&q);
      const float* qs = PARTS && p.Hckv <= NT * 8 ? reinterpret_cast<const float*>(s_pre)
                                                  : p.qs_ckv + f;
#pragma unroll
      for (int i = 0; i < 8; ++i) qb[i] = quant_i8(v[i], qs[i], -128, 127);
      *reinterpret_cast<uint2*>(static_cast<int8_t*>(p.kv_cache) + idx * p.Hckv + f) = q;
    } else {
      store8_bf16(static_cast<__nv_bfloat16*>(p.kv_cache) + idx * p.Hckv + f, v);
    }
  }
  // ---- k^R
  const float* hkr = h + p.Hcq + p.Hckv;
  const int half = p.Dr >> 1;
  for (int j = threadIdx.x; j < p.Dr; j += NT) {
    const float y = hkr[j];
    const float partner = j < half ? -hkr[j + half] : hkr[j - half];
    const bool pre = PARTS && p.Dr <= NT;           // (j == threadIdx.x then)
    const float c = __bfloat162float(pre ? cos_pre : p.cos[static_cast<size_t>(t) * p.Dr + j]);
    const float s = __bfloat162float(pre ? sin_pre : p.sin[static_cast<size_t>(t) * p.Dr + j]);
    const float v = y * c + partner * s;
    if (p.kr_int8)
      static_cast<int8_t*>(p.kr_cache)[idx * p.Dr + j] =
          quant_i8(v, pre ? qkr_pre : p.qs_ckr[j], -128, 127);
    else
      static_cast<__nv_bfloat16*>(p.kr_cache)[idx * p.Dr + j] = __float2bfloat16_rn(v);
  }
  finish();
}

// Without K splits (prefill): one warp per token, eight tokens per CTA.  Lane l holds the
// float4 columns l + 32 i of the token's row (down to NV per lane) in registers, so both sums of
// squares, the amax of the quantised c^Q and the RoPE partner exchange stay inside the warp: no
// block barrier between the load and the stores, and every warp keeps its whole row (8.4 KB at
// Ntot = 2112) in flight at once.  Same arithmetic as norm_rope_scatter_kernel, term by term;
// only the order of the two sums of squares differs (lane-strided, then a shuffle tree).
constexpr int kWarpTokens = 8;
constexpr int kWarpMaxDr = 256;
constexpr int kWarpNV = 17;   // Ntot <= 32 * 4 * 17 = 2176
constexpr int kWarpMaxGamma = 32 * 4 * kWarpNV;   // Hcq + Hckv

__device__ __forceinline__ void load4_bf16_smem(const __nv_bfloat16* p, float* out) {
  const uint2 r = *reinterpret_cast<const uint2*>(p);
  const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) out[i] = __bfloat162float(e[i]);
}

__device__ __forceinline__ void store4_f16(__half* p, const float* v) {
  uint2 r;
  __half2* e = reinterpret_cast<__half2*>(&r);
  e[0] = __floats2half2_rn(v[0], v[1]);
  e[1] = __floats2half2_rn(v[2], v[3]);
  *reinterpret_cast<uint2*>(p) = r;
}

__device__ __forceinline__ void store4_bf16(__nv_bfloat16* p, const float* v) {
  uint2 r;
  __nv_bfloat162* e = reinterpret_cast<__nv_bfloat162*>(&r);
  e[0] = __floats2bfloat162_rn(v[0], v[1]);
  e[1] = __floats2bfloat162_rn(v[2], v[3]);
  *reinterpret_cast<uint2*>(p) = r;
}

template <int NV>
__global__ void __launch_bounds__(32 * kWarpTokens, 2) norm_rope_scatter_warp_kernel(
    const FinalizeParams p) {
  // one slot per warp: the token's row (Ntot floats), then two buffers of its cos and sin rows
  // (Dr bf16 each; fill k uses buffer k & 1, so the next token's tables cannot overwrite the ones
  // this token's k^R still reads)
  extern __shared__ __align__(16) float row_s[];
  __shared__ float kr_s[kWarpTokens][kWarpMaxDr];
  __shared__ __align__(16) __nv_bfloat16 gamma_s[kWarpMaxGamma];      // gamma_cq | gamma_ckv
  __shared__ uint64_t full[kWarpTokens];
  __shared__ int abort_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int stride = gridDim.x * kWarpTokens;        // tokens per round of the grid
  int t = blockIdx.x * kWarpTokens + warp;
  const uint32_t row_bytes = static_cast<uint32_t>(p.Ntot) * 4u;   // (Ntot % 4 == 0)
  const uint32_t tab_bytes = static_cast<uint32_t>(p.Dr) * 2u;     // (Dr % 8 == 0)
  float* slot = row_s + static_cast<size_t>(warp) * (p.Ntot + 2 * p.Dr);
  // the gammas are inputs of the call: into shared memory before the wait
  for (int i = threadIdx.x; i < (p.Hcq + p.Hckv) / 8; i += 32 * kWarpTokens) {
    const int f = 8 * i;
    *reinterpret_cast<uint4*>(gamma_s + f) =
        f < p.Hcq ? __ldg(reinterpret_cast<const uint4*>(p.gamma_cq + f))
                  : __ldg(reinterpret_cast<const uint4*>(p.gamma_ckv + (f - p.Hcq)));
  }
  if (threadIdx.x == 0) {
    stamp(p.stamps, MLAP_STAMP_NORM, kStampStart);
    for (int i = 0; i < kWarpTokens; ++i) mbar_init(&full[i], 1);
    abort_sh = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  grid_launch_dependents();
  grid_dependency_wait();
  if (threadIdx.x == 0) stamp(p.stamps, MLAP_STAMP_NORM, kStampDep);
  // the warp's token rows go through its slot: the next row is requested as soon as the current
  // one is in registers, so its load overlaps this token's arithmetic and stores
  auto request = [&](int tt, int fill) {
    const bool tab = p.slots > 0;   // (the tables serve k^R, stored only with a cache)
    mbar_arrive_expect_tx(&full[warp], row_bytes + (tab ? 2 * tab_bytes : 0u));
    bulk_load_1d(slot, p.part + static_cast<size_t>(tt) * p.Ntot, row_bytes, &full[warp]);
    if (tab) {
      float* tb = slot + p.Ntot + (fill & 1) * p.Dr;
      bulk_load_1d(tb, p.cos + static_cast<size_t>(tt) * p.Dr, tab_bytes, &full[warp]);
      bulk_load_1d(tb + p.Dr / 2, p.sin + static_cast<size_t>(tt) * p.Dr, tab_bytes, &full[warp]);
    }
  };
  int fills = 0;
  if (t < p.T) {
    if (lane == 0) request(t, 0);
    fills = 1;
  }
  const int n4 = p.Ntot >> 2, q4 = p.Hcq >> 2, kv4 = (p.Hcq + p.Hckv) >> 2;
  for (int k = 0; t < p.T; ++k, t += stride) {
    const int64_t idx = p.slots > 0 ? p.cache_index[t] : -1;
    const bool landed = mbar_wait(&full[warp], static_cast<uint32_t>(k & 1), &abort_sh);
    if (!__all_sync(0xffffffffu, landed)) break;
    float4 v[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int c = lane + 32 * i;
      v[i] = c < n4 ? reinterpret_cast<const float4*>(slot)[c] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (p.dsx != nullptr) {   // full quant: dequant the exact integer products per token and column
      const float sx = p.dsx[t];
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int c = lane + 32 * i;
        if (c < n4) {   // (dsw_kv covers the c^KV and the k^R columns)
          const float* w = c < q4 ? p.dsw_q + 4 * c : p.dsw_kv + 4 * (c - q4);
          v[i].x *= sx * w[0];
          v[i].y *= sx * w[1];
          v[i].z *= sx * w[2];
          v[i].w *= sx * w[3];
        }
      }
    }
    float sq = 0.f, skv = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int c = lane + 32 * i;
      const float s4 = v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
      if (c < q4) sq += s4;
      else if (c < kv4) skv += s4;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sq += __shfl_xor_sync(0xffffffffu, sq, o);
      skv += __shfl_xor_sync(0xffffffffu, skv, o);
    }
    const float rq = 1.0f / sqrtf(sq / static_cast<float>(p.Hcq) + p.eps_cq);
    const float rkv = 1.0f / sqrtf(skv / static_cast<float>(p.Hckv) + p.eps_ckv);
    // every lane's reads of the slot have completed (the sums above consumed them): the slot
    // takes the next row while this one is normalised and stored
    __syncwarp();
    if (t + stride < p.T) {
      if (lane == 0) request(t + stride, k + 1);
      ++fills;
    }

    // ---- c^Q: bf16, or int8 codes held exactly in f16
    __nv_bfloat16* cq = p.cq_out + static_cast<size_t>(t) * p.Hcq;
    if (p.smooth == nullptr) {
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int c = lane + 32 * i;
        if (c < q4) {
          float g[4], o[4];
          load4_bf16_smem(gamma_s + 4 * c, g);
          o[0] = v[i].x * rq * g[0];
          o[1] = v[i].y * rq * g[1];
          o[2] = v[i].z * rq * g[2];
          o[3] = v[i].w * rq * g[3];
          store4_bf16(cq + 4 * c, o);
        }
      }
    } else {
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int c = lane + 32 * i;
        if (c < q4) {
          float* e = reinterpret_cast<float*>(&v[i]);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int f = 4 * c + k;
            const float cv = __bfloat162float(
                __float2bfloat16_rn(e[k] * rq * __bfloat162float(gamma_s[f])));
            e[k] = __fmul_rn(cv, p.smooth[f]);
            amax = fmaxf(amax, fabsf(e[k]));
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const float scale = __fdiv_rn(amax, 127.0f);
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int c = lane + 32 * i;
        if (c < q4) {
          const float* e = reinterpret_cast<const float*>(&v[i]);
          float o[4];
#pragma unroll
          for (int k = 0; k < 4; ++k)
            o[k] = static_cast<float>(scale > 0.f ? quant_i8(e[k], scale, -127, 127) : 0);
          store4_f16(reinterpret_cast<__half*>(cq) + 4 * c, o);   // f16 codes (exact)
        }
      }
      if (lane == 0) p.scale_t[t] = scale;
    }

    if (p.slots <= 0) continue;                     // empty caches: outputs only
    if (idx < 0 || idx >= p.slots) {
      if (idx != -1 && lane == 0) atomicOr(p.err, kErrIndexRange);
      continue;
    }
    // ---- c^KV, and k^R into this warp's shared row for the RoPE partner exchange
    float* kr = kr_s[warp];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int c = lane + 32 * i;
      if (c >= q4 && c < kv4) {
        const int f = 4 * (c - q4);
        float g[4], o[4];
        load4_bf16_smem(gamma_s + p.Hcq + f, g);
        o[0] = v[i].x * rkv * g[0];
        o[1] = v[i].y * rkv * g[1];
        o[2] = v[i].z * rkv * g[2];
        o[3] = v[i].w * rkv * g[3];
        if (p.kv_int8) {
          uint32_t q;
          int8_t* qb = reinterpret_cast<int8_t*>(&q);
#pragma unroll
          for (int k = 0; k < 4; ++k) qb[k] = quant_i8(o[k], p.qs_ckv[f + k], -128, 127);
          *reinterpret_cast<uint32_t*>(static_cast<int8_t*>(p.kv_cache) + idx * p.Hckv + f) = q;
        } else {
          store4_bf16(static_cast<__nv_bfloat16*>(p.kv_cache) + idx * p.Hckv + f, o);
        }
      } else if (c >= kv4 && c < n4) {
        *reinterpret_cast<float4*>(kr + 4 * (c - kv4)) = v[i];
      }
    }
    __syncwarp();
    const int half = p.Dr >> 1;
    for (int j = lane; j < p.Dr; j += 32) {
      const float y = kr[j];
      const float partner = j < half ? -kr[j + half] : kr[j - half];
      const __nv_bfloat16* tb =
          reinterpret_cast<const __nv_bfloat16*>(slot + p.Ntot + (k & 1) * p.Dr);
      const float c = __bfloat162float(tb[j]);
      const float s = __bfloat162float(tb[p.Dr + j]);
      const float o = y * c + partner * s;
      if (p.kr_int8)
        static_cast<int8_t*>(p.kr_cache)[idx * p.Dr + j] = quant_i8(o, p.qs_ckr[j], -128, 127);
      else
        static_cast<__nv_bfloat16*>(p.kr_cache)[idx * p.Dr + j] = __float2bfloat16_rn(o);
    }
  }
  if (abort_sh && lane == 0 && fills > 0) {
    // let this warp's last request land before the CTA exits (bounded)
    const uint32_t par = static_cast<uint32_t>(fills - 1) & 1u;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(&full[warp], par) && globaltimer_ns() - t0 < 20000000ull) {
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (abort_sh) atomicOr(p.err, kErrTimeout);
    stamp(p.stamps, MLAP_STAMP_NORM, kStampEnd);
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

// Full quant: 16 int8 values -> 16 f16 per thread and step (exact: |v| <= 128), the operand type
// of the int8-weight MMAs.
__global__ void widen_int8_kernel(const int8_t* __restrict__ x, __half* __restrict__ out,
                                  int64_t n16) {
  grid_dependency_wait();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n16;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 raw = reinterpret_cast<const uint4*>(x)[i];
    const int8_t* v = reinterpret_cast<const int8_t*>(&raw);
    uint4 o[2];
    __half* h = reinterpret_cast<__half*>(o);
#pragma unroll
    for (int k = 0; k < 16; ++k) h[k] = __short2half_rn(v[k]);
    reinterpret_cast<uint4*>(out + i * 16)[0] = o[0];
    reinterpret_cast<uint4*>(out + i * 16)[1] = o[1];
  }
  grid_launch_dependents();   // after this thread's loads: the next grid's prefetch waits for them
}

// int8 query per token and head (MlaPrologV2 README scenario matrix: query INT8 "pertoken_head"
// with dequant_scale_q_nope): one warp per (token, head) row of H values held in registers (up to
// 8 * 32 * kQqVec); scale = amax / 127, code = rne(v / scale) clamped to [-127, 127] (all-zero
// row: codes 0, scale 0), in fp32.
constexpr int kQqVec = 4;

__global__ void query_quant_kernel(const __nv_bfloat16* __restrict__ qn, int8_t* __restrict__ q,
                                   float* __restrict__ scale, int64_t rows, int32_t H) {
  const int64_t row = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  grid_dependency_wait();                         // q^N comes from the absorb GEMM
  if (row >= rows) return;                        // warp-uniform
  const __nv_bfloat16* src = qn + row * H;
  float v[kQqVec][8];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < kQqVec; ++i) {
    const int c = (lane + 32 * i) * 8;
    if (c < H) {
      load8_bf16(src + c, v[i]);
#pragma unroll
      for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(v[i][k]));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  grid_launch_dependents();
  const float sc = __fdiv_rn(amax, 127.0f);
  int8_t* dst = q + row * H;
#pragma unroll
  for (int i = 0; i < kQqVec; ++i) {
    const int c = (lane + 32 * i) * 8;
    if (c < H) {
      uint2 out;
      int8_t* o = reinterpret_cast<int8_t*>(&out);
#pragma unroll
      for (int k = 0; k < 8; ++k) o[k] = sc > 0.f ? quant_i8(v[i][k], sc, -127, 127) : 0;
      *reinterpret_cast<uint2*>(dst + c) = out;
    }
  }
  if (lane == 0) scale[row] = sc;
}

// Input RmsNormQuant (aclnnMlaPreprocessV2, "Formula": RMS, RmsNorm, RmsNormQuant), one CTA per
// token: x'[k] = bf16((gamma[k] * x[k] / RMS(x) + bias[k]) * deqScale[k]) with RMS(x) =
// sqrt(mean(x^2) + eps), all in fp32.  The row stays in registers between the sum of squares and
// the store: NV 16-byte vectors per thread cover He <= 8 * NT * NV.  PRE (few tokens) also holds
// gamma, bias and deqScale in registers, read before the wait on the preceding kernel; without it
// (many tokens) the kernel stays small enough for several CTAs per SM and reads them after the
// reduction.  The dependent down-projection is released once this CTA's row has arrived: an
// earlier release lets its weight prefetch queue ahead of these loads in DRAM.
template <int NT, int NV, bool PRE>
__global__ void __launch_bounds__(NT) rms_norm_quant_kernel(
    const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ gamma,
    const __nv_bfloat16* __restrict__ bias, const float* __restrict__ deq, int deq_per_channel,
    float eps, __nv_bfloat16* __restrict__ out, int32_t He) {
  __shared__ float2 red[NT / 32];
  const int nvec = He >> 3;
  auto load_params = [&](int i, float* g, float* b, float* d) {
    load8_bf16(gamma + i * 8, g);
    load8_bf16(bias + i * 8, b);
    if (deq_per_channel) {
      const float4 d0 = __ldg(reinterpret_cast<const float4*>(deq) + 2 * i);
      const float4 d1 = __ldg(reinterpret_cast<const float4*>(deq) + 2 * i + 1);
      d[0] = d0.x; d[1] = d0.y; d[2] = d0.z; d[3] = d0.w;
      d[4] = d1.x; d[5] = d1.y; d[6] = d1.z; d[7] = d1.w;
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) d[k] = __ldg(deq);
    }
  };
  constexpr int NP = PRE ? NV : 1;
  float g[NP][8], b[NP][8], d[NP][8];
  if constexpr (PRE) {
#pragma unroll
    for (int v = 0; v < NV; ++v)
      if (threadIdx.x + v * NT < nvec) load_params(threadIdx.x + v * NT, g[v], b[v], d[v]);
  }
  const uint4* row = reinterpret_cast<const uint4*>(x + static_cast<size_t>(blockIdx.x) * He);
  uint4 raw[NV];
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const int i = threadIdx.x + v * NT;
    if (i < nvec) raw[v] = __ldg(row + i);
  }
  float ss = 0.f;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    if (threadIdx.x + v * NT < nvec) {
      const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&raw[v]);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float f = __bfloat162float(e[k]);
        ss += f * f;
      }
    }
  }
  const float2 tot = block_sum2<NT>(make_float2(ss, 0.f), red);
  // token_x is an input of the call: its row and sum of squares come before the wait on the
  // preceding kernel; only the stores of x' (which that kernel may still read) wait
  grid_dependency_wait();
  grid_launch_dependents();
  const float r = 1.0f / sqrtf(tot.x / static_cast<float>(He) + eps);
  __nv_bfloat16* dst = out + static_cast<size_t>(blockIdx.x) * He;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const int i = threadIdx.x + v * NT;
    if (i < nvec) {
      const int p = PRE ? v : 0;
      if constexpr (!PRE) load_params(i, g[0], b[0], d[0]);
      const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&raw[v]);
      float y[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) y[k] = (g[p][k] * (__bfloat162float(e[k]) * r) + b[p][k]) * d[p][k];
      store8_bf16(dst + i * 8, y);
    }
  }
}

constexpr int kXnMaxHe = 10240;   // 8 * 256 * 5 = 8 * 128 * 10
constexpr int kXnFewTokens = 512;

// A launch, with programmatic stream serialization when pdl is set: the kernel may then start
// while the preceding kernel in the stream finishes (it waits for it with griddepcontrol.wait).
// Without it the kernel starts after the preceding one and its wait returns at once; its own
// griddepcontrol.launch_dependents still lets the next kernel start early.
template <class... KArgs, class... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, cudaStream_t stream, bool pdl,
                     Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

}  // namespace

cudaError_t launch_rms_norm_quant(const __nv_bfloat16* x, const __nv_bfloat16* gamma,
                                  const __nv_bfloat16* bias, const float* deq, bool deq_per_channel,
                                  float eps, __nv_bfloat16* out, int64_t T, int32_t He,
                                  cudaStream_t stream) {
  if ((He % 8) || He > kXnMaxHe) return cudaErrorInvalidValue;
  if (T < 1) return cudaSuccess;
  const int dpc = deq_per_channel ? 1 : 0;
  const dim3 grid(static_cast<unsigned>(T));
  if (T <= kXnFewTokens)
    return launch_k(rms_norm_quant_kernel<256, 5, true>, grid, dim3(256), stream, true, x, gamma,
                    bias, deq, dpc, eps, out, He);
  return launch_k(rms_norm_quant_kernel<128, 10, false>, grid, dim3(128), stream, true, x, gamma,
                  bias, deq, dpc, eps, out, He);
}

cudaError_t launch_widen_int8(const int8_t* x, __half* out, int64_t n, cudaStream_t stream) {
  if (n % 16) return cudaErrorInvalidValue;
  const int64_t n16 = n / 16;
  int64_t blocks = (n16 + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  // a plain launch measured 0.5 µs faster per full-quant call than an early one (with the query
  // quantisation below launched the same way)
  return launch_k(widen_int8_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), stream, false,
                  x, out, n16);
}

cudaError_t launch_query_quant(const __nv_bfloat16* qn, int8_t* q, float* scale, int64_t rows,
                               int32_t H, cudaStream_t stream) {
  if ((H % 8) || H > 8 * 32 * kQqVec) return cudaErrorInvalidValue;
  const int64_t blocks = (rows * 32 + 255) / 256;
  if (blocks < 1) return cudaSuccess;
  // (programmatic dependent launch: the kernel waits for q^N with griddepcontrol.wait)
  return launch_k(query_quant_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), stream,
                  true, qn, q, scale, rows, H);
}

cudaError_t launch_finalize(const FinalizeParams& p, cudaStream_t stream, bool pdl) {
  const size_t smem = static_cast<size_t>(p.Ntot) * sizeof(float);
  const bool split = p.splits > 1;
  if (!split && p.Ntot <= 32 * 4 * kWarpNV && p.Dr <= kWarpMaxDr) {
    // (Hcq, Hckv and Dr are multiples of 8: every float4 of a row lies in one part)
    auto wk = norm_rope_scatter_warp_kernel<kWarpNV>;
    const size_t wsmem = static_cast<size_t>(kWarpTokens) * (p.Ntot + 2 * p.Dr) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(wk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(wsmem));
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // persistent: two CTAs per SM (the register budget), no more than the tokens need
    int64_t blocks = 2 * static_cast<int64_t>(sms);
    const int64_t need = (p.T + kWarpTokens - 1) / kWarpTokens;
    if (blocks > need) blocks = need;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(32 * kWarpTokens);
    cfg.dynamicSmemBytes = wsmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, wk, p);
  }
  // up to 8 K-splits (decode): two CTAs per token, c^Q and c^KV/k^R
  const bool parts = split && p.splits <= 8;
  auto kern = !split ? norm_rope_scatter_kernel<1, 256>
              : parts ? norm_rope_scatter_kernel<8, 256, true>
                      : norm_rope_scatter_kernel<kMaxSplits, 512>;
  if (p.splits > kMaxSplits) return cudaErrorInvalidValue;
  if (smem > 48 * 1024) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(parts ? 2 * p.T : p.T));
  cfg.blockDim = dim3(split && !parts ? 512 : 256);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, p);
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
