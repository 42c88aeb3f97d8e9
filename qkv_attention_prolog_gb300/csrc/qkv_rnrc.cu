// QkvRmsNormRopeCache (aclnnQkvRmsNormRopeCache, "Formulas" (1)-(4) and "Other restrictions"):
//
//   q, k, v = SplitVD(qkv)                  heads [0,Nq) | [Nq, Nq+Nk) | [Nq+Nk, Nq+Nk+Nv)
//   y       = x / sqrt(mean(x^2) + eps) * gamma                      per q / k head, along D
//   y_embed = y * cos + cat(-y2, y1) * sin                           half-and-half, d = D
//   q_out   = y_embed(q);  k_cache[i] = Quant(y_embed(k));  v_cache[i] = Quant(v)
//   Quant   = identity, value / scale (symmetric) or value / scale + offset (asymmetric),
//             rounded half to even and saturated to int8 (computed as value * fp32(1/scale)
//             (+ offset) in fp32; the code can differ from the exact quotient's by one near a
//             rounding tie)
//   optional qBeforeQuant / kBeforeQuant / vBeforeQuant: the tensors entering Quant, dense per
//             token (the API function's optional outputs)
//
// A pure HBM stream: every token's qkv row is read once and its outputs written once.  What
// bounds it is how many bytes each SM keeps in flight, so every warp streams tokens on its own:
// one persistent CTA per SM holds one shared-memory slot per warp (the token's qkv row and its
// cos / sin rows), and a warp requests its next token with 1-D bulk copies as soon as it has read
// the current one out of its slot.  No CTA-wide barrier sits in the token loop, so a slow warp
// never holds the others, and with 16 warps about 200 KB of loads are in flight per SM.
#include "internal.h"

namespace mlap {

namespace {

constexpr int kD = 128;
constexpr int kMaxWarps = 16;
constexpr int kSmemBudget = 227 * 1024;

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

// int8 codes of x * (1/scale) (+ offset) (reciprocal of the per-channel scale in fp32), round
// half to even, saturated to [-128, 127].
template <bool ASYM>
__device__ __forceinline__ uint2 quant8_mul(const float (&x)[8], const float* inv, const float* off) {
  const float4 i0 = reinterpret_cast<const float4*>(inv)[0];
  const float4 i1 = reinterpret_cast<const float4*>(inv)[1];
  const float iv[8] = {i0.x, i0.y, i0.z, i0.w, i1.x, i1.y, i1.z, i1.w};
  float ov[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if constexpr (ASYM) {
    const float4 o0 = reinterpret_cast<const float4*>(off)[0];
    const float4 o1 = reinterpret_cast<const float4*>(off)[1];
    ov[0] = o0.x; ov[1] = o0.y; ov[2] = o0.z; ov[3] = o0.w;
    ov[4] = o1.x; ov[5] = o1.y; ov[6] = o1.z; ov[7] = o1.w;
  }
  uint2 out;
  int8_t* o = reinterpret_cast<int8_t*>(&out);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    int q = ASYM ? __float2int_rn(__fadd_rn(x[i] * iv[i], ov[i])) : __float2int_rn(x[i] * iv[i]);
    q = q < -128 ? -128 : (q > 127 ? 127 : q);
    o[i] = static_cast<int8_t>(q);
  }
  return out;
}

// Shared memory: the per-channel reciprocal quant scales of all k and v heads (and the
// asymmetric offsets), then one slot per warp: the token's qkv row ((Nq+Nk+Nv) * D elements,
// contiguous), its cos row and its sin row.  Inside a warp eight lanes own one head row: lane l
// holds elements 8l..8l+7 and 64+8l..64+8l+7, both members of its RoPE pairs, so the rotation
// needs no exchange and the RmsNorm sum is a 3-step shuffle; the warp covers four rows per step.
// QM: 0 no quant, 1 symmetric, 2 asymmetric.
template <bool BF16, int QM>
__global__ void __launch_bounds__(kMaxWarps * 32, 1) qkv_rnrc_kernel(const QkvParams p) {
  constexpr bool QUANT = QM != 0;
  constexpr bool ASYM = QM == 2;
  using E = Elem<BF16>;
  using T = typename E::T;
  extern __shared__ __align__(128) uint8_t qsm[];
  __shared__ uint64_t full[kMaxWarps];
  __shared__ int abort_sh;
  const int Nh = p.Nq + p.Nk + p.Nv;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const uint32_t row_bytes = static_cast<uint32_t>(Nh) * kD * sizeof(T);
  const uint32_t slot_bytes = row_bytes + 2 * kD * sizeof(T);     // qkv row, cos, sin
  const int l8 = lane & 7;
  const int sub = lane >> 3;                                       // row of the warp's step
  const unsigned mask = 0xffu << (lane & 24);                      // this row's 8 lanes
  const int ja = l8 * 8, jb = 64 + l8 * 8;                         // the two 8-element slices
  const int nscale = QUANT ? (p.Nk + p.Nv) * kD : 0;
  float* inv = reinterpret_cast<float*>(qsm);                      // reciprocal scales
  float* offs = inv + nscale;                                      // asymmetric offsets
  uint8_t* slots = qsm + static_cast<size_t>(nscale) * (ASYM ? 8 : 4);
  uint8_t* slot = slots + static_cast<size_t>(warp) * slot_bytes;

  if (threadIdx.x == 0) stamp(p.stamps, MLAP_STAMP_QKV, kStampStart);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kMaxWarps; ++i) mbar_init(&full[i], 1);
    abort_sh = 0;
    fence_mbarrier_init();
  }
  // per-lane gamma slices and the quant scales do not depend on an earlier kernel
  float ga_q[8], gb_q[8], ga_k[8], gb_k[8];
  unpack8<BF16>(reinterpret_cast<const uint4*>(p.gamma_q)[l8], ga_q);
  unpack8<BF16>(reinterpret_cast<const uint4*>(p.gamma_q)[8 + l8], gb_q);
  unpack8<BF16>(reinterpret_cast<const uint4*>(p.gamma_k)[l8], ga_k);
  unpack8<BF16>(reinterpret_cast<const uint4*>(p.gamma_k)[8 + l8], gb_k);
  if (QUANT) {
    for (int i = threadIdx.x; i < nscale; i += blockDim.x) {
      inv[i] = __frcp_rn(i < p.Nk * kD ? p.k_scale[i] : p.v_scale[i - p.Nk * kD]);
      if (ASYM) offs[i] = i < p.Nk * kD ? p.k_offset[i] : p.v_offset[i - p.Nk * kD];
    }
  }
  __syncthreads();
  grid_launch_dependents();

  const int stride = gridDim.x * nwarps;                           // tokens per round
  auto request = [&](int t) {
    mbar_arrive_expect_tx(&full[warp], slot_bytes);
    bulk_load_1d(slot, static_cast<const uint8_t*>(p.qkv) + static_cast<size_t>(t) * row_bytes,
                 row_bytes, &full[warp]);
    bulk_load_1d(slot + row_bytes,
                 static_cast<const uint8_t*>(p.cos) + static_cast<size_t>(t) * kD * sizeof(T),
                 kD * sizeof(T), &full[warp]);
    bulk_load_1d(slot + row_bytes + kD * sizeof(T),
                 static_cast<const uint8_t*>(p.sin) + static_cast<size_t>(t) * kD * sizeof(T),
                 kD * sizeof(T), &full[warp]);
  };
  int t = blockIdx.x * nwarps + warp;
  int fills = 0;                                                   // requests made on this slot
  // qkv and the tables are inputs the kernel only reads: each warp requests its first token
  // before the wait on the preceding kernel, so that the first loads overlap that kernel's tail
  // (68.4 -> 65.1 us per call at (16, 1024, 48, 128)); every store comes after the wait
  if (t < p.T && lane == 0) request(t);
  if (t < p.T) fills = 1;
  grid_dependency_wait();
  if (threadIdx.x == 0) stamp(p.stamps, MLAP_STAMP_QKV, kStampDep);

  for (int k = 0; t < p.T; ++k, t += stride) {
    // the slot holds token t once its k-th fill completes; a wait that gives up skips the
    // token's stores (its cache slots stay untouched) and ends this warp's loop
    // (every lane waits; the warp goes on only if all of them saw the fill complete)
    const bool landed = mbar_wait(&full[warp], static_cast<uint32_t>(k & 1), &abort_sh);
    if (!__all_sync(0xffffffffu, landed)) break;
    float ca[8], sa[8], cb[8], sb[8];
    const uint4* cs = reinterpret_cast<const uint4*>(slot + row_bytes);
    const uint4* sn = reinterpret_cast<const uint4*>(slot + row_bytes + kD * sizeof(T));
    unpack8<BF16>(cs[l8], ca);
    unpack8<BF16>(cs[8 + l8], cb);
    unpack8<BF16>(sn[l8], sa);
    unpack8<BF16>(sn[8 + l8], sb);
    const int64_t idx = p.index[t];
    const bool store = idx >= 0 && idx < p.slots;
    if (lane == 0 && idx != -1 && !store && p.slots > 0) atomicOr(p.err, kErrIndexRange);
    // read the whole row into registers step by step; the slot is free after the last step
    const int steps = (Nh + 3) >> 2;
    for (int st = 0; st < steps; ++st) {
      const int h = st * 4 + sub;
      uint4 rawa = make_uint4(0, 0, 0, 0), rawb = make_uint4(0, 0, 0, 0);
      if (h < Nh) {
        const uint4* row = reinterpret_cast<const uint4*>(slot + static_cast<size_t>(h) * kD * sizeof(T));
        rawa = row[l8];
        rawb = row[8 + l8];
      }
      if (st == steps - 1) {
        // every lane has read its last piece of the slot: request the next token into it
        __syncwarp();
        const int tn = t + stride;
        if (tn < p.T) {
          if (lane == 0) request(tn);
          ++fills;
        }
      }
      if (h >= Nh) continue;                                       // uniform in the 8 lanes
      float xa[8], xb[8];
      unpack8<BF16>(rawa, xa);
      unpack8<BF16>(rawb, xb);
      if (h < p.Nq + p.Nk) {
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) ss += xa[e] * xa[e] + xb[e] * xb[e];
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) ss += __shfl_xor_sync(mask, ss, o);
        const float rinv = rsqrtf(ss * (1.0f / static_cast<float>(kD)) + p.eps);
        const bool is_q = h < p.Nq;
        float oa[8], ob[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float ya = xa[e] * rinv * (is_q ? ga_q[e] : ga_k[e]);
          const float yb = xb[e] * rinv * (is_q ? gb_q[e] : gb_k[e]);
          oa[e] = ya * ca[e] - yb * sa[e];                         // j < 64: partner -y[j+64]
          ob[e] = yb * cb[e] + ya * sb[e];                         // j >= 64: partner y[j-64]
        }
        if (is_q) {
          const uint4 qa = pack8<BF16>(oa), qb = pack8<BF16>(ob);
          const size_t row = (static_cast<size_t>(t) * p.Nq + h) * kD;
          uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(p.q_out) + row);
          dst[l8] = qa;
          dst[8 + l8] = qb;
          if (p.q_before != nullptr) {
            uint4* bq = reinterpret_cast<uint4*>(static_cast<T*>(p.q_before) + row);
            bq[l8] = qa;
            bq[8 + l8] = qb;
          }
        } else {
          const int hk = h - p.Nq;
          if (p.k_before != nullptr) {   // dense, whatever the token's index
            uint4* bk = reinterpret_cast<uint4*>(static_cast<T*>(p.k_before) +
                                                 (static_cast<size_t>(t) * p.Nk + hk) * kD);
            bk[l8] = pack8<BF16>(oa);
            bk[8 + l8] = pack8<BF16>(ob);
          }
          if (store) {
            const size_t off = (static_cast<size_t>(idx) * p.Nk + hk) * kD;
            if (QUANT) {
              uint2* dst = reinterpret_cast<uint2*>(static_cast<int8_t*>(p.k_cache) + off);
              const float* iv = inv + hk * kD;
              const float* ov = offs + hk * kD;
              dst[l8] = quant8_mul<ASYM>(oa, iv + ja, ov + ja);
              dst[8 + l8] = quant8_mul<ASYM>(ob, iv + jb, ov + jb);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(p.k_cache) + off);
              dst[l8] = pack8<BF16>(oa);
              dst[8 + l8] = pack8<BF16>(ob);
            }
          }
        }
      } else {
        const int hv = h - p.Nq - p.Nk;
        if (p.v_before != nullptr) {
          uint4* bv = reinterpret_cast<uint4*>(static_cast<T*>(p.v_before) +
                                               (static_cast<size_t>(t) * p.Nv + hv) * kD);
          bv[l8] = rawa;
          bv[8 + l8] = rawb;
        }
        if (!store) continue;
        const size_t off = (static_cast<size_t>(idx) * p.Nv + hv) * kD;
        if (QUANT) {
          uint2* dst = reinterpret_cast<uint2*>(static_cast<int8_t*>(p.v_cache) + off);
          const float* iv = inv + (p.Nk + hv) * kD;
          const float* ov = offs + (p.Nk + hv) * kD;
          dst[l8] = quant8_mul<ASYM>(xa, iv + ja, ov + ja);
          dst[8 + l8] = quant8_mul<ASYM>(xb, iv + jb, ov + jb);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(p.v_cache) + off);
          dst[l8] = rawa;
          dst[8 + l8] = rawb;
        }
      }
    }
  }
  if (abort_sh && lane == 0 && fills > 0) {
    // let this warp's last request land before the CTA exits (bounded): fill number fills - 1
    // completes the phase of parity (fills - 1) & 1
    const uint32_t par = static_cast<uint32_t>(fills - 1) & 1u;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(&full[warp], par) && globaltimer_ns() - t0 < 20000000ull) {
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (abort_sh) atomicOr(p.err, kErrTimeout);
    stamp(p.stamps, MLAP_STAMP_QKV, kStampEnd);
  }
}

}  // namespace

cudaError_t launch_qkv_rnrc(const QkvParams& p, cudaStream_t stream, int sm_count) {
  const int Nh = p.Nq + p.Nk + p.Nv;
  const size_t elem = 2;   // fp16 and bf16
  const size_t slot = static_cast<size_t>(Nh) * kD * elem + 2 * kD * elem;
  const int qm = p.k_scale == nullptr ? 0 : (p.k_offset == nullptr ? 1 : 2);
  const size_t scales = static_cast<size_t>(p.Nk + p.Nv) * kD * (qm == 0 ? 0 : (qm == 1 ? 4 : 8));
  if (scales + slot > static_cast<size_t>(kSmemBudget)) return cudaErrorNotSupported;
  int warps = static_cast<int>((kSmemBudget - scales) / slot);
  if (warps > kMaxWarps) warps = kMaxWarps;
  // fewer tokens than warps: no idle warps
  int64_t blocks = sm_count;
  if (static_cast<int64_t>(blocks) * warps > p.T) {
    blocks = (p.T + warps - 1) / warps;
    if (blocks < 1) blocks = 1;
  }
  const size_t smem = scales + static_cast<size_t>(warps) * slot;
  auto pick = [&]() {
    if (p.bf16)
      return qm == 0 ? qkv_rnrc_kernel<true, 0> : (qm == 1 ? qkv_rnrc_kernel<true, 1>
                                                            : qkv_rnrc_kernel<true, 2>);
    return qm == 0 ? qkv_rnrc_kernel<false, 0> : (qm == 1 ? qkv_rnrc_kernel<false, 1>
                                                           : qkv_rnrc_kernel<false, 2>);
  };
  auto kern = pick();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(static_cast<unsigned>(warps * 32));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace mlap
