// Epilogue functors of the three MLA prolog contractions (see gemm.cuh for the calling contract).
//
// "SWAP" selects the decode orientation: A = the weight (its output features are the MMA's
// M = 128 rows), B = the activations (tokens are the MMA's N).  Without SWAP (prefill),
// A = activations (tokens are rows) and B = the weight.  The functors translate tile-space
// (row, column) back to (token, feature) and fuse the step that follows each contraction.
#pragma once
#include <cuda_bf16.h>
#include "ptx.cuh"

namespace mlap {

// ----------------------------------------------------------------------------------------------
// Down-projection  [h_q | h_kv | h_kr] = x · [W^DQ | W^DKV | W^KR]   (MlaPrologV2 README, c^Q and
// c^KV / k^R formulas).  The weight is two tensor maps (W^DQ, W^DKV|W^KR) seen as one operand
// with `seg_tiles` tiles in the first.  The fp32 result of K-split s goes to
// part[s][t][f], f in [0, Hcq + Hckv + Dr); the norm step sums the splits in order.
struct DownParams {
  float* part;
  int32_t T, Hcq, Nseg2, Ntot, seg_tiles;
};

template <bool SWAP, int TILE_W, int CH>
struct EpiDown {
  DownParams p;

  __device__ __forceinline__ int feature(int i) const {
    const int b0 = p.seg_tiles * TILE_W;
    if (i < b0) return i < p.Hcq ? i : -1;
    const int i2 = i - b0;
    return i2 < p.Nseg2 ? p.Hcq + i2 : -1;
  }

  __device__ __forceinline__ void operator()(int row, int col0, int, int s, const float* v) const {
    float* out = p.part + static_cast<size_t>(s) * p.T * p.Ntot;
    if constexpr (SWAP) {
      const int f = feature(row);
      if (f < 0) return;
#pragma unroll
      for (int j = 0; j < CH; ++j) {
        const int t = col0 + j;
        if (t < p.T) out[static_cast<size_t>(t) * p.Ntot + f] = v[j];
      }
    } else {
      const int t = row;
      if (t >= p.T) return;
      float* dst = out + static_cast<size_t>(t) * p.Ntot;
      const int f0 = feature(col0);
      const int fl = feature(col0 + CH - 1);
      const bool contiguous = f0 >= 0 && fl == f0 + CH - 1;
      const size_t off = static_cast<size_t>(s) * p.T * p.Ntot + static_cast<size_t>(t) * p.Ntot + f0;
      if (contiguous && (off % 4) == 0) {
        float4* d4 = reinterpret_cast<float4*>(dst + f0);
#pragma unroll
        for (int j = 0; j < CH / 4; ++j)
          d4[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
      } else {
#pragma unroll
        for (int j = 0; j < CH; ++j) {
          const int f = feature(col0 + j);
          if (f >= 0) dst[f] = v[j];
        }
      }
    }
  }
};

// ----------------------------------------------------------------------------------------------
// Up-projection  [q^C | q_r] = c^Q · W^UQ_QR  (MlaPrologV2 README q^C and q^R formulas) with the
// weight prepacked as rows [all heads' nope columns (n*D + d) | all heads' rope columns, each
// head's pair (j, j + Dr/2) stored adjacently].  Fused: bf16 rounding of q^C (the next matmul's
// input), half-and-half RoPE of q_r into query_rope, and for an int8 weight the dequant
// acc * scale_t[t] * dequant_scale_w_uq_qr[column].
struct UpParams {
  __nv_bfloat16* qc;            // (T, N*D)
  __nv_bfloat16* qrope;         // (T, N, Dr)
  const __nv_bfloat16* cos;     // (T, Dr)
  const __nv_bfloat16* sin;     // (T, Dr)
  const float* scale_t;         // (T) per-token dequant scale, int8 path
  const float* dqw;             // (N*(D+Dr)) per-column dequant scale, int8 path
  int32_t T, N, D, Dr;
};

template <bool SWAP, bool INT8, int CH>
struct EpiUp {
  UpParams p;

  // original column of weight_uq_qr for a prepacked row
  __device__ __forceinline__ int orig_col(int f) const {
    const int nd = p.N * p.D;
    if (f < nd) return (f / p.D) * (p.D + p.Dr) + (f % p.D);
    const int r = f - nd;
    const int n = r / p.Dr, q = r % p.Dr;
    return n * (p.D + p.Dr) + p.D + (q >> 1) + (q & 1) * (p.Dr >> 1);
  }

  __device__ __forceinline__ float cs(const __nv_bfloat16* tab, int t, int j) const {
    return __bfloat162float(tab[static_cast<size_t>(t) * p.Dr + j]);
  }

  __device__ __forceinline__ void operator()(int row, int col0, int, int, const float* v) const {
    const int nd = p.N * p.D;
    const int M = p.N * (p.D + p.Dr);
    if constexpr (SWAP) {
      const int f = row;
      if (f - (threadIdx.x & 31) < nd) {             // warp-uniform: nope rows (nd % 32 == 0)
        if (f >= nd) return;
        const float dq = INT8 ? p.dqw[orig_col(f)] : 1.f;
#pragma unroll
        for (int j = 0; j < CH; ++j) {
          const int t = col0 + j;
          if (t < p.T) {
            const float val = INT8 ? v[j] * p.scale_t[t] * dq : v[j];
            p.qc[static_cast<size_t>(t) * nd + f] = __float2bfloat16_rn(val);
          }
        }
      } else {                                        // rope rows: partner is lane ^ 1
        const bool valid = f < M;
        const int r = f - nd;
        const int n = r / p.Dr, q = r % p.Dr;
        const int e = q & 1;
        const int jj = (q >> 1) + e * (p.Dr >> 1);
        const float dq = (INT8 && valid) ? p.dqw[orig_col(f)] : 1.f;
#pragma unroll
        for (int j = 0; j < CH; ++j) {
          const int t = col0 + j;
          const bool tv = t < p.T;
          const float val = INT8 ? (tv && valid ? v[j] * p.scale_t[t] * dq : 0.f) : v[j];
          const float partner = __shfl_xor_sync(0xffffffffu, val, 1);
          if (valid && tv) {
            const float c = cs(p.cos, t, jj), s = cs(p.sin, t, jj);
            const float out = e ? (val * c + partner * s) : (val * c - partner * s);
            p.qrope[(static_cast<size_t>(t) * p.N + n) * p.Dr + jj] = __float2bfloat16_rn(out);
          }
        }
      }
    } else {
      const int t = row;
      if (t >= p.T) return;
      const float st = INT8 ? p.scale_t[t] : 1.f;
      if (col0 < nd) {
        __nv_bfloat16* dst = p.qc + static_cast<size_t>(t) * nd + col0;
        const bool full = col0 + CH <= nd;
        if (full && ((static_cast<size_t>(t) * nd + col0) % 8) == 0) {
#pragma unroll
          for (int j = 0; j < CH / 8; ++j) {
            uint4 pk;
            uint32_t* w = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              float a = v[8 * j + 2 * h], b = v[8 * j + 2 * h + 1];
              if (INT8) {
                a *= st * p.dqw[orig_col(col0 + 8 * j + 2 * h)];
                b *= st * p.dqw[orig_col(col0 + 8 * j + 2 * h + 1)];
              }
              __nv_bfloat162 h2 = __floats2bfloat162_rn(a, b);
              w[h] = *reinterpret_cast<uint32_t*>(&h2);
            }
            reinterpret_cast<uint4*>(dst)[j] = pk;
          }
        } else {
#pragma unroll
          for (int j = 0; j < CH; ++j) {
            if (col0 + j < nd) {
              float a = v[j];
              if (INT8) a *= st * p.dqw[orig_col(col0 + j)];
              dst[j] = __float2bfloat16_rn(a);
            }
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < CH; j += 2) {
          const int f = col0 + j;
          if (f >= M) continue;
          const int r = f - nd;
          const int n = r / p.Dr, pp = (r % p.Dr) >> 1;
          float y0 = v[j], y1 = v[j + 1];
          if (INT8) {
            y0 *= st * p.dqw[orig_col(f)];
            y1 *= st * p.dqw[orig_col(f + 1)];
          }
          const int j0 = pp, j1 = pp + (p.Dr >> 1);
          const float o0 = y0 * cs(p.cos, t, j0) - y1 * cs(p.sin, t, j0);
          const float o1 = y1 * cs(p.cos, t, j1) + y0 * cs(p.sin, t, j1);
          __nv_bfloat16* dst = p.qrope + (static_cast<size_t>(t) * p.N + n) * p.Dr;
          dst[j0] = __float2bfloat16_rn(o0);
          dst[j1] = __float2bfloat16_rn(o1);
        }
      }
    }
  }
};

// ----------------------------------------------------------------------------------------------
// Absorb  q^N[t, n, :] = q^C[t, n, :] · W^UK[n]  (MlaPrologV2 README q^N formula), batched over
// heads n; W^UK prepacked per head as (Hckv, D) so it is K-major.  Output query (T, N, Hckv) bf16.
struct AbsorbParams {
  __nv_bfloat16* query;
  int32_t T, N, Hckv;
};

template <bool SWAP, int CH>
struct EpiAbsorb {
  AbsorbParams p;

  __device__ __forceinline__ void operator()(int row, int col0, int n, int, const float* v) const {
    if constexpr (SWAP) {
      const int c = row;
      if (c >= p.Hckv) return;
#pragma unroll
      for (int j = 0; j < CH; ++j) {
        const int t = col0 + j;
        if (t < p.T)
          p.query[(static_cast<size_t>(t) * p.N + n) * p.Hckv + c] = __float2bfloat16_rn(v[j]);
      }
    } else {
      const int t = row;
      if (t >= p.T) return;
      __nv_bfloat16* dst = p.query + (static_cast<size_t>(t) * p.N + n) * p.Hckv + col0;
      const bool full = col0 + CH <= p.Hckv;
      if (full && (((static_cast<size_t>(t) * p.N + n) * p.Hckv + col0) % 8) == 0) {
#pragma unroll
        for (int j = 0; j < CH / 8; ++j) {
          uint4 pk;
          uint32_t* w = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            __nv_bfloat162 h2 = __floats2bfloat162_rn(v[8 * j + 2 * h], v[8 * j + 2 * h + 1]);
            w[h] = *reinterpret_cast<uint32_t*>(&h2);
          }
          reinterpret_cast<uint4*>(dst)[j] = pk;
        }
      } else {
#pragma unroll
        for (int j = 0; j < CH; ++j)
          if (col0 + j < p.Hckv) dst[j] = __float2bfloat16_rn(v[j]);
      }
    }
  }
};

}  // namespace mlap
