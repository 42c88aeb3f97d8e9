// Epilogue functors of the three MLA prolog contractions (see gemm.cuh for the calling contract).
//
// "SWAP" selects the decode orientation: A = the weight (its output features are the MMA's
// M = 128 rows), B = the activations (tokens are the MMA's N).  Without SWAP (prefill),
// A = activations (tokens are rows) and B = the weight.
//
// Every epilogue warp owns a 32 x CH block of the accumulator (32 TMEM lanes x CH columns).  The
// functor fuses the step that follows the contraction, writes the block into a per-warp shared
// memory staging tile laid out exactly as the TMA store box expects (token-major rows, the
// store map's swizzle applied), and returns the stores to issue.  Output tails (tokens beyond T,
// features beyond the matrix) are clipped by the store's tensor map, so no lane masks writes.
//
// In "direct" mode (template flag; the decode launches with tokens as MMA rows and the row-range
// schedule) the up-projection and absorb functors instead write their block from registers, each
// lane 64 contiguous bytes of its token's row, and return no TMA store: at decode sizes a TMA
// store of one 32 x 32 block costs a fraction of a microsecond to issue, which is most of an
// epilogue chunk, and the tail of the last tile is exposed.  Direct stores mask tokens >= T
// themselves.  The flag is compile-time so that the other launches keep their code unchanged.
#pragma once
#include <cuda_bf16.h>
#include "gemm.cuh"

namespace mlap {

// Swizzled staging addresses: element (row r, column c) of a tile whose rows are 128 B (fp32 x32,
// SWIZZLE_128B), 64 B (bf16 x32, SWIZZLE_64B) or 32 B (bf16 x16, SWIZZLE_32B).  The 16-byte chunk
// index is XORed with row bits as the TMA swizzle modes define; tiles start 1024-B aligned.
__device__ __forceinline__ uint32_t sw128_f32(int r, int c) {
  return r * 128 + ((((c >> 2) ^ (r & 7)) & 7) << 4) + (c & 3) * 4;
}
__device__ __forceinline__ uint32_t sw64_bf16(int r, int c) {
  return r * 64 + ((((c >> 3) ^ ((r >> 1) & 3)) & 3) << 4) + (c & 7) * 2;
}

__device__ __forceinline__ void st_f32(uint8_t* sb, uint32_t off, float v) {
  *reinterpret_cast<float*>(sb + off) = v;
}
__device__ __forceinline__ void st_bf16(uint8_t* sb, uint32_t off, float v) {
  *reinterpret_cast<__nv_bfloat16*>(sb + off) = __float2bfloat16_rn(v);
}

// Lane-as-row writes of 32 consecutive fp32 values (float4 chunks; the swizzle keeps the 32
// lanes' 16-byte writes on distinct banks).
__device__ __forceinline__ void stage_row_f32(uint8_t* sb, int r, const float* v) {
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<float4*>(sb + r * 128 + (((c ^ (r & 7)) & 7) << 4)) =
        make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint4 pack_bf16x8(const float* v) {
  return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                    pack_bf16x2(v[6], v[7]));
}

// Lane-as-row writes of 32 consecutive values rounded to bf16 (4 chunks of 8, SWIZZLE_64B).
__device__ __forceinline__ void stage_row_bf16x32(uint8_t* sb, int r, const float* v) {
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4*>(sb + r * 64 + (((c ^ ((r >> 1) & 3)) & 3) << 4)) = pack_bf16x8(v + 8 * c);
}

// Lane-as-row writes of 64 consecutive values rounded to bf16 (8 chunks of 8, SWIZZLE_128B).
__device__ __forceinline__ void stage_row_bf16x64(uint8_t* sb, int r, const float* v) {
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<uint4*>(sb + r * 128 + (((c ^ (r & 7)) & 7) << 4)) = pack_bf16x8(v + 8 * c);
}

// Lane-as-row writes of 16 consecutive values rounded to bf16 (2 chunks of 8, SWIZZLE_32B).
__device__ __forceinline__ void stage_row_bf16x16(uint8_t* sb, int r, const float* v) {
#pragma unroll
  for (int c = 0; c < 2; ++c)
    *reinterpret_cast<uint4*>(sb + r * 32 + (((c ^ ((r >> 2) & 1)) & 1) << 4)) = pack_bf16x8(v + 8 * c);
}

__device__ __forceinline__ void unpack_bf16x16(const uint4 (&q)[2], float* out) {
  const __nv_bfloat16* ea = reinterpret_cast<const __nv_bfloat16*>(&q[0]);
  const __nv_bfloat16* eb = reinterpret_cast<const __nv_bfloat16*>(&q[1]);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    out[i] = __bfloat162float(ea[i]);
    out[8 + i] = __bfloat162float(eb[i]);
  }
}

// ----------------------------------------------------------------------------------------------
// Down-projection  [h_q | h_kv | h_kr] = x · [W^DQ | W^DKV | W^KR]   (MlaPrologV2 README, c^Q and
// c^KV / k^R formulas).  The weight is two tensor maps (W^DQ, W^DKV|W^KR) seen as one operand
// with `seg_tiles` tiles in the first.  K-split s writes its fp32 partial to part[s][t][f]; the
// two output maps cover the W^DQ columns and the W^DKV|W^KR columns of part, 3-D (f, t, s).
struct DownParams {
  int32_t seg_tiles;
};

template <bool SWAP, int TILE_W, int CH>
struct EpiDown {
  static constexpr bool kDirect = false;
  static constexpr int kCols = CH;
  DownParams p;
  struct Pre {};
  __device__ __forceinline__ Pre preload(int, int) const { return {}; }

  __device__ __forceinline__ int operator()(int m0, int n0, int, int s, const float (&v)[CH],
                                            uint8_t* sb, StoreOp (&ops)[2], const Pre&) const {
    const int lane = threadIdx.x & 31;
    const int b0 = p.seg_tiles * TILE_W;
    if constexpr (SWAP) {
      const bool first = m0 < b0;
#pragma unroll
      for (int j = 0; j < CH; ++j) st_f32(sb, sw128_f32(j, lane), v[j]);
      ops[0] = {first ? 0 : 1, 3, first ? m0 : m0 - b0, n0, s, 0};
    } else {
      stage_row_f32(sb, lane, v);
      const bool first = n0 < b0;
      ops[0] = {first ? 0 : 1, 3, first ? n0 : n0 - b0, m0, s, 0};
    }
    return 1;
  }
};

// ----------------------------------------------------------------------------------------------
// Up-projection  [q^C | q_r] = c^Q · W^UQ_QR  (MlaPrologV2 README q^C and q^R formulas) with the
// weight prepacked as rows [all heads' nope columns (n*D + d) | all heads' rope columns, each
// head's pair (j, j + Dr/2) stored adjacently].  Fused: bf16 rounding of q^C (the next matmul's
// input, first output map: q^C (T, N*D)), half-and-half RoPE of q_r (aclnnQkvRmsNormRopeCache
// "Formulas" (3)) into query_rope (second output map: 3-D (Dr, N, T)), and for an int8 weight
// the dequant acc * scale_t[t] * dequant_scale_w_uq_qr[column].
struct UpParams {
  const __nv_bfloat16* cos;     // (T, Dr)
  const __nv_bfloat16* sin;     // (T, Dr)
  const float* scale_t;         // (T) per-token dequant scale, int8 path
  const float* dqw;             // (N*(D+Dr)) per-column dequant scale, int8 path
  int32_t T, N, D, Dr;
  __nv_bfloat16* qc_out;        // direct mode: q^C (T, N*D)
  __nv_bfloat16* qr_out;        //   and query_rope (T, N, Dr)
};

// DIRECT: the row-range decode launch (tokens as MMA rows, outputs written from registers).
template <bool SWAP, bool INT8, int CH, bool DIRECT = false>
struct EpiUp {
  static constexpr bool kDirect = DIRECT;
  static constexpr int kCols = CH;
  static_assert(!DIRECT || (!SWAP && !INT8), "direct stores: bf16 weight, tokens as MMA rows");
  UpParams p;

  // RoPE tables of one lane's token for one 32-row rope block: cos/sin of pairs p0..p0+15
  // (run a) and p0+Dr/2.. (run b), packed bf16.  Loaded ahead of use (see gemm.cuh).
  struct Pre {
    uint4 ca[2], sa[2], cb[2], sb[2];
  };

  __device__ __forceinline__ Pre preload(int m0, int n0) const {
    Pre r;
    const int nd = p.N * p.D;
    const int lane = threadIdx.x & 31;
    const int f0 = SWAP ? m0 : n0;        // first weight row of the block
    const int t = SWAP ? n0 + lane : m0 + lane;
    if (f0 >= nd && t < p.T) {
      const int p0 = ((f0 - nd) % p.Dr) >> 1;
      const uint4* c = reinterpret_cast<const uint4*>(p.cos + static_cast<size_t>(t) * p.Dr + p0);
      const uint4* s = reinterpret_cast<const uint4*>(p.sin + static_cast<size_t>(t) * p.Dr + p0);
      const int hb = p.Dr >> 4;           // uint4 offset of run b (Dr/2 bf16)
      r.ca[0] = __ldg(c);
      r.ca[1] = __ldg(c + 1);
      r.sa[0] = __ldg(s);
      r.sa[1] = __ldg(s + 1);
      r.cb[0] = __ldg(c + hb);
      r.cb[1] = __ldg(c + hb + 1);
      r.sb[0] = __ldg(s + hb);
      r.sb[1] = __ldg(s + hb + 1);
    } else {
      r.ca[0] = r.ca[1] = r.sa[0] = r.sa[1] = r.cb[0] = r.cb[1] = r.sb[0] = r.sb[1] =
          make_uint4(0, 0, 0, 0);
    }
    return r;
  }

  // original column of weight_uq_qr for a prepacked row
  __device__ __forceinline__ int orig_col(int f) const {
    const int nd = p.N * p.D;
    if (f < nd) return (f / p.D) * (p.D + p.Dr) + (f % p.D);
    const int r = f - nd;
    const int n = r / p.Dr, q = r % p.Dr;
    return n * (p.D + p.Dr) + p.D + (q >> 1) + (q & 1) * (p.Dr >> 1);
  }

  // RoPE of one token's 16 adjacent (j, j + Dr/2) pairs y[2i], y[2i+1], i < 16, i.e. pairs
  // p0 .. p0+15 of one head, with that token's preloaded tables; the results are staged at row r
  // of two 16-wide bf16 tiles holding output columns p0.. and p0+Dr/2.. (offsets 0 and 1024 of
  // the staging buffer).
  __device__ __forceinline__ void rope_pairs(const Pre& P, const float* y, float (&oa)[16],
                                             float (&ob)[16]) const {
    float c0[16], s0[16], c1[16], s1[16];
    unpack_bf16x16(P.ca, c0);
    unpack_bf16x16(P.sa, s0);
    unpack_bf16x16(P.cb, c1);
    unpack_bf16x16(P.sb, s1);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float y0 = y[2 * i], y1 = y[2 * i + 1];
      oa[i] = y0 * c0[i] - y1 * s0[i];
      ob[i] = y1 * c1[i] + y0 * s1[i];
    }
  }
  __device__ __forceinline__ void rope_row(uint8_t* sb, int r, const Pre& P, const float* y) const {
    float oa[16], ob[16];
    rope_pairs(P, y, oa, ob);
    stage_row_bf16x16(sb, r, oa);
    stage_row_bf16x16(sb + 1024, r, ob);
  }

  __device__ __forceinline__ int operator()(int m0, int n0, int, int, const float (&v)[CH],
                                            uint8_t* sb, StoreOp (&ops)[2], const Pre& P) const {
    const int lane = threadIdx.x & 31;
    const int nd = p.N * p.D;
    const int M = p.N * (p.D + p.Dr);
    if constexpr (SWAP) {
      // lane = weight row f = m0 + lane, v[j] = token n0 + j
      const int f = m0 + lane;
      float w[CH];
      if constexpr (INT8) {
        const float dq = f < M ? __ldg(p.dqw + orig_col(f)) : 0.f;
#pragma unroll
        for (int j = 0; j < CH; ++j) {
          const int t = n0 + j;
          w[j] = t < p.T ? v[j] * __ldg(p.scale_t + t) * dq : 0.f;
        }
      } else {
#pragma unroll
        for (int j = 0; j < CH; ++j) w[j] = v[j];
      }
      if (m0 < nd) {   // nope rows (nd is a multiple of 128: the whole block is nope)
#pragma unroll
        for (int j = 0; j < CH; ++j) st_bf16(sb, sw64_bf16(j, lane), w[j]);
        ops[0] = {0, 2, m0, n0, 0, 0};
        return 1;
      }
      // rope rows: transpose through the staging tile (fp32), then each lane takes one token
#pragma unroll
      for (int j = 0; j < CH; ++j) st_f32(sb, sw128_f32(j, lane), w[j]);
      __syncwarp();
      float y[32];
      if (lane < CH) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float4 q =
              *reinterpret_cast<const float4*>(sb + lane * 128 + (((c ^ (lane & 7)) & 7) << 4));
          y[4 * c] = q.x;
          y[4 * c + 1] = q.y;
          y[4 * c + 2] = q.z;
          y[4 * c + 3] = q.w;
        }
      }
      __syncwarp();
      const int r0 = m0 - nd;                 // first rope row of the block (Dr % 32 == 0)
      const int n = r0 / p.Dr, p0 = (r0 % p.Dr) >> 1;
      if (lane < CH) rope_row(sb, lane, P, y);
      ops[0] = {1, 3, p0, n, n0, 0};
      ops[1] = {1, 3, p0 + (p.Dr >> 1), n, n0, 1024};
      return 2;
    } else {
      // lane = token t = m0 + lane, v[j] = prepacked column n0 + j
      const int t = m0 + lane;
      float w[32];
      if constexpr (INT8) {
        const float st = t < p.T ? __ldg(p.scale_t + t) : 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int f = n0 + j;
          w[j] = f < M ? v[j] * st * __ldg(p.dqw + orig_col(f)) : 0.f;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) w[j] = v[j];
      }
      if constexpr (DIRECT) {   // lane = token, 64 contiguous bytes
        if (t >= p.T) return 0;
        if (n0 < nd) {
          uint4* dst = reinterpret_cast<uint4*>(p.qc_out + static_cast<size_t>(t) * nd + n0);
#pragma unroll
          for (int c = 0; c < 4; ++c) dst[c] = pack_bf16x8(w + 8 * c);
          return 0;
        }
        const int r0 = n0 - nd;
        const int n = r0 / p.Dr, p0 = (r0 % p.Dr) >> 1;
        float oa[16], ob[16];
        rope_pairs(P, w, oa, ob);
        __nv_bfloat16* row = p.qr_out + (static_cast<size_t>(t) * p.N + n) * p.Dr;
        uint4* da = reinterpret_cast<uint4*>(row + p0);
        uint4* db = reinterpret_cast<uint4*>(row + p0 + (p.Dr >> 1));
        da[0] = pack_bf16x8(oa);
        da[1] = pack_bf16x8(oa + 8);
        db[0] = pack_bf16x8(ob);
        db[1] = pack_bf16x8(ob + 8);
        return 0;
      }
      if (n0 < nd) {
        stage_row_bf16x32(sb, lane, w);
        ops[0] = {0, 2, n0, m0, 0, 0};
        return 1;
      }
      const int r0 = n0 - nd;
      const int n = r0 / p.Dr, p0 = (r0 % p.Dr) >> 1;
      rope_row(sb, lane, P, w);
      ops[0] = {1, 3, p0, n, m0, 0};
      ops[1] = {1, 3, p0 + (p.Dr >> 1), n, m0, 1024};
      return 2;
    }
  }
};

// ----------------------------------------------------------------------------------------------
// Absorb  q^N[t, n, :] = q^C[t, n, :] · W^UK[n]  (MlaPrologV2 README q^N formula), batched over
// heads n; W^UK prepacked per head as (Hckv, D) so it is K-major.  Output map: query as 3-D
// (Hckv, N, T) bf16.
struct AbsorbParams {
  __nv_bfloat16* out;           // direct mode: query (T, N, Hckv)
  int32_t T, N, Hckv;
};

// CH = 64 (prefill, TMA stores): each lane stages 128 contiguous bytes of its token's row and one
// store box covers 32 tokens x 64 columns, whole 128-byte lines of query.
template <bool SWAP, int CH, bool DIRECT = false>
struct EpiAbsorb {
  static constexpr bool kDirect = DIRECT;
  static constexpr int kCols = CH;
  static_assert(!DIRECT || !SWAP, "direct stores: tokens as MMA rows");
  static_assert(CH != 64 || (!SWAP && !DIRECT), "64-column chunks: TMA stores, tokens as rows");
  AbsorbParams p;
  struct Pre {};
  __device__ __forceinline__ Pre preload(int, int) const { return {}; }

  __device__ __forceinline__ int operator()(int m0, int n0, int n, int, const float (&v)[CH],
                                            uint8_t* sb, StoreOp (&ops)[2], const Pre&) const {
    const int lane = threadIdx.x & 31;
    if constexpr (SWAP) {
#pragma unroll
      for (int j = 0; j < CH; ++j) st_bf16(sb, sw64_bf16(j, lane), v[j]);
      ops[0] = {0, 3, m0, n, n0, 0};
    } else {
      if constexpr (DIRECT) {   // lane = token, 64 contiguous bytes
        const int t = m0 + lane;
        if (t < p.T) {
          uint4* dst = reinterpret_cast<uint4*>(
              p.out + (static_cast<size_t>(t) * p.N + n) * p.Hckv + n0);
#pragma unroll
          for (int c = 0; c < 4; ++c) dst[c] = pack_bf16x8(v + 8 * c);
        }
        return 0;
      }
      if constexpr (CH == 64) stage_row_bf16x64(sb, lane, v);
      else stage_row_bf16x32(sb, lane, v);
      ops[0] = {0, 3, n0, n, m0, 0};
    }
    return 1;
  }
};

}  // namespace mlap
