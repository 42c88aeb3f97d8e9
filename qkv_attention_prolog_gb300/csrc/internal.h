// Internal launch interfaces shared by the host API (api.cu) and the kernel translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "gemm.cuh"
#include "epilogues.cuh"
#include "stamps.cuh"

namespace mlap {

// One launch of umma_gemm_kernel: the four tensor maps (first/second segment of A and B),
// the tile geometry, the N tile width, the orientation and the grid.
struct GemmLaunch {
  CUtensorMap a0, a1, b0, b1;   // operand maps (first / second segment)
  CUtensorMap o0, o1;           // output maps for the epilogue's TMA stores
  GemmGeometry geo;
  int bn;
  int mt;            // 128-row tiles of A per unit (decode orientation: 1 or 2)
  bool swap;
  bool a_int8;       // A operand is an int8 weight converted to bf16 in shared memory
  bool rr;           // row-range schedule with direct epilogue stores (decode, tokens as rows)
  int cg;            // 2: CTA-pair tiles (256 rows of A, cta_group::2 MMAs); the grid counts CTAs
  int grid;
  cudaStream_t stream;
  bool pdl;
  uint32_t* err;
};

cudaError_t launch_down(const GemmLaunch& L, const DownParams& p);
cudaError_t launch_up(const GemmLaunch& L, const UpParams& p, bool int8);

// Fused decode up-projection + absorb, one CTA per head (up_absorb.cu): tokens as MMA rows,
// q^C kept in shared memory, query_rope and query written directly.
struct UpAbsorbParams {
  const __nv_bfloat16* cos;     // (T, Dr)
  const __nv_bfloat16* sin;     // (T, Dr)
  __nv_bfloat16* qr_out;        // query_rope (T, N, Dr)
  __nv_bfloat16* q_out;         // query (T, N, Hckv)
  int32_t T, N, Hcq, Hckv;
  const float* scale_t;         // int8 weight: per-token c^Q quant scale (T)
  const float* dqw;             // int8 weight: dequant_scale_w_uq_qr (N*(D+Dr))
  int32_t k;                    // W^QR blocks of 32 rows kept by each head CTA (0, 1 or 2)
  int32_t R;                    // CTAs after the head CTAs that take the other W^QR blocks
  uint64_t* stamps;             // optional execution stamps (stamps.cuh), slot MLAP_STAMP_UP
  int32_t pair;                 // 1: two CTAs (a cluster) per head, 2N head CTAs
  int32_t cq_rows;              // token rows of tmCq's box: T rounded up to 8, at most 128
};
// One CTA whose bounded mbarrier wait runs out (nothing completes the barrier) and latches
// kErrTimeout in err_word (selftest.cu).
cudaError_t launch_bounded_wait_selftest(uint32_t* err_word, cudaStream_t stream);

// k, R and pair for `sms` SMs and N heads (grid = N + R, or 2N + R for pairs)
void up_absorb_plan(int sms, int N, int* k, int* R, int* pair);
bool up_absorb_supported(int64_t T, int64_t N, int64_t D, int64_t Dr, int64_t Hckv);
// tmCq: c^Q (T, Hcq) bf16, box 64 x p.cq_rows, 128B-swizzled; tmW: prepacked W^UQ|W^QR
// (N*(D+Dr) rows of Hcq), box 64 x 32, bf16 128B-swizzled or int8 unswizzled (int8 = true);
// tmUk: prepacked W^UK (N*Hckv rows of D), box 64 x 32, 128B-swizzled.  tmW128 / tmUk128: the
// same two tensors with boxes of 128 rows, given for int8 weights (which selects the int8
// kernel) and null for bf16.
cudaError_t launch_up_absorb(const CUtensorMap& tmCq, const CUtensorMap& tmW,
                             const CUtensorMap& tmUk, const CUtensorMap* tmW128,
                             const CUtensorMap* tmUk128, const UpAbsorbParams& p, uint32_t* err,
                             cudaStream_t stream);
cudaError_t launch_absorb(const GemmLaunch& L, const AbsorbParams& p);

// RmsNorm of c^Q (+ dynamic int8 quant) and c^KV, RoPE of k^R, cache quant and scatter; one CTA
// per token, summing the down-projection's K-split partials in split order.
struct FinalizeParams {
  const float* part;
  int32_t splits, T, Hcq, Hckv, Dr, Ntot;
  const __nv_bfloat16* gamma_cq;
  const __nv_bfloat16* gamma_ckv;
  float eps_cq, eps_ckv;
  const __nv_bfloat16* cos;
  const __nv_bfloat16* sin;
  const int64_t* cache_index;
  int64_t slots;               // BlockNum * BlockSize (0: no cache update)
  void* kv_cache;
  void* kr_cache;
  int32_t kv_int8, kr_int8;
  const float* qs_ckv;
  const float* qs_ckr;
  __nv_bfloat16* cq_out;       // (T, Hcq): bf16 c^Q, or int8 codes held exactly in f16 bits
  const float* smooth;         // non-null: quantise c^Q per token
  float* scale_t;              // (T) per-token scale of the quantised c^Q
  uint32_t* err;
  const float* dsx;            // full quant: h *= dsx[t] * (dsw_q | dsw_kv)[column] (null: none)
  const float* dsw_q;
  const float* dsw_kv;
  uint64_t* stamps;            // optional execution stamps (stamps.cuh), slot MLAP_STAMP_NORM
};
cudaError_t launch_finalize(const FinalizeParams& p, cudaStream_t stream, bool pdl);

// Input RmsNormQuant ahead of the down-projection: out[t] = bf16((gamma * x[t] / RMS(x[t]) + bias)
// * deq) for T rows of He bf16 values (He a multiple of 8, at most 10240); deq holds He values, or
// one value for every channel when deq_per_channel is false.  Launched with programmatic
// dependent launch (waits for the preceding kernel before reading).
cudaError_t launch_rms_norm_quant(const __nv_bfloat16* x, const __nv_bfloat16* gamma,
                                  const __nv_bfloat16* bias, const float* deq, bool deq_per_channel,
                                  float eps, __nv_bfloat16* out, int64_t T, int32_t He,
                                  cudaStream_t stream);

// Full quant beyond 256 tokens: int8 token_x widened to f16 (exact), n elements (a multiple of
// 16).
cudaError_t launch_widen_int8(const int8_t* x, __half* out, int64_t n, cudaStream_t stream);

// int8 query per token and head: rows of H bf16 values -> int8 codes (scale = amax / 127, round
// half to even, clamp to [-127, 127]) and the per-row fp32 scale (dequant_scale_q_nope).
cudaError_t launch_query_quant(const __nv_bfloat16* qn, int8_t* q, float* scale, int64_t rows,
                               int32_t H, cudaStream_t stream);

// Weight prepack: dst[b][i][k] = src[b][k][perm(i)]  (a transpose with a row permutation).
enum PermKind : int32_t { kPermIdentity = 0, kPermUqQr = 1 };
struct PrepackParams {
  const void* src;
  void* dst;
  int32_t elem_bytes;          // 1 or 2
  int32_t K, C, R, batches;    // src (batches, K, C); dst (batches, R, K)
  int32_t perm;                // PermKind
  int32_t N, D, Dr;            // head geometry for kPermUqQr
};
cudaError_t launch_prepack(const PrepackParams& p, cudaStream_t stream);

// QkvRmsNormRopeCache streaming kernel.
struct QkvParams {
  const void* qkv;             // (T, (Nq+Nk+Nv)*D) fp16|bf16
  const void* gamma_q;
  const void* gamma_k;
  const void* cos;
  const void* sin;
  const int64_t* index;
  int64_t slots;
  void* k_cache;
  void* v_cache;
  const float* k_scale;        // null: no quant
  const float* v_scale;
  const float* k_offset;       // null: symmetric quant
  const float* v_offset;
  void* q_before;              // optional dense before-quant outputs (null: not written)
  void* k_before;
  void* v_before;
  void* q_out;
  int32_t T, Nq, Nk, Nv;
  float eps;
  int32_t bf16;                // element type of qkv: 0 fp16, 1 bf16
  uint32_t* err;
  uint64_t* stamps;            // optional execution stamps (stamps.cuh), slot MLAP_STAMP_QKV
};
cudaError_t launch_qkv_rnrc(const QkvParams& p, cudaStream_t stream, int sm_count);

}  // namespace mlap
