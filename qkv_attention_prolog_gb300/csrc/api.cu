// libmlaprolog host API: argument validation against the operator documentation, workspace
// planning, TMA descriptor encoding and the kernel launch sequence.
//
// Validation follows the MlaPrologV2 README parameter table (参数说明) and shape/dtype/scenario
// matrix (约束说明), and the aclnnQkvRmsNormRopeCache "Input shape restrictions"; the two-phase
// size-then-execute pattern follows the aclnn GetWorkspaceSize + execute pair.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"
#include "mlaprolog.h"

using namespace mlap;

namespace {

thread_local std::string g_last_error;

mlap_status_t fail(mlap_status_t code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

#define CHECK_STATUS(expr)              \
  do {                                  \
    mlap_status_t _s = (expr);          \
    if (_s != MLAP_OK) return _s;       \
  } while (0)

size_t dtype_bytes(int32_t dt) {
  switch (dt) {
    case MLAP_DTYPE_BF16:
    case MLAP_DTYPE_FP16: return 2;
    case MLAP_DTYPE_FP32: return 4;
    case MLAP_DTYPE_INT8: return 1;
    case MLAP_DTYPE_INT64: return 8;
    default: return 0;
  }
}

int64_t numel(const mlap_tensor_t& t) {
  int64_t n = 1;
  for (int i = 0; i < t.ndim; ++i) n *= t.shape[i];
  return n;
}

std::string shape_str(const mlap_tensor_t& t) {
  std::string s = "(";
  for (int i = 0; i < t.ndim; ++i) s += (i ? "," : "") + std::to_string(t.shape[i]);
  return s + ")";
}

bool present(const mlap_tensor_t& t) { return t.data != nullptr; }

mlap_status_t need(const mlap_tensor_t& t, const char* name, bool allow_empty) {
  if (t.ndim < 0 || t.ndim > 4) return fail(MLAP_ERR_SHAPE, std::string(name) + ": ndim out of range");
  for (int i = 0; i < t.ndim; ++i)
    if (t.shape[i] < 0) return fail(MLAP_ERR_SHAPE, std::string(name) + ": negative dimension");
  if (t.data == nullptr && !(allow_empty && numel(t) == 0))
    return fail(MLAP_ERR_NULL, std::string(name) + " is NULL");
  if (t.data != nullptr && (reinterpret_cast<uintptr_t>(t.data) & 15u) != 0)
    return fail(MLAP_ERR_UNSUPPORTED, std::string(name) + ": data pointer not 16-byte aligned");
  return MLAP_OK;
}

mlap_status_t want_dtype(const mlap_tensor_t& t, const char* name, int32_t dt) {
  if (t.dtype != dt) return fail(MLAP_ERR_DTYPE, std::string(name) + ": unexpected dtype");
  return MLAP_OK;
}

mlap_status_t want_shape(const mlap_tensor_t& t, const char* name, std::initializer_list<int64_t> s) {
  bool ok = t.ndim == static_cast<int32_t>(s.size());
  int i = 0;
  for (int64_t d : s) {
    if (!ok) break;
    ok = t.shape[i++] == d;
  }
  if (!ok) return fail(MLAP_ERR_SHAPE, std::string(name) + ": shape " + shape_str(t) + " does not match");
  return MLAP_OK;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// ----------------------------------------------------------------------------------------------
// MLA prolog shapes
struct MlaDims {
  int64_t T, B, S;
  bool bsh;
  int64_t He, Hcq, Hckv, N, D, Dr, BlockNum, BlockSize;
  bool w_int8, kv_int8, kr_int8;
  bool full;         // full quant: int8 token_x, W^DQ and W^DKV|W^KR (with dequant scales)
  bool query_int8;   // full quant with int8 kv_cache: int8 query + dequant_scale_q_nope
  bool xnorm;        // input RmsNormQuant ahead of the down-projection
  bool xnorm_deq_per_channel;
};

constexpr int kSwapMaxT = 256;   // decode orientation (weights as MMA rows) up to this many tokens
constexpr int kSplitMaxT = 256;  // down-projection K splits (few output tiles) up to this many tokens
constexpr int kMaxSplits = 16;
// The fused decode up/absorb runs one CTA per head (SMs left over take W^QR rows); from the
// smallest head count of the pages on it beats the separate kernels (16 heads, T = 8: 20.1 ->
// 15.0 µs per call).
constexpr int kFusedMinHeads = 16;
constexpr size_t kHeaderBytes = 256;    // the error word, padded to the workspace alignment

mlap_status_t validate_mla(const mlap_args_t* a, MlaDims* d) {
  if (a == nullptr) return fail(MLAP_ERR_NULL, "args is NULL");
  const mlap_tensor_t& x = a->token_x;
  // token_x: (T, He) or (B, S, He)  (约束说明: BS合轴 or not)
  if (x.ndim == 2) {
    d->bsh = false;
    d->T = x.shape[0];
    d->B = x.shape[0];
    d->S = 1;
    d->He = x.shape[1];
  } else if (x.ndim == 3) {
    d->bsh = true;
    d->B = x.shape[0];
    d->S = x.shape[1];
    d->T = d->B * d->S;
    d->He = x.shape[2];
  } else {
    return fail(MLAP_ERR_SHAPE, "token_x must be (T, He) or (B, S, He)");
  }
  CHECK_STATUS(need(x, "token_x", true));
  d->full = x.dtype == MLAP_DTYPE_INT8;   // 全量化: int8 token_x
  if (!d->full) CHECK_STATUS(want_dtype(x, "token_x", MLAP_DTYPE_BF16));
  const int wdt = d->full ? MLAP_DTYPE_INT8 : MLAP_DTYPE_BF16;   // W^DQ, W^DKV|W^KR dtype

  // weights (logical shapes (k, n); data = prepacked buffers)
  const mlap_tensor_t& wdq = a->weight_dq;
  CHECK_STATUS(need(wdq, "weight_dq", false));
  CHECK_STATUS(want_dtype(wdq, "weight_dq", wdt));
  if (wdq.ndim != 2 || wdq.shape[0] != d->He) return fail(MLAP_ERR_SHAPE, "weight_dq must be (He, Hcq)");
  d->Hcq = wdq.shape[1];

  const mlap_tensor_t& wuk = a->weight_uk;
  CHECK_STATUS(need(wuk, "weight_uk", false));
  CHECK_STATUS(want_dtype(wuk, "weight_uk", MLAP_DTYPE_BF16));
  if (wuk.ndim != 3) return fail(MLAP_ERR_SHAPE, "weight_uk must be (N, D, Hckv)");
  d->N = wuk.shape[0];
  d->D = wuk.shape[1];
  d->Hckv = wuk.shape[2];

  const mlap_tensor_t& sn = a->rope_sin;
  CHECK_STATUS(need(sn, "rope_sin", true));
  if (sn.ndim < 1) return fail(MLAP_ERR_SHAPE, "rope_sin must be (T, Dr) or (B, S, Dr)");
  d->Dr = sn.shape[sn.ndim - 1];

  if (d->D != 128) return fail(MLAP_ERR_UNSUPPORTED, "D (weight_uk dim 1) must be 128");
  if (d->Dr <= 0 || (d->Dr % 32)) return fail(MLAP_ERR_UNSUPPORTED, "Dr must be a positive multiple of 32");
  if (d->N <= 0 || d->Hckv <= 0 || d->Hcq <= 0 || d->He <= 0)
    return fail(MLAP_ERR_SHAPE, "N, Hckv, Hcq and He must be positive");
  if ((d->He % 8) || (d->Hcq % 8) || (d->Hckv % 8))
    return fail(MLAP_ERR_UNSUPPORTED, "He, Hcq and Hckv must be multiples of 8 (16-byte TMA pitch)");
  if (d->full && (d->He % 16))
    return fail(MLAP_ERR_UNSUPPORTED, "full quant needs He % 16 == 0 (16-byte int8 row pitch)");

  const mlap_tensor_t& wuq = a->weight_uq_qr;
  CHECK_STATUS(need(wuq, "weight_uq_qr", false));
  CHECK_STATUS(want_shape(wuq, "weight_uq_qr", {d->Hcq, d->N * (d->D + d->Dr)}));
  if (wuq.dtype == MLAP_DTYPE_INT8) {
    d->w_int8 = true;
    if (d->Hcq % 16)
      return fail(MLAP_ERR_UNSUPPORTED, "int8 weight_uq_qr needs Hcq % 16 == 0 (16-byte TMA row pitch)");
  }
  else if (wuq.dtype == MLAP_DTYPE_BF16) d->w_int8 = false;
  else return fail(MLAP_ERR_DTYPE, "weight_uq_qr must be bf16 or int8");

  const mlap_tensor_t& wkv = a->weight_dkv_kr;
  CHECK_STATUS(need(wkv, "weight_dkv_kr", false));
  CHECK_STATUS(want_dtype(wkv, "weight_dkv_kr", wdt));
  CHECK_STATUS(want_shape(wkv, "weight_dkv_kr", {d->He, d->Hckv + d->Dr}));

  CHECK_STATUS(need(a->rmsnorm_gamma_cq, "rmsnorm_gamma_cq", false));
  CHECK_STATUS(want_dtype(a->rmsnorm_gamma_cq, "rmsnorm_gamma_cq", MLAP_DTYPE_BF16));
  CHECK_STATUS(want_shape(a->rmsnorm_gamma_cq, "rmsnorm_gamma_cq", {d->Hcq}));
  CHECK_STATUS(need(a->rmsnorm_gamma_ckv, "rmsnorm_gamma_ckv", false));
  CHECK_STATUS(want_dtype(a->rmsnorm_gamma_ckv, "rmsnorm_gamma_ckv", MLAP_DTYPE_BF16));
  CHECK_STATUS(want_shape(a->rmsnorm_gamma_ckv, "rmsnorm_gamma_ckv", {d->Hckv}));

  // token-shaped inputs / outputs: BSH or TND, all in the same form as token_x
  const mlap_tensor_t& cs = a->rope_cos;
  CHECK_STATUS(need(cs, "rope_cos", true));
  CHECK_STATUS(want_dtype(sn, "rope_sin", MLAP_DTYPE_BF16));
  CHECK_STATUS(want_dtype(cs, "rope_cos", MLAP_DTYPE_BF16));
  const mlap_tensor_t& ci = a->cache_index;
  CHECK_STATUS(need(ci, "cache_index", true));
  CHECK_STATUS(want_dtype(ci, "cache_index", MLAP_DTYPE_INT64));
  const mlap_tensor_t& q = a->query;
  const mlap_tensor_t& qr = a->query_rope;
  CHECK_STATUS(need(q, "query", true));
  CHECK_STATUS(need(qr, "query_rope", true));
  d->query_int8 = q.dtype == MLAP_DTYPE_INT8;   // checked against the scenario below
  if (!d->query_int8) CHECK_STATUS(want_dtype(q, "query", MLAP_DTYPE_BF16));
  CHECK_STATUS(want_dtype(qr, "query_rope", MLAP_DTYPE_BF16));
  if (d->bsh) {
    CHECK_STATUS(want_shape(sn, "rope_sin", {d->B, d->S, d->Dr}));
    CHECK_STATUS(want_shape(cs, "rope_cos", {d->B, d->S, d->Dr}));
    CHECK_STATUS(want_shape(ci, "cache_index", {d->B, d->S}));
    CHECK_STATUS(want_shape(q, "query", {d->B, d->S, d->N, d->Hckv}));
    CHECK_STATUS(want_shape(qr, "query_rope", {d->B, d->S, d->N, d->Dr}));
  } else {
    CHECK_STATUS(want_shape(sn, "rope_sin", {d->T, d->Dr}));
    CHECK_STATUS(want_shape(cs, "rope_cos", {d->T, d->Dr}));
    CHECK_STATUS(want_shape(ci, "cache_index", {d->T}));
    CHECK_STATUS(want_shape(q, "query", {d->T, d->N, d->Hckv}));
    CHECK_STATUS(want_shape(qr, "query_rope", {d->T, d->N, d->Dr}));
  }

  // caches (BlockNum, BlockSize, Nkv = 1, H)
  const mlap_tensor_t& kv = a->kv_cache;
  const mlap_tensor_t& kr = a->kr_cache;
  if (kv.ndim != 4 || kr.ndim != 4) return fail(MLAP_ERR_SHAPE, "caches must be (BlockNum, BlockSize, Nkv, H)");
  d->BlockNum = kv.shape[0];
  d->BlockSize = kv.shape[1];
  CHECK_STATUS(need(kv, "kv_cache", true));
  CHECK_STATUS(need(kr, "kr_cache", true));
  if (kv.shape[2] != 1 || kr.shape[2] != 1) return fail(MLAP_ERR_UNSUPPORTED, "Nkv must be 1");
  CHECK_STATUS(want_shape(kv, "kv_cache", {d->BlockNum, d->BlockSize, 1, d->Hckv}));
  CHECK_STATUS(want_shape(kr, "kr_cache", {d->BlockNum, d->BlockSize, 1, d->Dr}));
  auto cache_dt = [](const mlap_tensor_t& c, const char* n, bool* i8) -> mlap_status_t {
    if (c.dtype == MLAP_DTYPE_INT8) *i8 = true;
    else if (c.dtype == MLAP_DTYPE_BF16) *i8 = false;
    else return fail(MLAP_ERR_DTYPE, std::string(n) + " must be bf16 or int8");
    return MLAP_OK;
  };
  CHECK_STATUS(cache_dt(kv, "kv_cache", &d->kv_int8));
  CHECK_STATUS(cache_dt(kr, "kr_cache", &d->kr_int8));

  // scenario matrix (约束说明)
  if (d->full) {
    // 全量化: per-token dequant of x, per-channel dequant of W^DQ and W^DKV|W^KR, int8 W^UQ|W^QR;
    // kr_cache stays bf16; an int8 kv_cache makes the query int8 per token and head
    const mlap_tensor_t& dsx = a->dequant_scale_x;
    CHECK_STATUS(need(dsx, "dequant_scale_x", false));
    CHECK_STATUS(want_dtype(dsx, "dequant_scale_x", MLAP_DTYPE_FP32));
    CHECK_STATUS(want_shape(dsx, "dequant_scale_x", {d->T, 1}));
    CHECK_STATUS(need(a->dequant_scale_w_dq, "dequant_scale_w_dq", false));
    CHECK_STATUS(want_dtype(a->dequant_scale_w_dq, "dequant_scale_w_dq", MLAP_DTYPE_FP32));
    CHECK_STATUS(want_shape(a->dequant_scale_w_dq, "dequant_scale_w_dq", {1, d->Hcq}));
    CHECK_STATUS(need(a->dequant_scale_w_dkv_kr, "dequant_scale_w_dkv_kr", false));
    CHECK_STATUS(want_dtype(a->dequant_scale_w_dkv_kr, "dequant_scale_w_dkv_kr", MLAP_DTYPE_FP32));
    CHECK_STATUS(want_shape(a->dequant_scale_w_dkv_kr, "dequant_scale_w_dkv_kr", {1, d->Hckv + d->Dr}));
    if (!d->w_int8) return fail(MLAP_ERR_UNSUPPORTED, "full quant needs an int8 weight_uq_qr");
    if (d->kr_int8) return fail(MLAP_ERR_UNSUPPORTED, "full quant keeps kr_cache bf16");
    if (present(a->quant_scale_ckr))
      return fail(MLAP_ERR_UNSUPPORTED, "quant_scale_ckr is not used in full quant");
    if (d->query_int8 != d->kv_int8)
      return fail(MLAP_ERR_UNSUPPORTED, "full quant: query is int8 exactly when kv_cache is int8");
    if (d->query_int8) {
      if (d->Hckv > 1024) return fail(MLAP_ERR_UNSUPPORTED, "an int8 query needs Hckv <= 1024");
      const mlap_tensor_t& sq = a->dequant_scale_q_nope;
      CHECK_STATUS(need(sq, "dequant_scale_q_nope", false));
      CHECK_STATUS(want_dtype(sq, "dequant_scale_q_nope", MLAP_DTYPE_FP32));
      CHECK_STATUS(want_shape(sq, "dequant_scale_q_nope", {d->T, d->N, 1}));
    }
  } else {
    if (present(a->dequant_scale_x) || present(a->dequant_scale_w_dq) ||
        present(a->dequant_scale_w_dkv_kr))
      return fail(MLAP_ERR_UNSUPPORTED,
                  "dequant_scale_x / _w_dq / _w_dkv_kr are reserved outside full quant and must be NULL");
    if (d->query_int8) return fail(MLAP_ERR_DTYPE, "int8 query is the full-quant scenario");
    if (d->kv_int8 != d->kr_int8)
      return fail(MLAP_ERR_UNSUPPORTED, "kv_cache and kr_cache must both be int8 or both bf16 outside full quant");
  }
  if (d->w_int8) {
    CHECK_STATUS(need(a->dequant_scale_w_uq_qr, "dequant_scale_w_uq_qr", false));
    CHECK_STATUS(want_dtype(a->dequant_scale_w_uq_qr, "dequant_scale_w_uq_qr", MLAP_DTYPE_FP32));
    CHECK_STATUS(want_shape(a->dequant_scale_w_uq_qr, "dequant_scale_w_uq_qr", {1, d->N * (d->D + d->Dr)}));
    CHECK_STATUS(need(a->smooth_scales_cq, "smooth_scales_cq", false));
    CHECK_STATUS(want_dtype(a->smooth_scales_cq, "smooth_scales_cq", MLAP_DTYPE_FP32));
    CHECK_STATUS(want_shape(a->smooth_scales_cq, "smooth_scales_cq", {1, d->Hcq}));
  } else {
    if (present(a->dequant_scale_w_uq_qr) || present(a->smooth_scales_cq))
      return fail(MLAP_ERR_UNSUPPORTED, "dequant_scale_w_uq_qr / smooth_scales_cq need an int8 weight_uq_qr");
    if (d->kv_int8) return fail(MLAP_ERR_UNSUPPORTED, "int8 caches need the partial-quant scenario");
  }
  if (d->kv_int8) {
    CHECK_STATUS(need(a->quant_scale_ckv, "quant_scale_ckv", false));
    CHECK_STATUS(want_dtype(a->quant_scale_ckv, "quant_scale_ckv", MLAP_DTYPE_FP32));
    CHECK_STATUS(want_shape(a->quant_scale_ckv, "quant_scale_ckv", {1, d->Hckv}));
  }
  if (d->kr_int8) {
    CHECK_STATUS(need(a->quant_scale_ckr, "quant_scale_ckr", false));
    CHECK_STATUS(want_dtype(a->quant_scale_ckr, "quant_scale_ckr", MLAP_DTYPE_FP32));
    CHECK_STATUS(want_shape(a->quant_scale_ckr, "quant_scale_ckr", {1, d->Dr}));
  }
  if ((!d->kv_int8 && present(a->quant_scale_ckv)) || (!d->kr_int8 && present(a->quant_scale_ckr))) {
    return fail(MLAP_ERR_UNSUPPORTED, "quant_scale_ckv / quant_scale_ckr need int8 caches");
  }
  // input RmsNormQuant (aclnnMlaPreprocessV2 "Formula"): all three parameters or none
  const int xn = present(a->rms_norm_quant_gamma) + present(a->rms_norm_quant_bias) +
                 present(a->rms_norm_quant_deq_scale);
  d->xnorm = xn == 3;
  d->xnorm_deq_per_channel = false;
  if (xn != 0 && xn != 3)
    return fail(MLAP_ERR_NULL, "rms_norm_quant_gamma, _bias and _deq_scale are given together or not at all");
  if (d->xnorm) {
    if (d->full) return fail(MLAP_ERR_UNSUPPORTED, "the input RmsNormQuant needs a bf16 token_x (not full quant)");
    if (d->He > 10240) return fail(MLAP_ERR_UNSUPPORTED, "the input RmsNormQuant supports He <= 10240");
    CHECK_STATUS(need(a->rms_norm_quant_gamma, "rms_norm_quant_gamma", false));
    CHECK_STATUS(want_dtype(a->rms_norm_quant_gamma, "rms_norm_quant_gamma", MLAP_DTYPE_BF16));
    CHECK_STATUS(want_shape(a->rms_norm_quant_gamma, "rms_norm_quant_gamma", {d->He}));
    CHECK_STATUS(need(a->rms_norm_quant_bias, "rms_norm_quant_bias", false));
    CHECK_STATUS(want_dtype(a->rms_norm_quant_bias, "rms_norm_quant_bias", MLAP_DTYPE_BF16));
    CHECK_STATUS(want_shape(a->rms_norm_quant_bias, "rms_norm_quant_bias", {d->He}));
    const mlap_tensor_t& dq = a->rms_norm_quant_deq_scale;
    CHECK_STATUS(need(dq, "rms_norm_quant_deq_scale", false));
    CHECK_STATUS(want_dtype(dq, "rms_norm_quant_deq_scale", MLAP_DTYPE_FP32));
    if (dq.ndim == 1 && dq.shape[0] == d->He) d->xnorm_deq_per_channel = true;
    else if (!(dq.ndim == 1 && dq.shape[0] == 1))
      return fail(MLAP_ERR_SHAPE, "rms_norm_quant_deq_scale must be (He) or (1)");
    if (!(a->rms_norm_quant_epsilon >= 0.0))
      return fail(MLAP_ERR_SHAPE, "rms_norm_quant_epsilon must be non-negative");
  }
  if (a->cache_mode != nullptr && std::strcmp(a->cache_mode, "PA_BSND") != 0)
    return fail(MLAP_ERR_UNSUPPORTED, std::string("cache_mode '") + a->cache_mode + "' not supported (PA_BSND only)");
  if (!(a->rmsnorm_epsilon_cq >= 0.0) || !(a->rmsnorm_epsilon_ckv >= 0.0))
    return fail(MLAP_ERR_SHAPE, "rmsnorm epsilons must be non-negative");
  if (d->T > (int64_t(1) << 30)) return fail(MLAP_ERR_UNSUPPORTED, "too many tokens");
  return MLAP_OK;
}

int swap_bn(int64_t T) {
  int bn = 16;
  while (bn < T) bn *= 2;
  return bn;
}

struct MlaWs {
  size_t part, cq, qc, scale, xb, qn, total;
  int split_cap;
};

MlaWs mla_ws_layout(const MlaDims& d) {
  MlaWs w;
  const bool swap = d.T <= kSwapMaxT;
  w.split_cap = d.T <= kSplitMaxT ? kMaxSplits : 1;
  const int64_t ntot = d.Hcq + d.Hckv + d.Dr;
  size_t off = kHeaderBytes;
  w.part = off;
  // the down-projection's K-split partials
  off += align_up(static_cast<size_t>(w.split_cap) * d.T * ntot * 4, 256);
  w.cq = off;
  off += align_up(static_cast<size_t>(d.T) * d.Hcq * 2, 256);
  w.qc = off;
  off += align_up(static_cast<size_t>(d.T) * d.N * d.D * 2, 256);
  w.scale = off;
  off += align_up(static_cast<size_t>(d.T) * 4, 256);
  w.xb = off;   // the down-projection's 16-bit operand when it is not token_x itself: token_x
                // widened (full quant outside the decode orientation) or after the input
                // RmsNormQuant
  if ((d.full && !swap) || d.xnorm) off += align_up(static_cast<size_t>(d.T) * d.He * 2, 256);
  w.qn = off;   // int8 query: q^N in bf16 before the per-token-head quant
  if (d.query_int8) off += align_up(static_cast<size_t>(d.T) * d.N * d.Hckv * 2, 256);
  w.total = off;
  return w;
}

// ----------------------------------------------------------------------------------------------
// TMA descriptors
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2D K-major bf16 operand: `rows` rows of `inner` elements, `pitch` elements apart; box of
// 64 elements x box_rows rows, 128-byte swizzle, zero fill outside the tensor.
mlap_status_t make_tmap(CUtensorMap* m, const void* base, int64_t inner, int64_t rows,
                        int64_t pitch_elems, int box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return fail(MLAP_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch_elems) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MLAP_ERR_CUDA, "cuTensorMapEncodeTiled failed (" + std::to_string(int(r)) + ")");
  return MLAP_OK;
}

// Output map for the epilogue's TMA stores: `rank` dims (innermost first), byte strides of dims
// 1.., box sizes, element type and swizzle matching the staging tile layout.
mlap_status_t make_out_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int rank,
                           std::initializer_list<int64_t> dims, std::initializer_list<int64_t> strides,
                           std::initializer_list<int> box, CUtensorMapSwizzle sw) {
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return fail(MLAP_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t d[3], st[2];
  cuuint32_t b[3], es[3] = {1, 1, 1};
  int i = 0;
  for (int64_t v : dims) d[i++] = static_cast<cuuint64_t>(v);
  i = 0;
  for (int64_t v : strides) st[i++] = static_cast<cuuint64_t>(v);
  i = 0;
  for (int v : box) b[i++] = static_cast<cuuint32_t>(v);
  CUresult r = enc(m, dt, rank, const_cast<void*>(base), d, st, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   sw, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MLAP_ERR_CUDA, "cuTensorMapEncodeTiled (output) failed (" + std::to_string(int(r)) + ")");
  return MLAP_OK;
}

// 2D int8 weight operand: `rows` rows of `inner` bytes; box of 64 bytes x box_rows rows, no
// swizzle (the converter warps write the bf16 swizzled layout), zero fill outside.
mlap_status_t make_tmap_i8(CUtensorMap* m, const void* base, int64_t inner, int64_t rows,
                           int box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return fail(MLAP_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner)};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MLAP_ERR_CUDA, "cuTensorMapEncodeTiled (int8) failed (" + std::to_string(int(r)) + ")");
  return MLAP_OK;
}

int ceil_div(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

// Token count from which the prefill-orientation bf16 GEMMs (down- and up-projection) run on CTA
// pairs with 256-row tiles of tokens.
constexpr int64_t kPairMinT = 1024;

// The decode-orientation activation operand, read by the GEMM's cp.async loader warps.
void set_act(GemmGeometry* g, const void* p, int64_t ld, int64_t rows, int64_t cols) {
  g->act = static_cast<const uint16_t*>(p);
  g->act_ld = ld;
  g->act_rows = static_cast<int32_t>(rows);
  g->act_cols = static_cast<int32_t>(cols);
}

// Persistent grid with equal work per CTA: the fewest CTAs that still finish the units in the
// minimum number of rounds (e.g. 192 units on 152 SMs -> 96 CTAs x 2 units instead of a second
// round that only 40 CTAs run).
int balanced_grid(int units, int sms) {
  if (units <= 0) return 1;
  const int rounds = ceil_div(units, sms);
  return ceil_div(units, rounds);
}



mlap_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(MLAP_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

mlap_status_t mla_run(const mlap_args_t* a, void* ws, size_t ws_bytes, cudaStream_t stream,
                      uint64_t* stamps) {
  MlaDims d;
  CHECK_STATUS(validate_mla(a, &d));
  if (d.T == 0) return MLAP_OK;
  const MlaWs L = mla_ws_layout(d);
  if (ws == nullptr || ws_bytes < L.total) return fail(MLAP_ERR_WORKSPACE, "workspace too small");
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return fail(MLAP_ERR_WORKSPACE, "workspace must be 256-byte aligned");

  int dev = 0, sms = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce == cudaSuccess) ce = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (ce != cudaSuccess) return cuda_fail(ce, "device query");

  uint8_t* wsb = static_cast<uint8_t*>(ws);
  uint32_t* err = reinterpret_cast<uint32_t*>(wsb);
  float* part = reinterpret_cast<float*>(wsb + L.part);
  __nv_bfloat16* cq = reinterpret_cast<__nv_bfloat16*>(wsb + L.cq);
  __nv_bfloat16* qc = reinterpret_cast<__nv_bfloat16*>(wsb + L.qc);
  float* scale_t = reinterpret_cast<float*>(wsb + L.scale);

  const bool swap = d.T <= kSwapMaxT;
  const int64_t Ntot = d.Hcq + d.Hckv + d.Dr;
  const int64_t Mup = d.N * (d.D + d.Dr);
  const int64_t slots = d.BlockNum * d.BlockSize;
  const int bn_t = swap_bn(d.T);
  // decode orientation: units of 256 weight rows (two accumulators) when they fit in TMEM
  const int mt = 1;                          // two-tile units pay off only with all SMs busy
  const int wrows = 128 * mt;

  // ---- 1. down-projection x·[W^DQ | W^DKV|W^KR]  (fp32 K-split partials)
  GemmLaunch g{};
  g.stream = stream;
  g.pdl = true;
  g.err = err;
  g.geo.stamps = stamps;
  g.geo.stamp_k = MLAP_STAMP_DOWN;
  // token_x itself is the activation (not normalised by a kernel of this call, and not widened:
  // in the decode orientation the converter warps expand full quant's int8 token_x tiles): the
  // down-projection streams before the preceding kernel finishes and waits only to store
  const bool widen = d.full && !swap;
  g.geo.act_ready = !(widen || d.xnorm);
  g.swap = swap;
  g.mt = swap ? mt : 1;
  DownParams dp{0};
  const int ch_t = swap ? (bn_t < 32 ? bn_t : 32) : 32;   // tokens per epilogue store box
  // full quant: the int8 weights (and, in the decode orientation, the int8 token_x tiles) are
  // expanded to f16 in shared memory by the GEMM's converter warps (exact); otherwise token_x is
  // widened to f16 by a kernel first.  The integer products are dequantised per token and
  // column after the K-split sum (norm kernel).
  const void* xact = widen || d.xnorm ? static_cast<const void*>(wsb + L.xb) : a->token_x.data;
  g.a_int8 = d.full;
  auto wmap = [&](CUtensorMap* m, const void* w, int64_t rows, int box) {
    return d.full ? make_tmap_i8(m, w, d.He, rows, box) : make_tmap(m, w, d.He, rows, d.He, box);
  };
  {
    const int kb = ceil_div(d.He, 64);
    if (swap) {
      const int seg = ceil_div(d.Hcq, wrows);
      CHECK_STATUS(wmap(&g.a0, a->weight_dq.data, d.Hcq, wrows));
      CHECK_STATUS(wmap(&g.a1, a->weight_dkv_kr.data, d.Hckv + d.Dr, wrows));
      if (d.full)
        CHECK_STATUS(make_tmap_i8(&g.b0, a->token_x.data, d.He, d.T, bn_t));
      else
        CHECK_STATUS(make_tmap(&g.b0, xact, d.He, d.T, d.He, bn_t));
      g.b1 = g.b0;
      g.bn = bn_t;
      g.geo.m_tiles = seg + ceil_div(d.Hckv + d.Dr, wrows);
      g.geo.n_tiles = 1;
      g.geo.a_seg_tiles = seg;
      g.geo.b_seg_tiles = 1;
      set_act(&g.geo, xact, d.He, d.T, d.He);
      int splits = sms / g.geo.m_tiles;
      if (splits > L.split_cap) splits = L.split_cap;
      if (splits > kb) splits = kb;
      if (splits < 1) splits = 1;
      g.geo.splits = splits;
      dp.seg_tiles = seg;
    } else {
      // N = 256 keeps the tensor pipe fed (N = 192 reached 0.68 of the sustained peak at
      // T = 8192); the int8 weights of full quant keep 192-row tiles for their converter warps.
      // Many tokens: CTA pairs, each CTA staging 128 tokens and half of a 256-row weight tile.
      const int bnd = d.full ? 192 : 256;
      const int seg = ceil_div(d.Hcq, bnd);
      g.cg = !d.full && d.T >= kPairMinT ? 2 : 1;
      CHECK_STATUS(make_tmap(&g.a0, xact, d.He, d.T, d.He, 128));
      g.a1 = g.a0;
      CHECK_STATUS(wmap(&g.b0, a->weight_dq.data, d.Hcq, bnd / g.cg));
      CHECK_STATUS(wmap(&g.b1, a->weight_dkv_kr.data, d.Hckv + d.Dr, bnd / g.cg));
      g.bn = bnd;
      g.geo.m_tiles = ceil_div(d.T, 128 * g.cg);
      g.geo.n_tiles = seg + ceil_div(d.Hckv + d.Dr, bnd);
      g.geo.a_seg_tiles = g.geo.m_tiles;
      g.geo.b_seg_tiles = seg;
      g.geo.n_fast = 1;   // each x tile (128 x He) is used by every weight tile while in L2
      int splits = sms / (g.geo.m_tiles * g.geo.n_tiles);
      if (splits > L.split_cap) splits = L.split_cap;
      if (splits > kb) splits = kb;
      if (splits < 1) splits = 1;
      g.geo.splits = splits;
      dp.seg_tiles = seg;
    }
    g.geo.batches = 1;
    g.geo.k_blocks = kb;
    g.geo.w_op = swap ? 0 : 1;
    g.geo.num_units = g.geo.m_tiles * g.geo.n_tiles * g.geo.splits;
    // partials part[s][t][f]: W^DQ columns and W^DKV|W^KR columns as two 3-D (f, t, s) maps
    const int64_t row_b = Ntot * 4, split_b = d.T * Ntot * 4;
    CHECK_STATUS(make_out_map(&g.o0, part, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                              {d.Hcq, d.T, g.geo.splits}, {row_b, split_b}, {32, ch_t, 1},
                              CU_TENSOR_MAP_SWIZZLE_128B));
    CHECK_STATUS(make_out_map(&g.o1, part + d.Hcq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                              {d.Hckv + d.Dr, d.T, g.geo.splits}, {row_b, split_b}, {32, ch_t, 1},
                              CU_TENSOR_MAP_SWIZZLE_128B));
    g.grid = g.cg == 2 ? 2 * balanced_grid(g.geo.num_units, sms / 2)
                       : balanced_grid(g.geo.num_units, sms);
    if (d.xnorm) {
      ce = launch_rms_norm_quant(static_cast<const __nv_bfloat16*>(a->token_x.data),
                                 static_cast<const __nv_bfloat16*>(a->rms_norm_quant_gamma.data),
                                 static_cast<const __nv_bfloat16*>(a->rms_norm_quant_bias.data),
                                 static_cast<const float*>(a->rms_norm_quant_deq_scale.data),
                                 d.xnorm_deq_per_channel,
                                 static_cast<float>(a->rms_norm_quant_epsilon),
                                 reinterpret_cast<__nv_bfloat16*>(wsb + L.xb), d.T,
                                 static_cast<int32_t>(d.He), stream);
      if (ce != cudaSuccess) return cuda_fail(ce, "input RmsNormQuant launch");
    }
    if (widen) {
      ce = launch_widen_int8(static_cast<const int8_t*>(a->token_x.data),
                             reinterpret_cast<__half*>(wsb + L.xb), d.T * d.He, stream);
      if (ce != cudaSuccess) return cuda_fail(ce, "token_x widening launch");
    }
    ce = launch_down(g, dp);
    if (ce != cudaSuccess) return cuda_fail(ce, "down-projection launch");
  }

  // ---- 2. RmsNorm(c^Q), RmsNorm(c^KV), RoPE(k^R), cache quant + scatter
  {
    FinalizeParams fp{};
    fp.part = part;
    fp.splits = g.geo.splits;
    fp.T = static_cast<int32_t>(d.T);
    fp.Hcq = static_cast<int32_t>(d.Hcq);
    fp.Hckv = static_cast<int32_t>(d.Hckv);
    fp.Dr = static_cast<int32_t>(d.Dr);
    fp.Ntot = static_cast<int32_t>(Ntot);
    fp.gamma_cq = static_cast<const __nv_bfloat16*>(a->rmsnorm_gamma_cq.data);
    fp.gamma_ckv = static_cast<const __nv_bfloat16*>(a->rmsnorm_gamma_ckv.data);
    fp.eps_cq = static_cast<float>(a->rmsnorm_epsilon_cq);
    fp.eps_ckv = static_cast<float>(a->rmsnorm_epsilon_ckv);
    fp.cos = static_cast<const __nv_bfloat16*>(a->rope_cos.data);
    fp.sin = static_cast<const __nv_bfloat16*>(a->rope_sin.data);
    fp.cache_index = static_cast<const int64_t*>(a->cache_index.data);
    fp.slots = slots;
    fp.kv_cache = a->kv_cache.data;
    fp.kr_cache = a->kr_cache.data;
    fp.kv_int8 = d.kv_int8;
    fp.kr_int8 = d.kr_int8;
    fp.qs_ckv = static_cast<const float*>(a->quant_scale_ckv.data);
    fp.qs_ckr = static_cast<const float*>(a->quant_scale_ckr.data);
    fp.cq_out = cq;
    fp.smooth = d.w_int8 ? static_cast<const float*>(a->smooth_scales_cq.data) : nullptr;
    fp.scale_t = scale_t;
    fp.err = err;
    fp.stamps = stamps;
    if (d.full) {
      fp.dsx = static_cast<const float*>(a->dequant_scale_x.data);
      fp.dsw_q = static_cast<const float*>(a->dequant_scale_w_dq.data);
      fp.dsw_kv = static_cast<const float*>(a->dequant_scale_w_dkv_kr.data);
    }
    ce = launch_finalize(fp, stream, true);
    if (ce != cudaSuccess) return cuda_fail(ce, "norm/rope/scatter launch");
  }

  // ---- 3+4 fused at decode: one CTA per head runs the up-projection, keeps q^C in shared
  // memory and multiplies it by the head's W^UK (up_absorb.cu)
  const bool fused = swap && d.N >= kFusedMinHeads &&
                     up_absorb_supported(d.T, d.N, d.D, d.Dr, d.Hckv);
  if (fused) {
    CUtensorMap tcq, tw, tw128, tuk, tuk128;   // (the wide maps serve int8 weights only: a head
                                               // CTA's W^UQ rows, 128 or 64 in a pair, and
                                               // 128 W^UK rows per box)
    // c^Q tiles of the token rows only (the MMA's other A rows feed accumulator lanes that are
    // never stored)
    const int cq_rows = d.T < 128 ? static_cast<int>((d.T + 7) / 8 * 8) : 128;
    CHECK_STATUS(make_tmap(&tcq, cq, d.Hcq, d.T, d.Hcq, cq_rows));
    int ua_k = 0, ua_r = 0, ua_pair = 0;
    up_absorb_plan(sms, static_cast<int>(d.N), &ua_k, &ua_r, &ua_pair);
    if (d.w_int8) {
      CHECK_STATUS(make_tmap_i8(&tw, a->weight_uq_qr.data, d.Hcq, Mup, 32));
      CHECK_STATUS(make_tmap_i8(&tw128, a->weight_uq_qr.data, d.Hcq, Mup, ua_pair ? 64 : 128));
      CHECK_STATUS(make_tmap(&tuk128, a->weight_uk.data, d.D, d.N * d.Hckv, d.D, 128));
    } else {
      CHECK_STATUS(make_tmap(&tw, a->weight_uq_qr.data, d.Hcq, Mup, d.Hcq, 32));
    }
    CHECK_STATUS(make_tmap(&tuk, a->weight_uk.data, d.D, d.N * d.Hckv, d.D, 32));
    // an int8 query is quantised per token and head from a bf16 q^N staged in the workspace
    __nv_bfloat16* qn_out = d.query_int8 ? reinterpret_cast<__nv_bfloat16*>(wsb + L.qn)
                                         : static_cast<__nv_bfloat16*>(a->query.data);
    UpAbsorbParams ua{static_cast<const __nv_bfloat16*>(a->rope_cos.data),
                      static_cast<const __nv_bfloat16*>(a->rope_sin.data),
                      static_cast<__nv_bfloat16*>(a->query_rope.data),
                      qn_out,
                      static_cast<int32_t>(d.T), static_cast<int32_t>(d.N),
                      static_cast<int32_t>(d.Hcq), static_cast<int32_t>(d.Hckv),
                      scale_t, static_cast<const float*>(a->dequant_scale_w_uq_qr.data), 2, 0,
                      stamps};
    ua.k = ua_k;
    ua.R = ua_r;
    ua.pair = ua_pair;
    ua.cq_rows = cq_rows;
    ce = launch_up_absorb(tcq, tw, tuk, d.w_int8 ? &tw128 : nullptr, d.w_int8 ? &tuk128 : nullptr,
                          ua, err, stream);
    if (ce != cudaSuccess) return cuda_fail(ce, "fused up-projection/absorb launch");
    if (d.query_int8) {
      ce = launch_query_quant(qn_out, static_cast<int8_t*>(a->query.data),
                              static_cast<float*>(a->dequant_scale_q_nope.data), d.T * d.N,
                              static_cast<int32_t>(d.Hckv), stream);
      if (ce != cudaSuccess) return cuda_fail(ce, "query quant launch");
    }
  }

  // ---- 3. up-projection c^Q·[W^UQ|W^QR] -> q^C (bf16 workspace) and query_rope
  if (!fused) {
    GemmLaunch u{};
    u.stream = stream;
    u.pdl = true;
    u.err = err;
    u.geo.stamps = stamps;
    u.geo.stamp_k = MLAP_STAMP_UP;
    // Decode with a bf16 weight and one 128-token tile: tokens as MMA rows and an equal range
    // of weight rows per SM (row-range schedule: 24576 rows on 152 SMs, 160 or 192 each).
    const bool up_var = swap && !d.w_int8 && d.T <= 128 && Mup % 32 == 0;
    u.swap = swap && !up_var;
    u.mt = u.swap ? mt : 1;
    if (up_var) {
      CHECK_STATUS(make_tmap(&u.a0, cq, d.Hcq, d.T, d.Hcq, 128));
      u.a1 = u.a0;
      CHECK_STATUS(make_tmap(&u.b0, a->weight_uq_qr.data, d.Hcq, Mup, d.Hcq, 32));
      u.b1 = u.b0;
      u.bn = 256;
      u.geo.m_tiles = 1;
      u.geo.n_tiles = 1;
      u.rr = true;
      u.geo.rr_rows = static_cast<int32_t>(Mup);
    } else if (swap) {
      if (d.w_int8)
        CHECK_STATUS(make_tmap_i8(&u.a0, a->weight_uq_qr.data, d.Hcq, Mup, wrows));
      else
        CHECK_STATUS(make_tmap(&u.a0, a->weight_uq_qr.data, d.Hcq, Mup, d.Hcq, wrows));
      u.a1 = u.a0;
      CHECK_STATUS(make_tmap(&u.b0, cq, d.Hcq, d.T, d.Hcq, bn_t));
      u.b1 = u.b0;
      set_act(&u.geo, cq, d.Hcq, d.T, d.Hcq);
      u.bn = bn_t;
      u.geo.m_tiles = ceil_div(Mup, wrows);
      u.geo.n_tiles = 1;
    } else {
      // many tokens, bf16 weight: CTA pairs (each CTA stages 128 tokens and 128 weight rows)
      u.cg = !d.w_int8 && d.T >= kPairMinT ? 2 : 1;
      CHECK_STATUS(make_tmap(&u.a0, cq, d.Hcq, d.T, d.Hcq, 128));
      u.a1 = u.a0;
      if (d.w_int8)
        CHECK_STATUS(make_tmap_i8(&u.b0, a->weight_uq_qr.data, d.Hcq, Mup, 256));
      else
        CHECK_STATUS(make_tmap(&u.b0, a->weight_uq_qr.data, d.Hcq, Mup, d.Hcq, 256 / u.cg));
      u.b1 = u.b0;
      u.bn = 256;
      u.geo.m_tiles = ceil_div(d.T, 128 * u.cg);
      u.geo.n_tiles = ceil_div(Mup, 256);
    }
    u.geo.a_seg_tiles = u.geo.m_tiles;
    u.geo.b_seg_tiles = u.geo.n_tiles;
    u.geo.batches = 1;
    u.geo.splits = 1;
    u.geo.w_op = u.swap ? 0 : 1;
    u.geo.k_blocks = ceil_div(d.Hcq, 64);
    u.geo.num_units = u.geo.m_tiles * u.geo.n_tiles;
    u.grid = up_var ? static_cast<int>(std::min<int64_t>(sms, Mup / 32))
             : u.cg == 2 ? 2 * balanced_grid(u.geo.num_units, sms / 2)
                         : balanced_grid(u.geo.num_units, sms);
    const int ch_u = u.swap ? ch_t : 32;   // tokens per store box: one per lane unless swapped
    CHECK_STATUS(make_out_map(&u.o0, qc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, {d.N * d.D, d.T},
                              {d.N * d.D * 2}, {32, ch_u}, CU_TENSOR_MAP_SWIZZLE_64B));
    CHECK_STATUS(make_out_map(&u.o1, a->query_rope.data, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                              {d.Dr, d.N, d.T}, {d.Dr * 2, d.N * d.Dr * 2}, {16, 1, ch_u},
                              CU_TENSOR_MAP_SWIZZLE_32B));
    UpParams up{static_cast<const __nv_bfloat16*>(a->rope_cos.data),
                static_cast<const __nv_bfloat16*>(a->rope_sin.data),
                scale_t,
                static_cast<const float*>(a->dequant_scale_w_uq_qr.data),
                static_cast<int32_t>(d.T), static_cast<int32_t>(d.N), static_cast<int32_t>(d.D),
                static_cast<int32_t>(d.Dr),
                up_var ? qc : nullptr,
                up_var ? static_cast<__nv_bfloat16*>(a->query_rope.data) : nullptr};
    ce = launch_up(u, up, d.w_int8);
    if (ce != cudaSuccess) return cuda_fail(ce, "up-projection launch");
  }

  // ---- 4. absorb q^N = q^C · W^UK per head -> query
  if (!fused) {
    GemmLaunch b{};
    b.stream = stream;
    b.pdl = true;
    b.err = err;
    b.geo.stamps = stamps;
    b.geo.stamp_k = MLAP_STAMP_ABSORB;
    // Decode with one 128-token tile: tokens as MMA rows and the row-range schedule over all
    // heads' W^UK rows (128 x 512 rows on 152 SMs: 416 or 448 each, cut at head boundaries).
    const bool ab_var = swap && d.T <= 128 && d.Hckv % 32 == 0;
    b.swap = swap && !ab_var;
    b.mt = b.swap ? mt : 1;
    if (ab_var) {
      CHECK_STATUS(make_tmap(&b.a0, qc, d.N * d.D, d.T, d.N * d.D, 128));
      b.a1 = b.a0;
      CHECK_STATUS(make_tmap(&b.b0, a->weight_uk.data, d.D, d.N * d.Hckv, d.D, 32));
      b.b1 = b.b0;
      b.bn = 256;
      b.geo.m_tiles = 1;
      b.geo.n_tiles = 1;
      b.geo.a_x_batch = static_cast<int32_t>(d.D);
      b.geo.a_y_batch = 0;
      b.geo.b_x_batch = 0;
      b.geo.b_y_batch = static_cast<int32_t>(d.Hckv);
      b.rr = true;
      b.geo.rr_rows = static_cast<int32_t>(d.Hckv);
    } else if (swap) {
      CHECK_STATUS(make_tmap(&b.a0, a->weight_uk.data, d.D, d.N * d.Hckv, d.D, wrows));
      b.a1 = b.a0;
      CHECK_STATUS(make_tmap(&b.b0, qc, d.N * d.D, d.T, d.N * d.D, bn_t));
      b.b1 = b.b0;
      set_act(&b.geo, qc, d.N * d.D, d.T, d.N * d.D);
      b.bn = bn_t;
      b.geo.m_tiles = ceil_div(d.Hckv, wrows);
      b.geo.n_tiles = 1;
      b.geo.a_x_batch = 0;
      b.geo.a_y_batch = static_cast<int32_t>(d.Hckv);
      b.geo.b_x_batch = static_cast<int32_t>(d.D);
      b.geo.b_y_batch = 0;
    } else {
      CHECK_STATUS(make_tmap(&b.a0, qc, d.N * d.D, d.T, d.N * d.D, 128));
      b.a1 = b.a0;
      CHECK_STATUS(make_tmap(&b.b0, a->weight_uk.data, d.D, d.N * d.Hckv, d.D, 256));
      b.b1 = b.b0;
      b.bn = 256;
      b.geo.m_tiles = ceil_div(d.T, 128);
      b.geo.n_tiles = ceil_div(d.Hckv, 256);
      b.geo.a_x_batch = static_cast<int32_t>(d.D);
      b.geo.a_y_batch = 0;
      b.geo.b_x_batch = 0;
      b.geo.b_y_batch = static_cast<int32_t>(d.Hckv);
    }
    b.geo.a_seg_tiles = b.geo.m_tiles;
    b.geo.b_seg_tiles = b.geo.n_tiles;
    b.geo.batches = static_cast<int32_t>(d.N);
    // tokens as rows: the two W^UK column tiles of a q^C tile run side by side, so the second
    // read of each q^C tile hits in L2
    if (!b.swap && !ab_var) b.geo.n_fast = 1;
    b.geo.splits = 1;
    b.geo.w_op = b.swap ? 0 : 1;
    b.geo.k_blocks = ceil_div(d.D, 64);
    b.geo.num_units = b.geo.m_tiles * b.geo.n_tiles * b.geo.batches;
    b.grid = ab_var ? static_cast<int>(std::min<int64_t>(sms, d.N * d.Hckv / 32))
                    : balanced_grid(b.geo.num_units, sms);
    // an int8 query is quantised per token and head from a bf16 q^N staged in the workspace
    __nv_bfloat16* qn_out = d.query_int8 ? reinterpret_cast<__nv_bfloat16*>(wsb + L.qn)
                                         : static_cast<__nv_bfloat16*>(a->query.data);
    // boxes of 32 tokens x 32 columns, or (tokens as rows, TMA stores) 32 x 64: whole lines
    const bool wide = !b.swap && !ab_var;
    CHECK_STATUS(make_out_map(&b.o0, qn_out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                              {d.Hckv, d.N, d.T}, {d.Hckv * 2, d.N * d.Hckv * 2},
                              {wide ? 64 : 32, 1, b.swap ? ch_t : 32},
                              wide ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B));
    b.o1 = b.o0;
    AbsorbParams ap{ab_var ? qn_out : nullptr,
                    static_cast<int32_t>(d.T), static_cast<int32_t>(d.N),
                    static_cast<int32_t>(d.Hckv)};
    ce = launch_absorb(b, ap);
    if (ce != cudaSuccess) return cuda_fail(ce, "absorb launch");
    if (d.query_int8) {
      ce = launch_query_quant(qn_out, static_cast<int8_t*>(a->query.data),
                              static_cast<float*>(a->dequant_scale_q_nope.data), d.T * d.N,
                              static_cast<int32_t>(d.Hckv), stream);
      if (ce != cudaSuccess) return cuda_fail(ce, "query quant launch");
    }
  }
  return MLAP_OK;
}

// ----------------------------------------------------------------------------------------------
// QkvRmsNormRopeCache
struct QkvDims {
  int64_t T, B, S;
  bool bsh;
  int64_t D, BlockNum, BlockSize;
  bool quant, asym, bf16;
};

mlap_status_t validate_qkv(const qkvrnrc_args_t* a, QkvDims* d) {
  if (a == nullptr) return fail(MLAP_ERR_NULL, "args is NULL");
  const int64_t Nq = a->Nq, Nk = a->Nk, Nv = a->Nv;
  if (Nq <= 0 || Nk <= 0 || Nv <= 0) return fail(MLAP_ERR_SHAPE, "Nq, Nk, Nv must be positive");
  if (Nk != Nv) return fail(MLAP_ERR_SHAPE, "SplitVD requires Nk == Nv");
  const mlap_tensor_t& x = a->qkv;
  int64_t width;
  if (x.ndim == 2) {
    d->bsh = false; d->T = x.shape[0]; d->B = x.shape[0]; d->S = 1; width = x.shape[1];
  } else if (x.ndim == 3) {
    d->bsh = true; d->B = x.shape[0]; d->S = x.shape[1]; d->T = d->B * d->S; width = x.shape[2];
  } else {
    return fail(MLAP_ERR_SHAPE, "qkv must be (T, Nqkv*D) or (B, S, Nqkv*D)");
  }
  CHECK_STATUS(need(x, "qkv", true));
  if (x.dtype == MLAP_DTYPE_FP16) d->bf16 = false;
  else if (x.dtype == MLAP_DTYPE_BF16) d->bf16 = true;
  else return fail(MLAP_ERR_DTYPE, "qkv must be fp16 or bf16");
  if (width % (Nq + Nk + Nv)) return fail(MLAP_ERR_SHAPE, "qkv width is not a multiple of Nq+Nk+Nv");
  d->D = width / (Nq + Nk + Nv);
  if (d->D != 128) return fail(MLAP_ERR_UNSUPPORTED, "head dim D must be 128");
  for (auto* pr : {&a->gamma_q, &a->gamma_k}) {
    CHECK_STATUS(need(*pr, "gamma", false));
    CHECK_STATUS(want_dtype(*pr, "gamma", x.dtype));
    CHECK_STATUS(want_shape(*pr, "gamma", {d->D}));
  }
  for (auto* pr : {&a->cos, &a->sin}) {
    CHECK_STATUS(need(*pr, "cos/sin", true));
    CHECK_STATUS(want_dtype(*pr, "cos/sin", x.dtype));
    if (d->bsh) CHECK_STATUS(want_shape(*pr, "cos/sin", {d->B, d->S, d->D}));
    else CHECK_STATUS(want_shape(*pr, "cos/sin", {d->T, d->D}));
  }
  CHECK_STATUS(need(a->index, "index", true));
  CHECK_STATUS(want_dtype(a->index, "index", MLAP_DTYPE_INT64));
  if (d->bsh) CHECK_STATUS(want_shape(a->index, "index", {d->B, d->S}));
  else CHECK_STATUS(want_shape(a->index, "index", {d->T}));
  CHECK_STATUS(need(a->q_out, "q_out", true));
  CHECK_STATUS(want_dtype(a->q_out, "q_out", x.dtype));
  if (d->bsh) CHECK_STATUS(want_shape(a->q_out, "q_out", {d->B, d->S, Nq, d->D}));
  else CHECK_STATUS(want_shape(a->q_out, "q_out", {d->T, Nq, d->D}));
  const mlap_tensor_t& kc = a->k_cache;
  const mlap_tensor_t& vc = a->v_cache;
  if (kc.ndim != 4 || vc.ndim != 4) return fail(MLAP_ERR_SHAPE, "caches must be (BlockNum, BlockSize, N, D)");
  d->BlockNum = kc.shape[0];
  d->BlockSize = kc.shape[1];
  CHECK_STATUS(need(kc, "k_cache", true));
  CHECK_STATUS(need(vc, "v_cache", true));
  CHECK_STATUS(want_shape(kc, "k_cache", {d->BlockNum, d->BlockSize, Nk, d->D}));
  CHECK_STATUS(want_shape(vc, "v_cache", {d->BlockNum, d->BlockSize, Nv, d->D}));
  if (kc.dtype != vc.dtype) return fail(MLAP_ERR_DTYPE, "k_cache and v_cache dtypes differ");
  d->quant = present(a->k_scale) || present(a->v_scale);
  d->asym = present(a->k_offset) || present(a->v_offset);
  if (d->asym) {
    if (!d->quant) return fail(MLAP_ERR_UNSUPPORTED, "k_offset / v_offset need k_scale / v_scale");
    CHECK_STATUS(need(a->k_offset, "k_offset", false));
    CHECK_STATUS(need(a->v_offset, "v_offset", false));
    CHECK_STATUS(want_dtype(a->k_offset, "k_offset", MLAP_DTYPE_FP32));
    CHECK_STATUS(want_dtype(a->v_offset, "v_offset", MLAP_DTYPE_FP32));
    CHECK_STATUS(want_shape(a->k_offset, "k_offset", {Nk, d->D}));
    CHECK_STATUS(want_shape(a->v_offset, "v_offset", {Nv, d->D}));
  }
  {   // optional before-quant outputs
    const mlap_tensor_t* outs[3] = {&a->q_before_quant, &a->k_before_quant, &a->v_before_quant};
    const char* names[3] = {"q_before_quant", "k_before_quant", "v_before_quant"};
    const int64_t heads[3] = {Nq, Nk, Nv};
    for (int i = 0; i < 3; ++i) {
      if (!present(*outs[i])) continue;
      CHECK_STATUS(need(*outs[i], names[i], true));
      CHECK_STATUS(want_dtype(*outs[i], names[i], x.dtype));
      if (d->bsh) CHECK_STATUS(want_shape(*outs[i], names[i], {d->B, d->S, heads[i], d->D}));
      else CHECK_STATUS(want_shape(*outs[i], names[i], {d->T, heads[i], d->D}));
    }
  }
  if (d->quant) {
    CHECK_STATUS(want_dtype(kc, "k_cache", MLAP_DTYPE_INT8));
    CHECK_STATUS(need(a->k_scale, "k_scale", false));
    CHECK_STATUS(need(a->v_scale, "v_scale", false));
    CHECK_STATUS(want_dtype(a->k_scale, "k_scale", MLAP_DTYPE_FP32));
    CHECK_STATUS(want_dtype(a->v_scale, "v_scale", MLAP_DTYPE_FP32));
    CHECK_STATUS(want_shape(a->k_scale, "k_scale", {Nk, d->D}));
    CHECK_STATUS(want_shape(a->v_scale, "v_scale", {Nv, d->D}));
  } else {
    CHECK_STATUS(want_dtype(kc, "k_cache", x.dtype));
  }
  if (a->cache_mode != nullptr && std::strcmp(a->cache_mode, "PA_BSND") != 0)
    return fail(MLAP_ERR_UNSUPPORTED, std::string("cache_mode '") + a->cache_mode + "' not supported (PA_BSND only)");
  if (d->bsh && d->BlockSize > 0 && d->T > 0 &&
      d->BlockNum < (d->S + d->BlockSize - 1) / d->BlockSize * d->B)
    return fail(MLAP_ERR_SHAPE, "BlockNum must be >= ceil(S / BlockSize) * B");
  if (!(a->epsilon >= 0.0)) return fail(MLAP_ERR_SHAPE, "epsilon must be non-negative");
  return MLAP_OK;
}

mlap_status_t qkv_run(const qkvrnrc_args_t* a, void* ws, size_t ws_bytes, cudaStream_t stream,
                      uint64_t* stamps) {
  QkvDims d;
  CHECK_STATUS(validate_qkv(a, &d));
  if (d.T == 0) return MLAP_OK;
  if (ws == nullptr || ws_bytes < 256) return fail(MLAP_ERR_WORKSPACE, "workspace too small");
  int dev = 0, sms = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce == cudaSuccess) ce = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (ce != cudaSuccess) return cuda_fail(ce, "device query");
  QkvParams p{};
  p.qkv = a->qkv.data;
  p.gamma_q = a->gamma_q.data;
  p.gamma_k = a->gamma_k.data;
  p.cos = a->cos.data;
  p.sin = a->sin.data;
  p.index = static_cast<const int64_t*>(a->index.data);
  p.slots = d.BlockNum * d.BlockSize;
  p.k_cache = a->k_cache.data;
  p.v_cache = a->v_cache.data;
  p.k_scale = d.quant ? static_cast<const float*>(a->k_scale.data) : nullptr;
  p.v_scale = d.quant ? static_cast<const float*>(a->v_scale.data) : nullptr;
  p.k_offset = d.asym ? static_cast<const float*>(a->k_offset.data) : nullptr;
  p.v_offset = d.asym ? static_cast<const float*>(a->v_offset.data) : nullptr;
  p.q_before = present(a->q_before_quant) ? a->q_before_quant.data : nullptr;
  p.k_before = present(a->k_before_quant) ? a->k_before_quant.data : nullptr;
  p.v_before = present(a->v_before_quant) ? a->v_before_quant.data : nullptr;
  p.q_out = a->q_out.data;
  p.T = static_cast<int32_t>(d.T);
  p.Nq = a->Nq;
  p.Nk = a->Nk;
  p.Nv = a->Nv;
  p.eps = static_cast<float>(a->epsilon);
  p.bf16 = d.bf16;
  p.err = static_cast<uint32_t*>(ws);
  p.stamps = stamps;
  ce = launch_qkv_rnrc(p, stream, sms);
  if (ce != cudaSuccess) return cuda_fail(ce, "QkvRmsNormRopeCache launch");
  return MLAP_OK;
}

}  // namespace

// ================================================================================================
extern "C" {

const char* mlap_status_string(mlap_status_t s) {
  switch (s) {
    case MLAP_OK: return "MLAP_OK";
    case MLAP_ERR_NULL: return "MLAP_ERR_NULL";
    case MLAP_ERR_SHAPE: return "MLAP_ERR_SHAPE";
    case MLAP_ERR_DTYPE: return "MLAP_ERR_DTYPE";
    case MLAP_ERR_UNSUPPORTED: return "MLAP_ERR_UNSUPPORTED";
    case MLAP_ERR_WORKSPACE: return "MLAP_ERR_WORKSPACE";
    case MLAP_ERR_CUDA: return "MLAP_ERR_CUDA";
    case MLAP_ERR_INDEX_RANGE: return "MLAP_ERR_INDEX_RANGE";
    case MLAP_ERR_TIMEOUT: return "MLAP_ERR_TIMEOUT";
    default: return "MLAP_ERR_UNKNOWN";
  }
}

const char* mlap_last_error(void) { return g_last_error.c_str(); }

mlap_status_t mlap_prepack_size(const mlap_tensor_t* w, int32_t which, int32_t N, int32_t D,
                                int32_t Dr, size_t* bytes) {
  if (w == nullptr || bytes == nullptr) return fail(MLAP_ERR_NULL, "NULL argument");
  const size_t eb = dtype_bytes(w->dtype);
  switch (which) {
    case MLAP_WEIGHT_DQ:
    case MLAP_WEIGHT_DKV_KR:
      if (w->dtype != MLAP_DTYPE_BF16 && w->dtype != MLAP_DTYPE_INT8)
        return fail(MLAP_ERR_DTYPE, "weight must be bf16 or int8 (full quant)");
      if (w->ndim != 2) return fail(MLAP_ERR_SHAPE, "weight must be 2-D (k, n)");
      break;
    case MLAP_WEIGHT_UQ_QR:
      if (w->dtype != MLAP_DTYPE_BF16 && w->dtype != MLAP_DTYPE_INT8)
        return fail(MLAP_ERR_DTYPE, "weight_uq_qr must be bf16 or int8");
      if (w->ndim != 2 || N <= 0 || D <= 0 || Dr <= 0 || (Dr & 1) ||
          w->shape[1] != int64_t(N) * (D + Dr))
        return fail(MLAP_ERR_SHAPE, "weight_uq_qr must be (Hcq, N*(D+Dr)) with even Dr");
      break;
    case MLAP_WEIGHT_UK:
      if (w->dtype != MLAP_DTYPE_BF16) return fail(MLAP_ERR_DTYPE, "weight_uk must be bf16");
      if (w->ndim != 3) return fail(MLAP_ERR_SHAPE, "weight_uk must be (N, D, Hckv)");
      break;
    default:
      return fail(MLAP_ERR_UNSUPPORTED, "unknown weight id");
  }
  for (int i = 0; i < w->ndim; ++i)
    if (w->shape[i] <= 0) return fail(MLAP_ERR_SHAPE, "weight dimensions must be positive");
  *bytes = static_cast<size_t>(numel(*w)) * eb;
  return MLAP_OK;
}

mlap_status_t mlap_prepack_weights(const mlap_tensor_t* w, int32_t which, int32_t N, int32_t D,
                                   int32_t Dr, void* dst, void* stream) {
  size_t bytes = 0;
  CHECK_STATUS(mlap_prepack_size(w, which, N, D, Dr, &bytes));
  if (w->data == nullptr || dst == nullptr) return fail(MLAP_ERR_NULL, "NULL weight or destination");
  PrepackParams p{};
  p.src = w->data;
  p.dst = dst;
  p.elem_bytes = static_cast<int32_t>(dtype_bytes(w->dtype));
  p.perm = kPermIdentity;
  p.N = N;
  p.D = D;
  p.Dr = Dr;
  if (which == MLAP_WEIGHT_UK) {
    p.batches = static_cast<int32_t>(w->shape[0]);
    p.K = static_cast<int32_t>(w->shape[1]);
    p.C = static_cast<int32_t>(w->shape[2]);
    p.R = p.C;
  } else {
    p.batches = 1;
    p.K = static_cast<int32_t>(w->shape[0]);
    p.C = static_cast<int32_t>(w->shape[1]);
    p.R = p.C;
    if (which == MLAP_WEIGHT_UQ_QR) p.perm = kPermUqQr;
  }
  cudaError_t e = launch_prepack(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "prepack launch");
  return MLAP_OK;
}

mlap_status_t mlap_get_workspace_size(const mlap_args_t* args, size_t* bytes) {
  if (bytes == nullptr) return fail(MLAP_ERR_NULL, "bytes is NULL");
  MlaDims d;
  CHECK_STATUS(validate_mla(args, &d));
  *bytes = mla_ws_layout(d).total;
  return MLAP_OK;
}

mlap_status_t mlap_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (ws == nullptr) return fail(MLAP_ERR_NULL, "workspace is NULL");
  if (ws_bytes < 256) return fail(MLAP_ERR_WORKSPACE, "workspace smaller than its 256-byte header");
  cudaError_t e = cudaMemsetAsync(ws, 0, kHeaderBytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  return MLAP_OK;
}

mlap_status_t mlap_execute(const mlap_args_t* args, void* ws, size_t ws_bytes, void* stream) {
  return mla_run(args, ws, ws_bytes, static_cast<cudaStream_t>(stream), nullptr);
}

mlap_status_t mlap_check_errors(void* ws, void* stream) {
  if (ws == nullptr) return fail(MLAP_ERR_NULL, "workspace is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws, 0, sizeof(word), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the error word");
  if (word & kErrIndexRange) return fail(MLAP_ERR_INDEX_RANGE, "a cache index was outside [-1, BlockNum*BlockSize)");
  if (word & kErrTimeout) return fail(MLAP_ERR_TIMEOUT, "a kernel wait timed out");
  return MLAP_OK;
}

mlap_status_t mlap_selftest_bounded_wait(void* ws, size_t ws_bytes, void* stream) {
  if (ws == nullptr) return fail(MLAP_ERR_NULL, "workspace is NULL");
  if (ws_bytes < 256) return fail(MLAP_ERR_WORKSPACE, "workspace smaller than 256 bytes");
  cudaError_t e = launch_bounded_wait_selftest(static_cast<uint32_t*>(ws),
                                               static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "bounded-wait self-test launch");
  return MLAP_OK;
}

mlap_status_t qkvrnrc_get_workspace_size(const qkvrnrc_args_t* args, size_t* bytes) {
  if (bytes == nullptr) return fail(MLAP_ERR_NULL, "bytes is NULL");
  QkvDims d;
  CHECK_STATUS(validate_qkv(args, &d));
  *bytes = 256;
  return MLAP_OK;
}

mlap_status_t qkvrnrc_execute(const qkvrnrc_args_t* a, void* ws, size_t ws_bytes, void* stream) {
  return qkv_run(a, ws, ws_bytes, static_cast<cudaStream_t>(stream), nullptr);
}

mlap_status_t mlap_execute_stamped(const mlap_args_t* args, void* ws, size_t ws_bytes, void* stream,
                                   uint64_t* stamps) {
  if (stamps == nullptr) return fail(MLAP_ERR_NULL, "stamps is NULL");
  return mla_run(args, ws, ws_bytes, static_cast<cudaStream_t>(stream), stamps);
}

mlap_status_t qkvrnrc_execute_stamped(const qkvrnrc_args_t* args, void* ws, size_t ws_bytes,
                                      void* stream, uint64_t* stamps) {
  if (stamps == nullptr) return fail(MLAP_ERR_NULL, "stamps is NULL");
  return qkv_run(args, ws, ws_bytes, static_cast<cudaStream_t>(stream), stamps);
}

}  // extern "C"

// ================================================================================================
// Allocation-free MLA prolog.
//
// Some callers cannot hand the library a workspace: a plugin whose host framework owns every
// device buffer and passes in only the tensors it manages, a latency-critical serving loop that
// may not pay cudaMalloc's implicit device synchronisation, or a plain C caller with no device
// allocator of its own.  mlap_execute_no_alloc runs the same kernels as mlap_execute with its
// scratch (K-split partials, c^Q, q^C, error word) in the fixed-size array below.  Every GPU that
// uses this entry point keeps the array until the process exits.
static __device__ __align__(256) uint8_t g_mlap_static_scratch[MLAP_NO_ALLOC_SCRATCH_BYTES];

extern "C" mlap_status_t mlap_execute_no_alloc(const mlap_args_t* args, void* stream) {
  MlaDims d;
  CHECK_STATUS(validate_mla(args, &d));
  const size_t need = mla_ws_layout(d).total;
  if (need > static_cast<size_t>(MLAP_NO_ALLOC_SCRATCH_BYTES))
    return fail(MLAP_ERR_WORKSPACE,
                "mlap_execute_no_alloc: these shapes need " + std::to_string(need) +
                    " bytes of scratch; the static scratch holds " +
                    std::to_string(static_cast<size_t>(MLAP_NO_ALLOC_SCRATCH_BYTES)) +
                    " (use mlap_execute with a caller workspace)");
  if (d.T == 0) return MLAP_OK;
  // The array's name is only a host-side stand-in: the kernels get the device address the runtime
  // reports for it on the current device.  The lookup is asked for on every call (a host-side
  // table lookup once the module is loaded), so a context that was torn down and made again
  // (cudaDeviceReset) gets the array's new address.
  void* scratch = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&scratch, g_mlap_static_scratch);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
  // The array keeps the previous call's contents; only the header (the error word) must start at
  // zero: every other scratch byte a call reads was written earlier in the same call.
  e = cudaMemsetAsync(scratch, 0, kHeaderBytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "clearing the static scratch header");
  return mla_run(args, scratch, static_cast<size_t>(MLAP_NO_ALLOC_SCRATCH_BYTES),
                 static_cast<cudaStream_t>(stream), nullptr);
}
