"""MLA prolog oracle (MlaPrologV2 / MlaPreprocess inference prolog) — TEST INFRASTRUCTURE ONLY.

Plain float64 restatement of the MlaPrologV2 README, "功能说明" (computation formulas):

    c^Q  = RmsNorm(x · W^DQ)                      q^C = c^Q · W^UQ        q^N = q^C · W^UK
    q^R  = ROPE(c^Q · W^QR)
    c^KV = RmsNorm(x · W^DKV)   -> kv_cache        k^R = ROPE(x · W^KR)  -> kr_cache

with the RmsNorm of the same section (epsilon added to the mean of squares, inside the root; the
aclnnMlaPreprocessV2 "Formula" RMS agrees) and the half-and-half RoPE of aclnnQkvRmsNormRopeCache,
"Formulas" (3), which the MLA pages name (ROPE) but do not define.

Readings where the pages are silent (each is also listed in the design notes):

* Rounding points.  float64 throughout, rounded to bf16 only where a tensor becomes the input of a
  bf16 matmul (c^Q; the q^C nope slice) and at the outputs (query, query_rope, the caches).
* Fused weights.  weight_dkv_kr columns are [W^DKV (Hckv) | W^KR (Dr)]; weight_uq_qr columns are
  grouped per head n as [W^UQ_n (D) | W^QR_n (Dr)].  The pages give only the fused shapes
  ("约束说明" dtype/shape matrix: (He, Hckv+Dr), (Hcq, N*(D+Dr))).
* Partial quant ("部分量化"): c^Q (bf16) is multiplied by smooth_scales_cq, quantised per token
  symmetrically with scale = amax/127, round half to even, clamp to [-127, 127]; the int8 matmul
  accumulates exactly and is dequantised by scale_t * dequant_scale_w_uq_qr[column].  Scale,
  quotient and code are float64 like everything else here: the pages state only the division.
* Cache quant: value / quant_scale (the aclnnQkvRmsNormRopeCache "Formulas" (4) rule
  kQuant = kRoPE / kScale), round half to even, clamp to [-128, 127], in float64.
* Full quant ("全量化", the scenario matrix of "约束说明"): token_x int8 with the per-token
  dequant_scale_x (T, 1), weight_dq and weight_dkv_kr int8 with per-channel dequant_scale_w_dq
  (1, Hcq) and dequant_scale_w_dkv_kr (1, Hckv+Dr).  Reading: the int8 matmuls accumulate
  exactly and are dequantised as acc * dequant_scale_x[t] * dequant_scale_w[column]; from there
  the path is the partial-quant one.  With the quantised kv_cache column, query is int8
  "pertoken_head": per token and head, scale = amax over Hckv of q^N / 127, code = q^N / scale
  rounded half to even and clamped to [-127, 127] (the c^Q rule), in float64;
  dequant_scale_q_nope (T, N, 1) returns the scale (0 and all-zero codes when amax = 0).  The
  pages call that cache quant "pertensor" but give quant_scale_ckv the shape (1, Hckv); the
  shape is followed (one scale per channel, the cache-quant rule above); kr_cache stays bf16
  there ("无需赋值" for quant_scale_ckr).
* Input RmsNormQuant (aclnnMlaPreprocessV2, "Formula", RmsNormQuant): when its parameters are
  given, x is replaced ahead of the down-projection by (gamma * x / RMS(x) + bias) * deqScale,
  RMS(x) = sqrt(mean over He of x^2 + epsilon).  Readings: gamma and bias are per hidden channel
  (He) bf16 values, deqScale is float32 per channel (He) or one value for all channels; the
  printed formula has no rounding to an integer grid, so the result is rounded to bf16, the type
  of the down-projection's operand (the rounding-point rule above), and the step composes with
  the bf16-x scenarios only (non-quant, partial quant).
* cache_index: slot i goes to block i // BlockSize, row i % BlockSize (Nkv = 1); i = -1 skips the
  row (aclnnQkvRmsNormRopeCache, "Other restrictions"); other out-of-range values are skipped too
  (the CUDA path also flags them).
"""
from __future__ import annotations

import numpy as np

from .rounding import round_bf16, saturate_int8_rne


def rms_norm(h: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """gamma * h / sqrt(mean(h^2) + eps) along the last axis (MlaPrologV2 README, RmsNorm公式)."""
    h = np.asarray(h, dtype=np.float64)
    mean_sq = np.mean(h * h, axis=-1, keepdims=True)
    return np.asarray(gamma, dtype=np.float64) * h / np.sqrt(mean_sq + eps)


def rope_half_and_half(y: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """y*cos + cat(-y2, y1)*sin with y1, y2 the two halves of the last axis
    (aclnnQkvRmsNormRopeCache, "Formulas" (3) RoPE (Half-and-Half))."""
    y = np.asarray(y, dtype=np.float64)
    half = y.shape[-1] // 2
    y1, y2 = y[..., :half], y[..., half:]
    rotated = np.concatenate([-y2, y1], axis=-1)
    return y * np.asarray(cos, np.float64) + rotated * np.asarray(sin, np.float64)


def rms_norm_quant(x: np.ndarray, gamma: np.ndarray, bias: np.ndarray, deq_scale,
                   eps: float) -> np.ndarray:
    """(gamma * x / RMS(x) + bias) * deqScale along the last axis with RMS(x) = sqrt(mean(x^2) +
    eps) (aclnnMlaPreprocessV2, "Formula": RMS, RmsNorm, RmsNormQuant).  float64, unrounded;
    deq_scale is one value per channel or a single value."""
    x = np.asarray(x, dtype=np.float64)
    rms = np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    normed = np.asarray(gamma, np.float64).reshape(-1) * x / rms
    return (normed + np.asarray(bias, np.float64).reshape(-1)) * np.asarray(deq_scale, np.float64).reshape(-1)


def dynamic_quant_per_token(c_q: np.ndarray, smooth: np.ndarray):
    """Per-token symmetric int8 quant of c^Q after smoothing (MlaPrologV2 README, parameter
    smooth_scales_cq: "RmsNormCq输出动态量化参数"; formula is the reading stated in the module
    docstring).  Returns (codes int8 (T,Hcq), scale float64 (T,)), all in float64."""
    s = np.asarray(c_q, np.float64) * np.asarray(smooth, np.float64).reshape(1, -1)
    amax = np.max(np.abs(s), axis=-1)
    scale = amax / 127.0
    safe = np.where(scale > 0, scale, 1.0)
    codes = saturate_int8_rne(s / safe[:, None], -127, 127)
    codes[scale == 0] = 0
    return codes, scale


def cache_quant(v: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """int8 code of v / scale per channel, round half to even, clamp to [-128,127], in float64
    (MlaPrologV2 README quant_scale_ckv / quant_scale_ckr; the division rule of
    aclnnQkvRmsNormRopeCache "Formulas" (4))."""
    q = np.asarray(v, np.float64) / np.asarray(scale, np.float64).reshape(1, -1)
    return saturate_int8_rne(q)


def quant_per_token_head(q_n: np.ndarray):
    """int8 query "pertoken_head" (MlaPrologV2 README, scenario matrix: query INT8 in full quant
    with quantised kv_cache; dequant_scale_q_nope (T, N, 1)): per token and head symmetric, scale
    = amax / 127, round half to even, clamp to [-127, 127], in float64.  Returns (codes (T, N, H)
    int8, scale (T, N) float64)."""
    s = np.asarray(q_n, np.float64)
    amax = np.max(np.abs(s), axis=-1)
    scale = amax / 127.0
    safe = np.where(scale > 0, scale, 1.0)
    codes = saturate_int8_rne(s / safe[..., None], -127, 127)
    codes[scale == 0] = 0
    return codes, scale


def up_projection_int8(codes, scale_t, weight_uq_qr, dequant_scale_w_uq_qr) -> np.ndarray:
    """c^Q · [W^UQ | W^QR] in partial / full quant: the int8 codes times the int8 weight,
    accumulated exactly, dequantised by scale_t[t] * dequant_scale_w_uq_qr[column] (MlaPrologV2
    README, 参数说明 dequant_scale_w_uq_qr; reading stated in the module docstring)."""
    acc = np.asarray(codes).astype(np.int64) @ np.asarray(weight_uq_qr).astype(np.int64)
    return (acc.astype(np.float64) * np.asarray(scale_t, np.float64).reshape(-1, 1)
            * np.asarray(dequant_scale_w_uq_qr, np.float64).reshape(1, -1))


def query_outputs(u, weight_uk, rope_cos, rope_sin, Dr: int, query_int8: bool = False):
    """From u = c^Q · [W^UQ | W^QR] (T, N*(D+Dr)), columns per head [D nope | Dr rope]: q^C =
    bf16(nope part) (input of the W^UK matmul), q^N = q^C · W^UK per head, query = bf16(q^N) (or
    the int8 "pertoken_head" query and its scales), query_rope = bf16(ROPE(rope part))
    (MlaPrologV2 README, 功能说明 q^C, q^N and q^R formulas).  Returns (query, query_rope,
    dequant_scale_q_nope or None)."""
    w_uk = np.asarray(weight_uk, np.float64)
    N, D, Hckv = w_uk.shape
    u = np.asarray(u, np.float64).reshape(-1, N, D + Dr)
    T = u.shape[0]
    cos = np.asarray(rope_cos, np.float64).reshape(T, 1, Dr)
    sin = np.asarray(rope_sin, np.float64).reshape(T, 1, Dr)
    q_c = round_bf16(u[:, :, :D])                  # q^C, input of the W^UK matmul
    q_r = u[:, :, D:]                              # c^Q · W^QR, before ROPE
    q_n = np.empty((T, N, Hckv), np.float64)
    for n in range(N):                             # q^N = q^C · W^UK, per head
        q_n[:, n, :] = q_c[:, n, :] @ w_uk[n]
    scale_q = None
    if query_int8:
        query, scale_q = quant_per_token_head(q_n)
    else:
        query = round_bf16(q_n)
    query_rope = round_bf16(rope_half_and_half(q_r, cos, sin))
    return query, query_rope, scale_q


def scatter_rows(cache: np.ndarray, rows: np.ndarray, cache_index: np.ndarray) -> np.ndarray:
    """Copy of ``cache`` (BlockNum, BlockSize, 1, H) with row t stored at slot cache_index[t]
    (MlaPrologV2 README k^C = Cache(c^KV), k^R = Cache(...); "-1 skips" from
    aclnnQkvRmsNormRopeCache "Other restrictions")."""
    out = cache.copy()
    block_num, block_size = cache.shape[0], cache.shape[1]
    for t, i in enumerate(np.asarray(cache_index).reshape(-1).tolist()):
        if i < 0 or i >= block_num * block_size:
            continue
        out[i // block_size, i % block_size, 0, :] = rows[t]
    return out


def mla_prolog(token_x, weight_dq, weight_uq_qr, weight_uk, weight_dkv_kr,
               rmsnorm_gamma_cq, rmsnorm_gamma_ckv, rope_sin, rope_cos, cache_index,
               kv_cache, kr_cache, rmsnorm_epsilon_cq, rmsnorm_epsilon_ckv,
               dequant_scale_w_uq_qr=None, smooth_scales_cq=None,
               quant_scale_ckv=None, quant_scale_ckr=None, dequant_scale_x=None,
               dequant_scale_w_dq=None, dequant_scale_w_dkv_kr=None,
               query_int8: bool = False, rms_norm_quant_gamma=None, rms_norm_quant_bias=None,
               rms_norm_quant_deq_scale=None, rms_norm_quant_epsilon=None) -> dict:
    """The whole prolog for T tokens.

    Inputs are numpy arrays holding the exact values of the operator inputs (bf16 values as
    float64; int8 weights/caches as int8).  token_x is (T, He) (the BSH form (B,S,He) is the same
    memory and is flattened by the caller).  Returns a dict with query (T,N,Hckv), query_rope
    (T,N,Dr) as float64 holding bf16 values, and the updated kv_cache / kr_cache (float64 bf16
    values, or int8 when the caches are quantised).  Full quant: token_x, weight_dq and
    weight_dkv_kr int8 with their dequant scales; query_int8 returns int8 query codes and
    dequant_scale_q_nope (T, N).  rms_norm_quant_*: the input RmsNormQuant of
    aclnnMlaPreprocessV2 applied to token_x first (bf16 x only).
    """
    x_int8 = np.asarray(token_x).dtype == np.int8
    x = np.asarray(token_x, np.float64)
    if rms_norm_quant_gamma is not None:           # x' = bf16((RmsNorm(x) + bias) * deqScale)
        x = round_bf16(rms_norm_quant(x, rms_norm_quant_gamma, rms_norm_quant_bias,
                                      rms_norm_quant_deq_scale, rms_norm_quant_epsilon))
    T, He = x.shape
    N, D, Hckv = weight_uk.shape
    Dr = np.asarray(rope_sin).shape[-1]
    Hcq = weight_dq.shape[1]
    sin = np.asarray(rope_sin, np.float64).reshape(T, Dr)
    cos = np.asarray(rope_cos, np.float64).reshape(T, Dr)

    def down(w, w_scale):
        """x · W, or for int8 x and W the exact integer product dequantised per token and column."""
        if not x_int8:
            return x @ np.asarray(w, np.float64)
        acc = np.asarray(token_x).astype(np.int64) @ np.asarray(w).astype(np.int64)   # exact
        return (acc.astype(np.float64)
                * np.asarray(dequant_scale_x, np.float64).reshape(-1, 1)
                * np.asarray(w_scale, np.float64).reshape(1, -1))

    # Query path: c^Q = RmsNorm(x · W^DQ), rounded to bf16 as the next matmul's input.
    h_q = down(weight_dq, dequant_scale_w_dq)
    c_q_exact = rms_norm(h_q, rmsnorm_gamma_cq, rmsnorm_epsilon_cq)
    c_q = round_bf16(c_q_exact)

    # c^Q · [W^UQ | W^QR]
    codes = scale_t = None
    if np.asarray(weight_uq_qr).dtype == np.int8:
        codes, scale_t = dynamic_quant_per_token(c_q, smooth_scales_cq)
        u = up_projection_int8(codes, scale_t, weight_uq_qr, dequant_scale_w_uq_qr)
    else:
        u = c_q @ np.asarray(weight_uq_qr, np.float64)
    query, query_rope, scale_q = query_outputs(u, weight_uk, cos, sin, Dr, query_int8)

    # Key path: c^KV = RmsNorm(x · W^DKV), k^R = ROPE(x · W^KR)
    h_kvr = down(weight_dkv_kr, dequant_scale_w_dkv_kr)
    c_kv = rms_norm(h_kvr[:, :Hckv], rmsnorm_gamma_ckv, rmsnorm_epsilon_ckv)
    k_r = rope_half_and_half(h_kvr[:, Hckv:Hckv + Dr], cos, sin)

    if np.asarray(kv_cache).dtype == np.int8:
        kv_rows = cache_quant(c_kv, quant_scale_ckv)
    else:
        kv_rows = round_bf16(c_kv)
    if np.asarray(kr_cache).dtype == np.int8:
        kr_rows = cache_quant(k_r, quant_scale_ckr)
    else:
        kr_rows = round_bf16(k_r)

    return {
        "query": query,
        "query_rope": query_rope,
        "kv_cache": scatter_rows(np.asarray(kv_cache), kv_rows, cache_index),
        "kr_cache": scatter_rows(np.asarray(kr_cache), kr_rows, cache_index),
        "dequant_scale_q_nope": scale_q,
        # intermediates, exposed for tests only
        "c_q_exact": c_q_exact,
        "c_q": c_q,
        "c_q_codes": codes,
        "c_q_scale": scale_t,
        "c_kv": c_kv,
        "k_r": k_r,
    }


def mla_prolog_tokens(inputs: dict, token_ids) -> dict:
    """The prolog restricted to a subset of tokens (tokens are independent).  Caches are not
    scattered; the rows that would be stored are returned instead."""
    ids = np.asarray(token_ids)
    sub = dict(inputs)
    sub["token_x"] = np.asarray(inputs["token_x"])[ids]
    sub["rope_sin"] = np.asarray(inputs["rope_sin"]).reshape(-1, np.asarray(inputs["rope_sin"]).shape[-1])[ids]
    sub["rope_cos"] = np.asarray(inputs["rope_cos"]).reshape(-1, np.asarray(inputs["rope_cos"]).shape[-1])[ids]
    sub["cache_index"] = -np.ones(len(ids), np.int64)   # no scatter
    if inputs.get("dequant_scale_x") is not None:
        sub["dequant_scale_x"] = np.asarray(inputs["dequant_scale_x"]).reshape(-1, 1)[ids]
    out = mla_prolog(**sub)
    kv_dtype = np.asarray(inputs["kv_cache"]).dtype
    kr_dtype = np.asarray(inputs["kr_cache"]).dtype
    out["kv_rows"] = (cache_quant(out["c_kv"], inputs["quant_scale_ckv"]) if kv_dtype == np.int8
                      else round_bf16(out["c_kv"]))
    out["kr_rows"] = (cache_quant(out["k_r"], inputs["quant_scale_ckr"]) if kr_dtype == np.int8
                      else round_bf16(out["k_r"]))
    return out


def mla_key_rows(token_x, weight_dkv_kr, rmsnorm_gamma_ckv, rope_sin, rope_cos,
                 rmsnorm_epsilon_ckv, Hckv, kv_dtype_int8=False, kr_dtype_int8=False,
                 quant_scale_ckv=None, quant_scale_ckr=None, dequant_scale_x=None,
                 dequant_scale_w_dkv_kr=None, rms_norm_quant_gamma=None,
                 rms_norm_quant_bias=None, rms_norm_quant_deq_scale=None,
                 rms_norm_quant_epsilon=None, **_unused) -> tuple:
    """Only the key path of ``mla_prolog`` (c^KV = RmsNorm(x·W^DKV), k^R = ROPE(x·W^KR)), as the
    rows the cache would receive for every token: (kv_rows, kr_rows).  Same formulas and
    rounding as ``mla_prolog``; used to check every written cache slot of large workloads."""
    x = np.asarray(token_x, np.float64)
    if rms_norm_quant_gamma is not None:
        x = round_bf16(rms_norm_quant(x, rms_norm_quant_gamma, rms_norm_quant_bias,
                                      rms_norm_quant_deq_scale, rms_norm_quant_epsilon))
    T = x.shape[0]
    Dr = np.asarray(rope_sin).shape[-1]
    sin = np.asarray(rope_sin, np.float64).reshape(T, Dr)
    cos = np.asarray(rope_cos, np.float64).reshape(T, Dr)
    if np.asarray(token_x).dtype == np.int8:      # full quant: exact product, then dequant
        acc = np.asarray(token_x).astype(np.int64) @ np.asarray(weight_dkv_kr).astype(np.int64)
        h_kvr = (acc.astype(np.float64) * np.asarray(dequant_scale_x, np.float64).reshape(-1, 1)
                 * np.asarray(dequant_scale_w_dkv_kr, np.float64).reshape(1, -1))
    else:
        h_kvr = x @ np.asarray(weight_dkv_kr, np.float64)
    c_kv = rms_norm(h_kvr[:, :Hckv], rmsnorm_gamma_ckv, rmsnorm_epsilon_ckv)
    k_r = rope_half_and_half(h_kvr[:, Hckv:Hckv + Dr], cos, sin)
    kv = cache_quant(c_kv, quant_scale_ckv) if kv_dtype_int8 else round_bf16(c_kv)
    kr = cache_quant(k_r, quant_scale_ckr) if kr_dtype_int8 else round_bf16(k_r)
    return kv, kr
