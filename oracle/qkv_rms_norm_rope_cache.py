"""QkvRmsNormRopeCache oracle — TEST INFRASTRUCTURE ONLY.

Plain float64 restatement of aclnnQkvRmsNormRopeCache, "Formulas":

  (1) SplitVD: q = qkv[..., :Nq*D], k = qkv[..., Nq*D:(Nq+Nk)*D], v = qkv[..., (Nq+Nk)*D:]
  (2) RmsNorm per head along D: y = x / sqrt(mean(x^2) + eps) * gamma      (q and k)
  (3) RoPE (half-and-half) on the RmsNorm output, d = D                    (q and k)
  (4) Quant: none (kQuant = kRoPE, vQuant = v), symmetric (kRoPE / kScale, v / vScale) or
      asymmetric (kRoPE / kScale + kOffset, v / vScale + vOffset)

and "Other restrictions": index in [-1, BlockNum*BlockSize), -1 skips the update.  The API
function's optional outputs qBeforeQuant, kBeforeQuant, vBeforeQuant are the three tensors that
enter "Quant": q and k after RmsNorm and RoPE, v as split.

Readings (the parameter table is lost from the page): gamma_q and gamma_k have shape (D,) and
are shared by all heads of their kind; sin and cos have shape (B*S, D) and are shared by all
heads; k_scale (Nk, D) and v_scale (Nv, D) are per channel; the cache layout is
(BlockNum, BlockSize, N, D) with slot i at block i // BlockSize, row i % BlockSize; qOut is
rounded to the dtype of qkv (fp16 or bf16); int8 codes round half to even, clamp to [-128, 127],
with the quotient in float64 (the page states only the division).
Asymmetric quant: k_offset (Nk, D) and v_offset (Nv, D) are per-channel float32 offsets added to
the float64 quotient before rounding.  The before-quant outputs are dense (T, N, D) tensors in
the dtype of qkv, one row per token whatever its index (they are not cache writes); qBeforeQuant
equals qOut because the formulas never quantise q.
"""
from __future__ import annotations

import numpy as np

from .mla_prolog import rms_norm, rope_half_and_half
from .rounding import round_bf16, round_fp16, saturate_int8_rne


def _quant(v: np.ndarray, scale: np.ndarray, offset=None) -> np.ndarray:
    """Quant of "Formulas" (4): v / scale (+ offset), round half to even, clamp, in float64."""
    q = np.asarray(v, np.float64) / np.asarray(scale, np.float64)
    if offset is not None:                               # asymmetric: + offset
        q = q + np.asarray(offset, np.float64)
    return saturate_int8_rne(q)


def qkv_rms_norm_rope_cache(qkv, gamma_q, gamma_k, cos, sin, index, k_cache, v_cache,
                            epsilon, Nq, Nk, Nv, k_scale=None, v_scale=None,
                            out_dtype: str = "fp16", k_offset=None, v_offset=None) -> dict:
    """qkv: (..., (Nq+Nk+Nv)*D) values; caches (BlockNum, BlockSize, Nk|Nv, D).

    Returns q_out (T, Nq, D) as float64 values of ``out_dtype`` ("fp16" or "bf16", the dtype of
    qkv), the updated caches (int8 when quantised, else float64 values of ``out_dtype``), and the
    before-quant tensors q_before (T, Nq, D), k_before (T, Nk, D), v_before (T, Nv, D).
    """
    rnd = round_fp16 if out_dtype == "fp16" else round_bf16
    qkv = np.asarray(qkv, np.float64)
    D = qkv.shape[-1] // (Nq + Nk + Nv)
    x = qkv.reshape(-1, Nq + Nk + Nv, D)
    T = x.shape[0]
    q, k, v = x[:, :Nq, :], x[:, Nq:Nq + Nk, :], x[:, Nq + Nk:, :]     # SplitVD
    cos = np.asarray(cos, np.float64).reshape(T, 1, D)
    sin = np.asarray(sin, np.float64).reshape(T, 1, D)
    q_emb = rope_half_and_half(rms_norm(q, gamma_q, epsilon), cos, sin)
    k_emb = rope_half_and_half(rms_norm(k, gamma_k, epsilon), cos, sin)

    quantised = np.asarray(k_cache).dtype == np.int8
    if quantised:
        ko = None if k_offset is None else np.asarray(k_offset).reshape(1, Nk, D)
        vo = None if v_offset is None else np.asarray(v_offset).reshape(1, Nv, D)
        k_rows = _quant(k_emb, np.asarray(k_scale).reshape(1, Nk, D), ko)
        v_rows = _quant(v, np.asarray(v_scale).reshape(1, Nv, D), vo)
    else:
        k_rows = rnd(k_emb)
        v_rows = rnd(v)

    k_out = np.asarray(k_cache).copy()
    v_out = np.asarray(v_cache).copy()
    block_num, block_size = k_out.shape[0], k_out.shape[1]
    for t, i in enumerate(np.asarray(index).reshape(-1).tolist()):
        if i < 0 or i >= block_num * block_size:
            continue
        k_out[i // block_size, i % block_size] = k_rows[t]
        v_out[i // block_size, i % block_size] = v_rows[t]
    return {"q_out": rnd(q_emb), "k_cache": k_out, "v_cache": v_out,
            "k_rows": k_rows, "v_rows": v_rows,
            "q_before": rnd(q_emb), "k_before": rnd(k_emb), "v_before": rnd(v)}
