"""QkvRmsNormRopeCache oracle — TEST INFRASTRUCTURE ONLY.

Plain float64 restatement of aclnnQkvRmsNormRopeCache, "Formulas":

  (1) SplitVD: q = qkv[..., :Nq*D], k = qkv[..., Nq*D:(Nq+Nk)*D], v = qkv[..., (Nq+Nk)*D:]
  (2) RmsNorm per head along D: y = x / sqrt(mean(x^2) + eps) * gamma      (q and k)
  (3) RoPE (half-and-half) on the RmsNorm output, d = D                    (q and k)
  (4) Quant: none (kQuant = kRoPE, vQuant = v) or symmetric (kRoPE / kScale, v / vScale)

and "Other restrictions": index in [-1, BlockNum*BlockSize), -1 skips the update.

Readings (the parameter table is lost from the page): gamma_q and gamma_k have shape (D,) and
are shared by all heads of their kind; sin and cos have shape (B*S, D) and are shared by all
heads; k_scale (Nk, D) and v_scale (Nv, D) are per channel; the cache layout is
(BlockNum, BlockSize, N, D) with slot i at block i // BlockSize, row i % BlockSize; qOut is
rounded to the dtype of qkv (fp16 or bf16); int8 codes round half to even, clamp to [-128, 127], decided in float32.
"""
from __future__ import annotations

import numpy as np

from .mla_prolog import rms_norm, rope_half_and_half
from .rounding import round_bf16, round_fp16, saturate_int8_rne


def _quant(v: np.ndarray, scale: np.ndarray) -> np.ndarray:
    q = (np.asarray(v, np.float64).astype(np.float32)
         / np.asarray(scale, np.float32)).astype(np.float32)
    return saturate_int8_rne(q)


def qkv_rms_norm_rope_cache(qkv, gamma_q, gamma_k, cos, sin, index, k_cache, v_cache,
                            epsilon, Nq, Nk, Nv, k_scale=None, v_scale=None,
                            out_dtype: str = "fp16") -> dict:
    """qkv: (..., (Nq+Nk+Nv)*D) values; caches (BlockNum, BlockSize, Nk|Nv, D).

    Returns q_out (T, Nq, D) as float64 values of ``out_dtype`` ("fp16" or "bf16", the dtype of
    qkv) and the updated caches (int8 when quantised, else float64 values of ``out_dtype``).
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
        k_rows = _quant(k_emb, np.asarray(k_scale).reshape(1, Nk, D))
        v_rows = _quant(v, np.asarray(v_scale).reshape(1, Nv, D))
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
            "k_rows": k_rows, "v_rows": v_rows}
