"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check the pins catch them.

Each mutation rewrites one line of ``oracle/mla_prolog.py`` or ``oracle/qkv_rms_norm_rope_cache.py``
in a private module copy; the brute-force pin must then fail.  The real oracle is untouched.
"""
import importlib.util
import os
import sys
import types

import numpy as np
import pytest

import oracle
from tests import bruteforce as bf
from tests.test_oracle_pins import _brute, _qkv_brute, _tiny_mla, _tiny_qkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _mutant(fname, old, new):
    path = os.path.join(ROOT, "oracle", fname)
    src = open(path).read()
    assert src.count(old) >= 1, (fname, old)
    mod = types.ModuleType("oracle._mutant")
    mod.__package__ = "oracle"
    exec(compile(src.replace(old, new), path, "exec"), mod.__dict__)
    return mod


MLA_MUTATIONS = [
    ("eps outside the root", "np.sqrt(mean_sq + eps)", "(np.sqrt(mean_sq) + eps * 1e5)"),
    ("sum instead of mean", "np.mean(h * h, axis=-1, keepdims=True)",
     "np.sum(h * h, axis=-1, keepdims=True)"),
    ("rope sign", "rotated = np.concatenate([-y2, y1], axis=-1)",
     "rotated = np.concatenate([y2, -y1], axis=-1)"),
    ("nope/rope order in a head", "q_c = round_bf16(u[:, :, :D])", "q_c = round_bf16(u[:, :, Dr:])"),
    ("rope slice", "q_r = u[:, :, D:]", "q_r = u[:, :, :Dr]"),
    ("kv/kr column order", "h_kvr[:, :Hckv], rmsnorm_gamma_ckv",
     "h_kvr[:, Dr:], rmsnorm_gamma_ckv"),
    ("gamma dropped", "return np.asarray(gamma, dtype=np.float64) * h / np.sqrt(mean_sq + eps)",
     "return h / np.sqrt(mean_sq + eps)"),
    ("slot block/offset swapped", "out[i // block_size, i % block_size, 0, :] = rows[t]",
     "out[i % block_num, i // block_num, 0, :] = rows[t]"),
    ("dequant scale dropped", "* np.asarray(dequant_scale_w_uq_qr, np.float64).reshape(1, -1))",
     ")"),
    ("cache quant multiplies", "q = np.asarray(v, np.float64) / np.asarray(scale, np.float64)",
     "q = np.asarray(v, np.float64) * np.asarray(scale, np.float64)"),
    ("missing bf16 round of q^C", "q_c = round_bf16(u[:, :, :D])", "q_c = u[:, :, :D] * (1 + 2**-9)"),
]


@pytest.mark.parametrize("label,old,new", MLA_MUTATIONS, ids=[m[0] for m in MLA_MUTATIONS])
def test_mla_pins_catch_mutation(label, old, new):
    mod = _mutant("mla_prolog.py", old, new)
    int8 = "dequant" in label or "quant" in label
    rng = np.random.default_rng(31)
    inp = _tiny_mla(rng, int8=int8, int8_cache="cache quant" in label)
    want = _brute(inp)
    got = mod.mla_prolog(**inp)
    same = True
    for key in ("query", "query_rope", "kv_cache", "kr_cache"):
        same &= np.allclose(np.asarray(got[key], np.float64), np.array(want[key], np.float64),
                            rtol=1e-12, atol=1e-14)
    assert not same, f"mutation '{label}' not detected"


FULL_QUANT_MUTATIONS = [
    ("x dequant dropped", "* np.asarray(dequant_scale_x, np.float64).reshape(-1, 1)", ""),
    ("W^DKV dequant from W^DQ", "h_kvr = down(weight_dkv_kr, dequant_scale_w_dkv_kr)",
     "h_kvr = down(weight_dkv_kr, np.full_like(dequant_scale_w_dkv_kr, np.mean(dequant_scale_w_dq)))"),
    ("query codes truncated", "codes = saturate_int8_rne(s / safe[..., None], -127, 127)",
     "codes = np.clip(np.trunc(s / safe[..., None]), -127, 127).astype(np.int8)"),
    ("query scale per token", "amax = np.max(np.abs(s), axis=-1)\n    scale = amax / 127.0\n    safe = np.where(scale > 0, scale, 1.0)\n    codes = saturate_int8_rne(s / safe[..., None]",
     "amax = np.max(np.abs(s), axis=(-2, -1), keepdims=True) + 0 * s[..., 0:1]\n    amax = amax[..., 0]\n    scale = amax / 127.0\n    safe = np.where(scale > 0, scale, 1.0)\n    codes = saturate_int8_rne(s / safe[..., None]"),
]


@pytest.mark.parametrize("label,old,new", FULL_QUANT_MUTATIONS, ids=[m[0] for m in FULL_QUANT_MUTATIONS])
def test_full_quant_pins_catch_mutation(label, old, new):
    mod = _mutant("mla_prolog.py", old, new)
    rng = np.random.default_rng(33)
    inp = _tiny_mla(rng, True, True, full=True)
    want = _brute(inp)
    got = mod.mla_prolog(**inp)
    same = np.array_equal(np.asarray(got["query"]), np.array(want["query"], np.int8))
    same &= np.array_equal(np.asarray(got["dequant_scale_q_nope"]),
                           np.array(want["dequant_scale_q_nope"], np.float64))
    for key in ("query_rope", "kr_cache"):
        same &= np.allclose(np.asarray(got[key], np.float64), np.array(want[key], np.float64),
                            rtol=1e-12, atol=1e-14)
    same &= np.array_equal(np.asarray(got["kv_cache"]), np.array(want["kv_cache"], np.int8))
    assert not same, f"mutation '{label}' not detected"


XNORM_MUTATIONS = [
    ("bias after deqScale", "return (normed + np.asarray(bias, np.float64).reshape(-1)) * np.asarray(deq_scale, np.float64).reshape(-1)",
     "return normed * np.asarray(deq_scale, np.float64).reshape(-1) + np.asarray(bias, np.float64).reshape(-1)"),
    ("x eps outside the root", "rms = np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)",
     "rms = np.sqrt(np.mean(x * x, axis=-1, keepdims=True)) + eps * 1e3"),
    ("x gamma dropped", "normed = np.asarray(gamma, np.float64).reshape(-1) * x / rms", "normed = x / rms"),
    ("x' not rounded", "x = round_bf16(rms_norm_quant(x, rms_norm_quant_gamma, rms_norm_quant_bias,\n                                      rms_norm_quant_deq_scale, rms_norm_quant_epsilon))\n    T, He",
     "x = rms_norm_quant(x, rms_norm_quant_gamma, rms_norm_quant_bias,\n                                      rms_norm_quant_deq_scale, rms_norm_quant_epsilon) * (1 + 2**-10)\n    T, He"),
]


@pytest.mark.parametrize("label,old,new", XNORM_MUTATIONS, ids=[m[0] for m in XNORM_MUTATIONS])
def test_rms_norm_quant_pins_catch_mutation(label, old, new):
    mod = _mutant("mla_prolog.py", old, new)
    rng = np.random.default_rng(34)
    inp = _tiny_mla(rng, xnorm="channel")
    want = _brute(inp)
    got = mod.mla_prolog(**inp)
    same = True
    for key in ("query", "query_rope", "kv_cache", "kr_cache"):
        same &= np.allclose(np.asarray(got[key], np.float64), np.array(want[key], np.float64),
                            rtol=1e-12, atol=1e-14)
    assert not same, f"mutation '{label}' not detected"


QKV_MUTATIONS = [
    ("split k/v swapped", "k, v = x[:, :Nq, :], x[:, Nq:Nq + Nk, :], x[:, Nq + Nk:, :]",
     "k, v = x[:, :Nq, :], x[:, Nq + Nk:, :], x[:, Nq:Nq + Nk, :]"),
    ("v normalised too", "v_rows = _quant(v, np.asarray(v_scale).reshape(1, Nv, D), vo)",
     "v_rows = _quant(rms_norm(v, 1.0, epsilon), np.asarray(v_scale).reshape(1, Nv, D), vo)"),
    ("offset subtracted", "q = q + np.asarray(offset, np.float64)",
     "q = q - np.asarray(offset, np.float64)"),
    ("v offset ignored", "vo = None if v_offset is None else np.asarray(v_offset).reshape(1, Nv, D)",
     "vo = None"),
    ("offset added after rounding", "return saturate_int8_rne(q)",
     "return saturate_int8_rne(q - (0 if offset is None else np.asarray(offset, np.float64))) + "
     "(0 if offset is None else np.rint(np.asarray(offset, np.float64)))"),
    ("v_before normalised", '"v_before": rnd(v)', '"v_before": rnd(rms_norm(v, 1.0, epsilon))'),
    ("k_before before RoPE", '"k_before": rnd(k_emb)', '"k_before": rnd(rms_norm(k, gamma_k, epsilon))'),
    ("k gamma from q", "k_emb = rope_half_and_half(rms_norm(k, gamma_k, epsilon), cos, sin)",
     "k_emb = rope_half_and_half(rms_norm(k, gamma_q, epsilon), cos, sin)"),
]


@pytest.mark.parametrize("label,old,new", QKV_MUTATIONS, ids=[m[0] for m in QKV_MUTATIONS])
def test_qkv_pins_catch_mutation(label, old, new):
    mod = _mutant("qkv_rms_norm_rope_cache.py", old, new)
    rng = np.random.default_rng(32)
    inp = _tiny_qkv(rng, quant="asym")
    got = mod.qkv_rms_norm_rope_cache(**inp)
    ref = oracle.qkv_rms_norm_rope_cache(**inp)
    want = _qkv_brute(inp)
    assert np.array_equal(ref["k_cache"], np.array(want["k_cache"], np.int8))
    detected = (not np.allclose(got["q_out"], np.array(want["q_out"]))
                or not np.array_equal(got["k_cache"], np.array(want["k_cache"], np.int8))
                or not np.array_equal(got["v_cache"], np.array(want["v_cache"], np.int8))
                or any(not np.allclose(got[k], np.array(want[k]), rtol=1e-12, atol=1e-14)
                       for k in ("q_before", "k_before", "v_before")))
    assert detected, f"mutation '{label}' not detected"
