"""Pins for the CPU oracle (no GPU).  Each test ties a piece of ``oracle/`` to something other than
itself: worked values derived by hand from the operator formulas (tests/golden), closed forms,
invariants, library routines on special cases, and a scalar brute force on tiny inputs.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle.mla_prolog import mla_key_rows, mla_prolog_tokens
from tests import bruteforce as bf

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _num(v):
    return math.inf if v == "inf" else float(v)


# ----------------------------------------------------------------------------- rounding

def test_rounding_golden():
    g = _golden("rounding_worked.json")
    for x, want in g["bf16"]:
        assert oracle.round_bf16(np.array([x]))[0] == _num(want), (x, want)
    for x, want in g["fp16"]:
        assert oracle.round_fp16(np.array([x]))[0] == _num(want), (x, want)
    for x, want in g["int8"]:
        assert int(oracle.saturate_int8_rne(np.array([x]))[0]) == want, (x, want)


def test_round_bf16_matches_library_cast_on_fp32_values():
    # On float32-representable inputs a float32 -> bfloat16 cast rounds once, to nearest even.
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(200000) * 10.0 ** rng.integers(-30, 30, 200000),
                        rng.standard_normal(1000)]).astype(np.float32)
    # add exact ties: bf16 value + half ulp
    base = torch.randn(5000).to(torch.bfloat16).to(torch.float32).numpy()
    ulp = np.ldexp(1.0, (np.frexp(base)[1] - 1) - 7).astype(np.float32)
    x = np.concatenate([x, base + ulp / 2, base - ulp / 2]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_bf16(x.astype(np.float64))
    assert np.array_equal(got, want)


def test_round_fp16_matches_library_cast_on_fp32_values():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(200000) * 10.0 ** rng.integers(-9, 5, 200000)).astype(np.float32)
    base = torch.randn(5000).to(torch.float16).to(torch.float32).numpy()
    ulp = np.ldexp(1.0, (np.frexp(base)[1] - 1) - 10).astype(np.float32)
    x = np.concatenate([x, base + ulp / 2, base - ulp / 2]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.float16).to(torch.float64).numpy()
    got = oracle.round_fp16(x.astype(np.float64))
    assert np.array_equal(got, want)


def test_round_fp32_matches_library_cast():
    rng = np.random.default_rng(2)
    x = rng.standard_normal(100000) * 10.0 ** rng.integers(-40, 38, 100000)
    assert np.array_equal(oracle.round_fp32(x), x.astype(np.float32).astype(np.float64))


def test_rounding_bit_brute_force_agrees():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(3000) * 8
    assert np.array_equal(oracle.round_bf16(x), np.array([bf.bf16(v) for v in x]))
    assert np.array_equal(oracle.round_fp16(x), np.array([bf.fp16(v) for v in x]))


# ----------------------------------------------------------------------------- RmsNorm

def test_rmsnorm_golden():
    for case in _golden("rmsnorm_worked.json")["cases"]:
        y = oracle.rms_norm(np.array(case["x"]), np.array(case["gamma"]), case["eps"])
        np.testing.assert_allclose(y, case["y"], rtol=1e-15, atol=1e-15)


def test_rmsnorm_closed_forms():
    rng = np.random.default_rng(4)
    h = rng.standard_normal((7, 96))
    g = -1.75
    y = oracle.rms_norm(h, np.full(96, g), 0.0)
    # constant gamma: root mean square of the output equals |gamma|
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), abs(g), rtol=1e-13)
    # invariant to positive scaling of the row when eps = 0
    gam = rng.uniform(0.5, 1.5, 96)
    np.testing.assert_allclose(oracle.rms_norm(h * 37.5, gam, 0.0), oracle.rms_norm(h, gam, 0.0),
                               rtol=1e-13)
    # textbook form through the Euclidean norm: h / (||h|| / sqrt(n))
    want = gam * h / (np.linalg.norm(h, axis=-1, keepdims=True) / math.sqrt(96))
    np.testing.assert_allclose(oracle.rms_norm(h, gam, 0.0), want, rtol=1e-13)


def test_rms_norm_quant_golden():
    for case in _golden("rms_norm_quant_worked.json")["cases"]:
        y = oracle.rms_norm_quant(np.array(case["x"]), np.array(case["gamma"]),
                                  np.array(case["bias"]), np.array(case["deq_scale"]), case["eps"])
        np.testing.assert_allclose(y, case["y"], rtol=1e-15, atol=1e-15)


def test_rms_norm_quant_closed_forms():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((6, 64))
    gam, b = rng.uniform(0.5, 1.5, 64), rng.uniform(-1, 1, 64)
    d = rng.uniform(0.5, 2.0, 64)
    y = oracle.rms_norm_quant(x, gam, b, d, 0.0)
    # invariant to positive scaling of the row when eps = 0
    np.testing.assert_allclose(oracle.rms_norm_quant(x * 19.0, gam, b, d, 0.0), y, rtol=1e-13)
    # bias 0 and deqScale 1: the textbook root-mean-square normalisation via the Euclidean norm
    want = gam * x / (np.linalg.norm(x, axis=-1, keepdims=True) / math.sqrt(64))
    np.testing.assert_allclose(oracle.rms_norm_quant(x, gam, np.zeros(64), np.ones(1), 0.0), want,
                               rtol=1e-13)
    # affine in the bias with slope deqScale, linear in deqScale
    np.testing.assert_allclose(oracle.rms_norm_quant(x, gam, b + 0.25, d, 0.0) - y, 0.25 * d
                               + 0 * y, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(oracle.rms_norm_quant(x, gam, b, 3.0 * d, 0.0), 3.0 * y, rtol=1e-13)
    # one deqScale for all channels equals the same value repeated per channel
    np.testing.assert_array_equal(oracle.rms_norm_quant(x, gam, b, np.array([1.5]), 1e-3),
                                  oracle.rms_norm_quant(x, gam, b, np.full(64, 1.5), 1e-3))


# ----------------------------------------------------------------------------- RoPE

def test_rope_golden():
    for case in _golden("rope_worked.json")["cases"]:
        out = oracle.rope_half_and_half(np.array(case["y"]), np.array(case["cos"]),
                                        np.array(case["sin"]))
        np.testing.assert_array_equal(out, case["out"])


def test_rope_is_complex_rotation():
    # With tables whose halves repeat, half-and-half RoPE multiplies z_j = y_j + i*y_{j+d/2} by
    # exp(i*theta_j): an independent (complex-number) statement of the same map.
    rng = np.random.default_rng(5)
    d = 64
    y = rng.standard_normal((9, d))
    theta = rng.uniform(-10, 10, (9, d // 2))
    cos = np.concatenate([np.cos(theta)] * 2, axis=-1)
    sin = np.concatenate([np.sin(theta)] * 2, axis=-1)
    out = oracle.rope_half_and_half(y, cos, sin)
    z = (y[:, : d // 2] + 1j * y[:, d // 2:]) * np.exp(1j * theta)
    np.testing.assert_allclose(out[:, : d // 2], z.real, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out[:, d // 2:], z.imag, rtol=1e-12, atol=1e-12)
    # identity, quarter turn, and pair-norm preservation
    one, zero = np.ones((9, d)), np.zeros((9, d))
    np.testing.assert_array_equal(oracle.rope_half_and_half(y, one, zero), y)
    np.testing.assert_array_equal(oracle.rope_half_and_half(y, zero, one),
                                  np.concatenate([-y[:, d // 2:], y[:, : d // 2]], axis=-1))
    n_in = y[:, : d // 2] ** 2 + y[:, d // 2:] ** 2
    n_out = out[:, : d // 2] ** 2 + out[:, d // 2:] ** 2
    np.testing.assert_allclose(n_out, n_in, rtol=1e-12)


# ----------------------------------------------------------------------------- quant

def test_cache_quant_roundtrip_within_half_scale():
    rng = np.random.default_rng(6)
    v = rng.standard_normal((50, 32))
    scale = rng.uniform(0.01, 0.05, (1, 32))
    q = oracle.cache_quant(v, scale)
    assert q.dtype == np.int8
    back = q.astype(np.float64) * scale
    inside = np.abs(v / scale) < 127
    assert np.all(np.abs(back - v)[inside] <= (scale / 2 * (1 + 1e-6) + 1e-12).repeat(50, 0)[inside])
    assert np.all(q[v / scale > 128] == 127) and np.all(q[v / scale < -129] == -128)


def test_dynamic_quant_properties():
    rng = np.random.default_rng(7)
    c = oracle.round_bf16(rng.standard_normal((6, 40)))
    smooth = rng.uniform(0.5, 1.5, (1, 40)).astype(np.float32)
    codes, scale = oracle.dynamic_quant_per_token(c, smooth)
    s = c * smooth.astype(np.float64)
    amax_pos = np.argmax(np.abs(s), axis=-1)
    for t in range(6):
        assert abs(int(codes[t, amax_pos[t]])) == 127
        assert np.sign(codes[t, amax_pos[t]]) == np.sign(s[t, amax_pos[t]])
        np.testing.assert_allclose(scale[t], np.max(np.abs(s[t])) / 127, rtol=1e-6)
        assert np.all(np.abs(codes[t] * np.float64(scale[t]) - s[t]) <= scale[t] * 0.5001 + 1e-7)
    # an all-zero row quantises to zeros with zero scale
    codes0, scale0 = oracle.dynamic_quant_per_token(np.zeros((1, 40)), smooth)
    assert scale0[0] == 0 and not codes0.any()


# ----------------------------------------------------------------------------- MLA prolog

def _tiny_mla(rng, int8=False, int8_cache=False, T=3, He=8, Hcq=6, Hckv=5, N=2, D=4, Dr=4,
              full=False, xnorm=None):
    bfr = lambda *s: oracle.round_bf16(rng.standard_normal(s) * 0.5)
    inp = dict(
        token_x=bfr(T, He), weight_dq=bfr(He, Hcq), weight_uk=bfr(N, D, Hckv),
        weight_dkv_kr=bfr(He, Hckv + Dr),
        rmsnorm_gamma_cq=oracle.round_bf16(rng.uniform(0.5, 1.5, Hcq)),
        rmsnorm_gamma_ckv=oracle.round_bf16(rng.uniform(0.5, 1.5, Hckv)),
        rope_sin=bfr(T, Dr), rope_cos=bfr(T, Dr),
        cache_index=np.array([3, -1, 4][:T], np.int64),
        rmsnorm_epsilon_cq=1e-6, rmsnorm_epsilon_ckv=1e-5,
    )
    if int8:
        inp["weight_uq_qr"] = rng.integers(-127, 128, (Hcq, N * (D + Dr))).astype(np.int8)
        inp["dequant_scale_w_uq_qr"] = rng.uniform(1e-3, 1e-2, (1, N * (D + Dr))).astype(np.float32)
        inp["smooth_scales_cq"] = rng.uniform(0.5, 1.5, (1, Hcq)).astype(np.float32)
    else:
        inp["weight_uq_qr"] = bfr(Hcq, N * (D + Dr))
    if full:   # full quant: int8 x and down-projection weights with their dequant scales
        i8 = lambda *s: rng.integers(-127, 128, s).astype(np.int8)
        inp["token_x"], inp["weight_dq"], inp["weight_dkv_kr"] = i8(T, He), i8(He, Hcq), i8(He, Hckv + Dr)
        inp["dequant_scale_x"] = rng.uniform(2e-3, 8e-3, (T, 1)).astype(np.float32)
        inp["dequant_scale_w_dq"] = rng.uniform(2e-3, 8e-3, (1, Hcq)).astype(np.float32)
        inp["dequant_scale_w_dkv_kr"] = rng.uniform(2e-3, 8e-3, (1, Hckv + Dr)).astype(np.float32)
    if int8_cache:
        inp["kv_cache"] = rng.integers(-128, 128, (3, 2, 1, Hckv)).astype(np.int8)
        inp["quant_scale_ckv"] = rng.uniform(0.01, 0.05, (1, Hckv)).astype(np.float32)
        if full:   # full quant keeps kr_cache bf16 and query becomes int8
            inp["kr_cache"] = bfr(3, 2, 1, Dr)
            inp["query_int8"] = True
        else:
            inp["kr_cache"] = rng.integers(-128, 128, (3, 2, 1, Dr)).astype(np.int8)
            inp["quant_scale_ckr"] = rng.uniform(0.01, 0.05, (1, Dr)).astype(np.float32)
    else:
        inp["kv_cache"] = bfr(3, 2, 1, Hckv)
        inp["kr_cache"] = bfr(3, 2, 1, Dr)
    if xnorm is not None:   # input RmsNormQuant: "channel" deqScale per He channel, else one value
        inp["rms_norm_quant_gamma"] = oracle.round_bf16(rng.uniform(0.5, 1.5, He))
        inp["rms_norm_quant_bias"] = oracle.round_bf16(rng.uniform(-0.5, 0.5, He))
        inp["rms_norm_quant_deq_scale"] = (rng.uniform(0.5, 2.0, He if xnorm == "channel" else 1)
                                           .astype(np.float32))
        inp["rms_norm_quant_epsilon"] = 1e-4
    return inp


def _brute(inp):
    L = lambda a: (np.asarray(a).astype(int).tolist() if np.asarray(a).dtype == np.int8
                   else np.asarray(a).tolist())
    f = lambda a: None if a is None else np.asarray(a, np.float64).reshape(-1).tolist()
    wuq = np.asarray(inp["weight_uq_qr"])
    wuq = wuq.astype(int).tolist() if wuq.dtype == np.int8 else wuq.tolist()
    kv = np.asarray(inp["kv_cache"])
    kr = np.asarray(inp["kr_cache"])
    return bf.mla_prolog_bruteforce(
        L(inp["token_x"]), L(inp["weight_dq"]), wuq, L(inp["weight_uk"]),
        L(inp["weight_dkv_kr"]), L(inp["rmsnorm_gamma_cq"]), L(inp["rmsnorm_gamma_ckv"]),
        L(inp["rope_sin"]), L(inp["rope_cos"]), L(inp["cache_index"]),
        kv.astype(int).tolist() if kv.dtype == np.int8 else kv.tolist(),
        kr.astype(int).tolist() if kr.dtype == np.int8 else kr.tolist(),
        inp["rmsnorm_epsilon_cq"], inp["rmsnorm_epsilon_ckv"],
        dqw=f(inp.get("dequant_scale_w_uq_qr")), smooth=f(inp.get("smooth_scales_cq")),
        qs_ckv=f(inp.get("quant_scale_ckv")), qs_ckr=f(inp.get("quant_scale_ckr")),
        dsx=f(inp.get("dequant_scale_x")), dsw_dq=f(inp.get("dequant_scale_w_dq")),
        dsw_dkv=f(inp.get("dequant_scale_w_dkv_kr")), query_int8=inp.get("query_int8", False),
        xg=f(inp.get("rms_norm_quant_gamma")), xb=f(inp.get("rms_norm_quant_bias")),
        xd=f(inp.get("rms_norm_quant_deq_scale")), eps_x=inp.get("rms_norm_quant_epsilon"))


@pytest.mark.parametrize("int8,int8_cache,full,xnorm", [
    (False, False, False, None), (True, False, False, None), (True, True, False, None),
    (True, False, True, None), (True, True, True, None), (False, False, False, "channel"),
    (True, True, False, "tensor")])
def test_mla_prolog_matches_brute_force(int8, int8_cache, full, xnorm):
    rng = np.random.default_rng(11 + int8 + 2 * int8_cache + 4 * full + 8 * (xnorm is not None))
    inp = _tiny_mla(rng, int8, int8_cache, full=full, xnorm=xnorm)
    got = oracle.mla_prolog(**inp)
    want = _brute(inp)
    for key in ("query", "query_rope"):
        if np.asarray(got[key]).dtype == np.int8:
            np.testing.assert_array_equal(got[key], np.array(want[key], np.int8))
        else:
            np.testing.assert_allclose(got[key], np.array(want[key]), rtol=1e-12, atol=1e-14)
    if inp.get("query_int8"):
        np.testing.assert_array_equal(got["dequant_scale_q_nope"],
                                      np.array(want["dequant_scale_q_nope"], np.float64))
    for key in ("kv_cache", "kr_cache"):
        if got[key].dtype == np.int8:
            np.testing.assert_array_equal(got[key], np.array(want[key], np.int8))
        else:
            np.testing.assert_allclose(got[key], np.array(want[key]), rtol=1e-12, atol=1e-14)


def test_mla_absorb_reassociates():
    # q^N = (c^Q W^UQ_n) W^UK_n = c^Q (W^UQ_n W^UK_n).  W^UQ is a signed selection matrix so
    # q^C is exact in bf16 and no intermediate rounding interferes.
    rng = np.random.default_rng(12)
    T, He, Hcq, Hckv, N, D, Dr = 4, 16, 12, 10, 3, 6, 4
    inp = _tiny_mla(rng, T=T, He=He, Hcq=Hcq, Hckv=Hckv, N=N, D=D, Dr=Dr)
    inp["cache_index"] = np.array([0, 1, 2, 3])
    w = np.zeros((Hcq, N * (D + Dr)))
    for col in range(N * (D + Dr)):
        w[rng.integers(Hcq), col] = rng.choice([-1.0, 1.0])
    inp["weight_uq_qr"] = w
    out = oracle.mla_prolog(**inp)
    c_q = out["c_q"]
    for n in range(N):
        w_n = w[:, n * (D + Dr): n * (D + Dr) + D]
        fused = c_q @ (w_n @ inp["weight_uk"][n])
        np.testing.assert_allclose(out["query"][:, n, :], oracle.round_bf16(fused), rtol=2 ** -8,
                                   atol=1e-30)
        # the rope part of head n comes from the D..D+Dr columns of the head's block
        w_r = w[:, n * (D + Dr) + D:(n + 1) * (D + Dr)]
        np.testing.assert_allclose(
            out["query_rope"][:, n, :],
            oracle.round_bf16(oracle.rope_half_and_half(c_q @ w_r, inp["rope_cos"],
                                                        inp["rope_sin"])), rtol=0, atol=0)


def test_mla_special_case_reduces_to_textbook():
    # N = 1, gamma = 1, cos = 1, sin = 0: the key path is a textbook GEMM + RmsNorm and the rope
    # outputs are plain matmuls of the fused weights' trailing columns.
    rng = np.random.default_rng(13)
    T, He, Hcq, Hckv, N, D, Dr = 5, 24, 16, 12, 1, 8, 6
    inp = _tiny_mla(rng, T=T, He=He, Hcq=Hcq, Hckv=Hckv, N=N, D=D, Dr=Dr)
    inp["rmsnorm_gamma_ckv"] = np.ones(Hckv)
    inp["rmsnorm_gamma_cq"] = np.ones(Hcq)
    inp["rope_cos"] = np.ones((T, Dr))
    inp["rope_sin"] = np.zeros((T, Dr))
    inp["rmsnorm_epsilon_ckv"] = 0.0
    inp["rmsnorm_epsilon_cq"] = 0.0
    inp["kv_cache"] = np.zeros((3, 2, 1, Hckv))
    inp["kr_cache"] = np.zeros((3, 2, 1, Dr))
    inp["cache_index"] = np.array([5, 0, 2, 1, 4])
    out = oracle.mla_prolog(**inp)
    x = inp["token_x"]
    h = np.einsum("tk,kn->tn", x, inp["weight_dkv_kr"])
    kv = h[:, :Hckv] / (np.linalg.norm(h[:, :Hckv], axis=-1, keepdims=True) / math.sqrt(Hckv))
    for t, i in enumerate([5, 0, 2, 1, 4]):
        np.testing.assert_allclose(out["kv_cache"][i // 2, i % 2, 0], oracle.round_bf16(kv[t]),
                                   rtol=2 ** -8)
        np.testing.assert_allclose(out["kr_cache"][i // 2, i % 2, 0],
                                   oracle.round_bf16(h[t, Hckv:]), rtol=2 ** -8)
    hq = np.einsum("tk,kn->tn", x, inp["weight_dq"])
    cq = oracle.round_bf16(hq / (np.linalg.norm(hq, axis=-1, keepdims=True) / math.sqrt(Hcq)))
    np.testing.assert_allclose(out["c_q"], cq, rtol=2 ** -7)
    np.testing.assert_allclose(out["query_rope"][:, 0, :],
                               oracle.round_bf16(out["c_q"] @ inp["weight_uq_qr"][:, D:]),
                               rtol=2 ** -7, atol=1e-12)


def test_cache_invariants():
    rng = np.random.default_rng(14)
    inp = _tiny_mla(rng, T=3)
    inp["kv_cache"] = oracle.round_bf16(rng.standard_normal((3, 2, 1, 5)))
    inp["kr_cache"] = oracle.round_bf16(rng.standard_normal((3, 2, 1, 4)))
    inp["cache_index"] = np.array([4, -1, 1])
    out = oracle.mla_prolog(**inp)
    named = {4: 0, 1: 2}
    for blk in range(3):
        for off in range(2):
            slot = blk * 2 + off
            for key in ("kv_cache", "kr_cache"):
                if slot in named:
                    continue
                # untouched slots are bit-identical to the prefill
                assert out[key][blk, off].tobytes() == inp[key][blk, off].tobytes()
    sub = mla_prolog_tokens(inp, [0, 2])
    for slot, t in named.items():
        k = [0, 2].index(t)
        np.testing.assert_array_equal(out["kv_cache"][slot // 2, slot % 2, 0], sub["kv_rows"][k])
        np.testing.assert_array_equal(out["kr_cache"][slot // 2, slot % 2, 0], sub["kr_rows"][k])


@pytest.mark.parametrize("kw", [dict(), dict(xnorm="channel"), dict(int8=True, int8_cache=True),
                                dict(int8=True, int8_cache=True, full=True)],
                         ids=["bf16", "rms_norm_quant", "partial_quant", "full_quant"])
def test_key_rows_agree_with_the_prolog(kw):
    # mla_key_rows (the key path alone, used for every cache slot of the large GPU workloads)
    # gives exactly the rows mla_prolog scatters
    rng = np.random.default_rng(16)
    inp = _tiny_mla(rng, T=3, **kw)
    inp["cache_index"] = np.array([0, 3, 5])
    out = oracle.mla_prolog(**inp)
    kv, kr = mla_key_rows(**inp, Hckv=inp["weight_uk"].shape[2],
                          kv_dtype_int8=np.asarray(inp["kv_cache"]).dtype == np.int8,
                          kr_dtype_int8=np.asarray(inp["kr_cache"]).dtype == np.int8)
    for t, slot in enumerate([0, 3, 5]):
        np.testing.assert_array_equal(out["kv_cache"][slot // 2, slot % 2, 0], kv[t])
        np.testing.assert_array_equal(out["kr_cache"][slot // 2, slot % 2, 0], kr[t])


def test_int8_matmul_is_exact_integer_product():
    # scale_t = 1-type check: the dequantised result divided by its scales is the integer product.
    rng = np.random.default_rng(15)
    inp = _tiny_mla(rng, int8=True, T=3, Hcq=6)
    out = oracle.mla_prolog(**inp)
    codes, scale = oracle.dynamic_quant_per_token(out["c_q"], inp["smooth_scales_cq"])
    acc = [[sum(int(codes[t, c]) * int(inp["weight_uq_qr"][c, j]) for c in range(6))
            for j in range(inp["weight_uq_qr"].shape[1])] for t in range(3)]
    N, D, Dr = 2, 4, 4
    u = np.array(acc) * scale[:, None].astype(np.float64) * inp["dequant_scale_w_uq_qr"].astype(np.float64)
    u = u.reshape(3, N, D + Dr)
    np.testing.assert_array_equal(
        out["query_rope"],
        oracle.round_bf16(oracle.rope_half_and_half(u[:, :, D:], inp["rope_cos"][:, None, :],
                                                    inp["rope_sin"][:, None, :])))


# ----------------------------------------------------------------------------- QKV entry

def _tiny_qkv(rng, quant, T=4, Nq=3, Nk=2, Nv=2, D=8, block_num=3, block_size=2):
    f16 = lambda *s: oracle.round_fp16(rng.standard_normal(s))
    inp = dict(qkv=f16(T, (Nq + Nk + Nv) * D), gamma_q=oracle.round_fp16(rng.uniform(.5, 1.5, D)),
               gamma_k=oracle.round_fp16(rng.uniform(.5, 1.5, D)), cos=f16(T, D), sin=f16(T, D),
               index=np.array([5, -1, 0, 2][:T]), epsilon=1e-6, Nq=Nq, Nk=Nk, Nv=Nv)
    if quant:
        inp["k_scale"] = rng.uniform(0.02, 0.1, (Nk, D)).astype(np.float32)
        inp["v_scale"] = rng.uniform(0.02, 0.1, (Nv, D)).astype(np.float32)
        if quant == "asym":
            inp["k_offset"] = rng.uniform(-8, 8, (Nk, D)).astype(np.float32)
            inp["v_offset"] = rng.uniform(-8, 8, (Nv, D)).astype(np.float32)
        inp["k_cache"] = rng.integers(-128, 128, (block_num, block_size, Nk, D)).astype(np.int8)
        inp["v_cache"] = rng.integers(-128, 128, (block_num, block_size, Nv, D)).astype(np.int8)
    else:
        inp["k_cache"] = f16(block_num, block_size, Nk, D)
        inp["v_cache"] = f16(block_num, block_size, Nv, D)
    return inp


def _qkv_brute(inp):
    L = lambda a: np.asarray(a).tolist()
    cache = lambda a: np.asarray(a).astype(int).tolist() if np.asarray(a).dtype == np.int8 else L(a)
    opt = lambda k: L(inp[k]) if inp.get(k) is not None else None
    return bf.qkv_bruteforce(L(inp["qkv"]), L(inp["gamma_q"]), L(inp["gamma_k"]), L(inp["cos"]),
                             L(inp["sin"]), L(inp["index"]), cache(inp["k_cache"]),
                             cache(inp["v_cache"]), inp["epsilon"], inp["Nq"], inp["Nk"],
                             inp["Nv"], ks=opt("k_scale"), vs=opt("v_scale"), ko=opt("k_offset"),
                             vo=opt("v_offset"))


@pytest.mark.parametrize("quant", [False, True, "asym"])
def test_qkv_matches_brute_force(quant):
    rng = np.random.default_rng(20 + (2 if quant == "asym" else int(quant)))
    inp = _tiny_qkv(rng, quant)
    got = oracle.qkv_rms_norm_rope_cache(**inp)
    want = _qkv_brute(inp)
    np.testing.assert_allclose(got["q_out"], np.array(want["q_out"]), rtol=1e-12, atol=1e-14)
    for key in ("q_before", "k_before", "v_before"):
        np.testing.assert_allclose(got[key], np.array(want[key]), rtol=1e-12, atol=1e-14)
    for key in ("k_cache", "v_cache"):
        if quant:
            np.testing.assert_array_equal(got[key], np.array(want[key], np.int8))
        else:
            np.testing.assert_allclose(got[key], np.array(want[key]), rtol=1e-12, atol=1e-14)


def test_qkv_split_positions():
    # SplitVD: q = first Nq heads, k = next Nk, v = last Nv.  Constant heads with distinct signed
    # values show which slice each output took: v is stored without normalisation.
    rng = np.random.default_rng(22)
    inp = _tiny_qkv(rng, quant=False, T=1)
    Nq, Nk, Nv, D = 3, 2, 2, 8
    vals = [1.0, 2.0, -3.0, -4.0, 5.0, 6.0, -7.0]
    inp["qkv"] = np.concatenate([np.full(D, v) for v in vals])[None, :]
    inp["cos"] = np.ones((1, D))
    inp["sin"] = np.zeros((1, D))
    inp["gamma_q"] = np.ones(D)
    inp["gamma_k"] = np.full(D, 2.0)
    inp["epsilon"] = 0.0
    inp["index"] = np.array([3])
    out = oracle.qkv_rms_norm_rope_cache(**inp)
    np.testing.assert_array_equal(out["q_out"][0], np.sign(np.array(vals[:Nq]))[:, None] * np.ones(D))
    np.testing.assert_array_equal(out["k_cache"][1, 1], 2 * np.sign(np.array(vals[Nq:Nq + Nk]))[:, None] * np.ones(D))
    np.testing.assert_array_equal(out["v_cache"][1, 1], np.array(vals[Nq + Nk:])[:, None] * np.ones(D))
    # the -1 / untouched slots keep their bytes
    assert out["k_cache"][0].tobytes() == inp["k_cache"][0].tobytes()


def test_qkv_asym_zero_offset_is_symmetric():
    # kRoPE / kScale + 0 is the symmetric rule
    rng = np.random.default_rng(23)
    inp = _tiny_qkv(rng, "asym")
    inp["k_offset"] = np.zeros_like(inp["k_offset"])
    inp["v_offset"] = np.zeros_like(inp["v_offset"])
    asym = oracle.qkv_rms_norm_rope_cache(**inp)
    sym = oracle.qkv_rms_norm_rope_cache(**{k: v for k, v in inp.items() if "offset" not in k})
    for key in ("k_cache", "v_cache", "k_rows", "v_rows"):
        np.testing.assert_array_equal(asym[key], sym[key])


def test_qkv_asym_integer_offset_shifts_codes():
    # With an integer offset o and no saturation, rne(x / s + o) = rne(x / s) + o: every code
    # moves by exactly o (checked away from the clamp by keeping |x / s| small).
    rng = np.random.default_rng(24)
    inp = _tiny_qkv(rng, "asym")
    Nk, Nv, D = inp["Nk"], inp["Nv"], 8
    inp["k_scale"] = np.full((Nk, D), 0.25, np.float32)
    inp["v_scale"] = np.full((Nv, D), 0.25, np.float32)
    inp["k_offset"] = rng.integers(-20, 21, (Nk, D)).astype(np.float32)
    inp["v_offset"] = rng.integers(-20, 21, (Nv, D)).astype(np.float32)
    asym = oracle.qkv_rms_norm_rope_cache(**inp)
    sym = oracle.qkv_rms_norm_rope_cache(**{k: v for k, v in inp.items() if "offset" not in k})
    assert np.abs(sym["k_rows"]).max() < 100 and np.abs(sym["v_rows"]).max() < 100
    np.testing.assert_array_equal(asym["k_rows"].astype(int),
                                  sym["k_rows"].astype(int) + inp["k_offset"].astype(int)[None])
    np.testing.assert_array_equal(asym["v_rows"].astype(int),
                                  sym["v_rows"].astype(int) + inp["v_offset"].astype(int)[None])


def test_qkv_asym_offset_saturates():
    rng = np.random.default_rng(25)
    inp = _tiny_qkv(rng, "asym")
    inp["k_offset"] = np.full_like(inp["k_offset"], 400.0)
    inp["v_offset"] = np.full_like(inp["v_offset"], -400.0)
    out = oracle.qkv_rms_norm_rope_cache(**inp)
    assert (out["k_rows"] == 127).all() and (out["v_rows"] == -128).all()


def test_qkv_before_quant_outputs():
    # vBeforeQuant is the split v slice itself; qBeforeQuant is qOut; kBeforeQuant is the k row
    # that the quantiser consumes, so requantising it reproduces the cache codes away from ties.
    rng = np.random.default_rng(26)
    inp = _tiny_qkv(rng, True)
    out = oracle.qkv_rms_norm_rope_cache(**inp)
    T, Nq, Nk, Nv, D = 4, inp["Nq"], inp["Nk"], inp["Nv"], 8
    x = np.asarray(inp["qkv"]).reshape(T, Nq + Nk + Nv, D)
    np.testing.assert_array_equal(out["v_before"], x[:, Nq + Nk:, :])
    np.testing.assert_array_equal(out["q_before"], out["q_out"])
    requant = np.clip(np.rint(out["k_before"] / np.asarray(inp["k_scale"], np.float64)[None]),
                      -128, 127)
    assert np.abs(requant - out["k_rows"]).max() <= 1


def test_full_quant_k_rope_is_linear_in_dequant_scale_x():
    # k^R = ROPE(x · W^KR) has no normalisation: doubling a token's dequant_scale_x doubles its
    # k^R row exactly (a power of two commutes with the bf16 rounding); c^KV, normalised, stays.
    rng = np.random.default_rng(40)
    inp = _tiny_mla(rng, True, False, full=True)
    inp["cache_index"] = np.array([0, 1, 2], np.int64)
    a = oracle.mla_prolog(**inp)
    inp2 = dict(inp)
    inp2["dequant_scale_x"] = inp["dequant_scale_x"] * np.array([[2.0], [1.0], [1.0]], np.float32)
    b = oracle.mla_prolog(**inp2)
    np.testing.assert_array_equal(b["kr_cache"][0, 0], 2 * a["kr_cache"][0, 0])
    np.testing.assert_array_equal(b["kr_cache"][0, 1], a["kr_cache"][0, 1])
    np.testing.assert_allclose(b["c_kv"][0], a["c_kv"][0], rtol=1e-3)   # up to eps


def test_full_quant_integer_products_are_exact():
    # with unit dequant scales the down-projection is the integer matrix product
    rng = np.random.default_rng(41)
    inp = _tiny_mla(rng, True, False, full=True)
    for k in ("dequant_scale_x", "dequant_scale_w_dq", "dequant_scale_w_dkv_kr"):
        inp[k] = np.ones_like(inp[k])
    out = oracle.mla_prolog(**inp)
    h = np.asarray(inp["token_x"]).astype(np.int64) @ np.asarray(inp["weight_dkv_kr"]).astype(np.int64)
    Hckv = 5
    want = oracle.rope_half_and_half(h[:, Hckv:].astype(np.float64),
                                     np.asarray(inp["rope_cos"], np.float64),
                                     np.asarray(inp["rope_sin"], np.float64))
    np.testing.assert_allclose(out["k_r"], want, rtol=1e-15)


def test_query_int8_per_token_head():
    # codes * scale reconstructs q^N within half a step, and the largest |q^N| of each (token,
    # head) maps to +-127
    rng = np.random.default_rng(42)
    inp = _tiny_mla(rng, True, True, full=True)
    out = oracle.mla_prolog(**inp)
    inp_f = dict(inp)
    inp_f["query_int8"] = False
    ref = oracle.mla_prolog(**inp_f)          # bf16 query of the same computation
    codes = out["query"].astype(np.float64)
    scale = out["dequant_scale_q_nope"].astype(np.float64)[..., None]
    assert (np.abs(codes).max(axis=-1) == 127).all()
    err = np.abs(codes * scale - ref["query"])
    assert (err <= 0.5 * scale * (1 + 1e-6) + np.abs(ref["query"]) * 2.0 ** -8).all()
