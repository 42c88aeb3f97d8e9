"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI and compare with
the oracle under the acceptance bars:

* float outputs (bf16 / fp16): |gpu - oracle| <= 1e-2*|oracle| + 1e-2*rms(oracle), elementwise;
* int8 outputs: within 1 LSB;
* cache slots that are not written (untouched, or index -1): bit-identical to their prefill.
"""
from __future__ import annotations

import numpy as np
import torch

import qkv_attention_prolog_gb300 as pkg

REL = 1e-2
RMS = 1e-2


def f64(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    return t.numpy() if t.dtype in (torch.int8, torch.int64) else t.to(torch.float64).numpy()


def assert_close(got, want, what, rel=REL, rms_frac=RMS):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    if want.size == 0:
        return
    rms = float(np.sqrt(np.mean(want * want)))
    err = np.abs(got - want)
    bad = ~(err <= rel * np.abs(want) + rms_frac * rms)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{bad.size} out of tolerance; first at {tuple(i)}: "
            f"gpu={got[tuple(i)]!r} oracle={want[tuple(i)]!r} rms={rms:.3g}")


def assert_int8_close(got, want, what, lsb=1):
    d = np.abs(np.asarray(got, np.int32) - np.asarray(want, np.int32))
    assert d.max(initial=0) <= lsb, f"{what}: int8 codes differ by up to {d.max()}"


def check_cache(got, prefill, want_rows, cache_index, what):
    """got/prefill: (BlockNum, BlockSize, N, H) torch tensors; want_rows: (T, N*H) oracle rows."""
    g = got.detach().cpu()
    p = prefill.detach().cpu()
    slots = g.shape[0] * g.shape[1]
    gflat = g.reshape(slots, -1)
    pflat = p.reshape(slots, -1)
    idx = np.asarray(cache_index).reshape(-1)
    written = np.zeros(slots, bool)
    valid = (idx >= 0) & (idx < slots)
    written[idx[valid]] = True
    # untouched slots: bit-identical
    untouched = torch.from_numpy(~written)
    assert torch.equal(gflat[untouched].view(torch.uint8) if g.dtype != torch.int8 else gflat[untouched],
                       pflat[untouched].view(torch.uint8) if p.dtype != torch.int8 else pflat[untouched]), \
        f"{what}: a slot not named by cache_index changed"
    rows_got = gflat[torch.from_numpy(idx[valid])]
    rows_want = np.asarray(want_rows).reshape(len(idx), -1)[valid]
    if g.dtype == torch.int8:
        assert_int8_close(rows_got.numpy(), rows_want, what)
    else:
        assert_close(f64(rows_got), rows_want, what)


def mla_device_tensors(cpu: dict, dims, device, bsh=False):
    t = {k: v.to(device) for k, v in cpu.items() if isinstance(v, torch.Tensor)}
    if bsh:
        shape = lambda *tail: (dims.B, dims.S) + tail
        for k in ("token_x", "rope_sin", "rope_cos"):
            t[k] = t[k].reshape(shape(t[k].shape[-1]))
        t["cache_index"] = t["cache_index"].reshape(dims.B, dims.S)
        t["query"] = torch.empty(shape(dims.N, dims.Hckv), dtype=torch.bfloat16, device=device)
        t["query_rope"] = torch.empty(shape(dims.N, dims.Dr), dtype=torch.bfloat16, device=device)
    else:
        t["query"] = torch.empty(dims.T, dims.N, dims.Hckv, dtype=torch.bfloat16, device=device)
        t["query_rope"] = torch.empty(dims.T, dims.N, dims.Dr, dtype=torch.bfloat16,
                                      device=device)
    # poison the outputs so unwritten elements show up
    t["query"].fill_(float("nan"))
    t["query_rope"].fill_(float("nan"))
    if query_int8(cpu):   # full quant with int8 kv_cache: int8 query per token and head
        t["query"] = torch.full(t["query"].shape, 99, dtype=torch.int8, device=device)
        t["dequant_scale_q_nope"] = torch.full((dims.T, dims.N, 1), float("nan"),
                                               dtype=torch.float32, device=device)
    return t


def query_int8(cpu: dict) -> bool:
    return cpu["token_x"].dtype == torch.int8 and cpu["kv_cache"].dtype == torch.int8


def run_mla(cpu: dict, dims, eps, device="cuda", bsh=False, prolog=None):
    t = mla_device_tensors(cpu, dims, device, bsh)
    if prolog is None:
        prolog = pkg.MlaProlog({k: t[k] for k in ("weight_dq", "weight_uq_qr", "weight_uk",
                                                  "weight_dkv_kr")}, dims.N, dims.D, dims.Dr)
    run_t = {k: v for k, v in t.items() if not k.startswith("weight_")}
    prolog.run(run_t, eps, eps, eps_x=cpu.get("rms_norm_quant_epsilon"))
    torch.cuda.synchronize()
    status = pkg.mlap_check_errors(prolog.ws)
    return t, prolog, status


def oracle_inputs(cpu: dict, eps: float) -> dict:
    inp = {k: f64(v) for k, v in cpu.items() if isinstance(v, torch.Tensor)}
    inp["rmsnorm_epsilon_cq"] = eps
    inp["rmsnorm_epsilon_ckv"] = eps
    inp["query_int8"] = query_int8(cpu)
    if "rms_norm_quant_gamma" in cpu:
        inp["rms_norm_quant_epsilon"] = cpu["rms_norm_quant_epsilon"]
    return inp


# ---- int8 c^Q (partial and full quant): where floating point decides an integer, several
# results are correct.  The dynamic quant of c^Q takes integer decisions from floating-point
# values: the bf16 rounding of c^Q (a stated rounding point) and rne(s / scale_t).  The kernels
# compute c^Q in fp32 (about 5e-7 relative error from the fp32 accumulation of the
# down-projection), the oracle in fp64, so an element of c^Q that lies within that error of a
# bf16 rounding midpoint, or a quotient within it of a code midpoint, may be decided either way;
# each flipped code moves the token's whole q^C by one weight row times scale_t, which re-rounds
# part of q^C to bf16 and moves query by up to about 1 % of its rms.  For a token whose row misses
# the tolerance against the oracle, the oracle is evaluated again for every combination of the
# token's ambiguous decisions (found from the oracle's own fp64 values, with bands far wider than
# the kernels' error), and the token passes if one of them is met within the same tolerance.
DELTA_CQ = 1e-5      # relative band around a bf16 rounding midpoint of the unrounded c^Q
DELTA_CODE = 1e-4    # band, in code units, around a rounding midpoint of s / scale_t
MAX_AMBIGUOUS = 6


def _bf16_alternative(c: np.ndarray, c_bf: np.ndarray):
    """For each value of c (fp64), the other bf16 neighbour when c lies within DELTA_CQ of the
    rounding midpoint between its two bf16 neighbours, else nan."""
    c = np.asarray(c, np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        e = np.frexp(np.abs(c))[1] - 1
        ulp = np.ldexp(1.0, e - 7)
        lower = np.floor(np.abs(c) / ulp) * ulp
        mid = lower + ulp / 2
        near = np.abs(np.abs(c) - mid) <= DELTA_CQ * np.abs(c)
        other = np.where(np.abs(c_bf) == lower, lower + ulp, lower) * np.sign(c)
    return np.where(near & (c != 0), other, np.nan)


def _code_candidates(s: np.ndarray, scale: float, lo=-127, hi=127):
    """Candidate codes of each element: rne(s / scale), and the neighbour when the quotient lies
    within DELTA_CODE of a rounding midpoint."""
    if scale == 0:
        return [[0] for _ in s]
    q = s / scale
    out = []
    for v in q:
        r = int(np.clip(np.rint(v), lo, hi))
        cand = {r}
        f = v - np.floor(v)
        if abs(f - 0.5) <= DELTA_CODE:
            cand.add(int(np.clip(np.floor(v), lo, hi)))
            cand.add(int(np.clip(np.floor(v) + 1, lo, hi)))
        out.append(sorted(cand))
    return out


def int8_token_variants(ref: dict, inp: dict, t: int):
    """Oracle results of token t for every combination of its ambiguous c^Q decisions: a list of
    (query (N, Hckv), query_rope (N, Dr), dequant_scale_q_nope (N) or None), or None when the
    token has more than MAX_AMBIGUOUS ambiguous decisions."""
    from oracle.mla_prolog import dynamic_quant_per_token, query_outputs, up_projection_int8
    import itertools
    smooth = np.asarray(inp["smooth_scales_cq"], np.float64).reshape(-1)
    c_exact = np.asarray(ref["c_q_exact"][t], np.float64)
    c_bf = np.asarray(ref["c_q"][t], np.float64)
    alt = _bf16_alternative(c_exact, c_bf)
    # the scale follows the largest |c^Q * smooth|: an ambiguous rounding there changes it
    s0 = np.abs(c_bf * smooth)
    bases = [c_bf]
    i_max = int(np.argmax(s0))
    if not np.isnan(alt[i_max]):
        c2 = c_bf.copy()
        c2[i_max] = alt[i_max]
        bases.append(c2)
    Dr = np.asarray(inp["rope_sin"]).shape[-1]
    cos = np.asarray(inp["rope_cos"], np.float64).reshape(-1, Dr)[t:t + 1]
    sin = np.asarray(inp["rope_sin"], np.float64).reshape(-1, Dr)[t:t + 1]
    variants = []
    for cb in bases:
        codes0, scale = dynamic_quant_per_token(cb[None, :], smooth)
        sc = float(scale[0])
        cands = _code_candidates(cb * smooth, sc)
        for i in np.nonzero(~np.isnan(alt))[0]:     # the other rounding of an ambiguous c^Q
            if i == i_max:
                continue
            for c in _code_candidates(np.array([alt[i] * smooth[i]]), sc)[0]:
                if c not in cands[i]:
                    cands[i] = sorted(set(cands[i]) | {c})
        amb = [i for i, c in enumerate(cands) if len(c) > 1]
        if len(amb) > MAX_AMBIGUOUS:
            return None
        for choice in itertools.product(*[cands[i] for i in amb]):
            codes = codes0.copy()
            for i, c in zip(amb, choice):
                codes[0, i] = c
            u = up_projection_int8(codes, scale, inp["weight_uq_qr"], inp["dequant_scale_w_uq_qr"])
            q, qr, sq = query_outputs(u, inp["weight_uk"], cos, sin, Dr,
                                      bool(inp.get("query_int8", False)))
            variants.append((q[0], qr[0], None if sq is None else sq[0]))
    return variants


def _rows_close(got, want, rms, rel=REL, rms_frac=RMS):
    return bool(np.all(np.abs(got - want) <= rel * np.abs(want) + rms_frac * rms))


def check_int8_query(t_gpu: dict, ref: dict, inp: dict, dims, what=""):
    """query / query_rope (and with an int8 query its codes and scales) of the int8-c^Q paths:
    every token within the tolerance of the oracle, or of the oracle under one combination of
    that token's ambiguous integer decisions (see above)."""
    T, N, Hckv, Dr = dims.T, dims.N, dims.Hckv, dims.Dr
    int8_q = t_gpu["query"].dtype == torch.int8
    gq = f64(t_gpu["query"]).reshape(T, N, Hckv)
    gr = f64(t_gpu["query_rope"]).reshape(T, N, Dr)
    gs = f64(t_gpu["dequant_scale_q_nope"]).reshape(T, N) if int8_q else None
    wq, wr = np.asarray(ref["query"], np.float64), np.asarray(ref["query_rope"], np.float64)
    ws = np.asarray(ref["dequant_scale_q_nope"], np.float64) if int8_q else None
    rms_q = float(np.sqrt(np.mean(wq * wq)))
    rms_r = float(np.sqrt(np.mean(wr * wr)))
    rms_s = float(np.sqrt(np.mean(ws * ws))) if int8_q else 0.0

    def ok(t, q, r, s):
        good = _rows_close(gr[t], r, rms_r)
        if int8_q:
            good &= int(np.abs(gq[t] - q).max(initial=0)) <= 1 and _rows_close(gs[t], s, rms_s)
        else:
            good &= _rows_close(gq[t], q, rms_q)
        return good

    failed = []
    resolved = 0
    for t in range(T):
        if ok(t, wq[t], wr[t], None if ws is None else ws[t]):
            continue
        var = int8_token_variants(ref, inp, t)
        if var is not None and any(ok(t, *v) for v in var):
            resolved += 1
            continue
        failed.append((t, None if var is None else len(var)))
    assert not failed, (f"{what} query: tokens {failed[:8]} match neither the oracle nor any "
                        f"combination of their ambiguous c^Q decisions (token, variants)")
    return resolved
