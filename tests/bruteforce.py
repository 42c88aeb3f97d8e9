"""Scalar brute-force restatements used to pin the oracle on tiny inputs (test helper).

Written independently of ``oracle/``: plain Python floats and ints, one output element at a time,
and a rounding routine that works on the IEEE-754 bit pattern with integer arithmetic (the oracle
rounds through frexp/ldexp instead).  Valid only for tiny shapes and normal-range values.
"""
from __future__ import annotations

import math
import struct


def _bits(x: float) -> int:
    return struct.unpack("<Q", struct.pack("<d", x))[0]


def _float(b: int) -> float:
    return struct.unpack("<d", struct.pack("<Q", b))[0]


def rne_keep_bits(x: float, keep: int) -> float:
    """Round a normal float64 to ``keep`` explicit mantissa bits, ties to even, on its bit pattern."""
    if x == 0.0 or math.isinf(x) or math.isnan(x):
        return x
    drop = 52 - keep
    b = _bits(x)
    lsb = (b >> drop) & 1
    b += (1 << (drop - 1)) - 1 + lsb
    b &= ~((1 << drop) - 1)
    return _float(b)


def bf16(x: float) -> float:
    return rne_keep_bits(x, 7)


def fp16(x: float) -> float:
    return rne_keep_bits(x, 10)


def int8_code(q: float, lo: int, hi: int) -> int:
    r = round(q)                    # Python rounds half to even
    return max(lo, min(hi, r))


def rope_element(y, cos, sin, j):
    d = len(y)
    h = d // 2
    partner = -y[j + h] if j < h else y[j - h]
    return y[j] * cos[j] + partner * sin[j]


def mla_prolog_bruteforce(x, wdq, wuq, wuk, wdkv, gcq, gckv, sin, cos, idx, kv_cache, kr_cache,
                          eps_cq, eps_ckv, dqw=None, smooth=None, qs_ckv=None, qs_ckr=None,
                          dsx=None, dsw_dq=None, dsw_dkv=None, query_int8=False, xg=None, xb=None,
                          xd=None, eps_x=None):
    """All arguments are nested Python lists.  Returns dict of nested lists.  Full quant: x, wdq,
    wdkv hold ints and dsx (T), dsw_dq (Hcq), dsw_dkv (Hckv+Dr) their dequant scales.  xg, xb,
    xd, eps_x: input RmsNormQuant gamma (He), bias (He), deqScale (He or one value), epsilon."""
    T, He = len(x), len(x[0])
    Hcq = len(wdq[0])
    N, D, Hckv = len(wuk), len(wuk[0]), len(wuk[0][0])
    Dr = len(sin[0])
    int8_w = isinstance(wuq[0][0], int)
    query = [[[0.0] * Hckv for _ in range(N)] for _ in range(T)]
    query_rope = [[[0.0] * Dr for _ in range(N)] for _ in range(T)]
    kv = [[[list(r) for r in row] for row in blk] for blk in kv_cache]
    kr = [[[list(r) for r in row] for row in blk] for blk in kr_cache]
    bs = len(kv_cache[0])
    scale_q = [[0.0] * N for _ in range(T)]
    for t in range(T):
        xt = x[t]
        if xg is not None:                    # (gamma*x/RMS(x) + bias) * deqScale, then bf16
            rms_x = math.sqrt(sum(v * v for v in xt) / He + eps_x)
            xt = [bf16((xg[k] * xt[k] / rms_x + xb[k]) * xd[k if len(xd) > 1 else 0])
                  for k in range(He)]
        hq = [sum(xt[k] * wdq[k][c] for k in range(He)) for c in range(Hcq)]
        if dsx is not None:                   # exact integer sums, dequantised
            hq = [hq[c] * dsx[t] * dsw_dq[c] for c in range(Hcq)]
        rms = math.sqrt(sum(v * v for v in hq) / Hcq + eps_cq)
        cq = [bf16(gcq[c] * hq[c] / rms) for c in range(Hcq)]
        if int8_w:
            s = [cq[c] * smooth[c] for c in range(Hcq)]
            amax = max(abs(v) for v in s)
            scale = amax / 127.0
            codes = [0 if scale == 0 else int8_code(v / scale, -127, 127) for v in s]
        for n in range(N):
            base = n * (D + Dr)
            u = []
            for jj in range(D + Dr):
                col = base + jj
                if int8_w:
                    acc = sum(codes[c] * wuq[c][col] for c in range(Hcq))
                    u.append(acc * scale * dqw[col])
                else:
                    u.append(sum(cq[c] * wuq[c][col] for c in range(Hcq)))
            qc = [bf16(v) for v in u[:D]]
            r = u[D:]
            qn = [sum(qc[d] * wuk[n][d][c2] for d in range(D)) for c2 in range(Hckv)]
            if query_int8:
                amax = max(abs(v) for v in qn)
                sc = amax / 127.0
                scale_q[t][n] = sc
                query[t][n] = [0 if sc == 0 else int8_code(v / sc, -127, 127) for v in qn]
            else:
                query[t][n] = [bf16(v) for v in qn]
            for j in range(Dr):
                query_rope[t][n][j] = bf16(rope_element(r, cos[t], sin[t], j))
        hkv = [sum(xt[k] * wdkv[k][c] for k in range(He)) for c in range(Hckv + Dr)]
        if dsx is not None:
            hkv = [hkv[c] * dsx[t] * dsw_dkv[c] for c in range(Hckv + Dr)]
        rms = math.sqrt(sum(v * v for v in hkv[:Hckv]) / Hckv + eps_ckv)
        ckv = [gckv[c] * hkv[c] / rms for c in range(Hckv)]
        kr_row = [rope_element(hkv[Hckv:], cos[t], sin[t], j) for j in range(Dr)]
        i = idx[t]
        if 0 <= i < len(kv_cache) * bs:
            if qs_ckv is not None:
                kv[i // bs][i % bs][0] = [int8_code(ckv[c] / qs_ckv[c], -128, 127)
                                          for c in range(Hckv)]
            else:
                kv[i // bs][i % bs][0] = [bf16(v) for v in ckv]
            if qs_ckr is not None:
                kr[i // bs][i % bs][0] = [int8_code(kr_row[j] / qs_ckr[j], -128, 127)
                                          for j in range(Dr)]
            else:
                kr[i // bs][i % bs][0] = [bf16(v) for v in kr_row]
    return {"query": query, "query_rope": query_rope, "kv_cache": kv, "kr_cache": kr,
            "dequant_scale_q_nope": scale_q}


def qkv_bruteforce(qkv, gq, gk, cos, sin, idx, k_cache, v_cache, eps, Nq, Nk, Nv, ks=None,
                   vs=None, ko=None, vo=None):
    """qkv: T rows of (Nq+Nk+Nv)*D floats."""
    T = len(qkv)
    D = len(qkv[0]) // (Nq + Nk + Nv)
    q_out = [[[0.0] * D for _ in range(Nq)] for _ in range(T)]
    k_before = [[[0.0] * D for _ in range(Nk)] for _ in range(T)]
    v_before = [[[0.0] * D for _ in range(Nv)] for _ in range(T)]
    kc = [[[list(r) for r in row] for row in blk] for blk in k_cache]
    vc = [[[list(r) for r in row] for row in blk] for blk in v_cache]
    bs = len(k_cache[0])
    for t in range(T):
        heads = [qkv[t][h * D:(h + 1) * D] for h in range(Nq + Nk + Nv)]
        k_rows, v_rows = [], []
        for h in range(Nq + Nk):
            xh = heads[h]
            g = gq if h < Nq else gk
            rms = math.sqrt(sum(v * v for v in xh) / D + eps)
            y = [xh[j] / rms * g[j] for j in range(D)]
            e = [rope_element(y, cos[t], sin[t], j) for j in range(D)]
            if h < Nq:
                q_out[t][h] = [fp16(v) for v in e]
            else:
                hk = h - Nq
                k_before[t][hk] = [fp16(v) for v in e]
                if ks is not None:
                    off = [0.0] * D if ko is None else ko[hk]
                    k_rows.append([int8_code(e[j] / ks[hk][j] + off[j], -128, 127)
                                   for j in range(D)])
                else:
                    k_rows.append([fp16(v) for v in e])
        for hv in range(Nv):
            vh = heads[Nq + Nk + hv]
            v_before[t][hv] = [fp16(v) for v in vh]
            if vs is not None:
                off = [0.0] * D if vo is None else vo[hv]
                v_rows.append([int8_code(vh[j] / vs[hv][j] + off[j], -128, 127)
                               for j in range(D)])
            else:
                v_rows.append([fp16(v) for v in vh])
        i = idx[t]
        if 0 <= i < len(k_cache) * bs:
            kc[i // bs][i % bs] = k_rows
            vc[i // bs][i % bs] = v_rows
    return {"q_out": q_out, "k_cache": kc, "v_cache": vc, "q_before": q_out,
            "k_before": k_before, "v_before": v_before}
