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
