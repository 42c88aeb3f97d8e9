"""Throughput of the MLA prolog on GB300 (and of the CPU oracle as the reference arm).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode|prefill|tiny|partial_quant|qkv]

One step = one full prolog call (down-projection, RmsNorm/RoPE/scatter, up-projection with query
RoPE, per-head absorb) over one batch of seeded synthetic inputs.  The default workload is the
bf16 decode configuration (T=128 tokens, He=7168, Hcq=1536, Hckv=512, N=128, D=128, Dr=64).

`value` is device-timed whole-job throughput (tokens/s over all ranks) with inputs resident in
HBM: K steps replayed from a CUDA graph of the C-ABI execute call, rotating over enough input sets
(weights, activations, caches) that each step's working set has left L2 by the time it recurs.
`e2e` is the same metric through the C-ABI call from pinned host buffers, host<->device copies of
the step's inputs and outputs inside the timed region.  Multi-GPU runs are independent replicas
(the prolog shards by tokens with no exchange step): one process per GPU, max time over ranks.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA-prolog µs/call & tokens/s; % of HBM (decode) / tensor (prefill) roofline"
UNIT = "tokens/s"
L2_BYTES = 129 * 1024 * 1024


def _parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode",
                    choices=["decode", "prefill", "tiny", "partial_quant", "full_quant", "xnorm",
                             "qkv", "qkv_asym"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--timer-calls", type=int, default=200,
                    help="calls timed kernel by kernel for the roofline entry")
    return ap.parse_args()


def _case(name):
    import synthetic
    return {"decode": synthetic.MLA_DECODE, "prefill": synthetic.MLA_PREFILL,
            "tiny": synthetic.MLA_TINY, "partial_quant": synthetic.MLA_PARTIAL_QUANT,
            "full_quant": synthetic.MLA_FULL_QUANT, "xnorm": synthetic.MLA_XNORM,
            "qkv": synthetic.QKV_EPILOGUE, "qkv_asym": synthetic.QKV_EPILOGUE_ASYM}[name]


# ------------------------------------------------------------------------------- byte/flop model
def mla_model(d, w_int8=False, cache_int8=False, full=False, xnorm=False):
    """Algorithmic bytes and FLOPs per call and per kernel (each tensor read or written once).
    full: full quant (int8 x and down weights; int8 kv_cache -> bf16 kr_cache, int8 query).
    xnorm: the input RmsNormQuant, whose gamma, bias and deqScale (He each) are read once more
    (its normalised x is an intermediate, like the K-split partials, and is not counted)."""
    T, He, Hcq, Hckv, N, D, Dr = d.T, d.He, d.Hcq, d.Hckv, d.N, d.D, d.Dr
    wb = 1 if w_int8 else 2
    db = 1 if full else 2                       # x and the down-projection weights
    kvb = 1 if cache_int8 else 2
    krb = 1 if cache_int8 and not full else 2
    qb = 1 if cache_int8 and full else 2        # query
    tables = 2 * T * Dr * 2
    xparams = He * (2 + 2 + 4) if xnorm else 0
    k = {}
    k["down"] = {"bytes": He * (Hcq + Hckv + Dr) * db + T * He * db + xparams,
                 "flops": 2 * T * He * (Hcq + Hckv + Dr)}
    k["norm_scatter"] = {"bytes": T * Hcq * 2 + T * (Hckv * kvb + Dr * krb) + tables, "flops": 0}
    k["up"] = {"bytes": Hcq * N * (D + Dr) * wb + T * Hcq * 2 + T * N * D * 2 + T * N * Dr * 2
               + tables, "flops": 2 * T * Hcq * N * (D + Dr)}
    k["absorb"] = {"bytes": N * D * Hckv * 2 + T * N * D * 2 + T * N * Hckv * qb,
                   "flops": 2 * T * N * D * Hckv}
    path_bytes = (He * (Hcq + Hckv + Dr) * db + Hcq * N * (D + Dr) * wb + N * D * Hckv * 2
                  + T * He * db + T * N * Hckv * qb + T * N * Dr * 2 + T * (Hckv * kvb + Dr * krb)
                  + tables + T * 8 + xparams)
    path_flops = sum(v["flops"] for v in k.values())
    return k, path_bytes, path_flops


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p.get("bf16_tflops_sustained", p["bf16_tflops"]), \
            "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# Sources of each timed kernel: a recorded DRAM traffic figure stays valid while they are unchanged.
KERNEL_SOURCES = {
    "up_absorb": ["up_absorb.cu", "ptx.cuh"],
    "down": ["gemm_down.cu", "gemm.cuh", "epilogues.cuh", "gemm_launch.cuh", "ptx.cuh"],
    "up": ["gemm_up.cu", "gemm.cuh", "epilogues.cuh", "gemm_launch.cuh", "ptx.cuh"],
    "absorb": ["gemm_absorb.cu", "gemm.cuh", "epilogues.cuh", "gemm_launch.cuh", "ptx.cuh"],
    "norm_scatter": ["mla_norm_scatter.cu"],
    "qkv_rnrc": ["qkv_rnrc.cu"],
}


def kernel_source_hash(kernel_key):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "qkv_attention_prolog_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel_key]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def _ncu_traffic(kernel_key, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this kernel's
    current sources."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        ent = rec[workload][kernel_key]
    except Exception:
        return None
    if ent.get("sources") != kernel_source_hash(kernel_key):
        return None
    return ent.get("bytes")


# ------------------------------------------------------------------------------- clocks
class ClockSampler:
    def __init__(self, index=0):
        self.index = index
        self.proc = None

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.rows = []
        if self.proc is None:
            return False
        time.sleep(0.2)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        for row in csv.reader(io.StringIO(out)):
            if len(row) >= 9:
                self.rows.append([c.strip() for c in row])
        return False

    def summary(self):
        if not getattr(self, "rows", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4)
                          if r[5 + i].lower().startswith("active")})
        loaded = [s for s in sm if smax and s > 0.5 * max(smax)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(self.rows)}


# ------------------------------------------------------------------------------- distributed
def _dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    return rank, local, world


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------- oracle baseline
def oracle_tokens_per_s(case, budget_s=12.0, sample_tokens=4):
    """Time the oracle as it stands on a bounded token sample of the workload (host cores)."""
    import numpy as np
    import oracle
    import synthetic
    from oracle.mla_prolog import mla_prolog_tokens

    if isinstance(case, synthetic.QkvCase):
        cpu = synthetic.make_qkv_inputs(case)
        d = case.dims
        f = lambda t: t.to(__import__("torch").float64).numpy()
        ntok = min(d.T, 64)
        qkv = f(cpu["qkv"]).reshape(d.T, -1)[:ntok]
        args = (qkv, f(cpu["gamma_q"]), f(cpu["gamma_k"]), f(cpu["cos"])[:ntok],
                f(cpu["sin"])[:ntok], cpu["index"].numpy()[:ntok], cpu["k_cache"].numpy(),
                cpu["v_cache"].numpy(), case.eps, d.Nq, d.Nk, d.Nv, cpu["k_scale"].numpy(),
                cpu["v_scale"].numpy())
        kw = {}
        if case.quant == "asymmetric":
            kw = {"k_offset": cpu["k_offset"].numpy(), "v_offset": cpu["v_offset"].numpy()}
        call = lambda: oracle.qkv_rms_norm_rope_cache(*args, **kw)
        sample = f"{ntok} tokens of the {case.name} workload per oracle call"
    else:
        import torch
        cpu = synthetic.make_mla_inputs(case)
        inp = {k: (v.numpy() if v.dtype in (torch.int8, torch.int64) else
                   v.to(torch.float64).numpy()) for k, v in cpu.items()
               if isinstance(v, torch.Tensor)}
        inp["rmsnorm_epsilon_cq"] = case.eps
        inp["rmsnorm_epsilon_ckv"] = case.eps
        inp["query_int8"] = case.full_quant and case.cache_dtype == "int8"
        if case.x_norm is not None:
            inp["rms_norm_quant_epsilon"] = case.eps
        ntok = min(case.dims.T, sample_tokens)
        ids = np.arange(ntok)
        call = lambda: mla_prolog_tokens(inp, ids)
        sample = f"{ntok} tokens of the {case.name} workload per oracle call"
    t0 = time.perf_counter()
    calls = 0
    while True:
        call()
        calls += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    try:
        cores = len(os.sched_getaffinity(0))
    except Exception:
        cores = os.cpu_count()
    return calls * ntok / el, cores, f"{sample}; {calls} calls in {el:.1f} s"


# ------------------------------------------------------------------------------- our arm
def _mla_sets(case, dev, n_sets):
    import torch
    import synthetic
    import qkv_attention_prolog_gb300 as pkg
    cpu = synthetic.make_mla_inputs(case)
    d = case.dims
    sets = []
    for _ in range(n_sets):
        t = {k: v.to(dev) for k, v in cpu.items() if isinstance(v, torch.Tensor)}
        t["query"] = torch.empty(d.T, d.N, d.Hckv, dtype=torch.bfloat16, device=dev)
        t["query_rope"] = torch.empty(d.T, d.N, d.Dr, dtype=torch.bfloat16, device=dev)
        if case.full_quant and case.cache_dtype == "int8":   # int8 query per token and head
            t["query"] = torch.empty(d.T, d.N, d.Hckv, dtype=torch.int8, device=dev)
            t["dequant_scale_q_nope"] = torch.empty(d.T, d.N, 1, dtype=torch.float32, device=dev)
        packed = pkg.prepack_mla_weights({k: t.pop(k) for k in ("weight_dq", "weight_uq_qr",
                                                                "weight_uk", "weight_dkv_kr")},
                                         d.N, d.D, d.Dr)
        t.update(packed)
        a = pkg.make_mla_args(t, case.eps, case.eps, eps_x=case.eps)
        ws = torch.empty(pkg.mlap_get_workspace_size(a), dtype=torch.uint8, device=dev)
        pkg.mlap_workspace_init(ws)
        sets.append((t, a, ws))
    torch.cuda.synchronize()
    return cpu, sets


def run_ours(args, rank, local, world):
    import torch
    import qkv_attention_prolog_gb300 as pkg
    from qkv_attention_prolog_gb300 import build as _build

    _build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    case = _case(args.workload)
    is_qkv = args.workload.startswith("qkv")
    hbm, tf_burst, tf_sus, peak_kind = _peaks()

    if is_qkv:
        return run_qkv(args, case, dev, rank, world, hbm, peak_kind)

    d = case.dims
    w_int8 = case.weight_uq_qr_dtype == "int8"
    c_int8 = case.cache_dtype == "int8"
    kern, path_bytes, path_flops = mla_model(d, w_int8, c_int8, case.full_quant,
                                             case.x_norm is not None)
    # down, norm/scatter, up, absorb; full quant adds the token_x widening and, with an int8
    # query, its per-token-head quantisation; the input RmsNormQuant adds its own kernel
    launches_per_call = (4 + (1 + c_int8 if case.full_quant else 0)
                         + (1 if case.x_norm is not None else 0))
    n_sets = max(1, math.ceil(3 * L2_BYTES / path_bytes) + 1) if path_bytes < 2 * L2_BYTES else 1
    cpu, sets = _mla_sets(case, dev, n_sets)
    stream = torch.cuda.Stream(dev)

    steps = args.steps or {"decode": 40000, "tiny": 40000, "partial_quant": 40000,
                           "full_quant": 40000, "xnorm": 40000, "prefill": 1500}[args.workload]
    warm = max(3, args.warmup)
    with torch.cuda.stream(stream):
        for i in range(warm):
            t, a, ws = sets[i % n_sets]
            pkg.mlap_execute(a, ws, stream)
    stream.synchronize()

    # CUDA graph of `per_graph` consecutive steps over the rotating sets
    per_graph = n_sets * max(1, 64 // n_sets) if steps >= 64 else n_sets
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(per_graph):
            t, a, ws = sets[i % n_sets]
            pkg.mlap_execute(a, ws, torch.cuda.current_stream())
    replays = max(1, round(steps / per_graph))
    steps = replays * per_graph
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()

    _barrier(world)
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(replays):
                g.replay()
            ev1.record(stream)
        stream.synchronize()
    torch.cuda.synchronize()
    _barrier(world)
    ms_total = ev0.elapsed_time(ev1)
    ms_total = _max_over_ranks(ms_total, world)
    ms_step = ms_total / steps
    value = d.T * world * steps / (ms_total / 1e3)
    for s in sets:
        assert pkg.mlap_check_errors(s[2], stream) == 0, "kernel error during the timed region"

    # per-kernel durations (CUDA events around each launch on the execute stream)
    n_timed = max(2, args.timer_calls)
    timer = pkg.Timer(n_timed)
    with torch.cuda.stream(stream):
        for i in range(n_timed):
            t, a, ws = sets[i % n_sets]
            timer.execute(a, ws, stream)
    per = timer.read()
    timer.close()
    names = ["down", "norm_scatter", "up", "absorb"]
    per = per[min(10, len(per) // 2):]
    avg_ms = {n: statistics.mean(r[k] for r in per) for k, n in enumerate(names)}
    if avg_ms["absorb"] == 0.0:
        # the decode launch fuses the absorb into the up-projection (the timer's absorb phase is
        # empty): one kernel, whose algorithmic bytes are both weights, c^Q and both outputs
        avg_ms = {"down": avg_ms["down"], "norm_scatter": avg_ms["norm_scatter"],
                  "up_absorb": avg_ms["up"]}
        names = list(avg_ms)
        launches_per_call -= 1
        kern["up_absorb"] = {
            "bytes": kern["up"]["bytes"] + kern["absorb"]["bytes"] - 2 * d.T * d.N * d.D * 2,
            "flops": kern["up"]["flops"] + kern["absorb"]["flops"]}
    dominant = max(names, key=lambda n: avg_ms[n])
    tensor_bound = args.workload == "prefill"
    if tensor_bound:
        achieved = kern[dominant]["flops"] / (avg_ms[dominant] / 1e3) / 1e12
        peak = tf_sus
        roof = {"bound": "tensor", "unit": "TFLOP/s", "peak": peak}
    else:
        achieved = kern[dominant]["bytes"] / (avg_ms[dominant] / 1e3) / 1e9
        peak = hbm
        roof = {"bound": "hbm", "unit": "GB/s", "peak": peak}
    roof.update({"kernel": dominant, "achieved": round(achieved, 1),
                 "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                 "traffic": _ncu_traffic(dominant, args.workload),
                 "algorithmic_per_launch": kern[dominant]["bytes"] if not tensor_bound
                 else kern[dominant]["flops"],
                 "avg_launch_us": round(avg_ms[dominant] * 1e3, 3),
                 "per_kernel_us": {n: round(avg_ms[n] * 1e3, 3) for n in names}})
    path_time = max(path_bytes / (hbm * 1e9), path_flops / (tf_sus * 1e12))
    path_roof = {"bytes": path_bytes, "flops": path_flops,
                 "roofline_us": round(path_time * 1e6, 3),
                 "frac": round(path_time / (ms_step / 1e3), 4),
                 "bound": "tensor" if path_flops / (tf_sus * 1e12) > path_bytes / (hbm * 1e9)
                 else "hbm"}

    e2e = run_e2e(args, case, cpu, sets[0], dev, stream)

    line = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": steps, "warmup": warm, "ms_per_step": round(ms_step, 6),
            "us_per_call": round(ms_step * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; shapes and distributions of the workload recipe)",
            "config": {"workload": case.name, "T": d.T, "B": d.B, "S": d.S, "He": d.He,
                       "Hcq": d.Hcq, "Hckv": d.Hckv, "N": d.N, "D": d.D, "Dr": d.Dr,
                       "weight_uq_qr": case.weight_uq_qr_dtype, "caches": case.cache_dtype,
                       "token_x_and_down_weights": "int8" if case.full_quant else "bf16",
                       "input_rms_norm_quant": case.x_norm,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": (f"rotating {n_sets} input sets of {path_bytes/1e6:.1f} MB "
                              f"({n_sets*path_bytes/1e6:.0f} MB > 129 MB L2)" if n_sets > 1
                              else f"inputs {path_bytes/1e6:.0f} MB > 129 MB L2"),
                       "timing": f"CUDA graph of {per_graph} execute calls replayed {replays}x"},
            "roofline": roof, "path_roofline": path_roof, "clocks": clk.summary(),
            "e2e": e2e, "gpu_launches": launches_per_call * steps}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, sample = oracle_tokens_per_s(case)
        line["cpu_baseline"] = {"value": round(v, 3), "unit": UNIT, "cores": cores,
                                "kind": "oracle", "sample": sample}
    return line


def _blob(tensors, names, device, pinned=False):
    """One contiguous byte buffer holding `names` (256-byte aligned) and views of it shaped and
    typed like `tensors[name]`."""
    import torch
    offs, off = {}, 0
    for k in names:
        nb = tensors[k].numel() * tensors[k].element_size()
        offs[k] = (off, nb)
        off += (nb + 255) // 256 * 256
    blob = torch.empty(off, dtype=torch.uint8, device=device)
    if pinned:
        blob = blob.pin_memory()
    views = {k: blob[o:o + nb].view(tensors[k].dtype).view(tensors[k].shape)
             for k, (o, nb) in offs.items()}
    return blob, views


def run_e2e(args, case, cpu, s0, dev, stream):
    """Same metric through the C-ABI call with every step's inputs copied from pinned host memory
    and its outputs read back (host<->device copies inside the timed region).  The per-call inputs
    and the outputs each live in one contiguous buffer (one copy per direction per step), and two
    buffer sets let step i's read-back and step i+1's upload overlap step i+1's execute call on
    separate copy streams."""
    import torch
    import qkv_attention_prolog_gb300 as pkg
    t, _, ws = s0
    ins = ["token_x", "rope_sin", "rope_cos", "cache_index"]
    outs = [k for k in ("query", "query_rope", "dequant_scale_q_nope") if k in t]
    host_in, hv = _blob(t, ins, "cpu", pinned=True)
    for k in ins:
        hv[k].copy_(cpu[k].reshape(hv[k].shape))
    host_out, _ = _blob(t, outs, "cpu", pinned=True)
    sets = []
    for _ in range(2):
        din, iv = _blob(t, ins, dev)
        dout, ov = _blob(t, outs, dev)
        tt = dict(t)
        tt.update(iv)
        tt.update(ov)
        sets.append((din, dout, pkg.make_mla_args(tt, case.eps, case.eps, eps_x=case.eps)))
    h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event(enable_timing=False)
    in_ready = [ev(), ev()]
    exec_done = [ev(), ev()]
    out_read = [ev(), ev()]
    steps = max(3, args.e2e_steps)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    for i in range(3 + steps):
        b = i % 2
        din, dout, a = sets[b]
        if i == 3:
            torch.cuda.synchronize()
            e0.record(h2d)
        if i >= 2:
            h2d.wait_event(exec_done[b])        # the execute that read this input set is done
        with torch.cuda.stream(h2d):
            din.copy_(host_in, non_blocking=True)
            in_ready[b].record(h2d)
        stream.wait_event(in_ready[b])
        if i >= 2:
            stream.wait_event(out_read[b])      # this output set has been read back
        pkg.mlap_execute(a, ws, stream)
        exec_done[b].record(stream)
        d2h.wait_event(exec_done[b])
        with torch.cuda.stream(d2h):
            host_out.copy_(dout, non_blocking=True)
            out_read[b].record(d2h)
    e1.record(d2h)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return {"value": round(case.dims.T / (ms / 1e3), 1), "unit": UNIT,
            "h2d_bytes_per_step": host_in.numel(), "d2h_bytes_per_step": host_out.numel(),
            "ms_per_step": round(ms, 6),
            "copies": "one host-to-device and one device-to-host copy per step (packed "
                      "buffers), overlapped with the next step's execute on two copy streams"}


def run_qkv(args, case, dev, rank, world, hbm, peak_kind):
    import torch
    import synthetic
    import qkv_attention_prolog_gb300 as pkg
    d = case.dims
    cpu = synthetic.make_qkv_inputs(case)
    t = {k: v.to(dev) for k, v in cpu.items() if isinstance(v, torch.Tensor)}
    t["q_out"] = torch.empty(d.B, d.S, d.Nq, d.D, dtype=torch.float16, device=dev)
    t["cos"] = t["cos"].reshape(d.B, d.S, d.D)
    t["sin"] = t["sin"].reshape(d.B, d.S, d.D)
    t["index"] = t["index"].reshape(d.B, d.S)
    if case.before_quant:
        for name, n in (("q_before_quant", d.Nq), ("k_before_quant", d.Nk), ("v_before_quant", d.Nv)):
            t[name] = torch.empty(d.B, d.S, n, d.D, dtype=torch.float16, device=dev)
    a = pkg.make_qkv_args(t, d.Nq, d.Nk, d.Nv, case.eps)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)
    nb = (d.T * (d.Nq + d.Nk + d.Nv) * d.D * 2 + d.T * d.Nq * d.D * 2
          + d.T * (d.Nk + d.Nv) * d.D + 2 * d.T * d.D * 2 + d.T * 8)
    if case.before_quant:        # the three dense before-quant outputs
        nb += d.T * (d.Nq + d.Nk + d.Nv) * d.D * 2
    steps = args.steps or 2000
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            pkg.qkvrnrc_execute(a, ws, stream)
        g = torch.cuda.CUDAGraph()
        stream.synchronize()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(10):
            pkg.qkvrnrc_execute(a, ws, torch.cuda.current_stream())
    replays = max(1, steps // 10)
    steps = replays * 10
    for _ in range(2):          # the first replays upload the graph
        g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(replays):
                g.replay()
            e1.record(stream)
        stream.synchronize()
    ms = _max_over_ranks(e0.elapsed_time(e1), world) / steps
    achieved = nb / (ms / 1e3) / 1e9
    e2e = run_qkv_e2e(args, case, cpu, t, d, dev, stream)
    return {"metric": METRIC, "value": round(d.T * world / (ms / 1e3), 1), "unit": UNIT,
            "n_gpus": world, "steps": steps, "warmup": args.warmup, "ms_per_step": round(ms, 6),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp16",
            "data": "synthetic", "config": {"workload": case.name, "B": d.B, "S": d.S,
                                            "Nq": d.Nq, "Nk": d.Nk, "Nv": d.Nv, "D": d.D,
                                            "quant": case.quant,
                                            "before_quant_outputs": case.before_quant,
                                            "l2": f"inputs {nb/1e6:.0f} MB > 129 MB L2"},
            "roofline": {"bound": "hbm", "kernel": "qkv_rnrc", "achieved": round(achieved, 1),
                         "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                         "peak_kind": peak_kind, "traffic": _ncu_traffic("qkv_rnrc", args.workload)},
            "clocks": clk.summary(), "e2e": e2e, "gpu_launches": steps}


def run_qkv_e2e(args, case, cpu, t, d, dev, stream):
    """The QKV entry end to end: qkv, cos, sin and index uploaded from pinned host memory and q_out
    (and the before-quant outputs) read back every step, packed and overlapped as run_e2e; the
    caches stay on the device (they are the operator's state)."""
    import torch
    import qkv_attention_prolog_gb300 as pkg
    ins = ["qkv", "cos", "sin", "index"]
    outs = [k for k in ("q_out", "q_before_quant", "k_before_quant", "v_before_quant") if k in t]
    host_in, hv = _blob(t, ins, "cpu", pinned=True)
    for k in ins:
        hv[k].copy_(cpu[k].reshape(hv[k].shape))
    host_out, _ = _blob(t, outs, "cpu", pinned=True)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    sets = []
    for _ in range(2):
        din, iv = _blob(t, ins, dev)
        dout, ov = _blob(t, outs, dev)
        tt = dict(t)
        tt.update(iv)
        tt.update(ov)
        sets.append((din, dout, pkg.make_qkv_args(tt, d.Nq, d.Nk, d.Nv, case.eps)))
    h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_ready = [torch.cuda.Event(), torch.cuda.Event()]
    exec_done = [torch.cuda.Event(), torch.cuda.Event()]
    out_read = [torch.cuda.Event(), torch.cuda.Event()]
    steps = max(3, args.e2e_steps)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    for i in range(3 + steps):
        b = i % 2
        din, dout, a = sets[b]
        if i == 3:
            torch.cuda.synchronize()
            e0.record(h2d)
        if i >= 2:
            h2d.wait_event(exec_done[b])
        with torch.cuda.stream(h2d):
            din.copy_(host_in, non_blocking=True)
            in_ready[b].record(h2d)
        stream.wait_event(in_ready[b])
        if i >= 2:
            stream.wait_event(out_read[b])
        pkg.qkvrnrc_execute(a, ws, stream)
        exec_done[b].record(stream)
        d2h.wait_event(exec_done[b])
        with torch.cuda.stream(d2h):
            host_out.copy_(dout, non_blocking=True)
            out_read[b].record(d2h)
    e1.record(d2h)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return {"value": round(d.T / (ms / 1e3), 1), "unit": UNIT,
            "h2d_bytes_per_step": host_in.numel(), "d2h_bytes_per_step": host_out.numel(),
            "ms_per_step": round(ms, 6),
            "copies": "one host-to-device and one device-to-host copy per step (packed "
                      "buffers), overlapped with the next step's execute on two copy streams"}


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle as it stands, timed on this host's cores."""
    if rank != 0:
        return None
    case = _case(args.workload)
    steps = args.steps or 3
    warm = max(0, min(args.warmup, 1))
    import synthetic
    per_step_budget = 5.0
    vals = []
    for i in range(warm + steps):
        v, cores, sample = oracle_tokens_per_s(case, budget_s=per_step_budget)
        if i >= warm:
            vals.append(v)
    v = statistics.mean(vals)
    cfg = {"workload": case.name}
    return {"impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": UNIT,
            "n_gpus": world, "steps": steps, "warmup": warm,
            "ms_per_step": round(per_step_budget * 1e3, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": cfg,
            "cpu_baseline": {"value": round(v, 3), "unit": UNIT, "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = _parse()
    rank, local, world = _dist_setup(args.gpus)
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, local, world)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
