"""Throughput of the MLA prolog on GB300 (and of the CPU oracle as the reference arm).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode|prefill|tiny|partial_quant|full_quant|xnorm|qkv|qkv_asym]

One step = one full prolog call (down-projection, RmsNorm/RoPE/scatter, up-projection with query
RoPE, per-head absorb) over one batch of seeded synthetic inputs.  The default workload is the
bf16 decode configuration (T=128 tokens, He=7168, Hcq=1536, Hckv=512, N=128, D=128, Dr=64); the
same run also measures the bf16 prefill configuration (T=8192) and reports it in a `prefill`
object of the same line.

`value` is device-timed whole-job throughput (tokens/s over all ranks) with inputs resident in
HBM: K steps replayed from a CUDA graph of the C-ABI execute call, rotating over enough input sets
(weights, activations, caches) that each step's working set has left L2 by the time it recurs.
Per-kernel times come from %globaltimer stamps the kernels write inside the same pipelined calls
(mlap_execute_stamped), not from events between launches.  `e2e` is the same metric through the
C-ABI call from pinned host buffers, host<->device copies of the step's inputs and outputs inside
the timed region.  Multi-GPU runs are independent replicas (the prolog shards by tokens with no
exchange step): one process per GPU (torchrun, or spawned here when --gpus N > 1 is given without
a launcher), max time over ranks.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import re
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
    ap.add_argument("--stamp-calls", type=int, default=64,
                    help="pipelined calls whose kernels record execution stamps (per-kernel times)")
    ap.add_argument("--no-prefill", action="store_true",
                    help="skip the prefill measurement that the default decode run adds")
    ap.add_argument("--prefill-steps", type=int, default=60)
    ap.add_argument("--oracle-full-call", action="store_true",
                    help="also time one oracle call over the whole workload (host cores)")
    ap.add_argument("--oracle-worker", default=None, help=argparse.SUPPRESS)
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
KERNEL_SOURCES = {   # (api.cu sets each MLA kernel's grid, schedule and unit order)
    "up_absorb": ["up_absorb.cu", "ptx.cuh", "api.cu"],
    "down": ["gemm_down.cu", "gemm.cuh", "epilogues.cuh", "gemm_launch.cuh", "ptx.cuh", "api.cu"],
    "up": ["gemm_up.cu", "gemm.cuh", "epilogues.cuh", "gemm_launch.cuh", "ptx.cuh", "api.cu"],
    "absorb": ["gemm_absorb.cu", "gemm.cuh", "epilogues.cuh", "gemm_launch.cuh", "ptx.cuh",
               "api.cu"],
    "norm_scatter": ["mla_norm_scatter.cu", "api.cu"],
    "qkv_rnrc": ["qkv_rnrc.cu"],
}


_COMMENT = re.compile(r"//[^\n]*|/\*.*?\*/", re.S)


def code_only(text):
    """A C++/CUDA source without its comments, trailing spaces and blank lines: what the compiler
    sees, so that editing a comment leaves a recorded traffic figure valid."""
    body = _COMMENT.sub("", text)
    return "\n".join(line.rstrip() for line in body.splitlines() if line.strip())


def kernel_source_hash(kernel_key):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "qkv_attention_prolog_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel_key]:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode() + code_only(fh.read()).encode())
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
    """Rank, local rank and world size.  Under a launcher (WORLD_SIZE set) the world must match
    --gpus; the ranks meet over gloo (host-side barrier and max-over-ranks only: the replicas
    exchange no data)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if "WORLD_SIZE" in os.environ and n_gpus not in (None, world):
        raise SystemExit(f"bench.py: --gpus {n_gpus} but WORLD_SIZE={world}")
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
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


def _spawned_rank(rank, world, port, argv):
    """One replica started by `--gpus N` without a launcher (torch.multiprocessing, spawn)."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
    sys.argv = [sys.argv[0]] + list(argv)
    main()


def _spawn_replicas(n, argv):
    import socket
    import torch.multiprocessing as mp
    sock = socket.socket()
    sock.bind(("127.0.0.1", 0))
    port = sock.getsockname()[1]
    sock.close()
    mp.start_processes(_spawned_rank, args=(n, port, argv), nprocs=n, join=True,
                       start_method="spawn")


# ------------------------------------------------------------------------------- oracle baseline
def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def _oracle_call(case, sample_tokens, offset=0):
    """A closure running the oracle as it stands on `sample_tokens` tokens of the workload
    (tokens are independent), and a description of the sample."""
    import numpy as np
    import oracle
    import synthetic
    from oracle.mla_prolog import mla_prolog_tokens

    if isinstance(case, synthetic.QkvCase):
        import torch
        cpu = synthetic.make_qkv_inputs(case)
        d = case.dims
        f = lambda t: t.to(torch.float64).numpy()
        ntok = min(d.T, sample_tokens)
        ids = (offset + np.arange(ntok)) % d.T
        qkv = f(cpu["qkv"]).reshape(d.T, -1)[ids]
        args = (qkv, f(cpu["gamma_q"]), f(cpu["gamma_k"]), f(cpu["cos"]).reshape(d.T, -1)[ids],
                f(cpu["sin"]).reshape(d.T, -1)[ids], cpu["index"].numpy().reshape(-1)[ids],
                cpu["k_cache"].numpy(), cpu["v_cache"].numpy(), case.eps, d.Nq, d.Nk, d.Nv,
                cpu["k_scale"].numpy(), cpu["v_scale"].numpy())
        kw = {}
        if case.quant == "asymmetric":
            kw = {"k_offset": cpu["k_offset"].numpy(), "v_offset": cpu["v_offset"].numpy()}
        return (lambda: oracle.qkv_rms_norm_rope_cache(*args, **kw)), ntok
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
    ids = (offset + np.arange(ntok)) % case.dims.T
    return (lambda: mla_prolog_tokens(inp, ids)), ntok


def _oracle_rate(case, budget_s, sample_tokens, offset=0):
    call, ntok = _oracle_call(case, sample_tokens, offset)
    t0 = time.perf_counter()
    calls = 0
    while True:
        call()
        calls += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return calls * ntok / el, calls, el, ntok


def _oracle_worker(spec):
    """Entry of a child process (single-threaded BLAS): time the oracle on its own token sample
    and print the rate as JSON."""
    a = json.loads(spec)
    rate, calls, el, ntok = _oracle_rate(_case(a["workload"]), a["budget"], a["tokens"], a["offset"])
    print(json.dumps({"rate": rate, "calls": calls, "elapsed": el, "tokens": ntok}), flush=True)


def _single_thread_env():
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS",
              "VECLIB_MAXIMUM_THREADS", "NUMEXPR_NUM_THREADS"):
        env[k] = "1"
    env.pop("WORLD_SIZE", None)
    env.pop("RANK", None)
    env.pop("LOCAL_RANK", None)
    return env


def oracle_baselines(workload, budget_s=10.0, sample_tokens=4):
    """The oracle as it stands, on the host cores, on bounded token samples of the workload:
    one single-threaded process, then one single-threaded process per core in the affinity set,
    each on its own sample (tokens are independent), run at once.  Returns the single-thread
    rate, the all-core rate (sum over processes), the core count and a description."""
    cores = _cores()
    env = _single_thread_env()

    def launch(offset):
        spec = json.dumps({"workload": workload, "budget": budget_s, "tokens": sample_tokens,
                           "offset": offset})
        return subprocess.Popen([sys.executable, os.path.abspath(__file__), "--oracle-worker",
                                 spec], stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                text=True, env=env, cwd=ROOT)

    def collect(ps):
        out = []
        for pr in ps:
            o, e = pr.communicate()
            if pr.returncode != 0:
                raise RuntimeError(f"oracle worker failed: {e[-2000:]}")
            out.append(json.loads(o.strip().splitlines()[-1]))
        return out

    single = collect([launch(0)])[0]
    allc = collect([launch(i * sample_tokens) for i in range(cores)])
    rate_all = sum(r["rate"] for r in allc)
    sample = (f"{single['tokens']} tokens of the {_case(workload).name} workload per oracle call, "
              f"{budget_s:.0f} s per process; single thread: {single['calls']} calls in "
              f"{single['elapsed']:.1f} s; all cores: {cores} single-threaded processes on "
              f"disjoint token samples at once")
    return single["rate"], rate_all, cores, sample


def oracle_full_call(workload):
    """Seconds for one oracle call over every token of the workload (default BLAS threads)."""
    call, ntok = _oracle_call(_case(workload), 1 << 30)
    t0 = time.perf_counter()
    call()
    return time.perf_counter() - t0, ntok


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


def _stamped_kernel_times(run_one, n_calls, stream, dev):
    """Per-kernel times inside pipelined calls: a CUDA graph of n_calls consecutive stamped calls
    (the same launches as the timed graph), replayed twice; the second replay's stamps are read.
    Returns {kernel: {"span_us", "dep_to_end_us"}} averaged over the calls (the first few, still
    ramping up after the graph launch, are dropped)."""
    import torch
    import qkv_attention_prolog_gb300 as pkg
    stamps = pkg.stamps_buffer(dev, n_calls)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n_calls):
            run_one(i, stamps[i], torch.cuda.current_stream())
    for _ in range(2):
        stamps.zero_()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
    skip = min(4, n_calls // 2)
    acc = {}
    for i in range(skip, n_calls):
        for k, v in pkg.read_stamps(stamps[i]).items():
            a = acc.setdefault(k, {"span": [], "dep": []})
            a["span"].append(v["span_ns"] / 1e3)
            if v["dep_to_end_ns"] is not None:
                a["dep"].append(v["dep_to_end_ns"] / 1e3)
    out = {k: {"span_us": round(statistics.mean(v["span"]), 3),
               "dep_to_end_us": round(statistics.mean(v["dep"]), 3) if v["dep"] else None}
           for k, v in acc.items()}
    last = pkg.read_stamps(stamps[n_calls - 1])
    timeline = {k: {"start_us": round(v["start_ns"] / 1e3, 3), "end_us": round(v["end_ns"] / 1e3, 3)}
                for k, v in last.items()}
    del g
    return out, timeline


def measure_mla(args, case, dev, stream, steps, warm, world, stamp_calls, sample_clocks=True):
    """Device-timed calls of one MLA workload and its per-kernel stamps."""
    import torch
    import qkv_attention_prolog_gb300 as pkg
    d = case.dims
    w_int8 = case.weight_uq_qr_dtype == "int8"
    c_int8 = case.cache_dtype == "int8"
    kern, path_bytes, path_flops = mla_model(d, w_int8, c_int8, case.full_quant,
                                             case.x_norm is not None)
    n_sets = max(1, math.ceil(3 * L2_BYTES / path_bytes) + 1) if path_bytes < 2 * L2_BYTES else 1
    cpu, sets = _mla_sets(case, dev, n_sets)
    with torch.cuda.stream(stream):
        for i in range(warm):
            t, a, ws = sets[i % n_sets]
            pkg.mlap_execute(a, ws, stream)
    stream.synchronize()

    # CUDA graph of `per_graph` consecutive steps over the rotating sets
    per_graph = n_sets * max(1, 64 // n_sets) if steps >= 64 else min(n_sets, steps)
    per_graph = max(1, per_graph)
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
    clk = ClockSampler(dev.index) if sample_clocks else None
    if clk is not None:
        clk.__enter__()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(replays):
            g.replay()
        ev1.record(stream)
    stream.synchronize()
    if clk is not None:
        clk.__exit__(None, None, None)
    torch.cuda.synchronize()
    _barrier(world)
    ms_total = _max_over_ranks(ev0.elapsed_time(ev1), world)
    ms_step = ms_total / steps
    del g
    for s_ in sets:
        assert pkg.mlap_check_errors(s_[2], stream) == 0, "kernel error during the timed region"

    def run_one(i, st, strm):
        t, a, ws = sets[i % n_sets]
        pkg.mlap_execute_stamped(a, ws, st, strm)

    per, timeline = _stamped_kernel_times(run_one, max(8, stamp_calls), stream, dev)
    for s_ in sets:
        assert pkg.mlap_check_errors(s_[2], stream) == 0, "kernel error during the stamped calls"
    if "up" in per and "absorb" not in per:
        # the decode launch runs the up-projection and the absorb in one kernel: its algorithmic
        # bytes are both weights, c^Q and both outputs (q^C stays on chip)
        per["up_absorb"] = per.pop("up")
        timeline["up_absorb"] = timeline.pop("up")
        kern["up_absorb"] = {
            "bytes": kern["up"]["bytes"] + kern["absorb"]["bytes"] - 2 * d.T * d.N * d.D * 2,
            "flops": kern["up"]["flops"] + kern["absorb"]["flops"]}
    # down, norm/scatter, up (+ absorb); full quant adds, with an int8 query, its per-token-head
    # quantisation, and beyond 256 tokens the token_x widening (up to 256 the down-projection's
    # converter warps expand token_x); the input RmsNormQuant adds its own kernel
    launches = (len(per) + ((int(c_int8) + int(d.T > 256)) if case.full_quant else 0)
                + (1 if case.x_norm is not None else 0))
    return {"case": case, "cpu": cpu, "sets": sets, "kern": kern, "path_bytes": path_bytes,
            "path_flops": path_flops, "ms_step": ms_step, "steps": steps, "n_sets": n_sets,
            "per_graph": per_graph, "replays": replays, "per_kernel": per,
            "timeline": timeline, "clocks": clk.summary() if clk is not None else None,
            "launches_per_call": launches}


def _roofline(m, tensor_bound, hbm, tf_sus, peak_kind, workload, tf_burst=None):
    """Roofline entry of the dominant kernel: algorithmic bytes (FLOPs) per launch over its mean
    span inside the pipelined calls (earliest CTA start to latest CTA end).  The dominant kernel
    is the one with the longest time from its dependency wait to its end: under programmatic
    dependent launch a kernel starts while its predecessor runs, so its span also holds time
    spent waiting, and the longest span need not be the kernel that takes the most of the call."""
    per, kern = m["per_kernel"], m["kern"]
    dominant = max(per, key=lambda n: per[n]["dep_to_end_us"] or per[n]["span_us"])
    span_s = per[dominant]["span_us"] / 1e6
    if tensor_bound:
        achieved = kern[dominant]["flops"] / span_s / 1e12
        roof = {"bound": "tensor", "unit": "TFLOP/s", "peak": tf_sus,
                "peak_note": "sustained bf16 (kernel timed inside a long step)",
                "frac_of_burst": round(achieved / tf_burst, 4) if tf_burst else None}
    else:
        achieved = kern[dominant]["bytes"] / span_s / 1e9
        roof = {"bound": "hbm", "unit": "GB/s", "peak": hbm}
    roof.update({"kernel": dominant, "achieved": round(achieved, 1),
                 "frac": round(achieved / roof["peak"], 4), "peak_kind": peak_kind,
                 "traffic": _ncu_traffic(dominant, workload),
                 "algorithmic_per_launch": kern[dominant]["flops" if tensor_bound else "bytes"],
                 "avg_launch_us": per[dominant]["span_us"],
                 "timing": "kernel span from %globaltimer stamps inside pipelined calls",
                 "per_kernel_us": {n: v["span_us"] for n, v in per.items()},
                 "per_kernel_dep_to_end_us": {n: v["dep_to_end_us"] for n, v in per.items()}})
    return roof


def _path_roofline(m, hbm, tf_sus):
    path_time = max(m["path_bytes"] / (hbm * 1e9), m["path_flops"] / (tf_sus * 1e12))
    return {"bytes": m["path_bytes"], "flops": m["path_flops"],
            "roofline_us": round(path_time * 1e6, 3),
            "frac": round(path_time / (m["ms_step"] / 1e3), 4),
            "bound": ("tensor" if m["path_flops"] / (tf_sus * 1e12) > m["path_bytes"] / (hbm * 1e9)
                      else "hbm")}


def run_ours(args, rank, local, world):
    import torch
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
    stream = torch.cuda.Stream(dev)
    steps = args.steps or {"decode": 40000, "tiny": 40000, "partial_quant": 40000,
                           "full_quant": 40000, "xnorm": 40000, "prefill": 1500}[args.workload]
    warm = max(3, args.warmup)
    m = measure_mla(args, case, dev, stream, steps, warm, world, args.stamp_calls)
    tensor_bound = args.workload == "prefill"
    roof = _roofline(m, tensor_bound, hbm, tf_sus, peak_kind, args.workload, tf_burst)
    path_roof = _path_roofline(m, hbm, tf_sus)
    e2e = run_e2e(args, case, m["cpu"], m["sets"][0], dev, stream)
    ms_step = m["ms_step"]
    line = {"metric": METRIC, "value": round(d.T * world * m["steps"] / (ms_step * m["steps"] / 1e3), 1),
            "unit": UNIT, "n_gpus": world, "steps": m["steps"], "warmup": warm,
            "ms_per_step": round(ms_step, 6), "us_per_call": round(ms_step * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; shapes and distributions of the workload recipe)",
            "config": {"workload": case.name, "T": d.T, "B": d.B, "S": d.S, "He": d.He,
                       "Hcq": d.Hcq, "Hckv": d.Hckv, "N": d.N, "D": d.D, "Dr": d.Dr,
                       "weight_uq_qr": case.weight_uq_qr_dtype, "caches": case.cache_dtype,
                       "token_x_and_down_weights": "int8" if case.full_quant else "bf16",
                       "input_rms_norm_quant": case.x_norm,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": (f"rotating {m['n_sets']} input sets of {m['path_bytes']/1e6:.1f} MB "
                              f"({m['n_sets']*m['path_bytes']/1e6:.0f} MB > 129 MB L2)"
                              if m["n_sets"] > 1
                              else f"inputs {m['path_bytes']/1e6:.0f} MB > 129 MB L2"),
                       "timing": (f"CUDA graph of {m['per_graph']} execute calls replayed "
                                  f"{m['replays']}x")},
            "roofline": roof, "path_roofline": path_roof, "clocks": m["clocks"],
            "timeline_us": m["timeline"],
            "e2e": e2e, "gpu_launches": m["launches_per_call"] * m["steps"]}
    del m
    if args.workload == "decode" and not args.no_prefill:
        torch.cuda.empty_cache()
        line["prefill"] = run_prefill_leg(args, dev, stream, world, hbm, tf_burst, tf_sus,
                                          peak_kind)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        single, allc, cores, sample = oracle_baselines(args.workload)
        line["cpu_baseline"] = {"value": round(allc, 3), "unit": UNIT, "cores": cores,
                                "kind": "oracle", "single_thread": round(single, 3),
                                "all_cores": round(allc, 3), "sample": sample}
    if args.oracle_full_call:
        sec, ntok = oracle_full_call(args.workload)
        line["oracle_full_call"] = {"seconds": round(sec, 2), "tokens": ntok,
                                    "tokens_per_s": round(ntok / sec, 2), "cores": _cores()}
    return line


def run_prefill_leg(args, dev, stream, world, hbm, tf_burst, tf_sus, peak_kind):
    """The bf16 prefill workload (T=8192) in the same process: microseconds per call, the path
    against the sustained tensor peak, and the per-kernel stamps."""
    import synthetic
    case = synthetic.MLA_PREFILL
    m = measure_mla(args, case, dev, stream, max(4, args.prefill_steps), 3, world,
                    min(16, args.stamp_calls))
    roof = _roofline(m, True, hbm, tf_sus, peak_kind, "prefill", tf_burst)
    path_roof = _path_roofline(m, hbm, tf_sus)
    ms = m["ms_step"]
    out = {"workload": case.name, "us_per_call": round(ms * 1e3, 3),
           "tokens_per_s": round(case.dims.T * world / (ms / 1e3), 1), "steps": m["steps"],
           "roofline": roof, "path_roofline": path_roof,
           "path_frac_of_burst": round(m["path_flops"] / (ms / 1e3) / 1e12 / tf_burst, 4),
           "timeline_us": m["timeline"], "clocks": m["clocks"],
           "timing": (f"CUDA graph of {m['per_graph']} execute calls replayed {m['replays']}x; "
                      f"inputs {m['path_bytes']/1e6:.0f} MB > 129 MB L2")}
    del m
    return out


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
    warm = max(3, args.warmup)
    with torch.cuda.stream(stream):
        for _ in range(warm):
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
    del g
    assert pkg.mlap_check_errors(ws, stream) == 0, "kernel error during the timed region"
    per, timeline = _stamped_kernel_times(
        lambda i, st, strm: pkg.qkvrnrc_execute_stamped(a, ws, st, strm), 16, stream, dev)
    span_us = per["qkv_rnrc"]["span_us"]
    achieved = nb / (span_us / 1e6) / 1e9
    e2e = run_qkv_e2e(args, case, cpu, t, d, dev, stream)
    return {"metric": METRIC, "value": round(d.T * world / (ms / 1e3), 1), "unit": UNIT,
            "n_gpus": world, "steps": steps, "warmup": warm, "ms_per_step": round(ms, 6),
            "us_per_call": round(ms * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp16",
            "data": "synthetic", "config": {"workload": case.name, "B": d.B, "S": d.S,
                                            "Nq": d.Nq, "Nk": d.Nk, "Nv": d.Nv, "D": d.D,
                                            "quant": case.quant,
                                            "before_quant_outputs": case.before_quant,
                                            "l2": f"inputs {nb/1e6:.0f} MB > 129 MB L2"},
            "roofline": {"bound": "hbm", "kernel": "qkv_rnrc", "achieved": round(achieved, 1),
                         "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                         "peak_kind": peak_kind, "traffic": _ncu_traffic("qkv_rnrc", args.workload),
                         "algorithmic_per_launch": nb, "avg_launch_us": span_us,
                         "timing": "kernel span from %globaltimer stamps inside pipelined calls",
                         "per_kernel_dep_to_end_us": {"qkv_rnrc": per["qkv_rnrc"]["dep_to_end_us"]}},
            "path_roofline": {"bytes": nb, "roofline_us": round(nb / (hbm * 1e9) * 1e6, 3),
                              "frac": round(nb / (hbm * 1e9) / (ms / 1e3), 4), "bound": "hbm"},
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
    """The reference arm: the CPU oracle as it stands, timed on this host's cores (rank 0 only;
    the other ranks exit without work)."""
    if rank != 0:
        return None
    case = _case(args.workload)
    steps = args.steps or 3
    warm = max(0, min(args.warmup, 1))
    per_step_budget = 5.0
    vals = []
    sample = ""
    for i in range(warm + steps):
        v, calls, el, ntok = _oracle_rate(case, per_step_budget, 4)
        sample = (f"{ntok} tokens of the {case.name} workload per oracle call; {calls} calls in "
                  f"{el:.1f} s per step")
        if i >= warm:
            vals.append(v)
    v = statistics.mean(vals)
    cores = _cores()
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
    if args.oracle_worker is not None:
        _oracle_worker(args.oracle_worker)
        return
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        # no launcher: start the N replicas here, one process per GPU
        _spawn_replicas(args.gpus, sys.argv[1:])
        return
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
