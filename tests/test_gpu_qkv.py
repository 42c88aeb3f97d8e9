"""GPU parity of QkvRmsNormRopeCache (CUDA path through the C ABI) against the fp64 oracle."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synthetic
import qkv_attention_prolog_gb300 as pkg
from tests.gpu_util import assert_close, check_cache, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    import __graft_entry__
    __graft_entry__.build()


def _run(case, dtype=torch.float16, tnd=False):
    cpu = synthetic.make_qkv_inputs(case)
    d = case.dims
    quant = case.quant in ("symmetric", "asymmetric")
    asym = case.quant == "asymmetric"
    if dtype != torch.float16:
        for k in ("qkv", "gamma_q", "gamma_k", "cos", "sin"):
            cpu[k] = cpu[k].to(dtype)
        if not quant:
            cpu["k_cache"] = cpu["k_cache"].to(dtype)
            cpu["v_cache"] = cpu["v_cache"].to(dtype)
    dev = torch.device("cuda")
    t = {k: v.to(dev) for k, v in cpu.items() if isinstance(v, torch.Tensor)}
    if tnd:
        t["qkv"] = t["qkv"].reshape(d.T, -1)
        t["cos"] = t["cos"].reshape(d.T, d.D)
        t["sin"] = t["sin"].reshape(d.T, d.D)
        t["q_out"] = torch.full((d.T, d.Nq, d.D), float("nan"), dtype=dtype, device=dev)
        lead = (d.T,)
    else:
        t["qkv"] = t["qkv"].reshape(d.B, d.S, -1)
        t["cos"] = t["cos"].reshape(d.B, d.S, d.D)
        t["sin"] = t["sin"].reshape(d.B, d.S, d.D)
        t["index"] = t["index"].reshape(d.B, d.S)
        t["q_out"] = torch.full((d.B, d.S, d.Nq, d.D), float("nan"), dtype=dtype, device=dev)
        lead = (d.B, d.S)
    if case.before_quant:
        for name, n in (("q_before_quant", d.Nq), ("k_before_quant", d.Nk), ("v_before_quant", d.Nv)):
            t[name] = torch.full(lead + (n, d.D), float("nan"), dtype=dtype, device=dev)
    a = pkg.make_qkv_args(t, d.Nq, d.Nk, d.Nv, case.eps)
    ws = torch.empty(pkg.qkvrnrc_get_workspace_size(a), dtype=torch.uint8, device=dev)
    pkg.mlap_workspace_init(ws)
    pkg.qkvrnrc_execute(a, ws)
    torch.cuda.synchronize()
    status = pkg.mlap_check_errors(ws)
    ref = oracle.qkv_rms_norm_rope_cache(
        f64(cpu["qkv"]), f64(cpu["gamma_q"]), f64(cpu["gamma_k"]), f64(cpu["cos"]),
        f64(cpu["sin"]), cpu["index"].numpy(), f64(cpu["k_cache"]), f64(cpu["v_cache"]),
        case.eps, d.Nq, d.Nk, d.Nv,
        cpu["k_scale"].numpy() if quant else None, cpu["v_scale"].numpy() if quant else None,
        out_dtype="bf16" if dtype == torch.bfloat16 else "fp16",
        k_offset=cpu["k_offset"].numpy() if asym else None,
        v_offset=cpu["v_offset"].numpy() if asym else None)
    return t, cpu, ref, status


def _check(case, dtype=torch.float16, tnd=False):
    t, cpu, ref, status = _run(case, dtype, tnd)
    d = case.dims
    assert status == 0
    assert_close(f64(t["q_out"]).reshape(d.T, d.Nq, d.D), ref["q_out"], "q_out")
    idx = cpu["index"].numpy()
    check_cache(t["k_cache"], cpu["k_cache"], ref["k_rows"].reshape(d.T, -1), idx, "k_cache")
    check_cache(t["v_cache"], cpu["v_cache"], ref["v_rows"].reshape(d.T, -1), idx, "v_cache")
    if case.before_quant:
        qb = t["q_before_quant"].reshape(d.T, d.Nq, d.D)
        assert torch.equal(qb.view(torch.int16), t["q_out"].reshape(d.T, d.Nq, d.D).view(torch.int16))
        assert_close(f64(t["k_before_quant"]).reshape(d.T, d.Nk, d.D), ref["k_before"], "k_before")
        # v is stored as split: bit-identical to the input slice
        v_in = cpu["qkv"].reshape(d.T, d.Nq + d.Nk + d.Nv, d.D)[:, d.Nq + d.Nk:, :]
        vb = t["v_before_quant"].reshape(d.T, d.Nv, d.D).cpu()
        assert torch.equal(vb.view(torch.int16), v_in.contiguous().view(torch.int16))


def test_qkv_full_workload():
    _check(synthetic.QKV_EPILOGUE)


@pytest.mark.parametrize("B,S,Nq,Nk", [(1, 1, 1, 1), (2, 3, 4, 2), (3, 129, 8, 1)])
def test_qkv_small(B, S, Nq, Nk):
    bn = max(1, -(-S // 128) * B)
    case = synthetic.QkvCase("small", synthetic.QkvDims(B=B, S=S, Nq=Nq, Nk=Nk, Nv=Nk,
                                                        block_num=bn + 1), seed=B * 100 + S)
    _check(case)
    _check(case, tnd=True)


def test_qkv_no_quant_fp16_caches():
    case = synthetic.QkvCase("noquant", synthetic.QkvDims(B=2, S=100, Nq=4, Nk=2, Nv=2,
                                                          block_num=3), seed=5, quant="none")
    _check(case)


def test_qkv_bf16():
    case = synthetic.QkvCase("bf16", synthetic.QkvDims(B=2, S=64, Nq=4, Nk=2, Nv=2,
                                                       block_num=2), seed=6)
    _check(case, dtype=torch.bfloat16)


def test_qkv_index_errors_reported():
    case = synthetic.QkvCase("oob", synthetic.QkvDims(B=1, S=8, Nq=2, Nk=1, Nv=1, block_num=1),
                             seed=8, skip_frac=0)
    cpu = synthetic.make_qkv_inputs(case)
    d = case.dims
    dev = torch.device("cuda")
    cpu["index"] = torch.tensor([0, 1, 128, -1, -5, 2, 3, 4], dtype=torch.int64)
    t = {k: v.to(dev) for k, v in cpu.items() if isinstance(v, torch.Tensor)}
    t["q_out"] = torch.empty(d.T, d.Nq, d.D, dtype=torch.float16, device=dev)
    t["qkv"] = t["qkv"].reshape(d.T, -1)
    t["cos"] = t["cos"].reshape(d.T, -1)
    t["sin"] = t["sin"].reshape(d.T, -1)
    a = pkg.make_qkv_args(t, d.Nq, d.Nk, d.Nv, case.eps)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    pkg.qkvrnrc_execute(a, ws)
    assert pkg.mlap_check_errors(ws) == 7
    ref = oracle.qkv_rms_norm_rope_cache(
        f64(cpu["qkv"]), f64(cpu["gamma_q"]), f64(cpu["gamma_k"]), f64(cpu["cos"]),
        f64(cpu["sin"]), cpu["index"].numpy(), cpu["k_cache"].numpy(), cpu["v_cache"].numpy(),
        case.eps, d.Nq, d.Nk, d.Nv, cpu["k_scale"].numpy(), cpu["v_scale"].numpy())
    check_cache(t["k_cache"], cpu["k_cache"], ref["k_rows"].reshape(d.T, -1),
                cpu["index"].numpy(), "k_cache")


def test_qkv_asymmetric_before_quant_full_workload():
    _check(synthetic.QKV_EPILOGUE_ASYM)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_qkv_asymmetric_before_quant_small(dtype):
    # ragged token count, -1 indices, both input dtypes, TND and BSH
    case = synthetic.QkvCase("small_asym", synthetic.QkvDims(B=3, S=37, Nq=4, Nk=2, Nv=2,
                                                             block_num=4), seed=77,
                             quant="asymmetric", before_quant=True, skip_frac=0.1)
    _check(case, dtype)
    _check(case, dtype, tnd=True)


def test_qkv_before_quant_without_quant():
    case = synthetic.QkvCase("small_bq", synthetic.QkvDims(B=2, S=5, Nq=2, Nk=1, Nv=1,
                                                           block_num=2), seed=78,
                             quant="none", before_quant=True)
    _check(case)


# every cos/sin element drawn on its own (no column repeats its partner j +- D/2): the
# half-and-half rule of "Formulas" (3) is applied with the tables elementwise
def test_qkv_rope_tables_independent_full_workload():
    _check(dataclasses.replace(synthetic.QKV_EPILOGUE, table_mode="independent", seed=2003))


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_qkv_rope_tables_independent_small(dtype):
    case = synthetic.QkvCase("tables", synthetic.QkvDims(B=2, S=37, Nq=4, Nk=2, Nv=2,
                                                         block_num=2), seed=79,
                             quant="asymmetric", before_quant=True, table_mode="independent")
    _check(case, dtype)
