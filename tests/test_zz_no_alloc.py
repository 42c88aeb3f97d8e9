"""The allocation-free entry point (mlap_execute_no_alloc) against the workspace entry point.

mlap_execute_no_alloc serves callers that cannot allocate device memory (a plugin whose host
framework owns every device buffer, a latency-critical loop that cannot pay cudaMalloc's device
synchronisation, a C caller without an allocator): its scratch is a static device array inside
the library.  Two calls in a row on different inputs must each give what mlap_execute gives on
the same inputs, within the parity tolerance; the second call checks that what the first left in
the shared scratch does not leak into its results.  This file sorts last so a failure here comes
after every other test has run.
"""
import dataclasses

import pytest
import torch

import synthetic
import qkv_attention_prolog_gb300 as pkg
from qkv_attention_prolog_gb300 import _lib
from tests.gpu_util import assert_close, check_cache, f64, mla_device_tensors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    import __graft_entry__
    __graft_entry__.build()


def _tensors(case, dev):
    cpu = synthetic.make_mla_inputs(case)
    t = mla_device_tensors(cpu, case.dims, dev)
    d = case.dims
    packed = pkg.prepack_mla_weights({k: t.pop(k) for k in ("weight_dq", "weight_uq_qr",
                                                            "weight_uk", "weight_dkv_kr")},
                                     d.N, d.D, d.Dr)
    t.update(packed)
    return cpu, t


def _fresh_outputs(t, cpu, dev):
    u = dict(t)
    for k in ("kv_cache", "kr_cache"):
        u[k] = cpu[k].to(dev)
    u["query"] = torch.full_like(t["query"], float("nan"))
    u["query_rope"] = torch.full_like(t["query_rope"], float("nan"))
    return u


def _decode_T300():
    # decode dimensions with 300 tokens: one K split and the tokens-as-rows GEMMs, so the
    # partials, c^Q, q^C and scale regions of the scratch sit at other offsets than at T = 128
    return dataclasses.replace(synthetic.MLA_DECODE, name="decode_T300",
                               dims=dataclasses.replace(synthetic.MLA_DECODE.dims, B=300))


CASES = {
    "decode_T128": lambda: synthetic.MLA_DECODE,
    "partial_quant_int8_caches_T64": lambda: synthetic.MLA_PARTIAL_QUANT,
    "decode_T300": _decode_T300,
}


@pytest.mark.parametrize("name", list(CASES))
def test_no_alloc_matches_workspace_entry_point_twice(name):
    dev = torch.device("cuda")
    case_a = CASES[name]()
    case_b = dataclasses.replace(case_a, seed=case_a.seed + 4242, n_skip=3)
    for case in (case_a, case_b):          # two calls in a row, different inputs
        cpu, t = _tensors(case, dev)
        ref = _fresh_outputs(t, cpu, dev)
        a_ref = pkg.make_mla_args(ref, case.eps, case.eps)
        need = pkg.mlap_get_workspace_size(a_ref)
        assert need <= 24 * 1024 * 1024, "case must fit the static scratch"
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
        pkg.mlap_workspace_init(ws)
        pkg.mlap_execute(a_ref, ws)

        out = _fresh_outputs(t, cpu, dev)
        a = pkg.make_mla_args(out, case.eps, case.eps)
        _lib.mlap_execute_no_alloc(a)
        torch.cuda.synchronize()

        assert_close(f64(out["query"]), f64(ref["query"]), "query")
        assert_close(f64(out["query_rope"]), f64(ref["query_rope"]), "query_rope")
        idx = cpu["cache_index"].numpy()
        T = case.dims.T
        check_cache(out["kv_cache"], cpu["kv_cache"], f64(ref["kv_cache"]).reshape(-1, case.dims.Hckv)[
            idx.clip(0)].reshape(T, -1), idx, "kv_cache")
        check_cache(out["kr_cache"], cpu["kr_cache"], f64(ref["kr_cache"]).reshape(-1, case.dims.Dr)[
            idx.clip(0)].reshape(T, -1), idx, "kr_cache")


def test_no_alloc_rejects_shapes_beyond_its_scratch():
    dev = torch.device("cuda")
    big = dataclasses.replace(synthetic.MLA_DECODE,
                              dims=dataclasses.replace(synthetic.MLA_DECODE.dims, B=200))
    cpu, t = _tensors(big, dev)
    a = pkg.make_mla_args(t, big.eps, big.eps)
    assert pkg.mlap_get_workspace_size(a) > 24 * 1024 * 1024
    with pytest.raises(pkg.MlapError) as e:
        _lib.mlap_execute_no_alloc(a)
    assert e.value.status == 5          # MLAP_ERR_WORKSPACE, before any device work
