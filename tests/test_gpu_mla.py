"""GPU parity of the MLA prolog (CUDA path through the C ABI) against the fp64 oracle."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synthetic
import qkv_attention_prolog_gb300 as pkg
from oracle.mla_prolog import mla_key_rows, mla_prolog_tokens
from tests.gpu_util import (assert_close, check_cache, check_int8_query, f64, oracle_inputs,
                            run_mla)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    import __graft_entry__
    __graft_entry__.build()


def _full_check(case, bsh=False):
    cpu = synthetic.make_mla_inputs(case)
    d = case.dims
    t, prolog, status = run_mla(cpu, d, case.eps, bsh=bsh)
    assert status == 0, f"kernel error status {status}"
    inp = oracle_inputs(cpu, case.eps)
    ref = oracle.mla_prolog(**inp)
    if cpu["weight_uq_qr"].dtype == torch.int8:
        # int8 c^Q: per token, the oracle or one of its ambiguous integer decisions (gpu_util);
        # an int8 query within 1 LSB with its scales in tolerance
        check_int8_query(t, ref, inp, d, case.name)
    else:
        assert_close(f64(t["query"]).reshape(d.T, d.N, d.Hckv), ref["query"], "query")
        assert_close(f64(t["query_rope"]).reshape(d.T, d.N, d.Dr), ref["query_rope"], "query_rope")
    idx = cpu["cache_index"].numpy()
    sub = mla_prolog_tokens(oracle_inputs(cpu, case.eps), np.arange(d.T))
    check_cache(t["kv_cache"], cpu["kv_cache"], sub["kv_rows"], idx, "kv_cache")
    check_cache(t["kr_cache"], cpu["kr_cache"], sub["kr_rows"], idx, "kr_cache")
    return t, prolog


def test_tiny_bf16():
    _full_check(synthetic.MLA_TINY)


SHAPES = [
    dict(B=1, S=1),                                   # single token
    dict(B=3, S=1, N=2),                              # ragged token tile
    dict(B=17, S=1, Hckv=256, N=4),                   # BN 32 in the decode orientation
    dict(B=2, S=65, He=512, Hcq=256, N=3),            # T=130: BN 256, ragged rope tail (N*Dr)
    dict(B=3, S=100, He=384, Hcq=192, Hckv=128, N=2),  # T=300: prefill orientation, ragged M
    dict(B=1, S=200, He=320, Hcq=136, Hckv=96, N=2, Dr=32),  # ragged K, Hcq, Hckv tiles
    dict(B=2, S=150, He=256, Hcq=128, Hckv=96, N=2, Dr=32),  # T=300: a query store box past Hckv
    dict(B=40, S=1, He=256, Hcq=1536, N=16),         # 16 heads, deep K (fused decode kernel)
    # from 1024 tokens the down- and up-projection run on CTA pairs (256-token tiles, each CTA
    # half of a 256-row weight tile): ragged token tile, a W^DQ tile and a W^UQ|W^QR tile whose
    # second half lies wholly past the weight rows
    dict(B=3, S=400, He=512, Hcq=320, Hckv=128, N=3),
    dict(B=2, S=512, He=384, Hcq=256, Hckv=256, N=2),  # T=1024: whole token tiles
]


@pytest.mark.parametrize("kw", SHAPES, ids=[str(i) for i in range(len(SHAPES))])
def test_shapes(kw):
    kw = dict(kw)
    block_num = max(1, (kw["B"] * kw["S"] + 127) // 128 + 1)
    case = synthetic.small_mla_case("shape", block_num=block_num, n_skip=1, **kw)
    _full_check(case)


def test_bsh_layout_matches_tnd():
    case = synthetic.small_mla_case("bsh", B=4, S=5, N=2, block_num=1)
    t_bsh, _ = _full_check(case, bsh=True)
    t_tnd, _ = _full_check(case, bsh=False)
    assert torch.equal(t_bsh["query"].reshape(-1), t_tnd["query"].reshape(-1))


def test_decode_T128():
    _full_check(synthetic.MLA_DECODE)


def test_prefill_T8192_sampled():
    case = synthetic.MLA_PREFILL
    cpu = synthetic.make_mla_inputs(case)
    d = case.dims
    t, _, status = run_mla(cpu, d, case.eps)
    assert status == 0
    inp = oracle_inputs(cpu, case.eps)
    rng = np.random.default_rng(0)
    sample = np.sort(np.concatenate([rng.choice(d.T, 254, replace=False), [0, d.T - 1]]))
    sub = mla_prolog_tokens(inp, sample)
    assert_close(f64(t["query"])[sample], sub["query"], "query (sampled tokens)")
    assert_close(f64(t["query_rope"])[sample], sub["query_rope"], "query_rope (sampled tokens)")
    kv, kr = mla_key_rows(**inp, Hckv=d.Hckv)
    idx = cpu["cache_index"].numpy()
    check_cache(t["kv_cache"], cpu["kv_cache"], kv, idx, "kv_cache (every slot)")
    check_cache(t["kr_cache"], cpu["kr_cache"], kr, idx, "kr_cache (every slot)")


def test_deterministic_bitwise():
    case = synthetic.MLA_DECODE
    cpu = synthetic.make_mla_inputs(case)
    t1, prolog, _ = run_mla(cpu, case.dims, case.eps)
    t2, _, _ = run_mla(cpu, case.dims, case.eps, prolog=prolog)
    for k in ("query", "query_rope", "kv_cache", "kr_cache"):
        assert torch.equal(t1[k].view(torch.uint8), t2[k].view(torch.uint8)), k


def test_empty_tokens():
    case = synthetic.small_mla_case("empty", B=0, S=1)
    cpu = synthetic.make_mla_inputs(case)
    t, _, status = run_mla(cpu, case.dims, case.eps)
    assert status == 0
    assert torch.equal(t["kv_cache"].cpu().view(torch.uint8), cpu["kv_cache"].view(torch.uint8))


def test_empty_cache_computes_outputs():
    case = synthetic.small_mla_case("skv0", B=4, S=1, block_num=0)
    cpu = synthetic.make_mla_inputs(case)
    cpu["cache_index"] = torch.full((4,), -1, dtype=torch.int64)
    cpu["cache_index"][1] = 5    # out of range of an empty cache: ignored, not an error
    t, _, status = run_mla(cpu, case.dims, case.eps)
    assert status == 0
    ref = oracle.mla_prolog(**oracle_inputs(cpu, case.eps))
    assert_close(f64(t["query"]), ref["query"], "query")


def test_out_of_range_index_is_skipped_and_reported():
    case = synthetic.small_mla_case("oob", B=4, S=1, block_num=2)
    cpu = synthetic.make_mla_inputs(case)
    cpu["cache_index"] = torch.tensor([3, 256, -7, 10], dtype=torch.int64)
    t, prolog, status = run_mla(cpu, case.dims, case.eps)
    assert status == 7       # MLAP_ERR_INDEX_RANGE
    sub = mla_prolog_tokens(oracle_inputs(cpu, case.eps), np.arange(4))
    check_cache(t["kv_cache"], cpu["kv_cache"], sub["kv_rows"], cpu["cache_index"].numpy(),
                "kv_cache")
    # the error word is cleared by the read
    assert pkg.mlap_check_errors(prolog.ws) == 0


@pytest.mark.parametrize("N", [3, 16], ids=["separate_kernels", "fused_kernel"])
def test_outputs_have_no_stray_writes(N):
    # outputs live inside larger poisoned buffers: bytes around them must not change
    case = synthetic.small_mla_case("canary", B=5, S=1, N=N, block_num=1)
    cpu = synthetic.make_mla_inputs(case)
    d = case.dims
    dev = torch.device("cuda")
    t = {k: v.to(dev) for k, v in cpu.items() if isinstance(v, torch.Tensor)}
    guard = 4096
    qbuf = torch.full((guard * 2 + d.T * d.N * d.Hckv,), 7.0, dtype=torch.bfloat16, device=dev)
    rbuf = torch.full((guard * 2 + d.T * d.N * d.Dr,), 7.0, dtype=torch.bfloat16, device=dev)
    t["query"] = qbuf[guard:guard + d.T * d.N * d.Hckv].view(d.T, d.N, d.Hckv)
    t["query_rope"] = rbuf[guard:guard + d.T * d.N * d.Dr].view(d.T, d.N, d.Dr)
    prolog = pkg.MlaProlog({k: t[k] for k in ("weight_dq", "weight_uq_qr", "weight_uk",
                                              "weight_dkv_kr")}, d.N, d.D, d.Dr)
    prolog.run({k: v for k, v in t.items() if not k.startswith("weight_")}, case.eps, case.eps)
    torch.cuda.synchronize()
    for buf, n in ((qbuf, d.T * d.N * d.Hckv), (rbuf, d.T * d.N * d.Dr)):
        assert bool((buf[:guard] == 7.0).all()) and bool((buf[guard + n:] == 7.0).all())
    ref = oracle.mla_prolog(**oracle_inputs(cpu, case.eps))
    assert_close(f64(t["query"]), ref["query"], "query")
    assert_close(f64(t["query_rope"]), ref["query_rope"], "query_rope")


def test_partial_quant_int8_caches():
    # int8 weight_uq_qr (per-channel dequant), dynamic per-token c^Q quant, int8 caches
    _full_check(synthetic.MLA_PARTIAL_QUANT)


def test_partial_quant_bf16_caches():
    _full_check(synthetic.MLA_PARTIAL_QUANT_BF16CACHE)


QUANT_SHAPES = [
    dict(B=5, S=1, He=256, Hcq=128, N=3, cache_dtype="int8"),             # decode orientation
    dict(B=3, S=100, He=384, Hcq=192, Hckv=128, N=2, cache_dtype="int8"),  # prefill orientation
    dict(B=2, S=150, He=256, Hcq=144, Hckv=96, N=2, Dr=32, cache_dtype="bf16"),
]


@pytest.mark.parametrize("kw", QUANT_SHAPES, ids=[str(i) for i in range(len(QUANT_SHAPES))])
def test_partial_quant_shapes(kw):
    kw = dict(kw)
    block_num = max(1, (kw["B"] * kw["S"] + 127) // 128 + 1)
    case = synthetic.small_mla_case("pq", block_num=block_num, n_skip=1,
                                    weight_uq_qr_dtype="int8", **kw)
    _full_check(case)


def test_full_quant_int8_cache():
    # int8 token_x / W^DQ / W^DKV|W^KR (per-token, per-channel dequant), int8 kv_cache, bf16
    # kr_cache, int8 query per token and head with dequant_scale_q_nope
    _full_check(synthetic.MLA_FULL_QUANT)


def test_full_quant_bf16_cache():
    _full_check(synthetic.MLA_FULL_QUANT_BF16CACHE)


FULL_QUANT_SHAPES = [
    dict(B=5, S=1, He=256, Hcq=128, N=3, cache_dtype="int8"),              # decode orientation
    # decode orientation, the int8 token_x tiles expanded by the converter warps at every token
    # tile width above 16 (32, 128 and 256 rows); He = 272 and 336 end in a partial K block
    dict(B=24, S=1, He=272, Hcq=128, N=2, cache_dtype="int8"),
    dict(B=100, S=1, He=512, Hcq=256, N=2, cache_dtype="bf16"),
    dict(B=200, S=1, He=336, Hcq=128, Hckv=96, N=2, Dr=32, cache_dtype="int8"),
    dict(B=3, S=100, He=384, Hcq=192, Hckv=128, N=2, cache_dtype="int8"),   # prefill orientation
    dict(B=2, S=150, He=256, Hcq=144, Hckv=96, N=2, Dr=32, cache_dtype="bf16"),
]


@pytest.mark.parametrize("kw", FULL_QUANT_SHAPES, ids=[str(i) for i in range(len(FULL_QUANT_SHAPES))])
def test_full_quant_shapes(kw):
    kw = dict(kw)
    block_num = max(1, (kw["B"] * kw["S"] + 127) // 128 + 1)
    case = synthetic.small_mla_case("fq", block_num=block_num, n_skip=1, full_quant=True,
                                    weight_uq_qr_dtype="int8", **kw)
    _full_check(case)


def test_full_quant_bsh():
    case = synthetic.small_mla_case("fq_bsh", B=4, S=5, N=2, block_num=1, full_quant=True,
                                    weight_uq_qr_dtype="int8", cache_dtype="int8")
    _full_check(case, bsh=True)


# ---- input RmsNormQuant (aclnnMlaPreprocessV2) ahead of the down-projection

def test_rms_norm_quant_decode():
    # the decode workload with the input RmsNormQuant (deqScale per channel)
    _full_check(synthetic.MLA_XNORM)


XNORM_SHAPES = [
    dict(B=3, S=1, He=264, N=2, x_norm="channel"),              # ragged He over the threads
    dict(B=2, S=1, He=10240, Hcq=256, N=2, x_norm="tensor"),    # largest He, one deqScale
    dict(B=3, S=100, He=384, Hcq=192, Hckv=128, N=2, x_norm="channel"),   # prefill orientation
    dict(B=5, S=1, He=256, Hcq=128, N=3, x_norm="tensor", weight_uq_qr_dtype="int8",
         cache_dtype="int8"),                                   # with partial quant
    dict(B=2, S=300, He=264, Hcq=128, N=2, x_norm="channel"),   # many tokens: the other kernel
]


@pytest.mark.parametrize("kw", XNORM_SHAPES, ids=[str(i) for i in range(len(XNORM_SHAPES))])
def test_rms_norm_quant_shapes(kw):
    kw = dict(kw)
    block_num = max(1, (kw["B"] * kw["S"] + 127) // 128 + 1)
    case = synthetic.small_mla_case("xnorm", block_num=block_num, n_skip=1, **kw)
    _full_check(case)


def test_rms_norm_quant_bsh_leaves_token_x():
    case = synthetic.small_mla_case("xnorm_bsh", B=4, S=5, N=2, block_num=1, x_norm="channel")
    cpu = synthetic.make_mla_inputs(case)
    t, _ = _full_check(case, bsh=True)
    # token_x is only read: the normalised copy lives in the workspace
    assert torch.equal(t["token_x"].reshape(cpu["token_x"].shape).cpu().view(torch.int16),
                       cpu["token_x"].view(torch.int16))


# ---- fused decode up-projection + absorb (T <= 128, N >= 16): one CTA per head, or two CTAs
# per head (a cluster pair splitting q^C and q^N) when 2N fits on the SMs

FUSED_SHAPES = [
    dict(B=1, S=1, N=64),                                          # single token
    dict(B=100, S=1, He=256, Hcq=136, Hckv=288, N=64),             # ragged K, absorb 256 + 32
    dict(B=33, S=1, He=320, Hcq=192, Hckv=96, N=80),               # 80 heads, one short chunk
    dict(B=4, S=32, He=256, Hcq=128, Hckv=512, N=64),              # BSH-shaped T = 128
    dict(B=3, S=1, He=256, Hcq=128, Hckv=64, N=128),               # heads keep one W^QR block
    dict(B=7, S=1, He=256, Hcq=320, Hckv=160, N=32),               # 32 heads + 64 rope CTAs
    # int8 weight_uq_qr (converter warps, dequant in the epilogue)
    dict(B=9, S=1, He=256, Hcq=192, Hckv=96, N=16, weight_uq_qr_dtype="int8",
         cache_dtype="int8"),                                       # partial quant
    dict(B=5, S=1, He=256, Hcq=144, Hckv=128, N=32, weight_uq_qr_dtype="int8",
         cache_dtype="bf16"),                                       # ragged K, bf16 caches
    dict(B=6, S=1, He=256, Hcq=128, Hckv=64, N=128, weight_uq_qr_dtype="int8",
         cache_dtype="int8", full_quant=True),                      # full quant, int8 query
    dict(B=9, S=1, He=256, Hcq=192, Hckv=96, N=96, weight_uq_qr_dtype="int8",
         cache_dtype="int8"),                                       # int8, one CTA per head
    # head pairs (2N <= SMs): the second CTA of each pair has no q^N columns
    dict(B=5, S=1, He=256, Hcq=128, Hckv=32, N=20),
    # head pairs on 144 of the SMs
    dict(B=3, S=1, He=256, Hcq=128, Hckv=64, N=72),
    # head pairs with the int8 query: the two CTAs write 64 and 32 columns of each (token, head)
    # row of the bf16 q^N that the query quant reads
    dict(B=7, S=1, He=256, Hcq=128, Hckv=96, N=20, weight_uq_qr_dtype="int8",
         cache_dtype="int8", full_quant=True),
]


@pytest.mark.parametrize("kw", FUSED_SHAPES, ids=[str(i) for i in range(len(FUSED_SHAPES))])
def test_fused_up_absorb_shapes(kw):
    kw = dict(kw)
    block_num = max(1, (kw["B"] * kw["S"] + 127) // 128 + 1)
    case = synthetic.small_mla_case("fused", block_num=block_num, n_skip=1, **kw)
    _full_check(case, bsh=kw["S"] > 1)


# ---- the full-width RoPE tables are used elementwise (aclnnQkvRmsNormRopeCache "Formulas" (3)):
# every table element drawn on its own, so cos[t, j] != cos[t, j + Dr/2]; a kernel that read
# only one half of a row, or paired the wrong columns, fails here

def test_rope_tables_independent_decode_fused():
    # the decode workload: fused up-projection/absorb (query_rope) and the norm kernel (kr_cache)
    _full_check(dataclasses.replace(synthetic.MLA_DECODE, table_mode="independent", seed=2001))


def test_rope_tables_independent_separate_kernels():
    # N = 3 heads: the up-projection and absorb run as separate GEMMs (row-range decode schedule)
    _full_check(synthetic.small_mla_case("tables_sep", B=9, S=1, He=256, Hcq=128, N=3,
                                         block_num=2, n_skip=1, table_mode="independent"))


def test_rope_tables_independent_prefill_orientation():
    # T = 300 tokens: tokens as MMA rows with TMA-staged stores (prefill orientation)
    _full_check(synthetic.small_mla_case("tables_pf", B=3, S=100, He=384, Hcq=192, Hckv=128,
                                         N=2, block_num=4, n_skip=1, table_mode="independent"))


def test_rope_tables_independent_int8():
    # partial quant with int8 caches through the fused int8 kernel
    _full_check(dataclasses.replace(synthetic.MLA_PARTIAL_QUANT, table_mode="independent",
                                    seed=2002))
