"""Seeded synthetic inputs for the MLA prolog and the QKV RmsNorm-RoPE-cache epilogue.

This module is shared by the oracle tests, the CUDA parity tests and ``bench.py``.  It draws
random numbers and lays them out in the shapes and dtypes that the operator documentation gives
(MlaPrologV2 README, "参数说明" parameter table and the dtype/shape matrix of "约束说明";
aclnnQkvRmsNormRopeCache, "Formulas" and "Input shape restrictions").  It holds none of the
operators' arithmetic: no RmsNorm, no RoPE rotation, no quantisation.  The only computation here is
the construction of the caller-supplied RoPE angle tables from positions, which the operators
receive as inputs.

Every tensor is a CPU ``torch`` tensor; callers move them where they need them.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch


@dataclass(frozen=True)
class MlaDims:
    """Shape symbols of the MLA prolog (MlaPrologV2 README, "约束说明")."""

    B: int
    S: int
    He: int
    Hcq: int
    Hckv: int
    N: int
    D: int = 128
    Dr: int = 64
    block_num: int = 4
    block_size: int = 128

    @property
    def T(self) -> int:
        return self.B * self.S


@dataclass(frozen=True)
class MlaCase:
    """One seeded MLA prolog workload."""

    name: str
    dims: MlaDims
    seed: int
    # "bf16" = non-quant scenario; "int8" = partial quant with int8 weight_uq_qr
    weight_uq_qr_dtype: str = "bf16"
    # "bf16" or "int8" (partial quant, kv_cache quantised)
    cache_dtype: str = "bf16"
    # "random": unique random slots; "paged": contiguous runs per sequence in random blocks
    index_mode: str = "random"
    n_skip: int = 0            # number of cache_index entries set to -1
    pos_mode: str = "random"   # "random": positions in [0,4096); "sequence": 0..S-1 per sequence
    eps: float = 1e-6
    # full quant ("全量化"): int8 token_x, weight_dq, weight_dkv_kr with their dequant scales
    # (weight_uq_qr_dtype must be "int8"); with cache_dtype "int8" only kv_cache is int8 and
    # the query is int8 per token and head
    full_quant: bool = False
    # input RmsNormQuant (aclnnMlaPreprocessV2) ahead of the down-projection: None (off),
    # "channel" (deqScale per hidden channel) or "tensor" (one deqScale)
    x_norm: str | None = None
    # "paired": rope_sin/rope_cos built from positions (columns j and j + Dr/2 share an angle);
    # "independent": every table element drawn on its own from U(-1, 1), so no column repeats
    # another and the elementwise use of the full-width tables is what is tested
    table_mode: str = "paired"


# The five workloads.  Sizes, distributions and cache layouts follow the stated workload recipe.
MLA_TINY = MlaCase("tiny_bf16_T8", MlaDims(B=8, S=1, He=2048, Hcq=512, Hckv=512, N=16,
                                           block_num=4), seed=1000, n_skip=2)
MLA_DECODE = MlaCase("decode_bf16_T128", MlaDims(B=128, S=1, He=7168, Hcq=1536, Hckv=512,
                                                 N=128, block_num=1024), seed=1001)
MLA_PREFILL = MlaCase("prefill_bf16_T8192", MlaDims(B=4, S=2048, He=7168, Hcq=1536, Hckv=512,
                                                    N=128, block_num=1024), seed=1002,
                      index_mode="paged", pos_mode="sequence")
MLA_PARTIAL_QUANT = MlaCase("partial_quant_int8cache_T64",
                            MlaDims(B=64, S=1, He=6144, Hcq=1536, Hckv=512, N=64,
                                    block_num=1024), seed=1003,
                            weight_uq_qr_dtype="int8", cache_dtype="int8")
# partial quant with bf16 kv_cache (the scenario's other column)
MLA_PARTIAL_QUANT_BF16CACHE = replace(MLA_PARTIAL_QUANT, name="partial_quant_bf16cache_T64",
                                      cache_dtype="bf16", seed=1005)
# full quant, both kv_cache columns, at the partial-quant shapes
MLA_FULL_QUANT = replace(MLA_PARTIAL_QUANT, name="full_quant_int8cache_T64", seed=1006,
                         full_quant=True)
MLA_FULL_QUANT_BF16CACHE = replace(MLA_PARTIAL_QUANT, name="full_quant_bf16cache_T64",
                                   seed=1007, full_quant=True, cache_dtype="bf16")
# the input RmsNormQuant of aclnnMlaPreprocessV2 ahead of the decode prolog
MLA_XNORM = replace(MLA_DECODE, name="decode_xnorm_T128", seed=1008, x_norm="channel")


@dataclass(frozen=True)
class QkvDims:
    """Shape symbols of QkvRmsNormRopeCache (aclnnQkvRmsNormRopeCache, "Input shape restrictions")."""

    B: int
    S: int
    Nq: int
    Nk: int
    Nv: int
    D: int = 128
    block_num: int = 160
    block_size: int = 128

    @property
    def T(self) -> int:
        return self.B * self.S


@dataclass(frozen=True)
class QkvCase:
    name: str
    dims: QkvDims
    seed: int
    quant: str = "symmetric"   # "none" (fp16 caches), "symmetric" or "asymmetric" (int8 caches)
    before_quant: bool = False # request the optional qBeforeQuant / kBeforeQuant / vBeforeQuant
    skip_frac: float = 0.01
    eps: float = 1e-6
    table_mode: str = "paired"  # as MlaCase.table_mode


QKV_EPILOGUE = QkvCase("qkv_rnrc_fp16_16x1024", QkvDims(B=16, S=1024, Nq=32, Nk=8, Nv=8),
                       seed=1004)
# Same shapes with asymmetric quant (offsets ~ U(-16, 16)) and the three before-quant outputs.
QKV_EPILOGUE_ASYM = QkvCase("qkv_rnrc_fp16_16x1024_asym_bq",
                            QkvDims(B=16, S=1024, Nq=32, Nk=8, Nv=8), seed=1005,
                            quant="asymmetric", before_quant=True)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _uniform(g, shape, lo, hi, dtype=torch.float32):
    return (torch.rand(shape, generator=g, dtype=torch.float64) * (hi - lo) + lo).to(dtype)


def rope_tables(positions: torch.Tensor, dim: int, dtype, base: float = 10000.0):
    """sin/cos tables in the half-and-half layout: column j and j+dim/2 share angle pos*base^(-2j/dim).

    The tables are operator inputs (rope_sin/rope_cos); only their construction lives here.
    """
    half = dim // 2
    j = torch.arange(half, dtype=torch.float64)
    inv = base ** (-2.0 * j / dim)
    ang = positions.to(torch.float64)[:, None] * inv[None, :]
    ang = torch.cat([ang, ang], dim=-1)
    return torch.sin(ang).to(dtype), torch.cos(ang).to(dtype)


def _slots(g, case_index_mode, T, B, S, block_num, block_size, n_skip):
    total = block_num * block_size
    if total == 0:
        return torch.full((T,), -1, dtype=torch.int64)   # empty cache: nothing can be stored
    if case_index_mode == "random":
        if T > total:
            raise ValueError("more tokens than cache slots")
        idx = torch.randperm(total, generator=g)[:T].to(torch.int64)
    elif case_index_mode == "paged":
        per_seq = math.ceil(S / block_size)
        blocks = torch.randperm(block_num, generator=g)[: B * per_seq].to(torch.int64)
        idx = torch.empty(T, dtype=torch.int64)
        for b in range(B):
            for s in range(S):
                blk = blocks[b * per_seq + s // block_size]
                idx[b * S + s] = blk * block_size + (s % block_size)
    else:
        raise ValueError(case_index_mode)
    if n_skip:
        where = torch.randperm(T, generator=g)[:n_skip]
        idx[where] = -1
    return idx


def make_mla_inputs(case: MlaCase) -> dict:
    """All operator inputs of one MLA prolog workload, keyed by the parameter-table names."""
    d = case.dims
    g = _gen(case.seed)
    T = d.T
    bf16 = torch.bfloat16
    inp: dict = {}
    inp["token_x"] = torch.randn(T, d.He, generator=g).to(bf16)

    def w(k, n):
        return (torch.randn(k, n, generator=g) / math.sqrt(k)).to(bf16)

    def i8(*shape):
        return torch.randint(-127, 128, shape, generator=g, dtype=torch.int8)

    if case.full_quant:
        # int8 x and down-projection weights; dequant scales sized so that x·W is O(1):
        # sum over He of U[-127,127]^2 products has std ~ 5e4*sqrt(He/100), times ~2.2e-6
        inp["token_x"] = i8(T, d.He)
        inp["dequant_scale_x"] = _uniform(g, (T, 1), 1e-3, 2e-3)
        inp["weight_dq"] = i8(d.He, d.Hcq)
        inp["dequant_scale_w_dq"] = _uniform(g, (1, d.Hcq), 1e-3, 2e-3)
    else:
        inp["weight_dq"] = w(d.He, d.Hcq)
    if case.weight_uq_qr_dtype == "int8":
        inp["weight_uq_qr"] = torch.randint(-127, 128, (d.Hcq, d.N * (d.D + d.Dr)), generator=g,
                                            dtype=torch.int8)
        inp["dequant_scale_w_uq_qr"] = _uniform(g, (1, d.N * (d.D + d.Dr)), 1e-3, 1e-2)
        inp["smooth_scales_cq"] = _uniform(g, (1, d.Hcq), 0.5, 1.5)
    else:
        inp["weight_uq_qr"] = w(d.Hcq, d.N * (d.D + d.Dr))
    inp["weight_uk"] = (torch.randn(d.N, d.D, d.Hckv, generator=g) / math.sqrt(d.D)).to(bf16)
    if case.full_quant:
        inp["weight_dkv_kr"] = i8(d.He, d.Hckv + d.Dr)
        inp["dequant_scale_w_dkv_kr"] = _uniform(g, (1, d.Hckv + d.Dr), 1e-3, 2e-3)
    else:
        inp["weight_dkv_kr"] = w(d.He, d.Hckv + d.Dr)
    inp["rmsnorm_gamma_cq"] = _uniform(g, (d.Hcq,), 0.5, 1.5, bf16)
    inp["rmsnorm_gamma_ckv"] = _uniform(g, (d.Hckv,), 0.5, 1.5, bf16)
    if case.pos_mode == "random":
        pos = torch.randint(0, 4096, (T,), generator=g)
    else:
        pos = torch.arange(d.S).repeat(d.B)
    inp["rope_sin"], inp["rope_cos"] = rope_tables(pos, d.Dr, bf16)
    inp["cache_index"] = _slots(g, case.index_mode, T, d.B, d.S, d.block_num, d.block_size,
                                case.n_skip)
    if case.cache_dtype == "int8" and case.full_quant:   # kv int8 per channel, kr stays bf16
        inp["kv_cache"] = torch.randint(-128, 128, (d.block_num, d.block_size, 1, d.Hckv),
                                        generator=g, dtype=torch.int8)
        inp["kr_cache"] = torch.randn(d.block_num, d.block_size, 1, d.Dr, generator=g).to(bf16)
        inp["quant_scale_ckv"] = _uniform(g, (1, d.Hckv), 0.01, 0.05)
    elif case.cache_dtype == "int8":
        inp["kv_cache"] = torch.randint(-128, 128, (d.block_num, d.block_size, 1, d.Hckv),
                                        generator=g, dtype=torch.int8)
        inp["kr_cache"] = torch.randint(-128, 128, (d.block_num, d.block_size, 1, d.Dr),
                                        generator=g, dtype=torch.int8)
        inp["quant_scale_ckv"] = _uniform(g, (1, d.Hckv), 0.01, 0.05)
        inp["quant_scale_ckr"] = _uniform(g, (1, d.Dr), 0.01, 0.05)
    else:
        inp["kv_cache"] = torch.randn(d.block_num, d.block_size, 1, d.Hckv, generator=g).to(bf16)
        inp["kr_cache"] = torch.randn(d.block_num, d.block_size, 1, d.Dr, generator=g).to(bf16)
    inp["rmsnorm_epsilon_cq"] = case.eps
    inp["rmsnorm_epsilon_ckv"] = case.eps
    if case.x_norm is not None:   # drawn last: the other inputs match the case without it
        inp["rms_norm_quant_gamma"] = _uniform(g, (d.He,), 0.5, 1.5, bf16)
        inp["rms_norm_quant_bias"] = _uniform(g, (d.He,), -0.25, 0.25, bf16)
        inp["rms_norm_quant_deq_scale"] = _uniform(g, (d.He if case.x_norm == "channel" else 1,),
                                                   0.5, 2.0)
        inp["rms_norm_quant_epsilon"] = case.eps
    if case.table_mode == "independent":   # drawn last, like the RmsNormQuant parameters
        inp["rope_sin"] = _uniform(g, (T, d.Dr), -1.0, 1.0, bf16)
        inp["rope_cos"] = _uniform(g, (T, d.Dr), -1.0, 1.0, bf16)
    return inp


def make_qkv_inputs(case: QkvCase) -> dict:
    """All inputs of one QkvRmsNormRopeCache workload."""
    d = case.dims
    g = _gen(case.seed)
    T = d.T
    f16 = torch.float16
    inp: dict = {}
    inp["qkv"] = torch.randn(d.B, d.S, (d.Nq + d.Nk + d.Nv) * d.D, generator=g).to(f16)
    inp["gamma_q"] = _uniform(g, (d.D,), 0.5, 1.5, f16)
    inp["gamma_k"] = _uniform(g, (d.D,), 0.5, 1.5, f16)
    pos = torch.arange(d.S).repeat(d.B)
    inp["sin"], inp["cos"] = rope_tables(pos, d.D, f16)
    total = d.block_num * d.block_size
    idx = torch.randperm(total, generator=g)[:T].to(torch.int64)
    n_skip = int(round(case.skip_frac * T))
    if n_skip:
        idx[torch.randperm(T, generator=g)[:n_skip]] = -1
    inp["index"] = idx
    if case.quant in ("symmetric", "asymmetric"):
        inp["k_scale"] = _uniform(g, (d.Nk, d.D), 0.02, 0.1)
        inp["v_scale"] = _uniform(g, (d.Nv, d.D), 0.02, 0.1)
        if case.quant == "asymmetric":
            inp["k_offset"] = _uniform(g, (d.Nk, d.D), -16.0, 16.0)
            inp["v_offset"] = _uniform(g, (d.Nv, d.D), -16.0, 16.0)
        inp["k_cache"] = torch.randint(-128, 128, (d.block_num, d.block_size, d.Nk, d.D),
                                       generator=g, dtype=torch.int8)
        inp["v_cache"] = torch.randint(-128, 128, (d.block_num, d.block_size, d.Nv, d.D),
                                       generator=g, dtype=torch.int8)
    else:
        inp["k_cache"] = torch.randn(d.block_num, d.block_size, d.Nk, d.D, generator=g).to(f16)
        inp["v_cache"] = torch.randn(d.block_num, d.block_size, d.Nv, d.D, generator=g).to(f16)
    inp["epsilon"] = case.eps
    if case.table_mode == "independent":   # drawn last: the other inputs stay as in "paired"
        inp["sin"] = _uniform(g, (T, d.D), -1.0, 1.0, f16)
        inp["cos"] = _uniform(g, (T, d.D), -1.0, 1.0, f16)
    return inp


def small_mla_case(name, B=2, S=3, He=256, Hcq=128, Hckv=128, N=2, D=128, Dr=64, block_num=2,
                   seed=7, **kw) -> MlaCase:
    """A hand-sized MLA workload for parity tests of tile edges and ragged tails."""
    return MlaCase(name, MlaDims(B=B, S=S, He=He, Hcq=Hcq, Hckv=Hckv, N=N, D=D, Dr=Dr,
                                 block_num=block_num), seed=seed, **kw)
