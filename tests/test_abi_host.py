"""C-ABI checks that need no GPU: the library loads, exports every symbol the header declares,
and phase-1 validation (no device work) accepts the documented shapes and rejects the rest."""
import ctypes
import os
import re

import pytest
import torch

import __graft_entry__
from qkv_attention_prolog_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    __graft_entry__.build()
    return _lib.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "mlaprolog.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b((?:mlap|qkvrnrc)_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(built):
    names = _declared()
    assert len(names) >= 14
    for n in names:
        assert hasattr(built, n), n
    assert sorted(_lib.EXPORTS) == names


class Fake:
    """Stands in for a device tensor: only shape, dtype and an aligned fake address."""

    _next = 1 << 20

    def __init__(self, shape, dtype):
        self.shape = tuple(shape)
        self.dtype = dtype
        Fake._next += 1 << 16
        self.addr = Fake._next

    def desc(self, shape=None):
        d = _lib.mlap_tensor_t()
        n = 1
        for s in self.shape:
            n *= s
        d.data = self.addr if n > 0 else None
        d.dtype = _lib._TORCH_DTYPE[self.dtype]
        d.ndim = len(self.shape)
        for i, s in enumerate(self.shape):
            d.shape[i] = s
        return d


def _mla(T=128, He=7168, Hcq=1536, Hckv=512, N=128, D=128, Dr=64, BN=16, bsh=False,
         w_int8=False, cache_int8=False, full=False, xnorm=None):
    bf, i8, f32 = torch.bfloat16, torch.int8, torch.float32
    tok = (T // 2, 2) if bsh else (T,)
    t = {
        "token_x": Fake(tok + (He,), bf), "weight_dq": Fake((He, Hcq), bf),
        "weight_uq_qr": Fake((Hcq, N * (D + Dr)), i8 if w_int8 else bf),
        "weight_uk": Fake((N, D, Hckv), bf), "weight_dkv_kr": Fake((He, Hckv + Dr), bf),
        "rmsnorm_gamma_cq": Fake((Hcq,), bf), "rmsnorm_gamma_ckv": Fake((Hckv,), bf),
        "rope_sin": Fake(tok + (Dr,), bf), "rope_cos": Fake(tok + (Dr,), bf),
        "cache_index": Fake(tok, torch.int64),
        "kv_cache": Fake((BN, 128, 1, Hckv), i8 if cache_int8 else bf),
        "kr_cache": Fake((BN, 128, 1, Dr), i8 if cache_int8 else bf),
        "query": Fake(tok + (N, Hckv), bf), "query_rope": Fake(tok + (N, Dr), bf),
    }
    if w_int8:
        t["dequant_scale_w_uq_qr"] = Fake((1, N * (D + Dr)), f32)
        t["smooth_scales_cq"] = Fake((1, Hcq), f32)
    if cache_int8:
        t["quant_scale_ckv"] = Fake((1, Hckv), f32)
        t["quant_scale_ckr"] = Fake((1, Dr), f32)
    if full:   # 全量化: int8 x and down weights with dequant scales, int8 W^UQ|W^QR
        t["token_x"] = Fake(tok + (He,), i8)
        t["weight_dq"] = Fake((He, Hcq), i8)
        t["weight_dkv_kr"] = Fake((He, Hckv + Dr), i8)
        t["dequant_scale_x"] = Fake((T, 1), f32)
        t["dequant_scale_w_dq"] = Fake((1, Hcq), f32)
        t["dequant_scale_w_dkv_kr"] = Fake((1, Hckv + Dr), f32)
        t["kr_cache"] = Fake((BN, 128, 1, Dr), bf)
        t.pop("quant_scale_ckr", None)
        if cache_int8:   # int8 kv_cache: int8 query per token and head
            t["query"] = Fake(tok + (N, Hckv), i8)
            t["dequant_scale_q_nope"] = Fake((T, N, 1), f32)
    if xnorm is not None:   # input RmsNormQuant; deqScale per channel or one value
        t["rms_norm_quant_gamma"] = Fake((He,), bf)
        t["rms_norm_quant_bias"] = Fake((He,), bf)
        t["rms_norm_quant_deq_scale"] = Fake((He if xnorm == "channel" else 1,), f32)
    return t


def _args(t, cache_mode=None, eps=1e-6, eps_x=1e-6):
    a = _lib.mlap_args_t()
    for name in _lib._MLA_TENSORS:
        v = t.get(name)
        setattr(a, name, v.desc() if v is not None else _lib.tensor_desc(None))
    a.rmsnorm_epsilon_cq = eps
    a.rmsnorm_epsilon_ckv = eps
    a.rms_norm_quant_epsilon = eps_x
    a.cache_mode = cache_mode.encode() if cache_mode else None
    return a


def _status(a):
    out = ctypes.c_size_t()
    return _lib.load().mlap_get_workspace_size(ctypes.byref(a), ctypes.byref(out)), out.value


def test_valid_scenarios_size_the_workspace():
    for kw in [{}, {"bsh": True}, {"w_int8": True}, {"w_int8": True, "cache_int8": True},
               {"T": 8, "He": 2048, "Hcq": 512, "N": 16, "BN": 4}, {"T": 8192}]:
        st, ws = _status(_args(_mla(**kw), cache_mode="PA_BSND"))
        assert st == 0, (kw, _lib.load().mlap_last_error())
        assert ws >= 256


def test_empty_token_count_is_accepted():
    st, _ = _status(_args(_mla(T=0)))
    assert st == 0


def test_workspace_grows_with_tokens():
    _, small = _status(_args(_mla(T=8)))
    _, big = _status(_args(_mla(T=8192)))
    assert big > small


@pytest.mark.parametrize("mutate,code", [
    (lambda t: t.__setitem__("query", Fake((128, 128, 256), torch.bfloat16)), 2),
    (lambda t: t.__setitem__("rope_sin", Fake((128, 32), torch.bfloat16)), 2),
    (lambda t: t.__setitem__("cache_index", Fake((128,), torch.int8)), 3),
    (lambda t: t.__setitem__("weight_uk", Fake((128, 64, 512), torch.bfloat16)), 4),   # D != 128
    (lambda t: t.__setitem__("dequant_scale_x", Fake((128, 1), torch.float32)), 4),
    (lambda t: t.__setitem__("token_x", Fake((128, 7168), torch.int8)), 3),   # full quant: int8 W^DQ
    (lambda t: t.__setitem__("kv_cache", Fake((16, 128, 2, 512), torch.bfloat16)), 4),  # Nkv != 1
    (lambda t: t.__setitem__("quant_scale_ckv", Fake((1, 512), torch.float32)), 4),
    (lambda t: t.__setitem__("query_rope", Fake((128, 128, 64), torch.float32)), 3),
    (lambda t: t.pop("weight_dq"), 1),
])
def test_rejections(mutate, code):
    t = _mla()
    mutate(t)
    if "weight_dq" not in t:
        a = _args(t)
        a.weight_dq = _lib.tensor_desc(None)
        a.weight_dq.ndim = 2
        a.weight_dq.shape[0] = 7168
        a.weight_dq.shape[1] = 1536
        a.weight_dq.dtype = _lib.MLAP_DTYPE_BF16
    else:
        a = _args(t)
    st, _ = _status(a)
    assert st == code, _lib.load().mlap_last_error()


def test_cache_mode_and_scenario_rules():
    assert _status(_args(_mla(), cache_mode="PA_NZ"))[0] == 4
    # int8 caches without the partial-quant weight are outside the scenario matrix
    assert _status(_args(_mla(cache_int8=True)))[0] == 4
    # int8 weight without its dequant scale
    t = _mla(w_int8=True)
    t.pop("dequant_scale_w_uq_qr")
    assert _status(_args(t))[0] == 1


def test_misaligned_pointer_rejected():
    t = _mla()
    t["query"].addr += 8
    assert _status(_args(t))[0] == 4


def test_prepack_size():
    d = _lib.mlap_tensor_t()
    d.data = None
    d.dtype = _lib.MLAP_DTYPE_BF16
    d.ndim = 2
    d.shape[0], d.shape[1] = 1536, 128 * 192
    out = ctypes.c_size_t()
    assert _lib.load().mlap_prepack_size(ctypes.byref(d), 1, 128, 128, 64, ctypes.byref(out)) == 0
    assert out.value == 1536 * 128 * 192 * 2
    # inconsistent head geometry
    assert _lib.load().mlap_prepack_size(ctypes.byref(d), 1, 100, 128, 64, ctypes.byref(out)) == 2


def _qkv(T=16, Nq=4, Nk=2, Nv=2, D=128, quant=True, bn=4, bs=8):
    f16, i8, f32 = torch.float16, torch.int8, torch.float32
    t = {"qkv": Fake((T, (Nq + Nk + Nv) * D), f16), "gamma_q": Fake((D,), f16),
         "gamma_k": Fake((D,), f16), "cos": Fake((T, D), f16), "sin": Fake((T, D), f16),
         "index": Fake((T,), torch.int64),
         "k_cache": Fake((bn, bs, Nk, D), i8 if quant else f16),
         "v_cache": Fake((bn, bs, Nv, D), i8 if quant else f16),
         "q_out": Fake((T, Nq, D), f16)}
    if quant:
        t["k_scale"] = Fake((Nk, D), f32)
        t["v_scale"] = Fake((Nv, D), f32)
    return t


def _qargs(t, Nq=4, Nk=2, Nv=2, mode=None):
    a = _lib.qkvrnrc_args_t()
    for name in _lib._QKV_TENSORS:
        v = t.get(name)
        setattr(a, name, v.desc() if v is not None else _lib.tensor_desc(None))
    a.Nq, a.Nk, a.Nv = Nq, Nk, Nv
    a.epsilon = 1e-6
    a.cache_mode = mode.encode() if mode else None
    return a


def _qstatus(a):
    out = ctypes.c_size_t()
    return _lib.load().qkvrnrc_get_workspace_size(ctypes.byref(a), ctypes.byref(out))


def test_qkv_validation():
    assert _qstatus(_qargs(_qkv())) == 0
    assert _qstatus(_qargs(_qkv(quant=False))) == 0
    assert _qstatus(_qargs(_qkv(), mode="PA_NZ")) == 4
    assert _qstatus(_qargs(_qkv(D=64))) == 4                 # only D = 128
    assert _qstatus(_qargs(_qkv(Nk=2, Nv=3), Nk=2, Nv=3)) == 2   # Nk must equal Nv
    t = _qkv()
    t["k_offset"] = Fake((2, 128), torch.float32)
    assert _qstatus(_qargs(t)) == 1                          # asymmetric needs both offsets
    t["v_offset"] = Fake((2, 128), torch.float32)
    assert _qstatus(_qargs(t)) == 0                          # asymmetric quant
    t["v_offset"] = Fake((2, 128), torch.float16)
    assert _qstatus(_qargs(t)) == 3                          # offsets are fp32
    t["v_offset"] = Fake((2, 64), torch.float32)
    assert _qstatus(_qargs(t)) == 2                          # per channel (Nv, D)
    t = _qkv(quant=False)
    t["k_offset"] = Fake((2, 128), torch.float32)
    t["v_offset"] = Fake((2, 128), torch.float32)
    assert _qstatus(_qargs(t)) == 4                          # offsets without scales
    t = _qkv()                                               # before-quant outputs
    t["q_before_quant"] = Fake((16, 4, 128), torch.float16)
    t["k_before_quant"] = Fake((16, 2, 128), torch.float16)
    t["v_before_quant"] = Fake((16, 2, 128), torch.float16)
    assert _qstatus(_qargs(t)) == 0
    t["k_before_quant"] = Fake((16, 4, 128), torch.float16)
    assert _qstatus(_qargs(t)) == 2
    t["k_before_quant"] = Fake((16, 2, 128), torch.bfloat16)
    assert _qstatus(_qargs(t)) == 3
    t = _qkv()
    t["q_out"] = Fake((16, 4, 128), torch.bfloat16)
    assert _qstatus(_qargs(t)) == 3


def test_full_quant_scenarios():
    assert _status(_args(_mla(w_int8=True, full=True)))[0] == 0               # kv_cache bf16
    assert _status(_args(_mla(w_int8=True, cache_int8=True, full=True)))[0] == 0
    assert _status(_args(_mla(w_int8=True, cache_int8=True, full=True, bsh=True)))[0] == 0
    t = _mla(w_int8=True, full=True)
    t.pop("dequant_scale_x")
    assert _status(_args(t))[0] == 1
    t = _mla(w_int8=True, full=True)
    t["dequant_scale_w_dq"] = Fake((1, 1536), torch.bfloat16)
    assert _status(_args(t))[0] == 3
    t = _mla(full=True)                                   # full quant needs an int8 W^UQ|W^QR
    t.pop("dequant_scale_w_uq_qr", None)
    assert _status(_args(t))[0] == 4
    t = _mla(w_int8=True, cache_int8=True, full=True)
    t["kr_cache"] = Fake((16, 128, 1, 64), torch.int8)    # kr_cache stays bf16
    assert _status(_args(t))[0] == 4
    t = _mla(w_int8=True, cache_int8=True, full=True)
    t["query"] = Fake((128, 128, 512), torch.bfloat16)    # int8 kv_cache -> int8 query
    assert _status(_args(t))[0] == 4
    t = _mla(w_int8=True, cache_int8=True, full=True)
    t["dequant_scale_q_nope"] = Fake((128, 128), torch.float32)
    assert _status(_args(t))[0] == 2
    t = _mla(w_int8=True)
    t["query"] = Fake((128, 128, 512), torch.int8)        # int8 query outside full quant
    assert _status(_args(t))[0] == 3
    # an int8 query row is quantised from registers: Hckv <= 1024
    assert _status(_args(_mla(Hckv=1024, w_int8=True, cache_int8=True, full=True)))[0] == 0
    assert _status(_args(_mla(Hckv=1032, w_int8=True, cache_int8=True, full=True)))[0] == 4
    # full quant's own workspace regions: q^N staged in bf16 ahead of the int8 query, and from
    # 257 tokens (prefill orientation) token_x widened to f16 for the down-projection; up to 256
    # tokens the down-projection's converter warps expand the int8 token_x tiles themselves
    for T, widened in ((128, 0), (256, 0), (512, 512 * 7168 * 2)):
        extra = (_status(_args(_mla(T=T, w_int8=True, cache_int8=True, full=True)))[1]
                 - _status(_args(_mla(T=T, w_int8=True, cache_int8=True)))[1])
        assert extra == T * 128 * 512 * 2 + widened, (T, extra)


def test_rms_norm_quant_validation():
    # accepted with the bf16-x scenarios, deqScale per channel or one value
    assert _status(_args(_mla(xnorm="channel")))[0] == 0
    assert _status(_args(_mla(xnorm="tensor", bsh=True)))[0] == 0
    assert _status(_args(_mla(xnorm="channel", w_int8=True, cache_int8=True)))[0] == 0
    # the down-projection reads the normalised copy from the workspace: T * He * 2 more bytes
    assert (_status(_args(_mla(xnorm="channel")))[1]
            - _status(_args(_mla()))[1]) == 128 * 7168 * 2
    # all three parameters or none
    for name in ("rms_norm_quant_gamma", "rms_norm_quant_bias", "rms_norm_quant_deq_scale"):
        t = _mla(xnorm="channel")
        t.pop(name)
        assert _status(_args(t))[0] == 1, name
    t = _mla(xnorm="channel")
    t["rms_norm_quant_gamma"] = Fake((7168,), torch.float32)
    assert _status(_args(t))[0] == 3
    t = _mla(xnorm="channel")
    t["rms_norm_quant_bias"] = Fake((7167,), torch.bfloat16)
    assert _status(_args(t))[0] == 2
    t = _mla(xnorm="channel")
    t["rms_norm_quant_deq_scale"] = Fake((2,), torch.float32)
    assert _status(_args(t))[0] == 2
    t = _mla(xnorm="channel")
    t["rms_norm_quant_deq_scale"] = Fake((7168,), torch.bfloat16)
    assert _status(_args(t))[0] == 3
    assert _status(_args(_mla(xnorm="channel"), eps_x=-1.0))[0] == 2
    # not with full quant (int8 token_x), nor above He = 10240
    assert _status(_args(_mla(xnorm="channel", w_int8=True, full=True)))[0] == 4
    assert _status(_args(_mla(He=10496, xnorm="channel")))[0] == 4
    assert _status(_args(_mla(He=10240, xnorm="channel")))[0] == 0


def test_no_alloc_checks_its_scratch_limit_before_device_work():
    # the allocation-free call validates and sizes like the workspace call, and refuses shapes
    # beyond its static scratch (MLAP_ERR_WORKSPACE) before touching a device; an empty call
    # returns at once
    lib = _lib.load()
    assert _status(_args(_mla(T=200)))[1] > 24 * 1024 * 1024
    assert lib.mlap_execute_no_alloc(ctypes.byref(_args(_mla(T=200))), None) == 5
    assert "static scratch" in lib.mlap_last_error().decode()
    assert lib.mlap_execute_no_alloc(ctypes.byref(_args(_mla(T=0))), None) == 0
    t = _mla(T=64)
    t.pop("token_x")                    # the same validation as the workspace call, first
    bad = _status(_args(t))[0]
    assert bad != 0 and lib.mlap_execute_no_alloc(ctypes.byref(_args(t)), None) == bad
