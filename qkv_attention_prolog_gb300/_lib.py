"""ctypes binding of libmlaprolog (include/mlaprolog.h): argument marshalling only.

Every compute step runs in the library's CUDA kernels; this module only turns torch tensors into
``mlap_tensor_t`` descriptors (device pointer, dtype, shape) and checks status codes.  Loading
fails loudly when the library has not been built: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmlaprolog.so")

MLAP_DTYPE_INVALID, MLAP_DTYPE_BF16, MLAP_DTYPE_FP16, MLAP_DTYPE_FP32, MLAP_DTYPE_INT8, \
    MLAP_DTYPE_INT64 = range(6)
MLAP_WEIGHT_DQ, MLAP_WEIGHT_UQ_QR, MLAP_WEIGHT_UK, MLAP_WEIGHT_DKV_KR = range(4)
# execution stamps (include/mlaprolog.h): slots of MLAP_STAMP_BLOCK uint64 words
MLAP_STAMP_KERNELS, MLAP_STAMP_BLOCK, MLAP_STAMP_CTAS = 5, 1024, 255
MLAP_STAMP_DOWN, MLAP_STAMP_NORM, MLAP_STAMP_UP, MLAP_STAMP_ABSORB, MLAP_STAMP_QKV = range(5)
STAMP_NAMES = {MLAP_STAMP_DOWN: "down", MLAP_STAMP_NORM: "norm_scatter", MLAP_STAMP_UP: "up",
               MLAP_STAMP_ABSORB: "absorb", MLAP_STAMP_QKV: "qkv_rnrc"}

STATUS_NAMES = {0: "MLAP_OK", 1: "MLAP_ERR_NULL", 2: "MLAP_ERR_SHAPE", 3: "MLAP_ERR_DTYPE",
                4: "MLAP_ERR_UNSUPPORTED", 5: "MLAP_ERR_WORKSPACE", 6: "MLAP_ERR_CUDA",
                7: "MLAP_ERR_INDEX_RANGE", 8: "MLAP_ERR_TIMEOUT"}

_TORCH_DTYPE = {torch.bfloat16: MLAP_DTYPE_BF16, torch.float16: MLAP_DTYPE_FP16,
                torch.float32: MLAP_DTYPE_FP32, torch.int8: MLAP_DTYPE_INT8,
                torch.int64: MLAP_DTYPE_INT64}

# Every symbol include/mlaprolog.h declares.
EXPORTS = ["mlap_prepack_size", "mlap_prepack_weights", "mlap_get_workspace_size",
           "mlap_workspace_init", "mlap_execute", "mlap_check_errors",
           "qkvrnrc_get_workspace_size", "qkvrnrc_execute", "mlap_status_string",
           "mlap_last_error", "mlap_execute_stamped", "qkvrnrc_execute_stamped",
           "mlap_execute_no_alloc", "mlap_selftest_bounded_wait"]


class MlapError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        self.name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{where}: {self.name}: {detail}")


class mlap_tensor_t(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4)]


_MLA_TENSORS = ["token_x", "weight_dq", "weight_uq_qr", "weight_uk", "weight_dkv_kr",
                "rmsnorm_gamma_cq", "rmsnorm_gamma_ckv", "rope_sin", "rope_cos", "cache_index",
                "kv_cache", "kr_cache", "dequant_scale_x", "dequant_scale_w_dq",
                "dequant_scale_w_uq_qr", "dequant_scale_w_dkv_kr", "quant_scale_ckv",
                "quant_scale_ckr", "smooth_scales_cq", "query", "query_rope",
                "dequant_scale_q_nope", "rms_norm_quant_gamma", "rms_norm_quant_bias",
                "rms_norm_quant_deq_scale"]


class mlap_args_t(ctypes.Structure):
    _fields_ = ([(n, mlap_tensor_t) for n in _MLA_TENSORS]
                + [("rmsnorm_epsilon_cq", ctypes.c_double),
                   ("rmsnorm_epsilon_ckv", ctypes.c_double),
                   ("rms_norm_quant_epsilon", ctypes.c_double), ("cache_mode", ctypes.c_char_p)])


_QKV_TENSORS = ["qkv", "gamma_q", "gamma_k", "cos", "sin", "index", "k_cache", "v_cache",
                "k_scale", "v_scale", "k_offset", "v_offset", "q_out", "q_before_quant",
                "k_before_quant", "v_before_quant"]


class qkvrnrc_args_t(ctypes.Structure):
    _fields_ = ([(n, mlap_tensor_t) for n in _QKV_TENSORS]
                + [("Nq", ctypes.c_int32), ("Nk", ctypes.c_int32), ("Nv", ctypes.c_int32),
                   ("epsilon", ctypes.c_double), ("cache_mode", ctypes.c_char_p)])


_lib = None


def load() -> ctypes.CDLL:
    """Load libmlaprolog.so (built by ``qkv_attention_prolog_gb300.build``); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libmlaprolog.so is not built ({LIB_PATH}); run "
                           "`python -c 'import __graft_entry__ as g; g.build()'` first")
    lib = ctypes.CDLL(LIB_PATH)
    st = ctypes.c_int32
    sz = ctypes.POINTER(ctypes.c_size_t)
    vp = ctypes.c_void_p
    T = ctypes.POINTER(mlap_tensor_t)
    A = ctypes.POINTER(mlap_args_t)
    Q = ctypes.POINTER(qkvrnrc_args_t)
    sig = {
        "mlap_prepack_size": (st, [T, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                   ctypes.c_int32, sz]),
        "mlap_prepack_weights": (st, [T, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                      ctypes.c_int32, vp, vp]),
        "mlap_get_workspace_size": (st, [A, sz]),
        "mlap_workspace_init": (st, [vp, ctypes.c_size_t, vp]),
        "mlap_execute": (st, [A, vp, ctypes.c_size_t, vp]),
        "mlap_check_errors": (st, [vp, vp]),
        "mlap_selftest_bounded_wait": (st, [vp, ctypes.c_size_t, vp]),
        "qkvrnrc_get_workspace_size": (st, [Q, sz]),
        "qkvrnrc_execute": (st, [Q, vp, ctypes.c_size_t, vp]),
        "mlap_status_string": (ctypes.c_char_p, [st]),
        "mlap_last_error": (ctypes.c_char_p, []),
        "mlap_execute_stamped": (st, [A, vp, ctypes.c_size_t, vp, vp]),
        "qkvrnrc_execute_stamped": (st, [Q, vp, ctypes.c_size_t, vp, vp]),
        "mlap_execute_no_alloc": (st, [A, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int, where: str):
    if status != 0:
        raise MlapError(status, where, load().mlap_last_error().decode())


def tensor_desc(t, shape=None, dtype=None) -> mlap_tensor_t:
    """Descriptor of a dense tensor; ``None`` gives an absent (NULL) parameter.  ``shape`` and
    ``dtype`` override the logical shape/dtype (used for prepacked weights, whose buffer holds
    the weight in the library's layout)."""
    d = mlap_tensor_t()
    if t is None:
        d.data = None
        d.dtype = MLAP_DTYPE_INVALID
        d.ndim = 0
        return d
    if not t.is_contiguous():
        raise ValueError("tensors passed to libmlaprolog must be contiguous")
    shp = list(t.shape if shape is None else shape)
    if len(shp) > 4:
        raise ValueError("at most 4 dimensions")
    d.data = t.data_ptr() if t.numel() > 0 else None
    d.dtype = _TORCH_DTYPE[t.dtype] if dtype is None else dtype
    d.ndim = len(shp)
    for i, s in enumerate(shp):
        d.shape[i] = int(s)
    return d


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


# --------------------------------------------------------------------------------- MLA prolog
def mlap_prepack_size(w_logical_shape, dtype, which: int, N=0, D=0, Dr=0) -> int:
    d = mlap_tensor_t()
    d.data = None
    d.dtype = _TORCH_DTYPE[dtype]
    d.ndim = len(w_logical_shape)
    for i, s in enumerate(w_logical_shape):
        d.shape[i] = int(s)
    out = ctypes.c_size_t()
    _check(load().mlap_prepack_size(ctypes.byref(d), which, N, D, Dr, ctypes.byref(out)),
           "mlap_prepack_size")
    return out.value


def mlap_prepack_weights(w: torch.Tensor, which: int, N=0, D=0, Dr=0, stream=None):
    """Repack a row-major device weight; returns a new device buffer in the library layout."""
    nbytes = mlap_prepack_size(tuple(w.shape), w.dtype, which, N, D, Dr)
    dst = torch.empty(nbytes // w.element_size(), dtype=w.dtype, device=w.device)
    d = tensor_desc(w)
    _check(load().mlap_prepack_weights(ctypes.byref(d), which, N, D, Dr, dst.data_ptr(),
                                       _stream_ptr(stream)), "mlap_prepack_weights")
    return dst


class PackedWeight:
    """A prepacked device buffer together with the logical (row-major) shape and dtype."""

    def __init__(self, buf: torch.Tensor, shape, dtype):
        self.buf, self.shape, self.dtype = buf, tuple(shape), dtype

    def desc(self) -> mlap_tensor_t:
        return tensor_desc(self.buf, shape=self.shape, dtype=_TORCH_DTYPE[self.dtype])


def prepack(w: torch.Tensor, which: int, N=0, D=0, Dr=0, stream=None) -> PackedWeight:
    return PackedWeight(mlap_prepack_weights(w, which, N, D, Dr, stream), w.shape, w.dtype)


def make_mla_args(tensors: dict, eps_cq=1e-6, eps_ckv=1e-6, cache_mode=None,
                  eps_x=None) -> mlap_args_t:
    """Fill mlap_args_t from a dict keyed by the parameter-table names; weights may be
    PackedWeight.  Missing optional keys are absent.  eps_x (the input RmsNormQuant epsilon)
    defaults to tensors["rms_norm_quant_epsilon"] when that key is present, else 1e-6."""
    a = mlap_args_t()
    for name in _MLA_TENSORS:
        v = tensors.get(name)
        setattr(a, name, v.desc() if isinstance(v, PackedWeight) else tensor_desc(v))
    a.rmsnorm_epsilon_cq = float(eps_cq)
    a.rmsnorm_epsilon_ckv = float(eps_ckv)
    a.rms_norm_quant_epsilon = float(tensors.get("rms_norm_quant_epsilon", 1e-6) if eps_x is None
                                     else eps_x)
    a.cache_mode = cache_mode.encode() if cache_mode else None
    return a


def mlap_get_workspace_size(args: mlap_args_t) -> int:
    out = ctypes.c_size_t()
    _check(load().mlap_get_workspace_size(ctypes.byref(args), ctypes.byref(out)),
           "mlap_get_workspace_size")
    return out.value


def mlap_workspace_init(ws: torch.Tensor, stream=None):
    _check(load().mlap_workspace_init(ws.data_ptr(), ws.numel() * ws.element_size(),
                                      _stream_ptr(stream)), "mlap_workspace_init")


def mlap_execute(args: mlap_args_t, ws: torch.Tensor, stream=None):
    _check(load().mlap_execute(ctypes.byref(args), ws.data_ptr(), ws.numel() * ws.element_size(),
                               _stream_ptr(stream)), "mlap_execute")


def mlap_execute_no_alloc(args: mlap_args_t, stream=None):
    """mlap_execute without a workspace: the library's static device scratch is used instead
    (for callers that cannot allocate device memory; see include/mlaprolog.h)."""
    _check(load().mlap_execute_no_alloc(ctypes.byref(args), _stream_ptr(stream)),
           "mlap_execute_no_alloc")


def mlap_check_errors(ws: torch.Tensor, stream=None) -> int:
    """Returns the status code (0 = OK); does not raise for kernel-reported errors."""
    return int(load().mlap_check_errors(ws.data_ptr(), _stream_ptr(stream)))


def mlap_selftest_bounded_wait(ws: torch.Tensor, stream=None):
    """Run the library's bounded wait on a barrier nothing completes (about 2 s on the GPU);
    mlap_check_errors(ws) then reports MLAP_ERR_TIMEOUT."""
    _check(load().mlap_selftest_bounded_wait(ws.data_ptr(), ws.numel() * ws.element_size(),
                                             _stream_ptr(stream)), "mlap_selftest_bounded_wait")


# --------------------------------------------------------------------------------- QKV entry
def make_qkv_args(tensors: dict, Nq, Nk, Nv, epsilon=1e-6, cache_mode=None) -> qkvrnrc_args_t:
    a = qkvrnrc_args_t()
    for name in _QKV_TENSORS:
        setattr(a, name, tensor_desc(tensors.get(name)))
    a.Nq, a.Nk, a.Nv = Nq, Nk, Nv
    a.epsilon = float(epsilon)
    a.cache_mode = cache_mode.encode() if cache_mode else None
    return a


def qkvrnrc_get_workspace_size(args: qkvrnrc_args_t) -> int:
    out = ctypes.c_size_t()
    _check(load().qkvrnrc_get_workspace_size(ctypes.byref(args), ctypes.byref(out)),
           "qkvrnrc_get_workspace_size")
    return out.value


def qkvrnrc_execute(args: qkvrnrc_args_t, ws: torch.Tensor, stream=None):
    _check(load().qkvrnrc_execute(ctypes.byref(args), ws.data_ptr(),
                                  ws.numel() * ws.element_size(), _stream_ptr(stream)),
           "qkvrnrc_execute")


# --------------------------------------------------------------------------------- profiling
def stamps_buffer(device, calls: int = 1) -> torch.Tensor:
    """Device buffer for the execution stamps of `calls` calls (one stamps area per call)."""
    return torch.zeros(calls, MLAP_STAMP_KERNELS * MLAP_STAMP_BLOCK, dtype=torch.int64,
                       device=device)


def mlap_execute_stamped(args: mlap_args_t, ws: torch.Tensor, stamps: torch.Tensor, stream=None):
    """mlap_execute whose kernels also record %globaltimer stamps into `stamps` (one row of
    stamps_buffer, zeroed by the caller beforehand)."""
    _check(load().mlap_execute_stamped(ctypes.byref(args), ws.data_ptr(),
                                       ws.numel() * ws.element_size(), _stream_ptr(stream),
                                       stamps.data_ptr()), "mlap_execute_stamped")


def qkvrnrc_execute_stamped(args: qkvrnrc_args_t, ws: torch.Tensor, stamps: torch.Tensor,
                            stream=None):
    _check(load().qkvrnrc_execute_stamped(ctypes.byref(args), ws.data_ptr(),
                                          ws.numel() * ws.element_size(), _stream_ptr(stream),
                                          stamps.data_ptr()), "qkvrnrc_execute_stamped")


def read_stamps(stamps_row) -> dict:
    """Per kernel that ran: its span (earliest CTA start to latest CTA end, ns), the time from
    the first wait on the preceding kernel returning to the latest end (ns), and the per-CTA
    stamps [start, dependency resolved, main work done, end] of the first CTAs (ns, relative to
    the earliest start of the call)."""
    import numpy as np
    w = np.asarray(stamps_row.detach().cpu().numpy(), dtype=np.int64).view(np.uint64)
    blocks = w.reshape(MLAP_STAMP_KERNELS, MLAP_STAMP_BLOCK)
    starts = [int(~b[0]) for b in blocks if b[1] != 0]
    if not starts:
        return {}
    t0 = min(starts)
    out = {}
    for k, b in enumerate(blocks):
        if b[1] == 0:
            continue
        first = int(~b[0])
        cta = b[4:4 + 4 * MLAP_STAMP_CTAS].reshape(MLAP_STAMP_CTAS, 4).astype(np.int64)
        used = cta[:, 0] != 0
        dep = cta[used, 1]
        dep = dep[dep != 0]
        out[STAMP_NAMES[k]] = {
            "start_ns": first - t0, "end_ns": int(b[1]) - t0, "span_ns": int(b[1]) - first,
            "dep_to_end_ns": (int(b[1]) - int(dep.min())) if dep.size else None,
            "ctas": np.where(cta[used] != 0, cta[used] - t0, -1).tolist()}
    return out
