"""GB300 (sm_103a) MLA prolog and QKV RmsNorm-RoPE-cache operators.

The compute lives in ``libmlaprolog.so`` (hand-written CUDA kernels behind the C ABI declared in
``include/mlaprolog.h``); this package holds the thin ctypes binding (``_lib``) and the build
script (``build``).
"""
from ._lib import (  # noqa: F401
    EXPORTS, MLAP_WEIGHT_DKV_KR, MLAP_WEIGHT_DQ, MLAP_WEIGHT_UK, MLAP_WEIGHT_UQ_QR, MlapError,
    PackedWeight, load, make_mla_args, make_qkv_args, mlap_check_errors, mlap_execute,
    mlap_get_workspace_size, mlap_prepack_size, mlap_prepack_weights, mlap_workspace_init,
    prepack, qkvrnrc_execute, qkvrnrc_get_workspace_size, tensor_desc, stamps_buffer,
    mlap_execute_stamped, qkvrnrc_execute_stamped, read_stamps)
from .prolog import MlaProlog, prepack_mla_weights  # noqa: F401
