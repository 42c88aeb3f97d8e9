"""Convenience wrappers over the C ABI: prepack the four MLA weights once, then call execute.

Marshalling only: prepacking and every step of the prolog run in libmlaprolog's kernels.
"""
from __future__ import annotations

import torch

from . import _lib


def prepack_mla_weights(weights: dict, N: int, D: int, Dr: int, stream=None) -> dict:
    """Prepack weight_dq, weight_uq_qr, weight_uk, weight_dkv_kr (row-major device tensors, the
    parameter-table shapes) into the library layout; returns PackedWeight objects by name."""
    ids = {"weight_dq": _lib.MLAP_WEIGHT_DQ, "weight_uq_qr": _lib.MLAP_WEIGHT_UQ_QR,
           "weight_uk": _lib.MLAP_WEIGHT_UK, "weight_dkv_kr": _lib.MLAP_WEIGHT_DKV_KR}
    return {name: _lib.prepack(weights[name], which, N, D, Dr, stream)
            for name, which in ids.items()}


class MlaProlog:
    """Holds prepacked weights and a workspace; ``run`` executes one prolog call.

    ``tensors`` passed to ``run`` are device tensors keyed by the parameter-table names
    (token_x, rmsnorm_gamma_*, rope_sin/cos, cache_index, kv_cache, kr_cache, query,
    query_rope and the optional scales).  Outputs and caches are written in place.
    """

    def __init__(self, weights: dict, N: int, D: int, Dr: int, stream=None):
        self.packed = prepack_mla_weights(weights, N, D, Dr, stream)
        self.ws = None

    def args(self, tensors: dict, eps_cq=1e-6, eps_ckv=1e-6, cache_mode=None, eps_x=None):
        merged = dict(tensors)
        merged.update(self.packed)
        return _lib.make_mla_args(merged, eps_cq, eps_ckv, cache_mode, eps_x)

    def ensure_workspace(self, args, device) -> torch.Tensor:
        need = _lib.mlap_get_workspace_size(args)
        if self.ws is None or self.ws.numel() < need:
            self.ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
            _lib.mlap_workspace_init(self.ws)
        return self.ws

    def run(self, tensors: dict, eps_cq=1e-6, eps_ckv=1e-6, cache_mode=None, stream=None,
            eps_x=None):
        """eps_x: epsilon of the input RmsNormQuant (used when its parameters are present)."""
        a = self.args(tensors, eps_cq, eps_ckv, cache_mode, eps_x)
        ws = self.ensure_workspace(a, tensors["token_x"].device)
        _lib.mlap_execute(a, ws, stream)
        return a
