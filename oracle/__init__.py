"""CPU oracle for the MLA prolog and the QKV RmsNorm-RoPE-cache epilogue — TEST INFRASTRUCTURE.

This package is the plain, slow, obviously correct definition that the CUDA path is checked
against.  Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
(and its ``--impl reference`` arm) may import it.  The library in ``qkv_attention_prolog_gb300``
never imports, calls or links anything here, and nothing here imports the library: the two share
no code.  Inputs come from the seeded generators in ``synthetic`` only.

Arithmetic is float64 (numpy), with rounding to bf16 / fp16 / int8 only at the points the
readings below fix.  Every function cites the passage of the operator documentation it follows:

* "MlaPrologV2 README" = gitcode ops-transformer ``attention/mla_prolog_v2/README.md``
  ("功能说明" formulas, "参数说明" parameter table, "约束说明" shape and scenario matrix);
* "aclnnQkvRmsNormRopeCache" = the CANN API page of that name ("Formulas" (1)-(4),
  "Other restrictions");
* "aclnnMlaPreprocessV2" = the CANN API page of that name ("Formula": RMS, RmsNorm and the input
  RmsNormQuant).

Pins: every function here is pinned by ``tests/test_oracle_pins.py`` against closed forms,
invariants, library routines for special cases and brute force on tiny inputs.  No function is
left with parity unpinned.
"""
from .rounding import round_bf16, round_fp16, round_fp32, saturate_int8_rne
from .mla_prolog import (rms_norm, rms_norm_quant, rope_half_and_half, dynamic_quant_per_token,
                         cache_quant, mla_prolog, scatter_rows)
from .qkv_rms_norm_rope_cache import qkv_rms_norm_rope_cache

__all__ = [
    "round_bf16", "round_fp16", "round_fp32", "saturate_int8_rne", "rms_norm", "rms_norm_quant",
    "rope_half_and_half", "dynamic_quant_per_token", "cache_quant", "mla_prolog",
    "scatter_rows", "qkv_rms_norm_rope_cache",
]
