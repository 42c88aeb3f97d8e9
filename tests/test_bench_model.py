"""The benchmark's algorithmic byte and FLOP model against hand-derived totals.

Each figure counts every weight, input and output once (intermediates such as c^Q and q^C stay
on chip), e.g. decode T=128: weights 122.55 MB (He·(Hcq+Hckv+Dr) + Hcq·N·(D+Dr) + N·D·Hckv, bf16)
+ x 1.84 + query 16.78 + query_rope 2.10 + cache rows 0.15 + sin/cos 0.03 + cache_index 0.001 MB.
"""
import pytest

import bench
import synthetic


@pytest.mark.parametrize("case,mb,gflop", [
    (synthetic.MLA_TINY, 9.89, 0.0776),
    (synthetic.MLA_DECODE, 143.44, 15.687),
    (synthetic.MLA_PREFILL, 1459.55, 1003.95),
    (synthetic.MLA_PARTIAL_QUANT, 58.77, 4.614),
], ids=["tiny", "decode", "prefill", "partial_quant"])
def test_path_bytes_and_flops(case, mb, gflop):
    _, path_bytes, path_flops = bench.mla_model(case.dims, case.weight_uq_qr_dtype == "int8",
                                                case.cache_dtype == "int8", case.full_quant)
    assert path_bytes / 1e6 == pytest.approx(mb, abs=0.01)
    assert path_flops / 1e9 == pytest.approx(gflop, rel=1e-3)


def test_decode_weights_dominate():
    d = synthetic.MLA_DECODE.dims
    weights = (d.He * (d.Hcq + d.Hckv + d.Dr) + d.Hcq * d.N * (d.D + d.Dr) + d.N * d.D * d.Hckv) * 2
    assert weights / 1e6 == pytest.approx(122.55, abs=0.01)
    kern, path_bytes, _ = bench.mla_model(d)
    # per-kernel figures add each intermediate once written and once read
    assert kern["down"]["bytes"] + kern["up"]["bytes"] + kern["absorb"]["bytes"] > path_bytes - 1e6


def test_kernel_source_hash_ignores_comments_only():
    # a recorded DRAM traffic figure stays valid across comment edits, not across code edits
    code = "int a = 1;  // one\n/* block\n   comment */\n\n__global__ void k() { a += 2; }\n"
    assert bench.code_only(code) == bench.code_only(code.replace("// one", "// the first"))
    assert bench.code_only(code) == bench.code_only("int a = 1;\n__global__ void k() { a += 2; }")
    assert bench.code_only(code) != bench.code_only(code.replace("a += 2", "a += 3"))
