"""The kernels' failure path on a GPU: a bounded wait that runs out is reported, not hung on.

The library's self-test kernel waits, with the same bounded mbarrier wait every kernel uses, on a
barrier nothing completes; the wait gives up after its limit and latches the timeout bit, which
mlap_check_errors reports.  The context stays usable: a prolog call right after still matches the
oracle.
"""
import pytest
import torch

import qkv_attention_prolog_gb300 as pkg
from qkv_attention_prolog_gb300 import _lib

pytestmark = pytest.mark.gpu

MLAP_ERR_TIMEOUT = 8


@pytest.fixture(scope="module", autouse=True)
def _build():
    import __graft_entry__
    __graft_entry__.build()


def test_bounded_wait_times_out_and_is_reported():
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    pkg.mlap_workspace_init(ws)
    assert pkg.mlap_check_errors(ws) == 0
    _lib.mlap_selftest_bounded_wait(ws)
    torch.cuda.synchronize()
    assert pkg.mlap_check_errors(ws) == MLAP_ERR_TIMEOUT
    assert pkg.mlap_check_errors(ws) == 0          # reading clears the word


def test_context_usable_after_a_timeout():
    import synthetic
    from tests.test_gpu_mla import _full_check
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    pkg.mlap_workspace_init(ws)
    _lib.mlap_selftest_bounded_wait(ws)
    torch.cuda.synchronize()
    assert pkg.mlap_check_errors(ws) == MLAP_ERR_TIMEOUT
    _full_check(synthetic.MLA_TINY)
