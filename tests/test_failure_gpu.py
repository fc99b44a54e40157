"""Failure detection without a GPU fault: a bounded device wait that is made to run
out (an ordering counter that no contributor will ever match) ends the kernels with
FA_ERR_DEVICE_TIMEOUT in the workspace status word, and the context stays usable."""

import pytest
import torch

from flashattention_backward_pass_gb300.workloads import custom, make_inputs
from tests.helpers import check_close, ensure_built, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    ensure_built()
    import flashattention_backward_pass_gb300 as fa
    from flashattention_backward_pass_gb300 import _abi
    fa.load()
    yield fa
    _abi.poison_ordering(False)
    _abi.set_wait_limit(2_000_000_000)
    _abi.set_algorithm(_abi.ALGO_AUTO)


def test_ordered_wait_times_out_and_recovers(fa):
    from flashattention_backward_pass_gb300 import _abi
    w = custom("poison", 1, 384, 384, 2, 2, 64, causal=True, seed=41)
    q, k, v, do = make_inputs(w, "cuda")
    out, lse = fa.attention_forward(q, k, v, w.scale, True)
    ws = fa.alloc_bwd_workspace(q, k, True)
    _abi.set_algorithm(_abi.ALGO_FUSED)    # the ordered dQ wait belongs to the fused path
    _abi.set_wait_limit(20_000_000)        # ~10 ms per wait
    _abi.poison_ordering(True)
    try:
        fa.attention_backward(do, q, k, v, out, lse, w.scale, True, deterministic=True, workspace=ws)
        torch.cuda.synchronize()
        status = fa.fa_bwd_status(ws)
    finally:
        _abi.poison_ordering(False)
        _abi.set_wait_limit(2_000_000_000)
        _abi.set_algorithm(_abi.ALGO_FUSED)
    assert status != 0, "the poisoned ordered wait should have reported a timeout"
    _abi.set_algorithm(_abi.ALGO_FUSED)
    # the context still works: a clean deterministic run gives the right answer
    dq1, dk1, dv1 = fa.attention_backward(do, q, k, v, out, lse, w.scale, True, deterministic=True,
                                          workspace=ws)
    torch.cuda.synchronize()
    assert fa.fa_bwd_status(ws) == 0
    dq2, dk2, dv2 = fa.attention_backward(do, q, k, v, out, lse, w.scale, True, deterministic=False)
    torch.cuda.synchronize()
    _abi.set_algorithm(_abi.ALGO_SPLIT)
    dq3, dk3, dv3 = fa.attention_backward(do, q, k, v, out, lse, w.scale, True)
    torch.cuda.synchronize()
    _abi.set_algorithm(_abi.ALGO_FUSED)
    for a, b in ((dq1, dq2), (dk1, dk2), (dv1, dv2), (dq1, dq3), (dk1, dk3), (dv1, dv3)):
        check_close("ordered vs unordered vs split", to64(a), to64(b), rel=1e-2, abs_=1e-3)
