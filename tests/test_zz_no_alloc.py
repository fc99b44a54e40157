"""fa_bwd_noalloc, the allocation-free backward for callers that cannot call cudaMalloc
(graph-captured regions, serving loops that must not synchronize, fixed-budget
embeddings): called through the C ABI twice in a row, its outputs must match fa_bwd's
(which uses a caller-provided workspace) within the parity bound of the other tests.
This file is collected last on purpose, and it builds and loads the library itself so
that it also passes alone in a fresh process."""

import pytest
import torch

from flashattention_backward_pass_gb300.workloads import WORKLOADS, custom, make_inputs
from tests.helpers import check_close, ensure_built, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    ensure_built()
    import flashattention_backward_pass_gb300 as fa
    fa.load()
    return fa


CASES = [WORKLOADS["tiny_mha"], WORKLOADS["mha_causal"],
         custom("noalloc_gqa_window_softcap", 1, 333, 517, 8, 2, 72, window_left=64,
                window_right=8, softcap=20.0, seed=51)]


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_noalloc_matches_fa_bwd_twice(fa, w):
    from flashattention_backward_pass_gb300 import _abi
    q, k, v, do = make_inputs(w, "cuda")
    out, lse = fa.attention_forward(q, k, v, w.scale, w.causal, w.window_left, w.window_right,
                                    w.softcap)
    ref = fa.attention_backward(do, q, k, v, out, lse, w.scale, w.causal, w.window_left,
                                w.window_right, w.softcap)
    torch.cuda.synchronize()
    for _ in range(2):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        _abi.fa_bwd_noalloc(do, q, k, v, out, lse, dq, dk, dv, w.scale, w.causal,
                            w.window_left, w.window_right, w.softcap)
        torch.cuda.synchronize()
        for name, got, want in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
            check_close(f"{w.name} noalloc {name}", to64(got), to64(want))
        assert _abi.fa_bwd_noalloc_status() == 0


@pytest.mark.parametrize("w", CASES[1:], ids=[w.name for w in CASES[1:]])
def test_noalloc_deterministic_is_bit_equal_to_fa_bwd(fa, w):
    """The ordered dQ mode on the shared scratch: its counters and accumulator must be
    cleared by every call, so three calls in a row give fa_bwd's deterministic result
    bit for bit."""
    from flashattention_backward_pass_gb300 import _abi
    q, k, v, do = make_inputs(w, "cuda")
    out, lse = fa.attention_forward(q, k, v, w.scale, w.causal, w.window_left, w.window_right,
                                    w.softcap)
    ref = fa.attention_backward(do, q, k, v, out, lse, w.scale, w.causal, w.window_left,
                                w.window_right, w.softcap, deterministic=True)
    torch.cuda.synchronize()
    for _ in range(3):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        _abi.fa_bwd_noalloc(do, q, k, v, out, lse, dq, dk, dv, w.scale, w.causal,
                            w.window_left, w.window_right, w.softcap, deterministic=True)
        torch.cuda.synchronize()
        assert _abi.fa_bwd_noalloc_status() == 0
        for name, got, want in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
            assert torch.equal(got.view(torch.int16), want.view(torch.int16)), name


def test_noalloc_timeout_is_readable(fa):
    """A bounded device wait that runs out inside fa_bwd_noalloc (an ordering counter no
    contributor matches) is reported by fa_bwd_noalloc_status and cleared by it; the next
    call on the same scratch is clean and correct."""
    from flashattention_backward_pass_gb300 import _abi
    w = custom("noalloc_poison", 1, 384, 384, 2, 2, 64, causal=True, seed=43)
    q, k, v, do = make_inputs(w, "cuda")
    out, lse = fa.attention_forward(q, k, v, w.scale, True)
    _abi.set_algorithm(_abi.ALGO_FUSED)    # the ordered dQ wait belongs to the fused path
    try:
        ref = fa.attention_backward(do, q, k, v, out, lse, w.scale, True, deterministic=True)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        _abi.set_wait_limit(20_000_000)        # ~10 ms per wait
        _abi.poison_ordering(True)
        try:
            _abi.fa_bwd_noalloc(do, q, k, v, out, lse, dq, dk, dv, w.scale, True, deterministic=True)
            torch.cuda.synchronize()
            status = _abi.fa_bwd_noalloc_status()
        finally:
            _abi.poison_ordering(False)
            _abi.set_wait_limit(2_000_000_000)
        assert status != 0, "the poisoned ordered wait should have reported a timeout"
        assert _abi.fa_bwd_noalloc_status() == 0   # read and cleared
        _abi.fa_bwd_noalloc(do, q, k, v, out, lse, dq, dk, dv, w.scale, True, deterministic=True)
        torch.cuda.synchronize()
    finally:
        _abi.set_algorithm(_abi.ALGO_AUTO)
    assert _abi.fa_bwd_noalloc_status() == 0
    for name, got, want in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), name


def test_noalloc_rejects_oversized_problem(fa):
    from flashattention_backward_pass_gb300 import _abi
    w = WORKLOADS["gqa_causal"]          # needs ~0.14 GB of scratch, above the 32 MiB limit
    q, k, v, do = make_inputs(w, "cuda")
    out, lse = torch.empty_like(q), torch.zeros(w.B, w.H, w.Sq, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    with pytest.raises(_abi.FaError) as e:
        _abi.fa_bwd_noalloc(do, q, k, v, out, lse, dq, dk, dv, w.scale, True)
    assert e.value.status == -7          # FA_ERR_WORKSPACE
