"""GPU parity of the wide kernels: head dims above 128 and a V head dim of its own (the
call-trace page's dispatch up to head dim 256; the `flash_bwd_sm90.py` page's
`head_dim` / `head_dim_v`), forward and backward through the C ABI against the fp64
oracle, element by element.  Shapes end in ragged tiles and cover causal, windowed and
softcapped masks, GQA / MQA head sharing, Dv below and above D, f16, and a call with no
keys.  Bound: max|gpu - oracle| <= 2e-2 * max|oracle| + 2e-3 per tensor, LSE within 1e-4.
"""

import pytest
import torch

from oracle import attention_backward, attention_forward
from flashattention_backward_pass_gb300.workloads import custom, make_inputs
from tests.helpers import check_close, check_lse, ensure_built, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    ensure_built()
    import flashattention_backward_pass_gb300 as fa
    fa.load()
    return fa


CASES = [
    custom("d192_causal_gqa", 1, 200, 333, 4, 2, 192, causal=True, seed=71),
    custom("d256_window_softcap", 2, 130, 257, 2, 1, 256, window_left=50, window_right=10,
           softcap=20.0, seed=72),
    custom("d192_dv128_causal", 1, 300, 300, 4, 1, 192, causal=True, seed=73, Dv=128),
    custom("d128_dv64", 1, 150, 200, 2, 2, 128, seed=74, Dv=64),
    custom("d64_dv256", 1, 129, 129, 2, 2, 64, seed=75, Dv=256),
    custom("d200_dv136_causal", 2, 97, 160, 3, 3, 200, causal=True, seed=76, Dv=136),
    custom("d256_mqa_rect_causal", 1, 64, 400, 4, 1, 256, causal=True, seed=77),
]


def run_and_compare(fa, w, dtype=torch.bfloat16):
    q, k, v, do = make_inputs(w, "cuda", dtype=dtype)
    kw = dict(causal=w.causal, window_left=w.window_left, window_right=w.window_right,
              softcap=w.softcap)
    out, lse = fa.attention_forward(q, k, v, w.scale, **kw)
    assert out.shape == (w.B, w.Sq, w.H, w.dv)
    ws = fa.alloc_bwd_workspace(q, k, False, v)
    dq, dk, dv = fa.attention_backward(do, q, k, v, out, lse, w.scale, workspace=ws, **kw)
    torch.cuda.synchronize()
    assert fa.fa_bwd_status(ws) == 0
    o_ref, lse_ref = attention_forward(to64(q), to64(k), to64(v), w.scale, **kw)
    dq_ref, dk_ref, dv_ref = attention_backward(to64(do), to64(q), to64(k), to64(v), w.scale, **kw)
    check_close(w.name + " O", to64(out), o_ref)
    check_lse(to64(lse), lse_ref)
    check_close(w.name + " dQ", to64(dq), dq_ref)
    check_close(w.name + " dK", to64(dk), dk_ref)
    check_close(w.name + " dV", to64(dv), dv_ref)


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_wide_parity(fa, w):
    run_and_compare(fa, w)


def test_wide_f16(fa):
    run_and_compare(fa, custom("d256_f16_causal", 1, 190, 190, 2, 1, 256, causal=True, seed=78),
                    dtype=torch.float16)


def test_wide_no_keys(fa):
    """Sk = 0: O = 0, LSE = +inf, dQ = 0 (dK / dV are empty)."""
    w = custom("d256_no_keys", 1, 70, 0, 2, 1, 256, seed=79, Dv=192)
    q, k, v, do = make_inputs(w, "cuda")
    out, lse = fa.attention_forward(q, k, v, w.scale)
    dq, dk, dv = fa.attention_backward(do, q, k, v, out, lse, w.scale)
    torch.cuda.synchronize()
    assert torch.all(out == 0) and torch.all(torch.isinf(lse)) and torch.all(dq == 0)


def test_wide_twice_same_workspace(fa):
    """A second call on the same workspace starts from a cleared accumulator."""
    w = CASES[2]
    q, k, v, do = make_inputs(w, "cuda")
    out, lse = fa.attention_forward(q, k, v, w.scale, w.causal)
    ws = fa.alloc_bwd_workspace(q, k, False, v)
    first = fa.attention_backward(do, q, k, v, out, lse, w.scale, w.causal, workspace=ws)
    second = fa.attention_backward(do, q, k, v, out, lse, w.scale, w.causal, workspace=ws)
    torch.cuda.synchronize()
    for a, b in zip(first, second):
        check_close("twice", to64(b), to64(a), rel=1e-2, abs_=1e-3)


@pytest.mark.parametrize("w", [CASES[0], CASES[2], CASES[6]], ids=[CASES[i].name for i in (0, 2, 6)])
def test_wide_deterministic(fa, w):
    """The ordered mode of the wide backward: oracle parity, and ten runs with identical
    bits."""
    q, k, v, do = make_inputs(w, "cuda")
    kw = dict(causal=w.causal, window_left=w.window_left, window_right=w.window_right,
              softcap=w.softcap)
    out, lse = fa.attention_forward(q, k, v, w.scale, **kw)
    ws = fa.alloc_bwd_workspace(q, k, True, v)
    first = None
    for _ in range(10):
        res = fa.attention_backward(do, q, k, v, out, lse, w.scale, deterministic=True,
                                    workspace=ws, **kw)
        torch.cuda.synchronize()
        assert fa.fa_bwd_status(ws) == 0
        bits = [x.view(torch.int16).clone() for x in res]
        if first is None:
            first = bits
            dq_ref, dk_ref, dv_ref = attention_backward(to64(do), to64(q), to64(k), to64(v),
                                                        w.scale, **kw)
            check_close(w.name + " det dQ", to64(res[0]), dq_ref)
            check_close(w.name + " det dK", to64(res[1]), dk_ref)
            check_close(w.name + " det dV", to64(res[2]), dv_ref)
        else:
            for a, b in zip(first, bits):
                assert torch.equal(a, b)


def test_wide_ordered_wait_times_out_and_recovers(fa):
    """A poisoned ordering counter makes the wide kernel's bounded wait run out: the status
    word reports it, and a clean call afterwards is correct."""
    from flashattention_backward_pass_gb300 import _abi
    w = custom("wide_poison", 1, 256, 256, 2, 1, 192, causal=True, seed=86)
    q, k, v, do = make_inputs(w, "cuda")
    out, lse = fa.attention_forward(q, k, v, w.scale, True)
    ws = fa.alloc_bwd_workspace(q, k, True, v)
    _abi.set_wait_limit(20_000_000)        # ~10 ms per wait
    _abi.poison_ordering(True)
    try:
        fa.attention_backward(do, q, k, v, out, lse, w.scale, True, deterministic=True, workspace=ws)
        torch.cuda.synchronize()
        status = fa.fa_bwd_status(ws)
    finally:
        _abi.poison_ordering(False)
        _abi.set_wait_limit(2_000_000_000)
    assert status != 0
    dq, dk, dv = fa.attention_backward(do, q, k, v, out, lse, w.scale, True, deterministic=True,
                                       workspace=ws)
    torch.cuda.synchronize()
    assert fa.fa_bwd_status(ws) == 0
    dq_ref, dk_ref, dv_ref = attention_backward(to64(do), to64(q), to64(k), to64(v), w.scale,
                                                causal=True)
    check_close("wide recovered dQ", to64(dq), dq_ref)
    check_close("wide recovered dK", to64(dk), dk_ref)
    check_close("wide recovered dV", to64(dv), dv_ref)
