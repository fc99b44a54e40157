"""Out-of-bounds write checks without compute-sanitizer: every output (O, LSE, dQ, dK, dV)
is a strided view into a larger buffer whose other elements hold a sentinel bit pattern.
After the forward and backward the sentinel must be intact everywhere outside the views,
and the views must hold the same results as contiguous outputs (bit for bit where the
path is deterministic).  Shapes end in ragged tiles (lengths that are not multiples of
128) so that the tail tiles' stores are exercised; batched calls run under both backward
algorithms, packed sequences under the fused one."""

import pytest
import torch

from flashattention_backward_pass_gb300.workloads import custom, make_inputs, make_varlen_inputs
from tests.helpers import algorithm_fixture_body, ensure_built

pytestmark = pytest.mark.gpu

SENT16 = 0x5A5A            # a bf16 / f16 bit pattern no kernel writes here
SENT32 = -123456.0         # fp32 LSE sentinel


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    ensure_built()
    import flashattention_backward_pass_gb300 as fa
    fa.load()
    return fa


def guarded16(shape, dtype=torch.bfloat16):
    """A view of `shape` (rows, ..., D) inside a buffer with one extra row before and two
    after, one extra head, and 8 + 16 extra columns around D (all 16-byte aligned)."""
    *lead, h, d = shape
    big_shape = (*lead[:-1], lead[-1] + 3, h + 1, d + 24)
    big = torch.full(big_shape, SENT16, dtype=torch.int16, device="cuda").view(dtype)
    idx = (*(slice(None),) * (len(lead) - 1), slice(1, 1 + lead[-1]), slice(0, h), slice(8, 8 + d))
    view = big[idx]
    mask = torch.ones(big_shape, dtype=torch.bool, device="cuda")
    mask[idx] = False
    return big, view, mask


def guarded_lse(shape):
    """A fp32 (..., H, S) view inside a buffer with one extra head and 4 + 4 extra columns."""
    *lead, h, s = shape
    big_shape = (*lead, h + 1, s + 8)
    big = torch.full(big_shape, SENT32, dtype=torch.float32, device="cuda")
    idx = (*(slice(None),) * len(lead), slice(1, 1 + h), slice(4, 4 + s))
    mask = torch.ones(big_shape, dtype=torch.bool, device="cuda")
    mask[idx] = False
    return big, big[idx], mask


def assert_intact(name, big, mask):
    if big.dtype == torch.float32:
        bad = (big[mask] != SENT32).sum().item()
    else:
        bad = (big.view(torch.int16)[mask] != SENT16).sum().item()
    assert bad == 0, f"{name}: {bad} elements outside the view were overwritten"


@pytest.fixture(params=[0, 1], ids=["split", "fused"])
def algorithm(request):
    yield from algorithm_fixture_body(request)


GUARD_CASES = [
    custom("guard_causal_gqa", 2, 201, 333, 4, 2, 72, causal=True, seed=61),
    custom("guard_window_softcap", 1, 300, 131, 2, 1, 128, window_left=40, window_right=7,
           softcap=15.0, seed=62),
]


@pytest.mark.parametrize("w", GUARD_CASES, ids=[w.name for w in GUARD_CASES])
def test_batched_outputs_stay_in_bounds(fa, algorithm, w):
    q, k, v, do = make_inputs(w, "cuda")
    ob, o, om = guarded16((w.B, w.Sq, w.H, w.D))
    lb, lse, lm = guarded_lse((w.B, w.H, w.Sq))
    fa.fa_fwd(q, k, v, o, lse, w.scale, w.causal, w.window_left, w.window_right, w.softcap)
    qb, dq, qm = guarded16((w.B, w.Sq, w.H, w.D))
    kb, dk, km = guarded16((w.B, w.Sk, w.Hk, w.D))
    vb, dv, vm = guarded16((w.B, w.Sk, w.Hk, w.D))
    ws = fa.alloc_bwd_workspace(q, k, True)
    fa.fa_bwd(do, q, k, v, o, lse, dq, dk, dv, w.scale, w.causal, w.window_left,
              w.window_right, w.softcap, deterministic=True, workspace=ws)
    torch.cuda.synchronize()
    assert fa.fa_bwd_status(ws) == 0
    for name, big, mask in (("O", ob, om), ("LSE", lb, lm), ("dQ", qb, qm), ("dK", kb, km),
                            ("dV", vb, vm)):
        assert_intact(f"{w.name} {name}", big, mask)
    # the views hold what contiguous outputs get (deterministic: bit for bit)
    o2, lse2 = fa.attention_forward(q, k, v, w.scale, w.causal, w.window_left, w.window_right,
                                    w.softcap)
    ref = fa.attention_backward(do, q, k, v, o2, lse2, w.scale, w.causal, w.window_left,
                                w.window_right, w.softcap, deterministic=True)
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(lse, lse2)
    for got, want in zip((dq, dk, dv), ref):
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))


def test_packed_outputs_stay_in_bounds(fa):
    lengths_q, lengths_k = [130, 0, 77, 256], [200, 50, 129, 256]
    H, Hk, D = 4, 2, 64
    q, k, v, do, cu_q, cu_k = make_varlen_inputs(lengths_q, lengths_k, H, Hk, D, seed=63,
                                                 device="cuda")
    tq, tk = q.shape[0], k.shape[0]
    mq, mk = max(lengths_q), max(lengths_k)
    scale = D ** -0.5
    ob, o, om = guarded16((tq, H, D))
    lb, lse, lm = guarded_lse((H, tq))
    fa.fa_fwd_varlen(q, k, v, o, lse, cu_q, cu_k, mq, mk, scale, True)
    qb, dq, qm = guarded16((tq, H, D))
    kb, dk, km = guarded16((tk, Hk, D))
    vb, dv, vm = guarded16((tk, Hk, D))
    ws = fa.fa_bwd_varlen(do, q, k, v, o, lse, dq, dk, dv, cu_q, cu_k, mq, mk, scale, True,
                          deterministic=True)
    torch.cuda.synchronize()
    assert fa.fa_bwd_status(ws) == 0
    for name, big, mask in (("O", ob, om), ("LSE", lb, lm), ("dQ", qb, qm), ("dK", kb, km),
                            ("dV", vb, vm)):
        assert_intact(f"packed {name}", big, mask)
    o2, lse2 = fa.attention_forward_varlen(q, k, v, cu_q, cu_k, mq, mk, scale, True)
    ref = fa.attention_backward_varlen(do, q, k, v, o2, lse2, cu_q, cu_k, mq, mk, scale, True,
                                       deterministic=True)
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(lse, lse2)
    for got, want in zip((dq, dk, dv), ref):
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("D,Dv", [(192, 128), (256, 256)])
def test_wide_outputs_stay_in_bounds(fa, D, Dv):
    """The wide kernels (head dims above 128, or Dv != D) write O, LSE, dQ, dK and dV only
    inside their views, and the views equal contiguous outputs bit for bit (ordered mode)."""
    w = custom(f"guard_wide_{D}_{Dv}", 1, 200, 330, 4, 2, D, causal=True, seed=64, Dv=Dv)
    q, k, v, do = make_inputs(w, "cuda")
    ob, o, om = guarded16((w.B, w.Sq, w.H, Dv))
    lb, lse, lm = guarded_lse((w.B, w.H, w.Sq))
    fa.fa_fwd(q, k, v, o, lse, w.scale, True)
    qb, dq, qm = guarded16((w.B, w.Sq, w.H, D))
    kb, dk, km = guarded16((w.B, w.Sk, w.Hk, D))
    vb, dv, vm = guarded16((w.B, w.Sk, w.Hk, Dv))
    ws = fa.alloc_bwd_workspace(q, k, True, v)
    fa.fa_bwd(do, q, k, v, o, lse, dq, dk, dv, w.scale, True, deterministic=True, workspace=ws)
    torch.cuda.synchronize()
    assert fa.fa_bwd_status(ws) == 0
    for name, big, mask in (("O", ob, om), ("LSE", lb, lm), ("dQ", qb, qm), ("dK", kb, km),
                            ("dV", vb, vm)):
        assert_intact(f"{w.name} {name}", big, mask)
    o2, lse2 = fa.attention_forward(q, k, v, w.scale, True)
    ref = fa.attention_backward(do, q, k, v, o2, lse2, w.scale, True, deterministic=True)
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(lse, lse2)
    for got, want in zip((dq, dk, dv), ref):
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))
