"""The torch.autograd wrappers: gradients taken through flash_attn_func /
flash_attn_varlen_func match the fp64 oracle (parity bound of the other tests), and a
loss that is not linear in O (so that dO is not the seed) still backpropagates."""

import pytest
import torch

from oracle import attention_backward, attention_forward
from flashattention_backward_pass_gb300.workloads import custom, make_inputs, make_varlen_inputs
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


def test_flash_attn_func_gradients(fa):
    w = custom("ag", 2, 300, 260, 8, 2, 64, causal=True, softcap=25.0, seed=71)
    q, k, v, do = make_inputs(w, "cuda")
    q, k, v = (t.clone().requires_grad_(True) for t in (q, k, v))
    out = fa.flash_attn_func(q, k, v, causal=True, softcap=25.0)
    out.backward(do)
    kw = dict(causal=True, softcap=25.0)
    o_ref, _ = attention_forward(to64(q), to64(k), to64(v), w.scale, **kw)
    dq, dk, dv = attention_backward(to64(do), to64(q), to64(k), to64(v), w.scale, **kw)
    check_close("autograd O", to64(out), o_ref)
    check_close("autograd dQ", to64(q.grad), dq)
    check_close("autograd dK", to64(k.grad), dk)
    check_close("autograd dV", to64(v.grad), dv)


def test_flash_attn_func_nonlinear_loss(fa):
    w = custom("ag2", 1, 200, 200, 4, 4, 64, seed=72)
    q, k, v, _ = make_inputs(w, "cuda")
    q, k, v = (t.clone().requires_grad_(True) for t in (q, k, v))
    out = fa.flash_attn_func(q, k, v)
    loss = (out.float() ** 2).sum()
    loss.backward()
    do = (2 * out.detach().float()).to(out.dtype)   # d loss / d out
    dq, dk, dv = attention_backward(to64(do), to64(q), to64(k), to64(v), w.scale)
    check_close("nonlinear dQ", to64(q.grad), dq)
    check_close("nonlinear dK", to64(k.grad), dk)
    check_close("nonlinear dV", to64(v.grad), dv)


def test_flash_attn_varlen_func_gradients(fa):
    lq, lk = [130, 0, 257], [200, 64, 257]
    q, k, v, do, cu_q, cu_k = make_varlen_inputs(lq, lk, 4, 2, 64, seed=73, device="cuda")
    q, k, v = (t.clone().requires_grad_(True) for t in (q, k, v))
    out = fa.flash_attn_varlen_func(q, k, v, cu_q, cu_k, max(lq), max(lk), causal=True)
    out.backward(do)
    scale = 64 ** -0.5
    q0 = k0 = 0
    for sq, sk in zip(lq, lk):
        if sq:
            qs, ks, vs, dos = (to64(t)[None] for t in (q[q0:q0 + sq], k[k0:k0 + sk], v[k0:k0 + sk], do[q0:q0 + sq]))
            dq, dk, dv = attention_backward(dos, qs, ks, vs, scale, causal=True)
            check_close("varlen autograd dQ", to64(q.grad[q0:q0 + sq])[None], dq)
            check_close("varlen autograd dK", to64(k.grad[k0:k0 + sk])[None], dk)
            check_close("varlen autograd dV", to64(v.grad[k0:k0 + sk])[None], dv)
        q0 += sq
        k0 += sk


def test_flash_attn_varlen_func_seqused(fa):
    """Used lengths through autograd: the used rows' output and gradients follow the oracle
    for each sequence as a batch of one of its used lengths; padding rows get a zero
    output and zero gradients."""
    cap_q, cap_k = [200, 130, 257], [256, 64, 300]
    used_q, used_k = [150, 0, 257], [256, 20, 299]
    q, k, v, do, cu_q, cu_k = make_varlen_inputs(cap_q, cap_k, 4, 2, 64, seed=79, device="cuda")
    q, k, v = (t.clone().requires_grad_(True) for t in (q, k, v))
    uq = torch.tensor(used_q, dtype=torch.int32, device="cuda")
    uk = torch.tensor(used_k, dtype=torch.int32, device="cuda")
    out = fa.flash_attn_varlen_func(q, k, v, cu_q, cu_k, max(used_q), max(used_k), causal=True,
                                    seqused_q=uq, seqused_k=uk)
    out.backward(do)
    scale = 64 ** -0.5
    q0 = k0 = 0
    for cq, ck, sq, sk in zip(cap_q, cap_k, used_q, used_k):
        if sq:
            qs, dos = to64(q[q0:q0 + sq])[None], to64(do[q0:q0 + sq])[None]
            ks, vs = to64(k[k0:k0 + sk])[None], to64(v[k0:k0 + sk])[None]
            o_ref, _ = attention_forward(qs, ks, vs, scale, causal=True)
            dq, dk, dv = attention_backward(dos, qs, ks, vs, scale, causal=True)
            check_close("seqused autograd O", to64(out[q0:q0 + sq].detach())[None], o_ref)
            check_close("seqused autograd dQ", to64(q.grad[q0:q0 + sq])[None], dq)
            check_close("seqused autograd dK", to64(k.grad[k0:k0 + sk])[None], dk)
            check_close("seqused autograd dV", to64(v.grad[k0:k0 + sk])[None], dv)
        else:
            assert torch.count_nonzero(k.grad[k0:k0 + sk]) == 0
            assert torch.count_nonzero(v.grad[k0:k0 + sk]) == 0
        assert torch.count_nonzero(out[q0 + sq:q0 + cq].detach()) == 0
        assert torch.count_nonzero(q.grad[q0 + sq:q0 + cq]) == 0
        assert torch.count_nonzero(k.grad[k0 + sk:k0 + ck]) == 0
        assert torch.count_nonzero(v.grad[k0 + sk:k0 + ck]) == 0
        q0 += cq
        k0 += ck
