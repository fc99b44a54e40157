"""GPU parity for block-sparse attention (fa_fwd_blocksparse / fa_bwd_blocksparse).

The oracle applies the same (B, H, Mb, Nb) block mask on top of the element mask (a
removed query-tile / key-tile pair is masked out entirely) and every output element is
compared under the bound of the other parity tests (max|gpu - oracle| <= 2e-2 *
max|oracle| + 2e-3 per tensor, LSE within 1e-4).  Cases mix random masks with rows and
columns of tiles removed entirely, causal / window / softcap element masks, GQA, a
padded head dim and lengths that are not multiples of 128.
"""

import pytest
import torch

from oracle import attention_backward, attention_forward
from flashattention_backward_pass_gb300.workloads import custom, make_block_mask, make_inputs
from tests.helpers import check_close, check_lse, ensure_built, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    ensure_built()
    import flashattention_backward_pass_gb300 as fa
    from flashattention_backward_pass_gb300 import _abi
    fa.load()
    _abi.set_algorithm(_abi.ALGO_FUSED)
    yield fa
    _abi.set_algorithm(_abi.ALGO_AUTO)


CASES = [
    (custom("bs_mha", 1, 640, 640, 2, 2, 64, seed=61), 0.5),
    (custom("bs_gqa_causal", 2, 513, 700, 8, 2, 128, causal=True, seed=62), 0.6),
    (custom("bs_window_softcap_d72", 1, 400, 400, 4, 1, 72, window_left=200, window_right=50,
            softcap=20.0, seed=63), 0.7),
]


def run(fa, w, bm_cpu, deterministic=False):
    q, k, v, do = make_inputs(w, "cuda")
    bm = bm_cpu.cuda()
    kw = dict(causal=w.causal, window_left=w.window_left, window_right=w.window_right,
              softcap=w.softcap)
    out = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.Sq, dtype=torch.float32, device="cuda")
    fa.fa_fwd_blocksparse(q, k, v, out, lse, bm, w.scale, **kw)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = fa.fa_bwd_blocksparse(do, q, k, v, out, lse, dq, dk, dv, bm, w.scale,
                               deterministic=deterministic, **kw)
    torch.cuda.synchronize()
    assert fa.fa_bwd_status(ws) == 0
    return (q, k, v, do), (out, lse, dq, dk, dv), kw


def compare(w, bm_cpu, tensors, gpu, kw):
    q, k, v, do = (to64(t) for t in tensors)
    out, lse, dq, dk, dv = gpu
    bm = bm_cpu.numpy().astype(bool)
    o_ref, lse_ref = attention_forward(q, k, v, w.scale, block_mask=bm, **kw)
    dq_ref, dk_ref, dv_ref = attention_backward(do, q, k, v, w.scale, block_mask=bm, **kw)
    check_close(w.name + " O", to64(out), o_ref)
    check_lse(to64(lse), lse_ref)
    check_close(w.name + " dQ", to64(dq), dq_ref)
    check_close(w.name + " dK", to64(dk), dk_ref)
    check_close(w.name + " dV", to64(dv), dv_ref)


@pytest.mark.parametrize("det", [False, True], ids=["unordered", "ordered"])
@pytest.mark.parametrize("case", CASES, ids=[c[0].name for c in CASES])
def test_blocksparse_matches_oracle(fa, case, det):
    w, density = case
    bm = make_block_mask(w.B, w.H, w.Sq, w.Sk, density, seed=w.seed)
    bm[0, 0, 0, :] = 0     # a query tile with no key tile at all
    bm[0, -1, :, -1] = 0   # a key tile no query tile of that head visits
    tensors, gpu, kw = run(fa, w, bm, deterministic=det)
    compare(w, bm, tensors, gpu, kw)


def test_blocksparse_deterministic_bitwise(fa):
    """Ordered mode on step lists: ten runs, identical bits."""
    w, density = CASES[1]
    bm = make_block_mask(w.B, w.H, w.Sq, w.Sk, density, seed=w.seed + 100)
    _, first, _ = run(fa, w, bm, deterministic=True)
    first = [x.view(torch.int16).clone() for x in first[2:]]
    for _ in range(9):
        _, again, _ = run(fa, w, bm, deterministic=True)
        for a, b in zip(first, again[2:]):
            assert torch.equal(a, b.view(torch.int16))


def test_blocksparse_all_kept_ordered_equals_dense_ordered(fa):
    """With every tile pair kept the step lists are the dense steps in the dense order, so
    the ordered sparse backward gives the fused ordered dense backward's bits."""
    from flashattention_backward_pass_gb300 import _abi
    w = custom("bs_all_ordered", 2, 384, 520, 4, 2, 64, causal=True, seed=65)
    ones = make_block_mask(w.B, w.H, w.Sq, w.Sk, 1.0)
    tensors, gpu, kw = run(fa, w, ones, deterministic=True)
    q, k, v, do = tensors
    _abi.set_algorithm(_abi.ALGO_FUSED)
    ref = fa.attention_backward(do, q, k, v, gpu[0], gpu[1], w.scale, deterministic=True, **kw)
    torch.cuda.synchronize()
    for a, b in zip(gpu[2:], ref):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_blocksparse_all_and_nothing(fa):
    w = custom("bs_edges", 1, 300, 260, 4, 2, 64, causal=True, seed=64)
    ones = make_block_mask(w.B, w.H, w.Sq, w.Sk, 1.0)
    tensors, gpu, kw = run(fa, w, ones)
    compare(w, ones, tensors, gpu, kw)
    # the dense forward gives the same bits when every pair is kept
    out_d, lse_d = fa.attention_forward(*tensors[:3], w.scale, True)
    assert torch.equal(out_d, gpu[0]) and torch.equal(lse_d, gpu[1])
    zeros = make_block_mask(w.B, w.H, w.Sq, w.Sk, 0.0)
    _, (out, lse, dq, dk, dv), _ = run(fa, w, zeros)
    assert torch.count_nonzero(out) == 0 and bool(torch.isposinf(lse).all())
    for g in (dq, dk, dv):
        assert torch.count_nonzero(g) == 0
