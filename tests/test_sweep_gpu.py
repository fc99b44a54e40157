"""A seeded sweep of small random problems through the forward and both backward
algorithms, against the fp64 oracle, element by element.

It reaches shapes the hand-picked cases do not: every head dim from 8 to 128 in steps
of 8 (padded inside to 64, 80, 96 or 128), lengths just below, at and above the 128-row
tiles, Sq > Sk and Sq < Sk, MQA / GQA / MHA head maps, and random causal / window /
softcap settings.  Bound: the parity bound of the other tests.
"""

import random

import pytest
import torch

from oracle import attention_backward, attention_forward
from flashattention_backward_pass_gb300.workloads import custom, make_inputs
from tests.helpers import check_close, check_lse, ensure_built, to64

pytestmark = pytest.mark.gpu


def _cases(n=24, seed=2024):
    rng = random.Random(seed)
    lengths = [1, 7, 64, 127, 128, 129, 200, 255, 256, 257, 390]
    out = []
    for idx in range(n):
        D = 8 * (idx % 16 + 1)               # every multiple of 8 up to 128 at least once
        Hk = rng.choice([1, 2, 3])
        G = rng.choice([1, 2, 4])
        Sq, Sk = rng.choice(lengths), rng.choice(lengths)
        causal = rng.random() < 0.4
        wl = rng.choice([-1, -1, 0, 5, 100])
        wr = -1 if causal else rng.choice([-1, -1, 0, 3, 64])
        cap = rng.choice([0.0, 0.0, 15.0])
        out.append(custom(f"sweep{idx}_D{D}_Sq{Sq}_Sk{Sk}_H{G * Hk}x{Hk}", rng.choice([1, 2]), Sq, Sk,
                          G * Hk, Hk, D, causal=causal, window_left=wl, window_right=wr,
                          softcap=cap, seed=100 + idx))
    return out


CASES = _cases()


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    ensure_built()
    import flashattention_backward_pass_gb300 as fa
    fa.load()
    return fa


@pytest.mark.parametrize("algo", [1, 0], ids=["fused", "split"])
@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_sweep(fa, w, algo):
    from flashattention_backward_pass_gb300 import _abi
    _abi.set_algorithm(algo)
    try:
        q, k, v, do = make_inputs(w, "cuda")
        kw = dict(causal=w.causal, window_left=w.window_left, window_right=w.window_right,
                  softcap=w.softcap)
        out, lse = fa.attention_forward(q, k, v, w.scale, **kw)
        ws = fa.alloc_bwd_workspace(q, k)
        dq, dk, dv = fa.attention_backward(do, q, k, v, out, lse, w.scale, workspace=ws, **kw)
        torch.cuda.synchronize()
        assert fa.fa_bwd_status(ws) == 0
    finally:
        _abi.set_algorithm(_abi.ALGO_AUTO)
    qs, ks, vs, dos = (to64(t) for t in (q, k, v, do))
    o_ref, lse_ref = attention_forward(qs, ks, vs, w.scale, **kw)
    dq_ref, dk_ref, dv_ref = attention_backward(dos, qs, ks, vs, w.scale, **kw)
    check_close(w.name + " O", to64(out), o_ref)
    check_lse(to64(lse), lse_ref)
    check_close(w.name + " dQ", to64(dq), dq_ref)
    check_close(w.name + " dK", to64(dk), dk_ref)
    check_close(w.name + " dV", to64(dv), dv_ref)
