"""The default backward algorithm (FA_BWD_ALGO_AUTO): deterministic batched bf16 calls on a
square shape run the split algorithm (bit for bit what FA_BWD_ALGO_SPLIT gives); every
other call runs the fused algorithm (bit for bit its ordered mode when deterministic)."""

import pytest
import torch

from flashattention_backward_pass_gb300.workloads import custom, make_inputs
from tests.helpers import ensure_built

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
    _abi.set_algorithm(_abi.ALGO_AUTO)


def _det_bits(fa, w, algo, dtype=torch.bfloat16):
    from flashattention_backward_pass_gb300 import _abi
    q, k, v, do = make_inputs(w, "cuda", dtype=dtype)
    kw = dict(causal=w.causal, window_left=w.window_left, window_right=w.window_right,
              softcap=w.softcap)
    out, lse = fa.attention_forward(q, k, v, w.scale, **kw)
    _abi.set_algorithm(algo)
    try:
        ws = fa.alloc_bwd_workspace(q, k, True)
        res = fa.attention_backward(do, q, k, v, out, lse, w.scale, deterministic=True,
                                    workspace=ws, **kw)
        torch.cuda.synchronize()
        assert fa.fa_bwd_status(ws) == 0
    finally:
        _abi.set_algorithm(_abi.ALGO_AUTO)
    return [x.view(torch.int16).clone() for x in res]


def _equal(a, b):
    return all(torch.equal(x, y) for x, y in zip(a, b))


def test_auto_is_the_default(fa):
    from flashattention_backward_pass_gb300 import _abi
    assert _abi.get_algorithm() == _abi.ALGO_AUTO


@pytest.mark.parametrize("w", [
    custom("auto_square", 2, 640, 640, 8, 2, 128, causal=True, seed=81),
    custom("auto_window", 1, 640, 640, 4, 2, 128, window_left=200, window_right=0, seed=82),
    custom("auto_noncausal", 1, 384, 384, 2, 2, 64, seed=84),
], ids=["causal", "window", "noncausal"])
def test_auto_square_runs_split(fa, w):
    from flashattention_backward_pass_gb300 import _abi
    assert _equal(_det_bits(fa, w, _abi.ALGO_AUTO), _det_bits(fa, w, _abi.ALGO_SPLIT))


@pytest.mark.parametrize("w", [
    custom("auto_rect", 1, 256, 640, 4, 4, 64, causal=True, seed=83),
    custom("auto_rect_tall", 1, 640, 300, 4, 2, 128, causal=True, seed=87),
], ids=["rectangular", "tall"])
def test_auto_rectangular_runs_fused(fa, w):
    from flashattention_backward_pass_gb300 import _abi
    assert _equal(_det_bits(fa, w, _abi.ALGO_AUTO), _det_bits(fa, w, _abi.ALGO_FUSED))


def test_auto_f16_square_causal_runs_fused(fa):
    from flashattention_backward_pass_gb300 import _abi
    w = custom("auto_f16", 1, 384, 384, 4, 2, 128, causal=True, seed=85)
    assert _equal(_det_bits(fa, w, _abi.ALGO_AUTO, torch.float16),
                  _det_bits(fa, w, _abi.ALGO_FUSED, torch.float16))
