"""deterministic=True: dQ additions are ordered by key tile, dK/dV are reduced inside
one CTA, so ten runs give bitwise-identical gradients."""

import pytest
import torch

from flashattention_backward_pass_gb300.workloads import WORKLOADS, custom, make_inputs
from tests.helpers import algorithm_fixture_body, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(params=[0, 1], ids=["split", "fused"], autouse=True)
def algorithm(request):
    yield from algorithm_fixture_body(request)


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    ensure_built()
    import flashattention_backward_pass_gb300 as fa
    fa.load()
    return fa


def _runs(fa, w, n):
    q, k, v, do = make_inputs(w, "cuda")
    out, lse = fa.attention_forward(q, k, v, w.scale, w.causal, w.window_left, w.window_right, w.softcap)
    ws = fa.alloc_bwd_workspace(q, k, True)
    res = []
    for _ in range(n):
        dq, dk, dv = fa.attention_backward(do, q, k, v, out, lse, w.scale, w.causal, w.window_left,
                                           w.window_right, w.softcap, True, ws)
        torch.cuda.synchronize()
        assert fa.fa_bwd_status(ws) == 0
        res.append(tuple(x.view(torch.int16).clone() for x in (dq, dk, dv)))
    return res


@pytest.mark.parametrize("name", ["mha_causal", "gqa_small"])
def test_bitwise_reproducible(fa, name):
    w = WORKLOADS.get(name) or custom("gqa_small", 2, 640, 640, 8, 2, 128, causal=True, seed=31)
    runs = _runs(fa, w, 10)
    for r in runs[1:]:
        for a, b in zip(runs[0], r):
            assert torch.equal(a, b)
