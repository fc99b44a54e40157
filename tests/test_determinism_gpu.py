"""deterministic=True: dQ additions are ordered by key tile, dK/dV are reduced inside
one CTA, so ten runs give bitwise-identical gradients.  Besides two small shapes, the
headline GQA workload, the windowed softcap workload and the rectangular (bottom-right
causal) workload run ten times each at full size, in the fused algorithm's ordered mode
(where the order of the dQ additions comes from counters) and in the split algorithm."""

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


def _check_runs(fa, w, n):
    """n deterministic backward calls on one workspace; each result must equal the first
    bit for bit."""
    q, k, v, do = make_inputs(w, "cuda")
    out, lse = fa.attention_forward(q, k, v, w.scale, w.causal, w.window_left, w.window_right, w.softcap)
    ws = fa.alloc_bwd_workspace(q, k, True)
    first = None
    for _ in range(n):
        dq, dk, dv = fa.attention_backward(do, q, k, v, out, lse, w.scale, w.causal, w.window_left,
                                           w.window_right, w.softcap, True, ws)
        torch.cuda.synchronize()
        assert fa.fa_bwd_status(ws) == 0
        cur = tuple(x.view(torch.int16) for x in (dq, dk, dv))
        if first is None:
            first = cur
        else:
            for name, a, b in zip(("dQ", "dK", "dV"), first, cur):
                assert torch.equal(a, b), f"{w.name} {name} differs between runs"


@pytest.mark.parametrize("name", ["mha_causal", "gqa_small", "gqa_causal", "swa_softcap",
                                  "ragged_d72"])
def test_bitwise_reproducible(fa, name):
    w = WORKLOADS.get(name) or custom("gqa_small", 2, 640, 640, 8, 2, 128, causal=True, seed=31)
    _check_runs(fa, w, 10)
