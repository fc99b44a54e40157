"""GPU parity: the CUDA forward/backward (through the C ABI) against the fp64 oracle.

Small cases compare every element and cover tile tails (lengths that are not multiples
of 128), Sq != Sk, fully masked query rows, no keys at all, key tiles with no visible
query, causal /
sliding-window / softcap masks, GQA and MQA head sharing, padded head dims and strided
inputs.  The five workloads run at full size in the launch configuration the benchmark
times; the oracle recomputes sampled (batch, kv-head group) slices of them, which is
exact because heads and batches are independent.

Bound: max|gpu - oracle| <= 2e-2 * max|oracle| + 2e-3 per tensor (dQ, dK, dV, O) and
|LSE_gpu - LSE_oracle| <= 1e-4.
"""

import numpy as np
import pytest
import torch

from oracle import attention_backward, attention_forward
from flashattention_backward_pass_gb300.workloads import WORKLOADS, custom, make_inputs
from tests.helpers import algorithm_fixture_body, check_close, check_lse, ensure_built, to64

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


def run_gpu(fa, w, q, k, v, do, deterministic=False):
    out, lse = fa.attention_forward(q, k, v, w.scale, w.causal, w.window_left, w.window_right,
                                    w.softcap)
    ws = fa.alloc_bwd_workspace(q, k, deterministic)
    dq, dk, dv = fa.attention_backward(do, q, k, v, out, lse, w.scale, w.causal, w.window_left,
                                       w.window_right, w.softcap, deterministic, ws)
    torch.cuda.synchronize()
    assert fa.fa_bwd_status(ws) == 0
    return out, lse, dq, dk, dv


def compare_slice(w, tensors, gpu, b, hk):
    """Oracle on batch b, kv-head hk and its G q-heads; compare that slice."""
    q, k, v, do = tensors
    out, lse, dq, dk, dv = gpu
    G = w.H // w.Hk
    hs = slice(hk * G, hk * G + G)
    qs, ks, vs, dos = (to64(q[b:b + 1, :, hs]), to64(k[b:b + 1, :, hk:hk + 1]),
                       to64(v[b:b + 1, :, hk:hk + 1]), to64(do[b:b + 1, :, hs]))
    kw = dict(causal=w.causal, window_left=w.window_left, window_right=w.window_right,
              softcap=w.softcap)
    o_ref, lse_ref = attention_forward(qs, ks, vs, w.scale, **kw)
    dq_ref, dk_ref, dv_ref = attention_backward(dos, qs, ks, vs, w.scale, **kw)
    tag = f"{w.name}[b={b},hk={hk}]"
    check_close(tag + " O", to64(out[b:b + 1, :, hs]), o_ref)
    check_lse(to64(lse[b:b + 1, hs]), lse_ref)
    check_close(tag + " dQ", to64(dq[b:b + 1, :, hs]), dq_ref)
    check_close(tag + " dK", to64(dk[b:b + 1, :, hk:hk + 1]), dk_ref)
    check_close(tag + " dV", to64(dv[b:b + 1, :, hk:hk + 1]), dv_ref)


def full_compare(w, tensors, gpu):
    for b in range(w.B):
        for hk in range(w.Hk):
            compare_slice(w, tensors, gpu, b, hk)


SMALL = [
    custom("tail_causal", 1, 77, 301, 4, 2, 64, causal=True, seed=11),
    custom("sq_gt_sk_causal", 2, 200, 130, 4, 4, 128, causal=True, seed=12),
    custom("mqa_d72", 1, 256, 256, 8, 1, 72, seed=13),
    custom("window", 1, 300, 300, 2, 1, 128, window_left=50, window_right=20, seed=14),
    custom("softcap_tail", 1, 257, 129, 2, 2, 64, softcap=5.0, seed=15),
    custom("d96", 1, 130, 200, 3, 3, 96, causal=True, seed=16),
    custom("d32", 2, 100, 100, 2, 1, 32, seed=17),
    custom("single", 1, 1, 1, 1, 1, 64, seed=18),
    custom("empty_key_tiles", 1, 64, 512, 2, 1, 64, window_left=10, window_right=0, seed=19),
    custom("gqa_window_softcap", 2, 384, 384, 8, 2, 128, window_left=100, window_right=0,
           softcap=30.0, seed=20),
    custom("d80_noncausal", 1, 129, 383, 2, 2, 80, seed=21),
    custom("no_keys", 2, 70, 0, 4, 2, 64, seed=23),
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_small_cases(fa, w):
    tensors = make_inputs(w, "cuda")
    gpu = run_gpu(fa, w, *tensors)
    full_compare(w, tensors, gpu)


def test_strided_inputs(fa):
    """q, k, v as views into packed (B, S, 3, H, D) buffers; outputs into padded rows."""
    B, S, H, D = 2, 200, 4, 64
    w = custom("strided", B, S, S, H, H, D, causal=True, seed=22)
    g = torch.Generator().manual_seed(22)
    qkv = torch.randn(B, S, 3, H, D, generator=g).to(torch.bfloat16).cuda()
    q, k, v = qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2]
    do = torch.randn(B, S, H, D, generator=g).to(torch.bfloat16).cuda()
    out = torch.empty(B, S, H, D + 64, dtype=torch.bfloat16, device="cuda")[..., :D]
    lse = torch.empty(B, H, S, dtype=torch.float32, device="cuda")
    fa.fa_fwd(q, k, v, out, lse, w.scale, True)
    dq = torch.empty(B, S, H, D + 8, dtype=torch.bfloat16, device="cuda")[..., :D]
    dk = torch.empty(B, S, H, D + 8, dtype=torch.bfloat16, device="cuda")[..., :D]
    dv = torch.empty(B, S, H, D + 8, dtype=torch.bfloat16, device="cuda")[..., :D]
    fa.fa_bwd(do, q, k, v, out, lse, dq, dk, dv, w.scale, True)
    torch.cuda.synchronize()
    full_compare(w, (q, k, v, do), (out, lse, dq, dk, dv))


# ------------------------------------------------------------------ the five workloads

def test_tiny_mha_full(fa):
    w = WORKLOADS["tiny_mha"]
    t = make_inputs(w, "cuda")
    full_compare(w, t, run_gpu(fa, w, *t))


@pytest.mark.parametrize("det", [False, True])
def test_mha_causal_full(fa, det):
    w = WORKLOADS["mha_causal"]
    t = make_inputs(w, "cuda")
    gpu = run_gpu(fa, w, *t, deterministic=det)
    for b in range(w.B):
        for hk in (0, 7, 15):
            compare_slice(w, t, gpu, b, hk)


@pytest.mark.parametrize("det", [False, True])
def test_gqa_causal_sampled(fa, det):
    w = WORKLOADS["gqa_causal"]
    t = make_inputs(w, "cuda")
    gpu = run_gpu(fa, w, *t, deterministic=det)
    for b, hk in ((0, 0), (3, 7)):
        compare_slice(w, t, gpu, b, hk)


@pytest.mark.parametrize("det", [False, True])
def test_swa_softcap_sampled(fa, det):
    w = WORKLOADS["swa_softcap"]
    t = make_inputs(w, "cuda")
    gpu = run_gpu(fa, w, *t, deterministic=det)
    compare_slice(w, t, gpu, 0, 0)   # batch 0, q-heads 0..7 (kv-head 0's group)


@pytest.mark.parametrize("det", [False, True])
def test_ragged_d72_sampled(fa, det):
    w = WORKLOADS["ragged_d72"]
    t = make_inputs(w, "cuda")
    gpu = run_gpu(fa, w, *t, deterministic=det)
    for b, h in ((0, 0), (7, 11), (4, 5)):
        compare_slice(w, t, gpu, b, h)
