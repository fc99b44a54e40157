"""GPU parity for packed variable-length sequences (fa_fwd_varlen / fa_bwd_varlen).

A packed batch is, by definition, a set of independent sequences: the oracle runs each
sequence alone as a batch of one (its own bottom-right aligned mask) and every output
row of that sequence is compared with it, under the bound of the other parity tests
(max|gpu - oracle| <= 2e-2 * max|oracle| + 2e-3 per tensor, LSE within 1e-4).  The cases
mix lengths that are not multiples of 128, empty query or key sequences, Sq != Sk per
sequence, GQA, windows, softcap, a padded head dim and f16.  In the ordered
(deterministic) mode a packed batch of equal lengths must give exactly the bits of the
batched entry points.
"""

import pytest
import torch

from oracle import attention_backward, attention_forward
from flashattention_backward_pass_gb300.workloads import make_varlen_inputs
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
    dict(name="mha_causal_mixed", lq=[300, 0, 129, 1024, 77], lk=[300, 0, 129, 1024, 77], H=4, Hk=4,
         D=64, causal=True),
    dict(name="gqa_rect_causal", lq=[200, 513, 64, 1], lk=[700, 128, 1, 300], H=8, Hk=2, D=128,
         causal=True),
    dict(name="window_softcap_d72", lq=[257, 400, 90], lk=[257, 400, 333], H=4, Hk=1, D=72,
         window_left=100, window_right=0, softcap=20.0),
    dict(name="noncausal_f16", lq=[129, 383], lk=[500, 64], H=2, Hk=2, D=96,
         dtype=torch.float16),
    dict(name="empty_keys", lq=[100, 50, 30], lk=[0, 70, 0], H=2, Hk=1, D=64, causal=True),
]


def run_case(fa, c, deterministic=False, seed=41):
    dtype = c.get("dtype", torch.bfloat16)
    q, k, v, do, cu_q, cu_k = make_varlen_inputs(c["lq"], c["lk"], c["H"], c["Hk"], c["D"],
                                                 seed=seed, device="cuda", dtype=dtype)
    kw = dict(causal=c.get("causal", False), window_left=c.get("window_left", -1),
              window_right=c.get("window_right", -1), softcap=c.get("softcap", 0.0))
    scale = c["D"] ** -0.5
    mq, mk = max(c["lq"]), max(c["lk"])
    out, lse = fa.attention_forward_varlen(q, k, v, cu_q, cu_k, mq, mk, scale, **kw)
    dq, dk, dv = fa.attention_backward_varlen(do, q, k, v, out, lse, cu_q, cu_k, mq, mk, scale,
                                              deterministic=deterministic, **kw)
    torch.cuda.synchronize()
    return (q, k, v, do), (out, lse, dq, dk, dv), scale, kw


def compare_sequences(c, tensors, gpu, scale, kw):
    q, k, v, do = tensors
    out, lse, dq, dk, dv = gpu
    q0 = k0 = 0
    for b, (sq, sk) in enumerate(zip(c["lq"], c["lk"])):
        if sq > 0:
            qs, dos = to64(q[q0:q0 + sq])[None], to64(do[q0:q0 + sq])[None]
            ks, vs = to64(k[k0:k0 + sk])[None], to64(v[k0:k0 + sk])[None]
            o_ref, lse_ref = attention_forward(qs, ks, vs, scale, **kw)
            dq_ref, dk_ref, dv_ref = attention_backward(dos, qs, ks, vs, scale, **kw)
            tag = f"{c['name']}[seq {b}: Sq={sq} Sk={sk}]"
            check_close(tag + " O", to64(out[q0:q0 + sq])[None], o_ref)
            check_lse(to64(lse[:, q0:q0 + sq])[None], lse_ref)
            check_close(tag + " dQ", to64(dq[q0:q0 + sq])[None], dq_ref)
            check_close(tag + " dK", to64(dk[k0:k0 + sk])[None], dk_ref)
            check_close(tag + " dV", to64(dv[k0:k0 + sk])[None], dv_ref)
        elif sk > 0:
            # no query: the sequence's dK / dV are zero
            assert torch.count_nonzero(dk[k0:k0 + sk]) == 0
            assert torch.count_nonzero(dv[k0:k0 + sk]) == 0
        q0 += sq
        k0 += sk


@pytest.mark.parametrize("c", CASES, ids=[c["name"] for c in CASES])
def test_varlen_matches_oracle_per_sequence(fa, c):
    tensors, gpu, scale, kw = run_case(fa, c)
    compare_sequences(c, tensors, gpu, scale, kw)


def test_varlen_deterministic_bitwise(fa):
    c = CASES[1]
    _, first, _, _ = run_case(fa, c, deterministic=True)
    for _ in range(3):
        _, again, _, _ = run_case(fa, c, deterministic=True)
        for a, b in zip(first, again):
            assert torch.equal(a, b)


def test_varlen_equal_lengths_match_batched_bitwise(fa):
    """Three sequences of 300 queries and 300 keys, packed, against the same data as a
    (3, 300, H, D) batch: in the ordered mode every output is bit-identical."""
    B, S, H, Hk, D = 3, 300, 4, 2, 128
    c = dict(name="equal", lq=[S] * B, lk=[S] * B, H=H, Hk=Hk, D=D, causal=True)
    (q, k, v, do), (out, lse, dq, dk, dv), scale, kw = run_case(fa, c, deterministic=True)
    qb, kb, vb, dob = (t.reshape(B, S, *t.shape[1:]) for t in (q, k, v, do))
    out_b, lse_b = fa.attention_forward(qb, kb, vb, scale, True)
    dq_b, dk_b, dv_b = fa.attention_backward(dob, qb, kb, vb, out_b, lse_b, scale, True,
                                             deterministic=True)
    torch.cuda.synchronize()
    assert torch.equal(out.reshape(B, S, H, D), out_b)
    assert torch.equal(lse.reshape(H, B, S).transpose(0, 1), lse_b)
    assert torch.equal(dq.reshape(B, S, H, D), dq_b)
    assert torch.equal(dk.reshape(B, S, Hk, D), dk_b)
    assert torch.equal(dv.reshape(B, S, Hk, D), dv_b)


# Padded packed sequences (seqused_q / seqused_k): sequence b owns the rows its offsets
# give but computes only the first used rows (clamped to the range), exactly as a batch
# of one of the used lengths; the remaining rows are padding and must come back
# untouched.  Padding rows hold their own random values, so any leak shows.
SEQUSED_CASES = [
    dict(name="causal_gqa", cap_q=[300, 200, 129, 64], used_q=[250, 0, 129, 1],
         cap_k=[300, 256, 140, 64], used_k=[290, 100, 1, 64], H=4, Hk=2, D=128, causal=True),
    dict(name="window_softcap_d72", cap_q=[257, 400, 50], used_q=[100, 399, 50],
         cap_k=[500, 400, 70], used_k=[257, 3, 0], H=2, Hk=1, D=72, window_left=64,
         window_right=0, softcap=20.0),
    # used lengths above the range are clamped to it
    dict(name="noncausal_f16_clamped", cap_q=[129, 383], used_q=[128, 1000], cap_k=[500, 64],
         used_k=[499, 65], H=2, Hk=2, D=64, dtype=torch.float16),
]
SENTINEL = dict(out=7.0, lse=-5.0, dq=3.0, dk=3.0, dv=3.0)


def run_seqused(fa, c, deterministic=False, seed=43, used=True):
    from flashattention_backward_pass_gb300 import _abi
    dtype = c.get("dtype", torch.bfloat16)
    q, k, v, do, cu_q, cu_k = make_varlen_inputs(c["cap_q"], c["cap_k"], c["H"], c["Hk"], c["D"],
                                                 seed=seed, device="cuda", dtype=dtype)
    kw = dict(causal=c.get("causal", False), window_left=c.get("window_left", -1),
              window_right=c.get("window_right", -1), softcap=c.get("softcap", 0.0))
    scale = c["D"] ** -0.5
    uq = torch.tensor(c["used_q"], dtype=torch.int32, device="cuda") if used else None
    uk = torch.tensor(c["used_k"], dtype=torch.int32, device="cuda") if used else None
    eff_q = [min(u, n) for u, n in zip(c["used_q"], c["cap_q"])] if used else c["cap_q"]
    eff_k = [min(u, n) for u, n in zip(c["used_k"], c["cap_k"])] if used else c["cap_k"]
    mq, mk = max(eff_q), max(eff_k)
    out = torch.full_like(q, SENTINEL["out"])
    lse = torch.full((c["H"], q.shape[0]), SENTINEL["lse"], dtype=torch.float32, device="cuda")
    _abi.fa_fwd_varlen(q, k, v, out, lse, cu_q, cu_k, mq, mk, scale, seqused_q=uq, seqused_k=uk,
                       **kw)
    dq = torch.full_like(q, SENTINEL["dq"])
    dk = torch.full_like(k, SENTINEL["dk"])
    dv = torch.full_like(v, SENTINEL["dv"])
    ws = _abi.fa_bwd_varlen(do, q, k, v, out, lse, dq, dk, dv, cu_q, cu_k, mq, mk, scale,
                            deterministic=deterministic, seqused_q=uq, seqused_k=uk, **kw)
    torch.cuda.synchronize()
    assert fa.fa_bwd_status(ws) == 0
    return (q, k, v, do), (out, lse, dq, dk, dv), (eff_q, eff_k), scale, kw


@pytest.mark.parametrize("c", SEQUSED_CASES, ids=[c["name"] for c in SEQUSED_CASES])
def test_seqused_matches_oracle_and_keeps_padding(fa, c):
    (q, k, v, do), (out, lse, dq, dk, dv), (eff_q, eff_k), scale, kw = run_seqused(fa, c)
    q0 = k0 = 0
    for b, (cq, ck, sq, sk) in enumerate(zip(c["cap_q"], c["cap_k"], eff_q, eff_k)):
        tag = f"{c['name']}[seq {b}: used {sq} of {cq} queries, {sk} of {ck} keys]"
        if sq > 0:
            qs, dos = to64(q[q0:q0 + sq])[None], to64(do[q0:q0 + sq])[None]
            ks, vs = to64(k[k0:k0 + sk])[None], to64(v[k0:k0 + sk])[None]
            o_ref, lse_ref = attention_forward(qs, ks, vs, scale, **kw)
            dq_ref, dk_ref, dv_ref = attention_backward(dos, qs, ks, vs, scale, **kw)
            check_close(tag + " O", to64(out[q0:q0 + sq])[None], o_ref)
            check_lse(to64(lse[:, q0:q0 + sq])[None], lse_ref)
            check_close(tag + " dQ", to64(dq[q0:q0 + sq])[None], dq_ref)
            if sk > 0:
                check_close(tag + " dK", to64(dk[k0:k0 + sk])[None], dk_ref)
                check_close(tag + " dV", to64(dv[k0:k0 + sk])[None], dv_ref)
        elif sk > 0:
            # no used query: the used key rows get zero gradients
            assert torch.count_nonzero(dk[k0:k0 + sk]) == 0, tag
            assert torch.count_nonzero(dv[k0:k0 + sk]) == 0, tag
        # padding rows are never written
        assert bool((out[q0 + sq:q0 + cq] == SENTINEL["out"]).all()), tag + " out padding"
        assert bool((lse[:, q0 + sq:q0 + cq] == SENTINEL["lse"]).all()), tag + " lse padding"
        assert bool((dq[q0 + sq:q0 + cq] == SENTINEL["dq"]).all()), tag + " dq padding"
        assert bool((dk[k0 + sk:k0 + ck] == SENTINEL["dk"]).all()), tag + " dk padding"
        assert bool((dv[k0 + sk:k0 + ck] == SENTINEL["dv"]).all()), tag + " dv padding"
        q0 += cq
        k0 += ck


def test_seqused_full_lengths_match_unpadded_bitwise(fa):
    """Used lengths equal to the ranges give exactly the bits of the call without them
    (ordered mode)."""
    c = dict(SEQUSED_CASES[0], used_q=SEQUSED_CASES[0]["cap_q"], used_k=SEQUSED_CASES[0]["cap_k"])
    _, a, _, _, _ = run_seqused(fa, c, deterministic=True, used=True)
    _, b, _, _, _ = run_seqused(fa, c, deterministic=True, used=False)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
