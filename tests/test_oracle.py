"""Pins for the fp64 oracle (CPU only).

Each check ties the oracle to something other than itself: central finite
differences of its own forward, a library autograd, hand-derived closed forms,
invariants of the softmax gradient, explicit brute-force loops and the special
cases where attention reduces to something elementary.  A plausible mistake in
the oracle (dropped term, sign, transposed operand, wrong head map, wrong mask
alignment) fails at least one of them.
"""

import json
import math
import os

import numpy as np
import pytest

from oracle import attention_backward, attention_forward, head_intermediates, visible_mask

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, rng, scale=1.0):
    return rng.standard_normal(shape) * scale


VARIANTS = [
    dict(causal=False, window_left=-1, window_right=-1, softcap=0.0),
    dict(causal=True, window_left=-1, window_right=-1, softcap=0.0),
    dict(causal=False, window_left=2, window_right=1, softcap=0.0),
    dict(causal=False, window_left=-1, window_right=-1, softcap=1.5),
    dict(causal=True, window_left=3, window_right=-1, softcap=2.0),
]


# ---------------------------------------------------------------- finite differences

@pytest.mark.parametrize("var", VARIANTS)
@pytest.mark.parametrize("H,Hk", [(2, 1), (2, 2)])
def test_finite_differences(var, H, Hk):
    """Central differences of L = sum(dO * O) against dQ, dK, dV (relative < 1e-6)."""
    rng = np.random.default_rng(1234)
    B, Sq, Sk, D = 1, 5, 7, 4
    q, k, v = _rand((B, Sq, H, D), rng), _rand((B, Sk, Hk, D), rng), _rand((B, Sk, Hk, D), rng)
    do = _rand((B, Sq, H, D), rng)
    scale = 0.7
    dq, dk, dv = attention_backward(do, q, k, v, scale, **var)

    def loss(qq, kk, vv):
        o, _ = attention_forward(qq, kk, vv, scale, **var)
        return float((do * o).sum())

    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            args_p = [q, k, v]; args_m = [q, k, v]
            pos = "qkv".index(name)
            args_p[pos] = xp; args_m[pos] = xm
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        err = np.abs(num - g).max() / max(np.abs(g).max(), 1e-300)
        assert err < 1e-6, (name, err)


# ---------------------------------------------------------------- library autograd

@pytest.mark.parametrize("var", VARIANTS)
def test_against_torch_autograd(var):
    """torch fp64 autograd of the forward definition agrees with the oracle's backward."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    B, Sq, Sk, H, Hk, D = 2, 9, 11, 4, 2, 8
    q, k, v = _rand((B, Sq, H, D), rng), _rand((B, Sk, Hk, D), rng), _rand((B, Sk, Hk, D), rng)
    do = _rand((B, Sq, H, D), rng)
    scale = D ** -0.5
    vis = torch.from_numpy(visible_mask(Sq, Sk, var["causal"], var["window_left"], var["window_right"]))
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    G = H // Hk
    kk = tk.repeat_interleave(G, dim=2)
    vv = tv.repeat_interleave(G, dim=2)
    a = torch.einsum("bihd,bjhd->bhij", tq, kk) * scale
    if var["softcap"] > 0:
        a = var["softcap"] * torch.tanh(a / var["softcap"])
    a = a.masked_fill(~vis, float("-inf"))
    p = torch.softmax(a, dim=-1)
    o = torch.einsum("bhij,bjhd->bihd", p, vv)
    o.backward(torch.from_numpy(do))
    dq, dk, dv = attention_backward(do, q, k, v, scale, **var)
    o_ref, _ = attention_forward(q, k, v, scale, **var)
    np.testing.assert_allclose(o_ref, o.detach().numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("var", VARIANTS)
def test_dz_rows_sum_to_zero(var):
    """sum_j dZ_ij = sum_j P_ij dP_ij - D_i = 0 because D_i = rowsum(dO*O) = sum_j P_ij dP_ij."""
    rng = np.random.default_rng(3)
    Sq, Sk, D = 16, 24, 8
    it = head_intermediates(_rand((Sq, D), rng), _rand((Sq, D), rng), _rand((Sk, D), rng),
                            _rand((Sk, D), rng), 0.5, **var)
    rs = it["dz"].sum(axis=1)
    ref = np.abs(it["p"] * it["dp"]).sum(axis=1) + 1e-300
    assert np.all(np.abs(rs) / ref < 1e-12)
    # D_i equals sum_j P_ij dP_ij (the identity the row-sum shortcut relies on)
    np.testing.assert_allclose(it["dsum"], (it["p"] * it["dp"]).sum(axis=1), rtol=1e-12, atol=1e-13)
    # P rows sum to one where any key is visible
    has = it["vis"].any(axis=1)
    np.testing.assert_allclose(it["p"].sum(axis=1)[has], 1.0, rtol=0, atol=1e-14)


@pytest.mark.parametrize("var", VARIANTS)
def test_gqa_equals_sum_of_mha(var):
    """dK/dV of a kv-head equal the sum of the MHA gradients of its q-heads with K, V
    replicated G times (call-trace page, GQA `sum_out`; GQA/MQA page head map)."""
    rng = np.random.default_rng(11)
    B, Sq, Sk, H, Hk, D = 2, 6, 10, 8, 2, 4
    G = H // Hk
    q, k, v = _rand((B, Sq, H, D), rng), _rand((B, Sk, Hk, D), rng), _rand((B, Sk, Hk, D), rng)
    do = _rand((B, Sq, H, D), rng)
    dq, dk, dv = attention_backward(do, q, k, v, 0.6, **var)
    k_rep = np.repeat(k, G, axis=2)       # q-head h -> kv-head h // G
    v_rep = np.repeat(v, G, axis=2)
    dq_m, dk_m, dv_m = attention_backward(do, q, k_rep, v_rep, 0.6, **var)
    np.testing.assert_allclose(dq, dq_m, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dk, dk_m.reshape(B, Sk, Hk, G, D).sum(axis=3), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dv, dv_m.reshape(B, Sk, Hk, G, D).sum(axis=3), rtol=1e-13, atol=1e-14)
    # the forward maps heads the same way
    o, lse = attention_forward(q, k, v, 0.6, **var)
    o_m, lse_m = attention_forward(q, k_rep, v_rep, 0.6, **var)
    np.testing.assert_allclose(o, o_m, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse, lse_m, rtol=1e-13)


# ---------------------------------------------------------------- masks

def test_mask_bottom_right_by_hand():
    """Sq=2, Sk=4 causal: row 0 sees keys 0..2, row 1 sees keys 0..3 (bottom-right)."""
    want = np.array([[1, 1, 1, 0], [1, 1, 1, 1]], dtype=bool)
    assert (visible_mask(2, 4, True, -1, -1) == want).all()
    # Sq=4, Sk=2 causal: rows 0, 1 see nothing; row 2 sees key 0; row 3 sees keys 0, 1
    want = np.array([[0, 0], [0, 0], [1, 0], [1, 1]], dtype=bool)
    assert (visible_mask(4, 2, True, -1, -1) == want).all()
    # window (1, 0) on a square: each row sees itself and one key back
    want = np.array([[1, 0, 0], [1, 1, 0], [0, 1, 1]], dtype=bool)
    assert (visible_mask(3, 3, False, 1, 0) == want).all()


def test_mask_brute_force_and_equivalences():
    for Sq, Sk in [(5, 5), (3, 8), (8, 3), (1, 1), (7, 13)]:
        for wl in (-1, 0, 2, 5):
            for wr in (-1, 0, 1, 4):
                m = visible_mask(Sq, Sk, False, wl, wr)
                for i in range(Sq):
                    for j in range(Sk):
                        ok = True
                        if wr >= 0 and j > i + Sk - Sq + wr:
                            ok = False
                        if wl >= 0 and j < i + Sk - Sq - wl:
                            ok = False
                        assert m[i, j] == ok
        assert (visible_mask(Sq, Sk, True, -1, -1) == visible_mask(Sq, Sk, False, -1, 0)).all()
        assert visible_mask(Sq, Sk, False, -1, -1).all()
        # causal forces window_right to 0 but keeps window_left
        assert (visible_mask(Sq, Sk, True, 2, 5) == visible_mask(Sq, Sk, False, 2, 0)).all()


def test_causal_equals_minus_inf_mask():
    """Causal attention equals full attention with -inf added above the (bottom-right)
    diagonal: computed here by giving the masked keys a huge negative score through
    an extra coordinate of Q and K, which the oracle treats as an ordinary dot product."""
    rng = np.random.default_rng(5)
    Sq, Sk, D = 6, 9, 4
    q, k, v, do = _rand((1, Sq, 1, D), rng), _rand((1, Sk, 1, D), rng), _rand((1, Sk, 1, D), rng), _rand((1, Sq, 1, D), rng)
    o_c, lse_c = attention_forward(q, k, v, 1.0, causal=True)
    dq_c, dk_c, dv_c = attention_backward(do, q, k, v, 1.0, causal=True)
    # extra column: q_i gets 1, k_j gets -1e4 for j > i + (Sk - Sq) -> needs a per-row
    # penalty, so do it one query row at a time
    for i in range(Sq):
        pen = np.where(np.arange(Sk) > i + Sk - Sq, -1e4, 0.0)
        qi = np.concatenate([q[:, i:i + 1], np.ones((1, 1, 1, 1))], axis=3)
        ki = np.concatenate([k, pen[None, :, None, None]], axis=3)
        vi = np.concatenate([v, np.zeros((1, Sk, 1, 1))], axis=3)
        o_i, lse_i = attention_forward(qi, ki, vi, 1.0)
        np.testing.assert_allclose(o_i[0, 0, 0, :D], o_c[0, i, 0], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse_i[0, 0, 0], lse_c[0, 0, i], rtol=1e-12)
        doi = np.concatenate([do[:, i:i + 1], np.zeros((1, 1, 1, 1))], axis=3)
        dq_i, dk_i, dv_i = attention_backward(doi, qi, ki, vi, 1.0)
        np.testing.assert_allclose(dq_i[0, 0, 0, :D], dq_c[0, i, 0], rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- closed forms

def test_two_keys_closed_form():
    """q=1, k=(0, ln3): exp scores (1, 3) so P=(1/4, 3/4).  v=(2, 6), dO=1:
    O=5, LSE=ln4, dV=P, dP=(2,6), D=5, dZ=(-3/4, 3/4), dQ=(3/4) ln3, dK=dZ*q."""
    q = np.array([1.0]).reshape(1, 1, 1, 1)
    k = np.array([0.0, math.log(3.0)]).reshape(1, 2, 1, 1)
    v = np.array([2.0, 6.0]).reshape(1, 2, 1, 1)
    do = np.ones((1, 1, 1, 1))
    o, lse = attention_forward(q, k, v, 1.0)
    assert abs(o[0, 0, 0, 0] - 5.0) < 1e-14
    assert abs(lse[0, 0, 0] - math.log(4.0)) < 1e-14
    dq, dk, dv, dsum = attention_backward(do, q, k, v, 1.0, return_dsum=True)
    assert abs(dsum[0, 0, 0] - 5.0) < 1e-14
    assert abs(dq[0, 0, 0, 0] - 0.75 * math.log(3.0)) < 1e-14
    np.testing.assert_allclose(dk[0, :, 0, 0], [-0.75, 0.75], atol=1e-14)
    np.testing.assert_allclose(dv[0, :, 0, 0], [0.25, 0.75], atol=1e-14)
    # scale enters dQ and dK once each: scale=2 with q halved gives the same scores
    dq2, dk2, dv2 = attention_backward(do, q / 2, k, v, 2.0)
    assert abs(dq2[0, 0, 0, 0] - 2.0 * 0.75 * math.log(3.0)) < 1e-13
    np.testing.assert_allclose(dk2[0, :, 0, 0], [-0.75, 0.75], atol=1e-14)


def test_two_keys_causal_closed_form():
    """Same keys with two queries (q=1 each) under causal masking: row 0 sees key 0
    only (P=(1,0), O=2, dZ=0); row 1 is the two-key case.  dV=(1+1/4, 3/4),
    dK=(-3/4, 3/4), dQ=(0, (3/4) ln3), LSE=(0, ln4)."""
    q = np.ones((1, 2, 1, 1))
    k = np.array([0.0, math.log(3.0)]).reshape(1, 2, 1, 1)
    v = np.array([2.0, 6.0]).reshape(1, 2, 1, 1)
    do = np.ones((1, 2, 1, 1))
    o, lse = attention_forward(q, k, v, 1.0, causal=True)
    np.testing.assert_allclose(o[0, :, 0, 0], [2.0, 5.0], atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], [0.0, math.log(4.0)], atol=1e-14)
    dq, dk, dv = attention_backward(do, q, k, v, 1.0, causal=True)
    np.testing.assert_allclose(dq[0, :, 0, 0], [0.0, 0.75 * math.log(3.0)], atol=1e-14)
    np.testing.assert_allclose(dk[0, :, 0, 0], [-0.75, 0.75], atol=1e-14)
    np.testing.assert_allclose(dv[0, :, 0, 0], [1.25, 0.75], atol=1e-14)


def test_two_keys_softcap_closed_form():
    """softcap c=2 with scores (0, ln3): tanh(ln3/2)=1/2, so z=(0, 1) and
    P=(1, e)/(1+e), O=(2+6e)/(1+e), dZ=(-4e, 4e)/(1+e)^2, dA=dZ*(1, 3/4),
    dQ=dA_2 ln3, dK=dA, LSE=ln(1+e)."""
    e = math.e
    q = np.array([1.0]).reshape(1, 1, 1, 1)
    k = np.array([0.0, math.log(3.0)]).reshape(1, 2, 1, 1)
    v = np.array([2.0, 6.0]).reshape(1, 2, 1, 1)
    do = np.ones((1, 1, 1, 1))
    o, lse = attention_forward(q, k, v, 1.0, softcap=2.0)
    assert abs(o[0, 0, 0, 0] - (2 + 6 * e) / (1 + e)) < 1e-14
    assert abs(lse[0, 0, 0] - math.log(1 + e)) < 1e-14
    dq, dk, dv = attention_backward(do, q, k, v, 1.0, softcap=2.0)
    dz = 4 * e / (1 + e) ** 2
    np.testing.assert_allclose(dk[0, :, 0, 0], [-dz, 0.75 * dz], atol=1e-14)
    assert abs(dq[0, 0, 0, 0] - 0.75 * dz * math.log(3.0)) < 1e-14
    np.testing.assert_allclose(dv[0, :, 0, 0], [1 / (1 + e), e / (1 + e)], atol=1e-14)


# ---------------------------------------------------------------- special cases

def test_single_key():
    """Sk=1: P=1, O=V, LSE=scale*q.k, dQ=dK=0 (dZ = dP - D = 0), dV = sum_i dO_i."""
    rng = np.random.default_rng(2)
    q, k, v, do = _rand((2, 5, 3, 4), rng), _rand((2, 1, 3, 4), rng), _rand((2, 1, 3, 4), rng), _rand((2, 5, 3, 4), rng)
    o, lse = attention_forward(q, k, v, 0.3)
    np.testing.assert_allclose(o, np.broadcast_to(v, o.shape), rtol=1e-14)
    np.testing.assert_allclose(lse, 0.3 * np.einsum("bihd,bjhd->bhi", q, k), rtol=1e-13)
    dq, dk, dv = attention_backward(do, q, k, v, 0.3)
    assert np.abs(dq).max() < 1e-14 and np.abs(dk).max() < 1e-13
    np.testing.assert_allclose(dv, do.sum(axis=1, keepdims=True), rtol=1e-13)


def test_zero_query_is_mean():
    """Q=0: all visible scores are 0, so O_i is the mean of the visible V rows and
    LSE_i = ln(number of visible keys)."""
    rng = np.random.default_rng(4)
    Sq, Sk = 6, 9
    q = np.zeros((1, Sq, 1, 4))
    k, v = _rand((1, Sk, 1, 4), rng), _rand((1, Sk, 1, 4), rng)
    for causal, wl in ((False, -1), (True, -1), (True, 2)):
        o, lse = attention_forward(q, k, v, 1.0, causal=causal, window_left=wl)
        vis = visible_mask(Sq, Sk, causal, wl, -1)
        for i in range(Sq):
            np.testing.assert_allclose(o[0, i, 0], v[0, vis[i], 0].mean(axis=0), rtol=1e-13)
            assert abs(lse[0, 0, i] - math.log(vis[i].sum())) < 1e-14


def test_large_softcap_is_no_softcap():
    rng = np.random.default_rng(6)
    q, k, v, do = _rand((1, 7, 2, 4), rng), _rand((1, 7, 2, 4), rng), _rand((1, 7, 2, 4), rng), _rand((1, 7, 2, 4), rng)
    a = attention_backward(do, q, k, v, 0.5, causal=True)
    b = attention_backward(do, q, k, v, 0.5, causal=True, softcap=1e7)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=1e-9, atol=1e-12)


def test_fully_masked_rows():
    """Sq > Sk with causal: rows i < Sq - Sk see no key: O=0, LSE=+inf, dQ=0."""
    rng = np.random.default_rng(8)
    Sq, Sk = 6, 3
    q, k, v, do = _rand((1, Sq, 1, 4), rng), _rand((1, Sk, 1, 4), rng), _rand((1, Sk, 1, 4), rng), _rand((1, Sq, 1, 4), rng)
    o, lse = attention_forward(q, k, v, 1.0, causal=True)
    dq, dk, dv = attention_backward(do, q, k, v, 1.0, causal=True)
    assert np.all(o[0, :3] == 0) and np.all(np.isinf(lse[0, 0, :3])) and np.all(lse[0, 0, :3] > 0)
    assert np.all(dq[0, :3] == 0)
    assert np.all(np.isfinite(lse[0, 0, 3:]))
    # the remaining rows equal an Sq=3 causal problem on the last three queries
    o3, _ = attention_forward(q[:, 3:], k, v, 1.0, causal=True)
    np.testing.assert_allclose(o[:, 3:], o3, rtol=1e-14)


def test_no_keys_at_all():
    """Sk = 0: every row is a row with no visible key (same reading as the fully masked
    rows above): O = 0, LSE = +inf, dQ = 0, and dK / dV are empty.  The rows must also
    equal the fully masked rows of a problem that has keys."""
    rng = np.random.default_rng(9)
    q, do = _rand((2, 5, 2, 4), rng), _rand((2, 5, 2, 4), rng)
    k = np.zeros((2, 0, 1, 4))
    v = np.zeros((2, 0, 1, 4))
    o, lse = attention_forward(q, k, v, 0.5)
    dq, dk, dv = attention_backward(do, q, k, v, 0.5)
    assert o.shape == q.shape and np.all(o == 0)
    assert np.all(np.isposinf(lse))
    assert dq.shape == q.shape and np.all(dq == 0)
    assert dk.shape == (2, 0, 1, 4) and dv.shape == (2, 0, 1, 4)
    # the rows a causal mask hides completely (Sq = 5 > Sk = 3: rows 0 and 1) are the same
    k1, v1 = _rand((2, 3, 1, 4), rng), _rand((2, 3, 1, 4), rng)
    o1, lse1 = attention_forward(q, k1, v1, 0.5, causal=True)
    dq1, _, _ = attention_backward(do, q, k1, v1, 0.5, causal=True)
    np.testing.assert_array_equal(o1[:, :2], o[:, :2])
    np.testing.assert_array_equal(lse1[:, :, :2], lse[:, :, :2])
    np.testing.assert_array_equal(dq1[:, :2], dq[:, :2])


# ---------------------------------------------------------------- brute force

def _brute(do, q, k, v, scale, causal, wl, wr, cap, block_mask=None, bs=1):
    """Explicit scalar loops from the definition, one (b, h) at a time."""
    B, Sq, H, D = q.shape
    Sk, Hk, Dv = k.shape[1], k.shape[2], v.shape[3]
    G = H // Hk
    O = np.zeros((B, Sq, H, Dv)); L = np.zeros((B, H, Sq))
    dQ = np.zeros(q.shape); dK = np.zeros(k.shape); dV = np.zeros(v.shape)
    if causal:
        wr = 0
    for b in range(B):
        for h in range(H):
            hk = h // G
            for i in range(Sq):
                z = {}; tt = {}
                for j in range(Sk):
                    if wr >= 0 and j > i + Sk - Sq + wr:
                        continue
                    if wl >= 0 and j < i + Sk - Sq - wl:
                        continue
                    if block_mask is not None and not block_mask[b, h, i // bs, j // bs]:
                        continue
                    s = sum(q[b, i, h, d] * k[b, j, hk, d] for d in range(D))
                    a = scale * s
                    if cap > 0:
                        tt[j] = math.tanh(a / cap)
                        z[j] = cap * tt[j]
                    else:
                        z[j] = a
                if not z:
                    L[b, h, i] = math.inf
                    continue
                m = max(z.values())
                den = sum(math.exp(x - m) for x in z.values())
                L[b, h, i] = m + math.log(den)
                P = {j: math.exp(z[j] - L[b, h, i]) for j in z}
                for d in range(Dv):
                    O[b, i, h, d] = sum(P[j] * v[b, j, hk, d] for j in P)
                Di = sum(do[b, i, h, d] * O[b, i, h, d] for d in range(Dv))
                for j in P:
                    dp = sum(do[b, i, h, d] * v[b, j, hk, d] for d in range(Dv))
                    dz = P[j] * (dp - Di)
                    da = dz * (1 - tt[j] ** 2) if cap > 0 else dz
                    for d in range(D):
                        dQ[b, i, h, d] += scale * da * k[b, j, hk, d]
                        dK[b, j, hk, d] += scale * da * q[b, i, h, d]
                    for d in range(Dv):
                        dV[b, j, hk, d] += P[j] * do[b, i, h, d]
    return O, L, dQ, dK, dV


@pytest.mark.parametrize("var", VARIANTS)
def test_brute_force_loops(var):
    rng = np.random.default_rng(9)
    B, Sq, Sk, H, Hk, D = 1, 3, 4, 2, 1, 3
    q, k, v, do = _rand((B, Sq, H, D), rng), _rand((B, Sk, Hk, D), rng), _rand((B, Sk, Hk, D), rng), _rand((B, Sq, H, D), rng)
    O, L, dQ, dK, dV = _brute(do, q, k, v, 0.8, var["causal"], var["window_left"], var["window_right"], var["softcap"])
    o, lse = attention_forward(q, k, v, 0.8, **var)
    dq, dk, dv = attention_backward(do, q, k, v, 0.8, **var)
    np.testing.assert_allclose(o, O, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse, L, rtol=1e-13)
    np.testing.assert_allclose(dq, dQ, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dk, dK, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dv, dV, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- block sparsity

def _bs_inputs(seed, B=1, Sq=5, Sk=7, H=2, Hk=1, D=3):
    rng = np.random.default_rng(seed)
    return (_rand((B, Sq, H, D), rng), _rand((B, Sk, Hk, D), rng), _rand((B, Sk, Hk, D), rng),
            _rand((B, Sq, H, D), rng), rng)


@pytest.mark.parametrize("var", VARIANTS[:3])
def test_block_mask_brute_force(var):
    """A random block mask (blocks of 2) against the scalar loops that skip the pairs
    of removed blocks."""
    q, k, v, do, rng = _bs_inputs(21)
    bm = rng.random((1, 2, 3, 4)) < 0.6
    bm[0, 1, 0, :] = False            # a query block with no key block at all
    O, L, dQ, dK, dV = _brute(do, q, k, v, 0.7, var["causal"], var["window_left"],
                              var["window_right"], var["softcap"], block_mask=bm, bs=2)
    o, lse = attention_forward(q, k, v, 0.7, block_mask=bm, block_size=2, **var)
    dq, dk, dv = attention_backward(do, q, k, v, 0.7, block_mask=bm, block_size=2, **var)
    np.testing.assert_allclose(o, O, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse, L, rtol=1e-13)
    np.testing.assert_allclose(dq, dQ, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dk, dK, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dv, dV, rtol=1e-12, atol=1e-13)
    assert np.all(np.isposinf(lse[0, 1, :2])) and np.all(o[0, :2, 1] == 0)


def test_block_mask_special_cases():
    q, k, v, do, rng = _bs_inputs(22)
    # all ones: no effect
    ones = np.ones((1, 2, 1, 1), dtype=bool)
    np.testing.assert_array_equal(attention_forward(q, k, v, 0.5, block_mask=ones)[0],
                                  attention_forward(q, k, v, 0.5)[0])
    # blocks of one element, lower-triangular (bottom-right aligned): the causal mask
    tri = np.zeros((1, 2, 5, 7), dtype=bool)
    for i in range(5):
        tri[0, :, i, :i + 2 + 1] = True   # j <= i + (Sk - Sq)
    o1, l1 = attention_forward(q, k, v, 0.5, block_mask=tri, block_size=1)
    o2, l2 = attention_forward(q, k, v, 0.5, causal=True)
    np.testing.assert_allclose(o1, o2, rtol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=1e-14)
    g1 = attention_backward(do, q, k, v, 0.5, block_mask=tri, block_size=1)
    g2 = attention_backward(do, q, k, v, 0.5, causal=True)
    for a, b in zip(g1, g2):
        np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-15)
    # nothing kept: O = 0, LSE = +inf, every gradient 0
    none = np.zeros((1, 2, 1, 1), dtype=bool)
    o, lse = attention_forward(q, k, v, 0.5, block_mask=none)
    assert np.all(o == 0) and np.all(np.isposinf(lse))
    for g in attention_backward(do, q, k, v, 0.5, block_mask=none):
        assert np.all(g == 0)


def test_block_mask_finite_differences():
    """The block-masked loss L = sum(dO * O) has the oracle's gradients."""
    q, k, v, do, rng = _bs_inputs(23, Sq=4, Sk=5)
    bm = np.array([[[[True, False, True], [False, True, True]],
                    [[False, True, True], [True, True, False]]]])  # (1, 2, 2, 3), blocks of 2
    kw = dict(block_mask=bm, block_size=2, softcap=1.5)
    loss = lambda q_, k_, v_: float((attention_forward(q_, k_, v_, 0.6, **kw)[0] * do).sum())
    dq, dk, dv = attention_backward(do, q, k, v, 0.6, **kw)
    eps = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = [xp if y is x else y for y in (q, k, v)]
            args_m = [xm if y is x else y for y in (q, k, v)]
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8)


# ---------------------------------------------------------------- stored regression values

def test_golden_regression():
    """Values written by tests/golden/make_golden.py (which calls only the oracle):
    guards the oracle's arithmetic against unnoticed changes."""
    with open(os.path.join(GOLDEN, "oracle_small.json")) as f:
        cases = json.load(f)
    for c in cases:
        arr = {n: np.array(c[n]) for n in ("q", "k", "v", "do")}
        o, lse = attention_forward(arr["q"], arr["k"], arr["v"], c["scale"], **c["variant"])
        dq, dk, dv = attention_backward(arr["do"], arr["q"], arr["k"], arr["v"], c["scale"], **c["variant"])
        lse_want = np.array([[[math.inf if x == "inf" else x for x in row] for row in bh] for bh in c["lse"]])
        np.testing.assert_allclose(o, np.array(c["o"]), rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(lse, lse_want, rtol=1e-12)
        for n, got in (("dq", dq), ("dk", dk), ("dv", dv)):
            np.testing.assert_allclose(got, np.array(c[n]), rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- a V head dim of its own

DV_SHAPES = [(4, 6), (6, 3)]   # (D of q and k, Dv of v, o, dO and dV)


@pytest.mark.parametrize("var", VARIANTS)
@pytest.mark.parametrize("D,Dv", DV_SHAPES)
def test_finite_differences_own_v_dim(var, D, Dv):
    """Central differences of L = sum(dO * O) with v's head dim different from q's and k's
    (the sm90 page's `head_dim` / `head_dim_v`): relative error < 1e-6 for dQ, dK and dV."""
    rng = np.random.default_rng(4321)
    B, Sq, Sk, H, Hk = 1, 4, 6, 2, 1
    q, k, v = _rand((B, Sq, H, D), rng), _rand((B, Sk, Hk, D), rng), _rand((B, Sk, Hk, Dv), rng)
    do = _rand((B, Sq, H, Dv), rng)
    scale = 0.6
    dq, dk, dv = attention_backward(do, q, k, v, scale, **var)
    assert dq.shape == q.shape and dk.shape == k.shape and dv.shape == v.shape

    def loss(qq, kk, vv):
        o, _ = attention_forward(qq, kk, vv, scale, **var)
        assert o.shape == (B, Sq, H, Dv)
        return float((do * o).sum())

    h = 1e-6
    for pos, (x, g) in enumerate(((q, dq), (k, dk), (v, dv))):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            args_p, args_m = [q, k, v], [q, k, v]
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            args_p[pos], args_m[pos] = xp, xm
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        err = np.abs(num - g).max() / max(np.abs(g).max(), 1e-300)
        assert err < 1e-6, ("qkv"[pos], err)


@pytest.mark.parametrize("var", VARIANTS)
def test_torch_autograd_own_v_dim(var):
    """torch fp64 autograd of the definition with D = 8 for q/k and Dv = 5 for v."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(17)
    B, Sq, Sk, H, Hk, D, Dv = 2, 7, 9, 4, 2, 8, 5
    q, k, v = _rand((B, Sq, H, D), rng), _rand((B, Sk, Hk, D), rng), _rand((B, Sk, Hk, Dv), rng)
    do = _rand((B, Sq, H, Dv), rng)
    scale = D ** -0.5
    vis = torch.from_numpy(visible_mask(Sq, Sk, var["causal"], var["window_left"], var["window_right"]))
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    G = H // Hk
    a = torch.einsum("bihd,bjhd->bhij", tq, tk.repeat_interleave(G, dim=2)) * scale
    if var["softcap"] > 0:
        a = var["softcap"] * torch.tanh(a / var["softcap"])
    p = torch.softmax(a.masked_fill(~vis, float("-inf")), dim=-1)
    o = torch.einsum("bhij,bjhd->bihd", p, tv.repeat_interleave(G, dim=2))
    o.backward(torch.from_numpy(do))
    o_ref, _ = attention_forward(q, k, v, scale, **var)
    dq, dk, dv = attention_backward(do, q, k, v, scale, **var)
    np.testing.assert_allclose(o_ref, o.detach().numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("var", VARIANTS)
@pytest.mark.parametrize("D,Dv", DV_SHAPES)
def test_brute_force_own_v_dim(var, D, Dv):
    rng = np.random.default_rng(19)
    B, Sq, Sk, H, Hk = 1, 3, 4, 2, 1
    q, k, v = _rand((B, Sq, H, D), rng), _rand((B, Sk, Hk, D), rng), _rand((B, Sk, Hk, Dv), rng)
    do = _rand((B, Sq, H, Dv), rng)
    O, L, dQ, dK, dV = _brute(do, q, k, v, 0.8, var["causal"], var["window_left"], var["window_right"], var["softcap"])
    o, lse = attention_forward(q, k, v, 0.8, **var)
    dq, dk, dv = attention_backward(do, q, k, v, 0.8, **var)
    np.testing.assert_allclose(o, O, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse, L, rtol=1e-13)
    np.testing.assert_allclose(dq, dQ, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dk, dK, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dv, dV, rtol=1e-12, atol=1e-13)


def test_own_v_dim_special_cases():
    """Sk = 1 with Dv != D: O = V, dQ = dK = 0, dV = sum_i dO_i.  GQA with Dv != D: dK / dV
    are the sums over the q-heads of the MHA gradients with K and V replicated.  And the
    columns of V are independent: O[..., c] depends on V[..., c] only (a split of V by
    columns gives the matching split of O and dV, and the same dQ / dK sums)."""
    rng = np.random.default_rng(23)
    q, k, v, do = (_rand((2, 5, 3, 4), rng), _rand((2, 1, 3, 4), rng), _rand((2, 1, 3, 7), rng),
                   _rand((2, 5, 3, 7), rng))
    o, lse = attention_forward(q, k, v, 0.3)
    np.testing.assert_allclose(o, np.broadcast_to(v, o.shape), rtol=1e-14)
    dq, dk, dv = attention_backward(do, q, k, v, 0.3)
    assert np.abs(dq).max() < 1e-14 and np.abs(dk).max() < 1e-13
    np.testing.assert_allclose(dv, do.sum(axis=1, keepdims=True), rtol=1e-13)

    B, Sq, Sk, H, Hk, D, Dv = 2, 6, 10, 8, 2, 4, 6
    G = H // Hk
    q, k, v = _rand((B, Sq, H, D), rng), _rand((B, Sk, Hk, D), rng), _rand((B, Sk, Hk, Dv), rng)
    do = _rand((B, Sq, H, Dv), rng)
    for var in VARIANTS:
        dq, dk, dv = attention_backward(do, q, k, v, 0.6, **var)
        dq_m, dk_m, dv_m = attention_backward(do, q, np.repeat(k, G, axis=2), np.repeat(v, G, axis=2),
                                              0.6, **var)
        np.testing.assert_allclose(dq, dq_m, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(dk, dk_m.reshape(B, Sk, Hk, G, D).sum(axis=3), rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(dv, dv_m.reshape(B, Sk, Hk, G, Dv).sum(axis=3), rtol=1e-13, atol=1e-14)
        # column split of V: forward and dV split, dQ / dK add up
        o, lse = attention_forward(q, k, v, 0.6, **var)
        oa, la = attention_forward(q, k, v[..., :2], 0.6, **var)
        ob, _ = attention_forward(q, k, v[..., 2:], 0.6, **var)
        np.testing.assert_allclose(o, np.concatenate([oa, ob], axis=-1), rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(lse, la, rtol=1e-14)
        dqa, dka, dva = attention_backward(do[..., :2], q, k, v[..., :2], 0.6, **var)
        dqb, dkb, dvb = attention_backward(do[..., 2:], q, k, v[..., 2:], 0.6, **var)
        np.testing.assert_allclose(dv, np.concatenate([dva, dvb], axis=-1), rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(dq, dqa + dqb, rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(dk, dka + dkb, rtol=1e-11, atol=1e-13)
    with pytest.raises(ValueError):
        attention_backward(do[..., :3], q, k, v, 0.6)     # dO must have v's head dim
