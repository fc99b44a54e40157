"""fp64 CPU oracle for softmax attention: forward (O, LSE) and backward (dQ, dK, dV).

TEST INFRASTRUCTURE ONLY.  Only the test-suite, the package's smoke check and the
benchmark's CPU-baseline leg may import this module.  The product path (the CUDA
library and its Python binding) never calls it, and this module imports nothing
from the product.

What it computes is the plain definition of softmax attention and of its gradient,
written out densely per (batch, q-head) with NumPy float64 matrices.  No tiling,
no online softmax, no recompute tricks: the (Sq, Sk) score matrix is formed whole.

Sources (web pages on the FlashAttention backward pass):

* "Fused Attention (Flash Attention v2)" Triton page, forward inner loop
  `_attn_fwd_inner` and `_attn_fwd_kernel`: scores q.k^T, masked entries set to
  -inf, exp-normalised rows, O = P V, and the saved row statistic LSE
  (that page stores it in log2 units; this oracle returns natural-log LSE, the
  `softmax_lse` convention of the call-trace page's `mha_bwd`).
* Same page, `_bwd_kernel_dk` / `_bwd_kernel_dv` / `_bwd_kernel_dq`: D_i = rowsum(dO*O),
  dS = P*(dP - D), dV = P^T dO, dK = scale * dS^T Q, dQ = scale * dS K.
* "backward call trace" page, `mha_bwd` signature (layouts (B,S,H,D) for q/k/v/out/dout,
  (B,H,Sq) for softmax_lse), `softmax_d` = row sums of dout*out, and the GQA
  `sum_out` reduction of expanded dK/dV over the q-heads of each kv-head.
* "GQA/MQA" page, KV-head mapping bidh_kv = bidh / (H / Hk) and the bottom-right
  aligned causal block range (n_idx = m_idx + seqlen_k - seqlen_q).
* `flash_bwd_sm90.py` page, `mma_one_m_block`: P = exp2(S*scale*log2e - LSE_log2),
  dS = P*(dP - dPsum); MHA dK multiplied by softmax_scale after the m-block loop.

Readings where the pages are silent (listed with reasons in the design notes):

* softcap c > 0: z = c * tanh(scale*s / c), applied before masking; its derivative
  multiplies dZ by (1 - tanh^2).  c == 0 disables it.
* masking: key j is visible to query i iff j <= i + (Sk - Sq) + window_right (when
  window_right >= 0) and j >= i + (Sk - Sq) - window_left (when window_left >= 0);
  causal forces window_right = 0.  A negative window bound is unbounded.
* a query row with no visible key has O = 0, LSE = +inf, P = 0 and dQ = 0.
* head dims: q and k share a head dim D; v may have its own head dim Dv (the sm90 page's
  `__init__` takes `head_dim` and `head_dim_v`), which o, dO and dV then have.
* block sparsity (the sm90 page's `blocksparse_tensors` give, per key block, the query
  blocks to visit): an optional (B, H, ceil(Sq/bs), ceil(Sk/bs)) boolean block mask; a
  (query block, key block) pair with a 0 entry is masked out entirely, on top of the
  element mask above.  All ones changes nothing.

Parity of every public function here is pinned by tests/test_oracle.py against
finite differences, closed forms, invariants and brute-force loops.
"""

from __future__ import annotations

import numpy as np

LOG2E = 1.4426950408889634


def visible_mask(Sq: int, Sk: int, causal: bool, window_left: int, window_right: int) -> np.ndarray:
    """Boolean (Sq, Sk) matrix: True where key j is visible to query i.

    Bottom-right alignment: the diagonal offset is Sk - Sq, as in the GQA/MQA page's
    causal block range (`n_idx = m_idx_max + seqlen_k - seqlen_q`) and the Triton
    page's forward (`offs_n_causal = offs_m + seqlen_k - seqlen_q`).
    """
    if causal:
        window_right = 0
    i = np.arange(Sq)[:, None]
    j = np.arange(Sk)[None, :]
    delta = Sk - Sq
    vis = np.ones((Sq, Sk), dtype=bool)
    if window_right >= 0:
        vis &= j <= i + delta + window_right
    if window_left >= 0:
        vis &= j >= i + delta - window_left
    return vis


def _head_forward(q, k, v, scale, vis, softcap):
    """One (batch, q-head): q (Sq,D), k/v (Sk,D) fp64.  Returns O, LSE and the
    intermediates the backward needs.

    Triton page `_attn_fwd_inner`: qk = q k^T, masked entries -> -inf, P = exp(qk - m)
    normalised by the row sum, acc = P V.  Here the whole row is normalised at once.
    """
    s = q @ k.T                                   # s_ij = sum_d Q_id K_jd
    a = scale * s                                 # a_ij = scale * s_ij
    if softcap > 0.0:
        t = np.tanh(a / softcap)
        z = softcap * t
    else:
        t = None
        z = a
    z = np.where(vis, z, -np.inf)
    rowmax = z.max(axis=1, initial=-np.inf)      # no key at all (Sk = 0): -inf, as masked
    has_key = np.isfinite(rowmax)
    safe_max = np.where(has_key, rowmax, 0.0)
    e = np.exp(z - safe_max[:, None])             # exp(-inf) = 0 for masked entries
    rowsum = e.sum(axis=1)
    lse = np.where(has_key, safe_max + np.log(np.where(has_key, rowsum, 1.0)), np.inf)
    p = np.where(has_key[:, None], e / np.where(has_key, rowsum, 1.0)[:, None], 0.0)
    o = p @ v
    return o, lse, p, t


def _head_backward(do, q, k, v, scale, vis, softcap):
    """One (batch, q-head) backward.  Returns dq, dk, dv, D and the intermediates.

    Triton page `_bwd_kernel_dv`: dV += P^T dO.  `_bwd_kernel_dk`: D_i = sum(dO*O),
    dS = P*(dO V^T - D), dK += dS^T Q (scaled).  `_bwd_kernel_dq`: dQ += dS K, times
    sm_scale.  With softcap the chain rule adds the factor (1 - tanh^2).
    """
    o, lse, p, t = _head_forward(q, k, v, scale, vis, softcap)
    dv = p.T @ do                                 # dV_j = sum_i P_ij dO_i
    dp = do @ v.T                                 # dP_ij = dO_i . V_j
    dsum = (do * o).sum(axis=1)                   # D_i = sum_d dO_id O_id
    dz = p * (dp - dsum[:, None])                 # dZ_ij = P_ij (dP_ij - D_i)
    if softcap > 0.0:
        da = dz * (1.0 - t * t)                   # d z / d a = 1 - tanh^2(a/c)
    else:
        da = dz
    dq = scale * (da @ k)                         # dQ_i = scale sum_j dA_ij K_j
    dk = scale * (da.T @ q)                       # dK_j = scale sum_i dA_ij Q_i
    return dq, dk, dv, dsum, dict(o=o, lse=lse, p=p, dp=dp, dz=dz, da=da)


def _block_vis(vis, block_mask_bh, block_size):
    """The element mask restricted to the kept (query block, key block) pairs."""
    if block_mask_bh is None:
        return vis
    Sq, Sk = vis.shape
    bm = np.asarray(block_mask_bh, dtype=bool)
    rows = np.arange(Sq) // block_size
    cols = np.arange(Sk) // block_size
    return vis & bm[rows[:, None], cols[None, :]]


def _check_block_mask(block_mask, B, H, Sq, Sk, block_size):
    if block_mask is None:
        return None
    bm = np.asarray(block_mask, dtype=bool)
    want = (B, H, -(-Sq // block_size), -(-Sk // block_size))
    if bm.shape != want:
        raise ValueError(f"block_mask must be {want}, got {bm.shape}")
    return bm


def _check_shapes(q, k, v):
    """(B, Sq, Sk, H, Hk, D, Dv) of q (B,Sq,H,D), k (B,Sk,Hk,D) and v (B,Sk,Hk,Dv)."""
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be (B, S, H, D)")
    B, Sq, H, D = q.shape
    Bk, Sk, Hk, Dk = k.shape
    if v.shape[:3] != k.shape[:3] or Bk != B or Dk != D:
        raise ValueError("k must be (B, Sk, Hk, D) matching q and v (B, Sk, Hk, Dv)")
    if Hk == 0 or H % Hk != 0:
        raise ValueError("H must be a multiple of Hk")
    return B, Sq, Sk, H, Hk, D, v.shape[3]


def attention_forward(q, k, v, scale, causal=False, window_left=-1, window_right=-1,
                      softcap=0.0, block_mask=None, block_size=128):
    """O (B,Sq,H,Dv) and natural-log LSE (B,H,Sq), both float64.

    q (B,Sq,H,D), k (B,Sk,Hk,D), v (B,Sk,Hk,Dv).  q-head h reads kv-head h // (H/Hk)
    (GQA/MQA page, `bidh_kv = bidh / qhead_per_khead`; Triton page
    `off_h_k = off_h // (HQ // HK)`).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Sq, Sk, H, Hk, D, Dv = _check_shapes(q, k, v)
    G = H // Hk
    vis = visible_mask(Sq, Sk, causal, window_left, window_right)
    bm = _check_block_mask(block_mask, B, H, Sq, Sk, block_size)
    o = np.zeros((B, Sq, H, Dv))
    lse = np.zeros((B, H, Sq))
    for b in range(B):
        for h in range(H):
            hk = h // G
            vbh = _block_vis(vis, None if bm is None else bm[b, h], block_size)
            oh, lh, _, _ = _head_forward(q[b, :, h], k[b, :, hk], v[b, :, hk], scale, vbh, softcap)
            o[b, :, h] = oh
            lse[b, h] = lh
    return o, lse


def attention_backward(do, q, k, v, scale, causal=False, window_left=-1, window_right=-1,
                       softcap=0.0, return_dsum=False, block_mask=None, block_size=128):
    """dQ (B,Sq,H,D), dK (B,Sk,Hk,D) and dV (B,Sk,Hk,Dv), float64; optionally D (B,H,Sq).

    do is (B,Sq,H,Dv), like O.  O and P are this module's own fp64 forward (no GPU value
    enters).  dK/dV of a kv-head are the sums of the per-q-head gradients over its H/Hk
    q-heads: the call-trace page's `sum_out` over the reshaped (B,S,Hk,H/Hk,D) expansion.
    """
    do = np.asarray(do, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Sq, Sk, H, Hk, D, Dv = _check_shapes(q, k, v)
    if do.shape != (B, Sq, H, Dv):
        raise ValueError("do must be (B, Sq, H, Dv), like O")
    G = H // Hk
    vis = visible_mask(Sq, Sk, causal, window_left, window_right)
    bm = _check_block_mask(block_mask, B, H, Sq, Sk, block_size)
    dq = np.zeros((B, Sq, H, D))
    dk = np.zeros((B, Sk, Hk, D))
    dv = np.zeros((B, Sk, Hk, Dv))
    dsum = np.zeros((B, H, Sq))
    for b in range(B):
        for h in range(H):
            hk = h // G
            vbh = _block_vis(vis, None if bm is None else bm[b, h], block_size)
            dqh, dkh, dvh, dh, _ = _head_backward(do[b, :, h], q[b, :, h], k[b, :, hk],
                                                  v[b, :, hk], scale, vbh, softcap)
            dq[b, :, h] = dqh
            dk[b, :, hk] += dkh
            dv[b, :, hk] += dvh
            dsum[b, h] = dh
    if return_dsum:
        return dq, dk, dv, dsum
    return dq, dk, dv


def head_intermediates(do, q, k, v, scale, causal=False, window_left=-1, window_right=-1,
                       softcap=0.0):
    """Single-head (S, D) inputs: the dense matrices P, dP, dZ, dA and O, LSE, D.

    Exposed so that tests can check invariants (for example sum_j dZ_ij = 0) on the
    very arrays the backward uses.
    """
    do, q, k, v = (np.asarray(x, dtype=np.float64) for x in (do, q, k, v))
    vis = visible_mask(q.shape[0], k.shape[0], causal, window_left, window_right)
    dq, dk, dv, dsum, inter = _head_backward(do, q, k, v, scale, vis, softcap)
    inter.update(dq=dq, dk=dk, dv=dv, dsum=dsum, vis=vis)
    return inter
