"""Seeded synthetic workloads: shapes and input generators, nothing else.

Shared by the tests (GPU path and oracle alike) and the benchmark.  It holds none
of the attention arithmetic: it only draws seeded random bf16 tensors with the
shapes, value distributions and mask settings of the five backward workloads.
The pages measure on no public dataset; these shapes are the whole workload
definition.
"""

from __future__ import annotations

import itertools
import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Sq: int
    Sk: int
    H: int
    Hk: int
    D: int
    causal: bool = False
    window_left: int = -1
    window_right: int = -1
    softcap: float = 0.0
    do_std: float = 1.0
    seed: int = 0
    deterministic_modes: tuple = field(default=(False,))
    Dv: int = 0          # v's head dim (0: the same as D)

    @property
    def dv(self) -> int:
        return self.Dv or self.D

    @property
    def scale(self) -> float:
        # default softmax scale 1/sqrt(D) (Triton page, `flash_attn_func`)
        return 1.0 / math.sqrt(self.D)

    @property
    def nominal_flops(self) -> float:
        """Backward FLOPs by the stated convention: 10*B*H*Sq*Sk*D, halved when causal
        (with a v head dim of its own: 2*(3*D + 2*Dv) in place of 10*D).  A window with
        window_right == 0 is causal (no key after the diagonal) and is counted as such."""
        f = 2.0 * (3 * self.D + 2 * self.dv) * self.B * self.H * self.Sq * self.Sk
        return f / 2 if (self.causal or self.window_right == 0) else f

    @property
    def forward_flops(self) -> float:
        """Forward FLOPs per visible pair: S = QK^T over D and O += PV over Dv."""
        return 2.0 * (self.D + self.dv) * self.B * self.H * self.visible_pairs_per_head()

    def visible_pairs_per_head(self) -> int:
        """Number of (query, key) pairs the mask keeps (closed form per row)."""
        wr = 0 if self.causal else self.window_right
        wl = self.window_left
        delta = self.Sk - self.Sq
        total = 0
        for i in range(self.Sq):
            hi = self.Sk - 1 if wr < 0 else min(self.Sk - 1, i + delta + wr)
            lo = 0 if wl < 0 else max(0, i + delta - wl)
            if hi >= lo:
                total += hi - lo + 1
        return total

    @property
    def algorithmic_flops(self) -> float:
        """Per visible pair, 2 flops per multiply-add of the five products: S and dK and
        dQ over D, dP and dV over Dv (10*D when Dv == D); logical head dims."""
        return 2.0 * (3 * self.D + 2 * self.dv) * self.B * self.H * self.visible_pairs_per_head()

    def describe(self) -> dict:
        d = dict(workload=self.name, B=self.B, Sq=self.Sq, Sk=self.Sk, H=self.H, Hk=self.Hk,
                 D=self.D, causal=self.causal, window_left=self.window_left,
                 window_right=self.window_right, softcap=self.softcap)
        if self.Dv:
            d["Dv"] = self.Dv
        return d


WORKLOADS = {
    "tiny_mha": Workload("tiny_mha", 1, 128, 128, 2, 2, 64, seed=0),
    "mha_causal": Workload("mha_causal", 2, 1024, 1024, 16, 16, 128, causal=True, seed=1,
                           deterministic_modes=(False, True)),
    "gqa_causal": Workload("gqa_causal", 4, 2048, 2048, 32, 8, 128, causal=True, do_std=0.1,
                           seed=2),
    "swa_softcap": Workload("swa_softcap", 1, 8192, 8192, 16, 2, 128, window_left=1024,
                            window_right=0, softcap=30.0, seed=3),
    "ragged_d72": Workload("ragged_d72", 8, 512, 4096, 12, 12, 72, causal=True, seed=4),
}

HEADLINE = "gqa_causal"

# Wider heads (the wide kernels): the headline's GQA causal shape with head dims 256 and
# (192 for q / k, 128 for v).  Bench lines of their own; parity cases live in the tests.
EXTRA_WORKLOADS = {
    "gqa_causal_d256": Workload("gqa_causal_d256", 2, 2048, 2048, 16, 4, 256, causal=True,
                                do_std=0.1, seed=5),
    "gqa_causal_d192_dv128": Workload("gqa_causal_d192_dv128", 4, 2048, 2048, 32, 8, 192,
                                      causal=True, do_std=0.1, seed=6, Dv=128),
}
# A non-causal square shape (for the choice between the deterministic algorithms).
EXTRA_WORKLOADS["mha_full"] = Workload("mha_full", 2, 2048, 2048, 16, 16, 128, seed=7)
ALL_WORKLOADS = {**WORKLOADS, **EXTRA_WORKLOADS}


def make_inputs(w: Workload, device="cpu", seed: int | None = None, dtype=torch.bfloat16):
    """q, k, v, do as 16-bit tensors (bf16 by default, or f16) in the (B, S, H, D)
    layout (v and do with the workload's v head dim), drawn from N(0, 1) (dO from
    N(0, do_std^2)) with a CPU generator so that every device sees the same values."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed if seed is None else seed)
    q = torch.randn(w.B, w.Sq, w.H, w.D, generator=g, dtype=torch.float32)
    k = torch.randn(w.B, w.Sk, w.Hk, w.D, generator=g, dtype=torch.float32)
    v = torch.randn(w.B, w.Sk, w.Hk, w.dv, generator=g, dtype=torch.float32)
    do = torch.randn(w.B, w.Sq, w.H, w.dv, generator=g, dtype=torch.float32) * w.do_std
    out = [t.to(dtype) for t in (q, k, v, do)]
    if device != "cpu":
        out = [t.to(device) for t in out]
    return out


def custom(name, B, Sq, Sk, H, Hk, D, **kw) -> Workload:
    return Workload(name, B, Sq, Sk, H, Hk, D, **kw)


def make_varlen_inputs(lengths_q, lengths_k, H, Hk, D, seed=0, device="cpu", dtype=torch.bfloat16,
                       do_std=1.0):
    """Packed sequences: q, do (sum(lengths_q), H, D), k, v (sum(lengths_k), Hk, D), drawn
    like make_inputs (N(0, 1), dO scaled by do_std) from a seeded CPU generator, and the
    int32 offsets cu_q, cu_k (length batch + 1, starting at 0)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    tq, tk = int(sum(lengths_q)), int(sum(lengths_k))
    q = torch.randn(tq, H, D, generator=g, dtype=torch.float32)
    k = torch.randn(tk, Hk, D, generator=g, dtype=torch.float32)
    v = torch.randn(tk, Hk, D, generator=g, dtype=torch.float32)
    do = torch.randn(tq, H, D, generator=g, dtype=torch.float32) * do_std
    cu_q = torch.tensor([0] + list(itertools.accumulate(lengths_q)), dtype=torch.int32)
    cu_k = torch.tensor([0] + list(itertools.accumulate(lengths_k)), dtype=torch.int32)
    out = [t.to(dtype) for t in (q, k, v, do)] + [cu_q, cu_k]
    if device != "cpu":
        out = [t.to(device) for t in out]
    return out


def make_block_mask(B, H, Sq, Sk, density=0.5, seed=0, block=128):
    """A seeded random block mask: uint8 (B, H, ceil(Sq/block), ceil(Sk/block)), each entry
    1 with probability `density` (1 = the query-tile / key-tile pair is kept)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    shape = (B, H, -(-Sq // block), -(-Sk // block))
    return (torch.rand(shape, generator=g) < density).to(torch.uint8)
