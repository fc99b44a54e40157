"""Writes tests/golden/oracle_small.json from the fp64 oracle (and nothing else).

The pages print no worked numeric example, so the stored values here are regression
values of the oracle itself, written by this script; the oracle's independent pins
are the closed forms, finite differences, invariants and brute-force loops in
tests/test_oracle.py.  Run from the repository root:  python tests/golden/make_golden.py
"""

import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
from oracle import attention_backward, attention_forward  # noqa: E402

CASES = [
    dict(shape=(1, 3, 2, 1, 4), scale=0.5, variant=dict(causal=False, window_left=-1, window_right=-1, softcap=0.0)),
    dict(shape=(1, 4, 3, 2, 4), scale=0.5, variant=dict(causal=True, window_left=-1, window_right=-1, softcap=0.0)),
    dict(shape=(1, 3, 5, 2, 4), scale=0.5, variant=dict(causal=False, window_left=1, window_right=0, softcap=3.0)),
]


def main():
    rng = np.random.default_rng(20261202)
    out = []
    for c in CASES:
        B, Sq, Sk, H, D = c["shape"]
        Hk = 1
        q = np.round(rng.standard_normal((B, Sq, H, D)), 3)
        k = np.round(rng.standard_normal((B, Sk, Hk, D)), 3)
        v = np.round(rng.standard_normal((B, Sk, Hk, D)), 3)
        do = np.round(rng.standard_normal((B, Sq, H, D)), 3)
        o, lse = attention_forward(q, k, v, c["scale"], **c["variant"])
        dq, dk, dv = attention_backward(do, q, k, v, c["scale"], **c["variant"])
        out.append(dict(scale=c["scale"], variant=c["variant"], q=q.tolist(), k=k.tolist(),
                        v=v.tolist(), do=do.tolist(), o=o.tolist(),
                        lse=[[["inf" if np.isinf(x) else x for x in row] for row in bh] for bh in lse.tolist()],
                        dq=dq.tolist(), dk=dk.tolist(), dv=dv.tolist()))
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_small.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
