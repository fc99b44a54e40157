"""Shared test helpers: library build/load, the parity bound, oracle slicing."""

from __future__ import annotations

import math

import numpy as np

# Parity bound for bf16 outputs: max|gpu - oracle| <= 2e-2 * max|oracle| + 2e-3 per tensor;
# LSE (fp32) within 1e-4 absolute.
REL_TOL = 2e-2
ABS_TOL = 2e-3
LSE_TOL = 1e-4


def ensure_built():
    from flashattention_backward_pass_gb300.build import build
    return build()


def check_close(name, got, want, rel=REL_TOL, abs_=ABS_TOL):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (name, got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values in GPU output"
    err = float(np.abs(got - want).max()) if got.size else 0.0
    bound = rel * (float(np.abs(want).max()) if want.size else 0.0) + abs_
    assert err <= bound, f"{name}: max|gpu-oracle|={err:.3e} > bound {bound:.3e}"
    return err, bound


def check_lse(got, want, tol=LSE_TOL):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape
    inf_w = np.isinf(want)
    assert np.array_equal(np.isinf(got), inf_w), "LSE: +inf rows differ"
    if (~inf_w).any():
        err = float(np.abs(got[~inf_w] - want[~inf_w]).max())
        assert err <= tol, f"LSE: max abs err {err:.3e} > {tol}"


def to64(t):
    return t.detach().float().cpu().double().numpy()


def algorithm_fixture_body(request):
    """Runs the test under the requested backward algorithm, then restores the default."""
    ensure_built()
    from flashattention_backward_pass_gb300 import _abi
    _abi.load()
    _abi.set_algorithm(request.param)
    yield request.param
    _abi.set_algorithm(_abi.ALGO_AUTO)
