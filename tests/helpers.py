"""Shared test helpers: tolerances and comparisons against the oracle."""

import numpy as np

# GPU-vs-oracle tolerances (bf16 tensor-core path / fp32 CUDA-core path)
TOL_O_BF16 = 2e-2       # max |O_gpu - O_oracle|
TOL_LSE_BF16 = 1e-2     # max |LSE_gpu - LSE_oracle|
TOL_FP32 = 1e-4         # max abs error of every fp32-path output
TOL_GRAD_REL = 3e-2     # ||g_gpu - g_oracle||_F / ||g_oracle||_F


def f64(t):
    return t.detach().to("cpu").double().numpy()


def max_abs(a, b):
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64)))) if np.size(a) else 0.0


def check_lse(got, ref, tol):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.array_equal(np.isneginf(got), np.isneginf(ref)), "empty-row pattern differs"
    fin = np.isfinite(ref)
    assert not np.any(np.isnan(got))
    if fin.any():
        err = float(np.max(np.abs(got[fin] - ref[fin])))
        assert err <= tol, f"LSE max abs err {err} > {tol}"


def check_close(got, ref, tol, what="O"):
    got = np.asarray(got, np.float64)
    assert not np.any(np.isnan(got)), f"{what} has NaN"
    err = max_abs(got, ref)
    assert err <= tol, f"{what} max abs err {err} > {tol}"


def rel_fro(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
