"""Shared test helpers: tolerances and comparisons against the oracle."""

import numpy as np

# GPU-vs-oracle tolerances (bf16 tensor-core path / fp32 CUDA-core path)
TOL_O_BF16 = 2e-2       # max |O_gpu - O_oracle|
TOL_LSE_BF16 = 1e-2     # max |LSE_gpu - LSE_oracle|
TOL_FP32 = 1e-4         # max abs error of every fp32-path output
TOL_GRAD_REL = 3e-2     # ||g_gpu - g_oracle||_F / ||g_oracle||_F
# The same bound applied to every 128-row tile of a gradient.  The global
# Frobenius figure alone cannot see one wrong tile among a thousand (a lost
# or doubled key-tile contribution moves it by ~3%); such a tile is wrong by
# the order of its own norm, while the rounding of P and dS to bf16 leaves
# every tile within the same few 1e-3 as the whole.  Tiles whose reference
# norm is under a tenth of the tensor's RMS tile norm (keys that only a few
# queries see) are held to that tenth instead of their own norm.
TOL_TILE_REL = 3e-2
TILE_ROWS = 128


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


def check_tiles(got, ref, what="grad", tol=TOL_TILE_REL, rows=TILE_ROWS):
    """Per-tile relative Frobenius bound over [..., N, d] arrays: every tile of
    `rows` consecutive rows of every leading index."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    n, d = ref.shape[-2], ref.shape[-1]
    g2 = got.reshape(-1, n, d)
    r2 = ref.reshape(-1, n, d)
    errs, norms = [], []
    for a in range(r2.shape[0]):
        for t0 in range(0, n, rows):
            errs.append(np.linalg.norm(g2[a, t0:t0 + rows] - r2[a, t0:t0 + rows]))
            norms.append(np.linalg.norm(r2[a, t0:t0 + rows]))
    errs, norms = np.array(errs), np.array(norms)
    if norms.size == 0 or not np.any(norms > 0):
        assert np.all(errs == 0), f"{what}: nonzero where the reference is zero"
        return 0.0
    floor = 0.1 * np.sqrt(np.mean(norms ** 2))
    rel = errs / np.maximum(norms, floor)
    worst = int(np.argmax(rel))
    assert rel[worst] <= tol, (f"{what}: tile {worst} (of {rel.size}) relative error "
                               f"{rel[worst]:.3e} > {tol}")
    return float(rel[worst])


def _oracle_bwd_part(args):
    from oracle import attention as A
    q, k, v, d_o, q_off, kv_off, causal, rows = args
    return A.attn_bwd(q, k, v, d_o, q_off, kv_off, causal, rows=rows)


def oracle_bwd_rows(q, k, v, d_o, q_off, kv_off, causal, rows, workers=8):
    """The oracle's attn_bwd over `rows`, split into `workers` groups of rows
    run in spawned processes (the oracle itself is unchanged; its dk / dv are
    sums over query rows, so the groups' contributions add up)."""
    import concurrent.futures as cf
    import multiprocessing as mp
    groups = [g for g in np.array_split(np.asarray(rows), workers) if g.size]
    with cf.ProcessPoolExecutor(len(groups), mp_context=mp.get_context("spawn")) as ex:
        parts = list(ex.map(_oracle_bwd_part,
                            [(q, k, v, d_o, q_off, kv_off, causal, g) for g in groups]))
    dq = np.concatenate([p_[0] for p_ in parts], axis=2)
    dk = sum(p_[1] for p_ in parts)
    dv = sum(p_[2] for p_ in parts)
    return dq, dk, dv
