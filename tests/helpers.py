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


def check_tiles(got, ref, what="grad", tol=TOL_TILE_REL, rows=TILE_ROWS, round_rows=None):
    """Per-tile relative Frobenius bound over [..., N, d] arrays: every tile of
    `rows` consecutive rows of every leading index.

    round_rows, optional, [..., N]: per-row scales of the error that the
    method's own bf16 roundings produce (bf16_rounding_scales).  A tile then
    also passes when its error is within ROUND_MULT times the root sum of
    squares of its rows' scales: a tile whose exact value is a cancellation
    residue of the rounded quantities (a row that sees two keys of nearly
    equal dP) has no more correct digits than that."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    n, d = ref.shape[-2], ref.shape[-1]
    g2 = got.reshape(-1, n, d)
    r2 = ref.reshape(-1, n, d)
    s2 = None if round_rows is None else np.asarray(round_rows, np.float64).reshape(-1, n)
    errs, norms, rnd = [], [], []
    for a in range(r2.shape[0]):
        for t0 in range(0, n, rows):
            errs.append(np.linalg.norm(g2[a, t0:t0 + rows] - r2[a, t0:t0 + rows]))
            norms.append(np.linalg.norm(r2[a, t0:t0 + rows]))
            rnd.append(0.0 if s2 is None else np.sqrt(np.sum(s2[a, t0:t0 + rows] ** 2)))
    errs, norms, rnd = np.array(errs), np.array(norms), np.array(rnd)
    if norms.size == 0 or not np.any(norms > 0):
        assert np.all(errs == 0), f"{what}: nonzero where the reference is zero"
        return 0.0
    floor = 0.1 * np.sqrt(np.mean(norms ** 2))
    rel = errs / np.maximum(np.maximum(norms, floor), ROUND_MULT * rnd / tol)
    worst = int(np.argmax(rel))
    assert rel[worst] <= tol, (f"{what}: tile {worst} (of {rel.size}) relative error "
                               f"{rel[worst]:.3e} > {tol}")
    return float(rel[worst])


BF16_U = 2.0 ** -8  # unit roundoff of bf16 (8 significant bits)
ROUND_MULT = 4.0    # standard deviations of the rounding model a tile may reach


def bf16_rounding_scales(q, k, v, d_o, o, lse, q_off=0, kv_off=0, causal=False, scale=None,
                         block_mask=None):
    """Per-row standard deviations of the gradient error that the bf16
    roundings of the tensor-core backward produce, to first order, taking
    every rounding as an independent relative error of at most u = 2^-8:

    - P rounded for the dV product (u), P and dS = P (dP - delta) rounded for
      the dK and dQ products (2u);
    - O rounded to bf16 by the forward, on top of the rounding of P in its
      P V product (2u per element of O), entering delta = sum_c dO_c O_c.

    With a2_r = sum_c (dO_rc O_rc)^2, for query row r and key row j:
      dQ_r: 2u scale sqrt(a2_r |sum_j P_rj k_j|^2 + sum_j dS_rj^2 |k_j|^2)
      dK_j: 2u scale sqrt(sum_r (dS_rj^2 + P_rj^2 a2_r) |q_r|^2)
      dV_j: u sqrt(sum_r P_rj^2 |dO_r|^2)
    (the sums over r run over the query rows of every head of j's group).
    Arguments are float64 arrays as given to the oracle (block_mask as
    well); o and lse are the oracle's exact forward.  Returns ([B,Hq,Lq],
    [B,Hkv,Lk], [B,Hkv,Lk])."""
    from oracle import attention as A
    b, hq, lq, d = q.shape
    hkv, lk = k.shape[1], k.shape[2]
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    c = 2.0 * BF16_U * scale
    vis = A.visible(q_off + np.arange(lq), kv_off + np.arange(lk), causal)
    if block_mask is not None:
        vis = vis & A.block_visible(np.arange(lq), np.arange(lk), block_mask)
    kn2, qn2, don2 = (k ** 2).sum(-1), (q ** 2).sum(-1), (d_o ** 2).sum(-1)
    sq = np.zeros((b, hq, lq))
    sk2 = np.zeros((b, hkv, lk))
    sv2 = np.zeros((b, hkv, lk))
    for bi in range(b):
        for h in range(hq):
            g = A.kv_head_of(h, hq, hkv)
            fin = np.isfinite(lse[bi, h])
            s = scale * (q[bi, h] @ k[bi, g].T)
            with np.errstate(over="ignore", invalid="ignore"):
                p = np.where(vis & fin[:, None],
                             np.exp(s - np.where(fin, lse[bi, h], 0.0)[:, None]), 0.0)
            dp = d_o[bi, h] @ v[bi, g].T
            delta = (d_o[bi, h] * o[bi, h]).sum(-1)
            a2 = ((d_o[bi, h] * o[bi, h]) ** 2).sum(-1)
            ds = p * (dp - delta[:, None])
            pk = p @ k[bi, g]
            sq[bi, h] = c * np.sqrt(a2 * (pk ** 2).sum(-1) + (ds ** 2) @ kn2[bi, g])
            sk2[bi, g] += c ** 2 * ((ds ** 2).T @ qn2[bi, h] + (p ** 2).T @ (a2 * qn2[bi, h]))
            sv2[bi, g] += BF16_U ** 2 * ((p ** 2).T @ don2[bi, h])
    return sq, np.sqrt(sk2), np.sqrt(sv2)


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
