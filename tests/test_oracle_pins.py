"""Pins for the fp64 oracle: each check depends on something other than the
oracle itself (scalar brute force, closed forms, algebraic invariants, finite
differences, exact symbolic evaluation, an independent library routine).

The planted-mistake tests at the end patch a deliberate error into the oracle
(on the CPU) and assert that at least one pin catches it.
"""

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import attention as A

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(shape, seed, scale=1.0):
    return scale * np.random.default_rng(seed).standard_normal(shape)


# --------------------------------------------------------------------------
# scalar brute force: loops + math.fsum, written independently of the oracle
# --------------------------------------------------------------------------

def brute_fwd(q, k, v, q_off, kv_off, causal, scale):
    b_, hq, lq, d = q.shape
    hkv, lk, dv = k.shape[1], k.shape[2], v.shape[3]
    grp = hq // hkv
    out = np.zeros((b_, hq, lq, dv))
    lse = np.full((b_, hq, lq), -math.inf)
    for b in range(b_):
        for h in range(hq):
            g = h // grp
            for i in range(lq):
                keys = [j for j in range(lk)
                        if (not causal) or (kv_off + j <= q_off + i)]
                if not keys:
                    continue
                s = [scale * math.fsum(float(q[b, h, i, c]) * float(k[b, g, j, c])
                                       for c in range(d)) for j in keys]
                m = max(s)
                e = [math.exp(x - m) for x in s]
                tot = math.fsum(e)
                for c in range(dv):
                    out[b, h, i, c] = math.fsum(
                        e[t] * float(v[b, g, j, c]) for t, j in enumerate(keys)) / tot
                lse[b, h, i] = m + math.log(tot)
    return out, lse


BRUTE_CASES = [
    # (Hq, Hkv, Lq, Lk, d, q_off, kv_off, causal, scale)
    (2, 2, 5, 7, 3, 0, 0, False, None),
    (2, 2, 5, 7, 3, 4, 0, True, 0.7),
    (4, 2, 6, 5, 4, 0, 3, True, None),   # GQA, first rows fully masked
    (3, 1, 4, 8, 2, 10, 2, True, 1.3),  # offsets beyond the key chunk
    (2, 1, 1, 9, 4, 0, 0, False, None),  # decode-shaped: one query
]


@pytest.mark.parametrize("case", BRUTE_CASES)
def test_fwd_matches_scalar_brute_force(case):
    hq, hkv, lq, lk, d, q_off, kv_off, causal, scale = case
    q = rnd((2, hq, lq, d), 1)
    k = rnd((2, hkv, lk, d), 2)
    v = rnd((2, hkv, lk, d + 1), 3)
    sc = scale if scale is not None else 1.0 / math.sqrt(d)
    o, lse = A.attn_fwd(q, k, v, q_off, kv_off, causal, scale)
    ob, lb = brute_fwd(q, k, v, q_off, kv_off, causal, sc)
    assert np.array_equal(np.isfinite(lse), np.isfinite(lb))
    fin = np.isfinite(lb)
    np.testing.assert_allclose(lse[fin], lb[fin], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(o, ob, rtol=1e-13, atol=1e-13)


def test_rows_subset_equals_full():
    q, k, v = rnd((1, 2, 40, 8), 4), rnd((1, 2, 40, 8), 5), rnd((1, 2, 40, 8), 6)
    rows = np.array([0, 3, 17, 39])
    o, lse = A.attn_fwd(q, k, v, 3, 0, True, None)
    o2, lse2 = A.attn_fwd(q, k, v, 3, 0, True, None, rows=rows, block=3)
    np.testing.assert_allclose(o2, o[:, :, rows], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(lse2, lse[:, :, rows], rtol=1e-14)


# --------------------------------------------------------------------------
# softmax normalisation, closed forms
# --------------------------------------------------------------------------

def test_probabilities_sum_to_one_and_are_nonnegative():
    lk = 12
    q = rnd((1, 2, 9, 5), 7, 3.0)
    k = rnd((1, 2, lk, 5), 8, 3.0)
    eye = np.broadcast_to(np.eye(lk), (1, 2, lk, lk))  # O = P when V = I
    p, lse = A.attn_fwd(q, k, eye, 2, 0, True, None)
    ok = np.isfinite(lse)
    assert np.all(p >= 0.0)
    np.testing.assert_allclose(p.sum(-1)[ok], 1.0, rtol=0, atol=1e-14)
    assert np.all(p[~ok] == 0.0)


@pytest.mark.parametrize("q_off,kv_off,causal", [(0, 0, False), (0, 0, True),
                                                 (3, 5, True), (20, 0, True)])
def test_zero_queries_give_mean_of_visible_values(q_off, kv_off, causal):
    lq, lk = 8, 10
    q = np.zeros((1, 2, lq, 4))
    k = rnd((1, 2, lk, 4), 9)
    v = rnd((1, 2, lk, 6), 10)
    o, lse = A.attn_fwd(q, k, v, q_off, kv_off, causal, None)
    for i in range(lq):
        n = lk if not causal else int(np.clip(q_off + i - kv_off + 1, 0, lk))
        if n == 0:
            assert np.all(o[:, :, i] == 0) and np.all(lse[:, :, i] == -np.inf)
        else:
            np.testing.assert_allclose(o[:, :, i], v[:, :, :n].mean(axis=2),
                                       rtol=1e-14, atol=1e-14)
            np.testing.assert_allclose(lse[:, :, i], math.log(n), rtol=1e-14)


def test_one_hot_score_row_returns_that_value_row():
    d, lk = 8, 16
    scale = 1.0 / math.sqrt(d)
    q = rnd((1, 1, 3, d), 11)
    k = rnd((1, 1, lk, d), 12, 0.01)
    v = rnd((1, 1, lk, d), 13)
    picks = [5, 0, 15]
    for i, j in enumerate(picks):
        # score of key j becomes 200 while the others stay near 0
        k[0, 0, j] = (200.0 / scale) * q[0, 0, i] / np.dot(q[0, 0, i], q[0, 0, i])
    rows_ok = [0, 2]  # row 1 may see another planted key; check rows 0 and 2
    o, _ = A.attn_fwd(q, k, v, 0, 0, False, scale)
    for i in rows_ok:
        others = [kk for kk in range(lk) if kk != picks[i]]
        s_other = scale * k[0, 0, others] @ q[0, 0, i]
        assert s_other.max() < 50.0
        np.testing.assert_allclose(o[0, 0, i], v[0, 0, picks[i]], rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# merge algebra and the chunk-merge invariant
# --------------------------------------------------------------------------

def _partial(seed, shape=(2, 3, 5), d=4, empty_rows=()):
    o = rnd(shape + (d,), seed)
    lse = rnd(shape, seed + 100, 30.0)
    for r in empty_rows:
        lse[..., r] = -np.inf
        o[..., r, :] = 0.0
    return o, lse


def test_merge_commutative_associative_identity():
    a, b, c = _partial(1, empty_rows=(0,)), _partial(2, empty_rows=(0, 1)), _partial(3)
    ab = A.lse_merge(*a, *b)
    ba = A.lse_merge(*b, *a)
    np.testing.assert_allclose(ab[0], ba[0], rtol=1e-14, atol=1e-15)
    np.testing.assert_array_equal(ab[1], ba[1])
    left = A.lse_merge(*ab, *c)
    right = A.lse_merge(*a, *A.lse_merge(*b, *c))
    np.testing.assert_allclose(left[0], right[0], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(left[1], right[1], rtol=1e-14)
    ident = (np.zeros_like(a[0]), np.full_like(a[1], -np.inf))
    ai = A.lse_merge(*a, *ident)
    np.testing.assert_array_equal(ai[0], a[0])
    np.testing.assert_array_equal(ai[1], a[1])
    # empty + empty stays empty, never NaN
    assert np.all(ab[1][..., 0] == -np.inf) and np.all(ab[0][..., 0, :] == 0)


def test_merge_huge_lse_gap_and_closed_form():
    o_a, o_b = np.ones((1, 4)), -np.ones((1, 4))
    o, lse = A.lse_merge(o_a, np.array([700.0]), o_b, np.array([-700.0]))
    np.testing.assert_allclose(o, o_a, atol=1e-300)
    np.testing.assert_allclose(lse, 700.0, rtol=1e-15)
    # equal LSEs: plain average, LSE + log 2
    o, lse = A.lse_merge(o_a, np.array([1.5]), o_b, np.array([1.5]))
    np.testing.assert_allclose(o, 0.0, atol=1e-15)
    np.testing.assert_allclose(lse, 1.5 + math.log(2.0), rtol=1e-15)


def test_tree_merge_equals_sequential_fold():
    parts = [_partial(10 + i, empty_rows=((i,) if i < 3 else ())) for i in range(7)]
    o_p = np.stack([p[0] for p in parts])
    l_p = np.stack([p[1] for p in parts])
    o_t, l_t = A.tree_merge(o_p, l_p)
    acc = parts[0]
    for p in parts[1:]:
        acc = A.lse_merge(*acc, *p)
    np.testing.assert_allclose(o_t, acc[0], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(l_t, acc[1], rtol=1e-14)


@pytest.mark.parametrize("causal", [True, False])
def test_chunk_partials_merged_equal_unchunked(causal):
    # the 4 x 4 chunk split of a 256-token sequence (64-row chunks), ring order
    n, c = 256, 64
    q, k, v = rnd((1, 2, n, 64), 21), rnd((1, 2, n, 64), 22), rnd((1, 2, n, 64), 23)
    o_full, lse_full = A.attn_fwd(q, k, v, 0, 0, causal, None)
    for qc in range(n // c):
        acc = None
        kcs = range(qc, -1, -1) if causal else range(n // c)
        for kc in kcs:
            part = A.attn_fwd(q[:, :, qc * c:(qc + 1) * c], k[:, :, kc * c:(kc + 1) * c],
                              v[:, :, kc * c:(kc + 1) * c], qc * c, kc * c, causal, None)
            acc = part if acc is None else A.lse_merge(*acc, *part)
        np.testing.assert_allclose(acc[0], o_full[:, :, qc * c:(qc + 1) * c],
                                   rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(acc[1], lse_full[:, :, qc * c:(qc + 1) * c],
                                   rtol=1e-12)


def test_uneven_key_splits_tree_merged_equal_unchunked():
    rng = np.random.default_rng(5)
    lq, lk = 30, 97
    q, k, v = rnd((1, 2, lq, 16), 31), rnd((1, 1, lk, 16), 32), rnd((1, 1, lk, 16), 33)
    q_off = 70
    o_full, lse_full = A.attn_fwd(q, k, v, q_off, 0, True, None)
    cuts = np.sort(rng.choice(np.arange(1, lk), size=6, replace=False))
    bounds = [0] + list(cuts) + [lk]
    parts = [A.attn_fwd(q, k[:, :, s:e], v[:, :, s:e], q_off, s, True, None)
             for s, e in zip(bounds[:-1], bounds[1:])]
    o_t, l_t = A.tree_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    np.testing.assert_allclose(o_t, o_full, rtol=1e-12, atol=1e-12)
    fin = np.isfinite(lse_full)
    assert np.array_equal(np.isfinite(l_t), fin)
    np.testing.assert_allclose(l_t[fin], lse_full[fin], rtol=1e-12)


def test_key_permutation_invariance_noncausal():
    q, k, v = rnd((1, 2, 7, 5), 41), rnd((1, 2, 11, 5), 42), rnd((1, 2, 11, 5), 43)
    perm = np.random.default_rng(1).permutation(11)
    o1, l1 = A.attn_fwd(q, k, v)
    o2, l2 = A.attn_fwd(q, k[:, :, perm], v[:, :, perm])
    np.testing.assert_allclose(o1, o2, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=1e-14)


# --------------------------------------------------------------------------
# energy view (Tree Attention abstract): the gradient of the scalar
# log-sum-exp "energy" is the attention block
# --------------------------------------------------------------------------

def test_energy_gradient_gives_attention_output():
    d, lq, lk = 6, 5, 9
    scale = 0.4
    q, k, v = rnd((1, 1, lq, d), 51), rnd((1, 1, lk, d), 52), rnd((1, 1, lk, d), 53)
    u = rnd((d,), 54)
    uv = v[0, 0] @ u  # u . v_j

    def lse_with(eps):
        # one extra feature: q' = [q, eps], k'_j = [k_j, (u.v_j)/scale]
        qa = np.concatenate([q, np.full((1, 1, lq, 1), eps)], axis=-1)
        ka = np.concatenate([k, (uv / scale)[None, None, :, None]], axis=-1)
        return A.attn_fwd(qa, ka, v, 4, 0, True, scale)[1]

    h = 1e-5
    deriv = (lse_with(h) - lse_with(-h)) / (2 * h)
    o, _ = A.attn_fwd(q, k, v, 4, 0, True, scale)
    np.testing.assert_allclose(deriv[0, 0], o[0, 0] @ u, rtol=1e-8, atol=1e-9)


# --------------------------------------------------------------------------
# backward: finite differences, identities
# --------------------------------------------------------------------------

def _loss(q, k, v, d_o, q_off, kv_off, causal, scale):
    return float((A.attn_fwd(q, k, v, q_off, kv_off, causal, scale)[0] * d_o).sum())


def test_backward_matches_elementwise_central_differences():
    q = rnd((1, 2, 4, 3), 61)
    k = rnd((1, 1, 5, 3), 62)
    v = rnd((1, 1, 5, 3), 63)
    d_o = rnd((1, 2, 4, 3), 64)
    args = (2, 0, True, 0.9)
    dq, dk, dv = A.attn_bwd(q, k, v, d_o, *args)
    h = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + h
            lp = _loss(q, k, v, d_o, *args)
            x[idx] = old - h
            lm = _loss(q, k, v, d_o, *args)
            x[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8)


@pytest.mark.parametrize("causal", [True, False])
def test_backward_directional_derivative_tiny_config(causal):
    # the 1 x 2 x 256 x 64 shape of the fp32 tiny case
    q, k, v = rnd((1, 2, 256, 64), 71), rnd((1, 2, 256, 64), 72), rnd((1, 2, 256, 64), 73)
    d_o = rnd((1, 2, 256, 64), 74)
    args = (0, 0, causal, None)
    grads = A.attn_bwd(q, k, v, d_o, *args)
    h = 1e-5
    for which in range(3):
        u = rnd(q.shape, 80 + which)
        xs = [q, k, v]
        plus = [x.copy() for x in xs]
        minus = [x.copy() for x in xs]
        plus[which] += h * u
        minus[which] -= h * u
        num = (_loss(*plus, d_o, *args) - _loss(*minus, d_o, *args)) / (2 * h)
        ana = float((grads[which] * u).sum())
        assert abs(num - ana) <= 1e-6 * max(1.0, abs(ana))


def test_backward_identities():
    n = 48
    q, k, v = rnd((2, 3, n, 8), 91), rnd((2, 3, n, 8), 92), rnd((2, 3, n, 8), 93)
    d_o = rnd((2, 3, n, 8), 94)
    q_off = 5  # every query sees at least key 0
    o, _ = A.attn_fwd(q, k, v, q_off, 0, True, None)
    dq, dk, dv = A.attn_bwd(q, k, v, d_o, q_off, 0, True, None)
    # rows of dS sum to zero  ->  sum_j dK_j = 0 for every head
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)
    # rows of P sum to one    ->  sum_j dV_j = sum_i dO_i
    np.testing.assert_allclose(dv.sum(axis=2), d_o.sum(axis=2), rtol=1e-12, atol=1e-12)
    # <Q, dQ> = <K, dK> and <V, dV> = <dO, O>, per head
    np.testing.assert_allclose((q * dq).sum(axis=(2, 3)), (k * dk).sum(axis=(2, 3)),
                               rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose((v * dv).sum(axis=(2, 3)), (d_o * o).sum(axis=(2, 3)),
                               rtol=1e-11, atol=1e-12)


def test_backward_row_subset_is_exact_for_tail_keys():
    n = 64
    q, k, v, d_o = (rnd((1, 2, n, 8), s) for s in (101, 102, 103, 104))
    dq, dk, dv = A.attn_bwd(q, k, v, d_o, 0, 0, True, None)
    tail = np.arange(n - 10, n)
    dq_t, dk_t, dv_t = A.attn_bwd(q, k, v, d_o, 0, 0, True, None, rows=tail, block=4)
    np.testing.assert_allclose(dq_t, dq[:, :, tail], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dk_t[:, :, tail], dk[:, :, tail], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dv_t[:, :, tail], dv[:, :, tail], rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------
# an independent library routine: torch SDPA on CPU in float64
# --------------------------------------------------------------------------

@pytest.mark.parametrize("q_off,kv_off,causal", [(0, 0, False), (0, 0, True), (9, 4, True)])
def test_matches_torch_sdpa_float64(q_off, kv_off, causal):
    torch = pytest.importorskip("torch")
    lq, lk, d = 12, 15, 8
    q, k, v = rnd((2, 4, lq, d), 111), rnd((2, 2, lk, d), 112), rnd((2, 2, lk, d), 113)
    d_o = rnd((2, 4, lq, d), 114)
    qt = torch.tensor(q, requires_grad=True)
    kt = torch.tensor(np.repeat(k, 2, axis=1), requires_grad=True)
    vt = torch.tensor(np.repeat(v, 2, axis=1), requires_grad=True)
    mask = None
    if causal:
        mask = torch.tensor((kv_off + np.arange(lk))[None, :] <= (q_off + np.arange(lq))[:, None])
        assert bool(mask.any(dim=1).all())  # SDPA gives NaN on empty rows
    ot = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask)
    (ot * torch.tensor(d_o)).sum().backward()
    o, _ = A.attn_fwd(q, k, v, q_off, kv_off, causal, None)
    dq, dk, dv = A.attn_bwd(q, k, v, d_o, q_off, kv_off, causal, None)
    np.testing.assert_allclose(o, ot.detach().numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dq, qt.grad.numpy(), rtol=1e-11, atol=1e-12)
    gk = kt.grad.numpy().reshape(2, 2, 2, lk, d).sum(axis=2)
    gv = vt.grad.numpy().reshape(2, 2, 2, lk, d).sum(axis=2)
    np.testing.assert_allclose(dk, gk, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dv, gv, rtol=1e-11, atol=1e-12)


# --------------------------------------------------------------------------
# exact symbolic worked example (tests/golden/worked_example.json)
# --------------------------------------------------------------------------

def test_worked_example_exact_symbolic():
    sp = pytest.importorskip("sympy")
    with open(os.path.join(GOLDEN, "worked_example.json")) as f:
        ex = json.load(f)
    fr = lambda m: [[sp.Rational(Fraction(x)) for x in row] for row in m]  # noqa: E731
    qv, kv, vv, dov = fr(ex["q"]), fr(ex["k"]), fr(ex["v"]), fr(ex["d_o"])
    scale = sp.Rational(Fraction(ex["scale"]))
    lq, lk, d = len(qv), len(kv), len(qv[0])
    Q = sp.Matrix(lq, d, lambda i, c: sp.Symbol(f"q{i}{c}"))
    K = sp.Matrix(lk, d, lambda j, c: sp.Symbol(f"k{j}{c}"))
    V = sp.Matrix(lk, d, lambda j, c: sp.Symbol(f"v{j}{c}"))
    subs = {}
    for M, val in ((Q, qv), (K, kv), (V, vv)):
        for i in range(M.rows):
            for c in range(M.cols):
                subs[M[i, c]] = val[i][c]
    O, LSE = [], []
    for i in range(lq):
        keys = [j for j in range(lk) if ex["kv_off"] + j <= ex["q_off"] + i]
        s = [scale * sum(Q[i, c] * K[j, c] for c in range(d)) for j in keys]
        z = sum(sp.exp(x) for x in s)
        O.append([sum(sp.exp(s[t]) * V[j, c] for t, j in enumerate(keys)) / z
                  for c in range(d)])
        LSE.append(sp.log(z))
    L = sum(sp.Rational(Fraction(0)) + dov[i][c] * O[i][c] for i in range(lq) for c in range(d))
    arr = lambda x: np.array(x, dtype=np.float64)  # noqa: E731
    q, k, v, d_o = arr(qv)[None, None], arr(kv)[None, None], arr(vv)[None, None], arr(dov)[None, None]
    o, lse = A.attn_fwd(q, k, v, ex["q_off"], ex["kv_off"], True, float(scale))
    dq, dk, dv = A.attn_bwd(q, k, v, d_o, ex["q_off"], ex["kv_off"], True, float(scale))
    ev = lambda e: float(sp.N(e.subs(subs), 30))  # noqa: E731
    for i in range(lq):
        assert abs(lse[0, 0, i] - ev(LSE[i])) < 1e-14
        for c in range(d):
            assert abs(o[0, 0, i, c] - ev(O[i][c])) < 1e-14
    for M, g in ((Q, dq), (K, dk), (V, dv)):
        for i in range(M.rows):
            for c in range(M.cols):
                assert abs(g[0, 0, i, c] - ev(sp.diff(L, M[i, c]))) < 1e-13


# --------------------------------------------------------------------------
# planted mistakes: each must be caught by a pin above
# --------------------------------------------------------------------------

def _fails(fn, *a, **kw):
    try:
        fn(*a, **kw)
    except AssertionError:
        return True
    return False


def test_planted_wrong_gqa_mapping_is_caught(monkeypatch):
    monkeypatch.setattr(A, "kv_head_of", lambda h, hq, hkv: h % hkv)
    assert _fails(test_fwd_matches_scalar_brute_force, BRUTE_CASES[2])


def test_planted_off_by_one_causal_mask_is_caught(monkeypatch):
    monkeypatch.setattr(A, "visible", lambda qp, kp, causal: (
        np.asarray(kp)[None, :] < np.asarray(qp)[:, None]) if causal else
        np.ones((len(qp), len(kp)), bool))
    assert _fails(test_zero_queries_give_mean_of_visible_values, 0, 0, True)
    assert _fails(test_fwd_matches_scalar_brute_force, BRUTE_CASES[1])


def test_planted_dropped_jacobian_term_is_caught(monkeypatch):
    monkeypatch.setattr(A, "_apply_softmax_jacobian", lambda p, dp: p * dp)
    assert _fails(test_backward_matches_elementwise_central_differences)
    assert _fails(test_backward_identities)


def test_planted_transposed_score_operand_is_caught(monkeypatch):
    real = A._scores

    def wrong(qh, kh, q_pos, k_pos, causal, scale, bvis=None):
        s = real(qh, kh, q_pos, k_pos, causal, scale, bvis)
        return s[:, ::-1].copy()  # keys in the wrong order
    monkeypatch.setattr(A, "_scores", wrong)
    assert _fails(test_fwd_matches_scalar_brute_force, BRUTE_CASES[0])


def test_planted_wrong_merge_weight_is_caught(monkeypatch):
    real = A.lse_merge

    def wrong(o_a, lse_a, o_b, lse_b):
        o, lse = real(o_a, lse_a, o_b, lse_b)
        return o, lse - 0.0 + (np.isfinite(lse) * 1e-3)
    monkeypatch.setattr(A, "lse_merge", wrong)
    assert _fails(test_chunk_partials_merged_equal_unchunked, True)


# --------------------------------------------------------------------------
# block masks (block-sparse attention)
# --------------------------------------------------------------------------

def brute_fwd_allowed(q, k, v, allowed, scale):
    """Scalar brute force over an explicit predicate allowed(i, j)."""
    b_, hq, lq, d = q.shape
    hkv, lk, dv = k.shape[1], k.shape[2], v.shape[3]
    grp = hq // hkv
    out = np.zeros((b_, hq, lq, dv))
    lse = np.full((b_, hq, lq), -math.inf)
    for b in range(b_):
        for h in range(hq):
            g = h // grp
            for i in range(lq):
                keys = [j for j in range(lk) if allowed(i, j)]
                if not keys:
                    continue
                s = [scale * math.fsum(float(q[b, h, i, c]) * float(k[b, g, j, c])
                                       for c in range(d)) for j in keys]
                m = max(s)
                e = [math.exp(x - m) for x in s]
                tot = math.fsum(e)
                for c in range(dv):
                    out[b, h, i, c] = math.fsum(
                        e[t] * float(v[b, g, j, c]) for t, j in enumerate(keys)) / tot
                lse[b, h, i] = m + math.log(tot)
    return out, lse


@pytest.mark.parametrize("causal", [False, True])
def test_block_mask_matches_scalar_brute_force(causal):
    lq, lk, blk, d = 9, 11, 2, 3
    q, k, v = rnd((2, 4, lq, d), 201), rnd((2, 2, lk, d), 202), rnd((2, 2, lk, d + 1), 203)
    mask = (np.random.default_rng(204).random((5, 6)) < 0.5).astype(np.uint8)
    mask[1, :] = 0  # queries 2, 3 see nothing
    sc = 0.8

    def allowed(i, j):
        return bool(mask[i // blk, j // blk]) and ((not causal) or j <= i)

    o, lse = A.attn_fwd(q, k, v, 0, 0, causal, sc, block_mask=mask, mask_block=blk)
    ob, lb = brute_fwd_allowed(q, k, v, allowed, sc)
    assert np.array_equal(np.isfinite(lse), np.isfinite(lb))
    assert np.all(o[:, :, 2:4] == 0) and np.all(lse[:, :, 2:4] == -np.inf)
    fin = np.isfinite(lb)
    np.testing.assert_allclose(lse[fin], lb[fin], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(o, ob, rtol=1e-13, atol=1e-13)


def test_full_and_block_causal_masks_reduce_to_the_plain_cases():
    n, blk = 40, 8
    q, k, v = rnd((1, 2, n, 4), 211), rnd((1, 2, n, 4), 212), rnd((1, 2, n, 4), 213)
    nb = n // blk
    full = np.ones((nb, nb), np.uint8)
    for causal in (False, True):
        a = A.attn_fwd(q, k, v, 0, 0, causal, None)
        b = A.attn_fwd(q, k, v, 0, 0, causal, None, block_mask=full, mask_block=blk)
        np.testing.assert_array_equal(a[0], b[0])
        np.testing.assert_array_equal(a[1], b[1])
    # blocks on and below the diagonal, plus the causal rule inside them
    tril = np.tril(np.ones((nb, nb), np.uint8))
    a = A.attn_fwd(q, k, v, 0, 0, True, None)
    b = A.attn_fwd(q, k, v, 0, 0, True, None, block_mask=tril, mask_block=blk)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_block_mask_backward_directional_derivative():
    lq = lk = 24
    blk = 4
    q, k, v = rnd((1, 2, lq, 5), 221), rnd((1, 1, lk, 5), 222), rnd((1, 1, lk, 5), 223)
    d_o = rnd((1, 2, lq, 5), 224)
    mask = (np.random.default_rng(225).random((6, 6)) < 0.6).astype(np.uint8)
    mask[:, 0] = 1
    kw = dict(block_mask=mask, mask_block=blk)

    def loss(q_, k_, v_):
        return float((A.attn_fwd(q_, k_, v_, 0, 0, True, 0.6, **kw)[0] * d_o).sum())

    grads = A.attn_bwd(q, k, v, d_o, 0, 0, True, 0.6, **kw)
    h = 1e-6
    for which in range(3):
        u = rnd((q, k, v)[which].shape, 230 + which)
        xs = [q.copy(), k.copy(), v.copy()]
        xm = [x.copy() for x in xs]
        xs[which] += h * u
        xm[which] -= h * u
        num = (loss(*xs) - loss(*xm)) / (2 * h)
        ana = float((grads[which] * u).sum())
        assert abs(num - ana) <= 1e-6 * max(1.0, abs(ana))


def test_planted_transposed_block_mask_is_caught(monkeypatch):
    real = A.block_visible

    def wrong(q_idx, k_idx, block_mask, block=128):
        return real(q_idx, k_idx, np.asarray(block_mask).T.copy()
                    if np.asarray(block_mask).shape[0] == np.asarray(block_mask).shape[1]
                    else block_mask, block)

    monkeypatch.setattr(A, "block_visible", wrong)

    def square_case():
        lq = lk = 9
        blk = 2
        q, k, v = rnd((1, 2, lq, 3), 241), rnd((1, 2, lk, 3), 242), rnd((1, 2, lk, 3), 243)
        mask = (np.random.default_rng(244).random((5, 5)) < 0.5).astype(np.uint8)

        def allowed(i, j):
            return bool(mask[i // blk, j // blk])
        o, _ = A.attn_fwd(q, k, v, 0, 0, False, 0.8, block_mask=mask, mask_block=blk)
        ob, _ = brute_fwd_allowed(q, k, v, allowed, 0.8)
        np.testing.assert_allclose(o, ob, rtol=1e-13, atol=1e-13)

    with pytest.raises(AssertionError):
        square_case()
