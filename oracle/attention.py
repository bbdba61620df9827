"""fp64 definition of exact softmax attention, its backward, and the LSE merge.

TEST INFRASTRUCTURE ONLY (see the package docstring): the oracle that the CUDA
path is checked against.  Plain numpy in float64; inputs are upcast copies of
exactly the values the GPU sees (bf16 or fp32).

What is computed, and where the pages fix it
--------------------------------------------
* Exact attention.  DistFlashAttn ("Effiziente verteilte Aufmerksamkeit fuer
  das Training von LLMs mit langem Kontext", core concepts) calls the method an
  *exact* attention mechanism, and BurstAttention (abstract) distributes that
  same exact computation.  The pages print no formula, so the oracle is the
  textbook definition: scores s_ij = scale * <q_i, k_j>, a softmax over the
  keys visible to query i, O_i = sum_j P_ij v_j, and the row log-sum-exp
  LSE_i = log sum_j exp(s_ij) in natural-log units.
* Chunks and offsets.  BurstAttention (method section: local attention
  computation plus global aggregation) splits the sequence into chunks; a
  chunk of queries starts at absolute position q_off and a chunk of keys at
  kv_off.  Reading taken where the pages are silent: with a causal mask, key j
  is visible to query i iff kv_off + j <= q_off + i (diagonal included).
* A query with no visible key gets O_i = 0 and LSE_i = -inf, which makes such
  a partial the identity of the merge below (the merge must be a reduction:
  LeanAttention abstract, "associative property of online softmax").
* Grouped query heads: query head h reads key/value head h // (H_q / H_kv)
  (contiguous groups; plainest reading, the pages do not define GQA).
* Merge.  Two partial results over disjoint key sets combine by the
  LSE-weighted sum; many partials combine in one pass by the same rule
  (Tree Attention abstract: the reduction across the sequence axis is a tree
  reduction; BurstAttention abstract: local results aggregated into global
  ones).
* Backward.  DistFlashAttn (core concepts, rematerialization-aware
  checkpointing) states the backward can run from the saved attention output
  without numerical differences.  The oracle does NOT use that shortcut: it
  rebuilds the softmax rows from Q and K and applies the softmax Jacobian
  explicitly, dS_ij = P_ij * (dP_ij - sum_k P_ik dP_ik).

* Block-sparse attention.  The Fine-grained Attention I/O Complexity page
  (abstract) extends the analysis to sparse attention, and the related-work
  list of the BriefGPT BurstAttention page names FlashAttention extended to
  a broad class of sparsity patterns.  Neither fixes a mask format; reading
  taken: a block mask over (query block, key block) of BLOCK x BLOCK
  positions, counted from the start of the chunks, shared by every batch row
  and head.  Key j is visible to query i iff the mask entry of their blocks
  is set AND the causal rule (if any) holds; a query left with no visible
  key gets O = 0, LSE = -inf as above.

The rows are processed in blocks only to bound memory (the full score matrix
of a 128K sequence is 128 GiB in fp64); each block holds complete score rows
and applies the two-pass softmax, so the blocking changes nothing.
"""

from __future__ import annotations

import math

import numpy as np

NEG_INF = -np.inf


def kv_head_of(h: int, n_q_heads: int, n_kv_heads: int) -> int:
    """Key/value head read by query head ``h`` (contiguous GQA groups)."""
    if n_kv_heads <= 0 or n_q_heads % n_kv_heads != 0:
        raise ValueError("query heads must be a multiple of key/value heads")
    return h // (n_q_heads // n_kv_heads)


def visible(q_pos: np.ndarray, k_pos: np.ndarray, causal: bool) -> np.ndarray:
    """Boolean [len(q_pos), len(k_pos)] visibility from ABSOLUTE positions."""
    q_pos = np.asarray(q_pos)
    k_pos = np.asarray(k_pos)
    if not causal:
        return np.ones((q_pos.shape[0], k_pos.shape[0]), dtype=bool)
    return k_pos[None, :] <= q_pos[:, None]


def _softmax_rows(s: np.ndarray):
    """Two-pass softmax of complete score rows; -inf entries are masked keys.

    Returns (P, LSE).  A row with no finite score yields P = 0, LSE = -inf.
    """
    m = s.max(axis=1)
    has = np.isfinite(m)
    m_safe = np.where(has, m, 0.0)
    e = np.exp(s - m_safe[:, None])  # exp(-inf) = 0 for masked keys
    denom = e.sum(axis=1)
    p = e / np.where(has, denom, 1.0)[:, None]
    with np.errstate(divide="ignore"):
        lse = np.where(has, m_safe + np.log(np.where(has, denom, 1.0)), NEG_INF)
    return p, lse


def _apply_softmax_jacobian(p: np.ndarray, dp: np.ndarray) -> np.ndarray:
    """dS = J^T dP for row-wise softmax, J = diag(p) - p p^T (symmetric)."""
    return p * (dp - (p * dp).sum(axis=1, keepdims=True))


def _shapes(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B, H, N, d]")
    b, hq, lq, d = q.shape
    bk, hkv, lk, dk = k.shape
    if bk != b or dk != d or v.shape[:3] != k.shape[:3]:
        raise ValueError("inconsistent q/k/v shapes")
    kv_head_of(0, hq, hkv)  # validates the grouping
    return b, hq, hkv, lq, lk, d


def block_visible(q_idx: np.ndarray, k_idx: np.ndarray, block_mask, block: int = 128):
    """Boolean [len(q_idx), len(k_idx)]: the mask entry of block
    (q // block, k // block) is set (indices from the start of the chunks)."""
    m = np.asarray(block_mask) != 0
    return m[np.asarray(q_idx)[:, None] // block, np.asarray(k_idx)[None, :] // block]


def _scores(qh, kh, q_pos, k_pos, causal, scale, bvis=None):
    s = scale * (qh @ kh.T)
    vis = visible(q_pos, k_pos, causal)
    if bvis is not None:
        vis = vis & bvis
    return np.where(vis, s, NEG_INF)


def attn_fwd(q, k, v, q_off=0, kv_off=0, causal=False, scale=None,
             rows=None, block=256, block_mask=None, mask_block=128):
    """Exact attention of a query chunk against a key/value chunk.

    q: [B, H_q, L_q, d]; k, v: [B, H_kv, L_k, d] (v may have its own last dim).
    q_off / kv_off: absolute position of row 0 of the chunk (causal mask only).
    rows: optional indices into L_q; only those query rows are computed.
    block_mask: optional [ceil(L_q/mask_block), ceil(L_k/mask_block)] array;
    only keys of set blocks are visible (see the module docstring).
    Returns (O [B, H_q, len(rows), d_v] float64, LSE [B, H_q, len(rows)]).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    b, hq, hkv, lq, lk, d = _shapes(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    rows = np.arange(lq) if rows is None else np.asarray(rows, dtype=np.int64)
    k_pos = kv_off + np.arange(lk)
    out = np.zeros((b, hq, rows.shape[0], v.shape[-1]))
    lse = np.full((b, hq, rows.shape[0]), NEG_INF)
    for bi in range(b):
        for h in range(hq):
            g = kv_head_of(h, hq, hkv)
            for r0 in range(0, rows.shape[0], block):
                ri = rows[r0:r0 + block]
                bv = None if block_mask is None else block_visible(
                    ri, np.arange(lk), block_mask, mask_block)
                s = _scores(q[bi, h, ri], k[bi, g], q_off + ri, k_pos, causal,
                            scale, bv)
                p, l_ = _softmax_rows(s)
                out[bi, h, r0:r0 + ri.shape[0]] = p @ v[bi, g]
                lse[bi, h, r0:r0 + ri.shape[0]] = l_
    return out, lse


def attn_bwd(q, k, v, d_o, q_off=0, kv_off=0, causal=False, scale=None,
             rows=None, block=256, block_mask=None, mask_block=128):
    """Gradients of L = sum(d_o * O) with respect to q, k, v.

    Rebuilds each softmax row from q and k and applies the softmax Jacobian
    explicitly (no saved O or LSE is used).  With ``rows`` given, only those
    query rows contribute: dq is returned for those rows, and dk/dv hold the
    contributions of those rows only (exact for key rows whose every visible
    query lies in ``rows``).
    Returns (dq [B,H_q,len(rows),d], dk [B,H_kv,L_k,d], dv [B,H_kv,L_k,d_v]).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    d_o = np.asarray(d_o, dtype=np.float64)
    b, hq, hkv, lq, lk, d = _shapes(q, k, v)
    if d_o.shape != q.shape[:3] + (v.shape[-1],):
        raise ValueError("d_o must be [B, H_q, L_q, d_v]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    rows = np.arange(lq) if rows is None else np.asarray(rows, dtype=np.int64)
    k_pos = kv_off + np.arange(lk)
    dq = np.zeros((b, hq, rows.shape[0], d))
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for bi in range(b):
        for h in range(hq):
            g = kv_head_of(h, hq, hkv)
            kh, vh = k[bi, g], v[bi, g]
            for r0 in range(0, rows.shape[0], block):
                ri = rows[r0:r0 + block]
                qh = q[bi, h, ri]
                bv = None if block_mask is None else block_visible(
                    ri, np.arange(lk), block_mask, mask_block)
                p, _ = _softmax_rows(_scores(qh, kh, q_off + ri, k_pos, causal,
                                             scale, bv))
                doh = d_o[bi, h, ri]
                dp = doh @ vh.T
                ds = _apply_softmax_jacobian(p, dp)
                dv[bi, g] += p.T @ doh
                dq[bi, h, r0:r0 + ri.shape[0]] = scale * (ds @ kh)
                dk[bi, g] += scale * (ds.T @ qh)
    return dq, dk, dv


def lse_merge(o_a, lse_a, o_b, lse_b):
    """Combine two partials over disjoint key sets into one.

    LSE = max + log(exp(LSE_a - max) + exp(LSE_b - max)); each O is weighted by
    exp(LSE_x - LSE).  Two empty partials (-inf, -inf) give (O = 0, -inf).
    """
    o_a = np.asarray(o_a, dtype=np.float64)
    o_b = np.asarray(o_b, dtype=np.float64)
    lse_a = np.asarray(lse_a, dtype=np.float64)
    lse_b = np.asarray(lse_b, dtype=np.float64)
    m = np.maximum(lse_a, lse_b)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    wa = np.exp(lse_a - m_safe)
    wb = np.exp(lse_b - m_safe)
    tot = np.where(empty, 1.0, wa + wb)
    lse = np.where(empty, NEG_INF, m_safe + np.log(tot))
    o = (wa / tot)[..., None] * o_a + (wb / tot)[..., None] * o_b
    return o, lse


def tree_merge(o_parts, lse_parts):
    """One-pass combination of k partials: o_parts [k, ...,d], lse_parts [k, ...].

    Same rule as ``lse_merge`` applied to all k at once (max over the k LSEs,
    weights exp(LSE_k - max), renormalised).
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    if o_parts.shape[:-1] != lse_parts.shape or o_parts.shape[0] < 1:
        raise ValueError("o_parts must be [k, ..., d] and lse_parts [k, ...]")
    m = lse_parts.max(axis=0)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    w = np.exp(lse_parts - m_safe[None])
    tot = np.where(empty, 1.0, w.sum(axis=0))
    lse = np.where(empty, NEG_INF, m_safe + np.log(tot))
    o = ((w / tot[None])[..., None] * o_parts).sum(axis=0)
    return o, lse
