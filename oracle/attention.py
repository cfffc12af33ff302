"""fp64 reference of exact softmax attention, forward and backward.

TEST INFRASTRUCTURE ONLY (see the package docstring): nothing on the product path
imports this module, and this module imports nothing from the product path.

Sources, cited by page title and section:

* [FA-chapter]  "Flash Attention" (mlx.void.app, chapter 4 deep dive), sections
  "地基：流式 softmax" (streaming softmax), "FlashAttention——把整件事分块塞进 SRAM",
  "FlashAttention-2——让每个核心都忙起来".
* [FA-review]   review of "FlashAttention: Fast and Memory-Efficient Exact Attention
  with IO-Awareness" (trdm.cn/news/294627), sections "方法细节" and "常见问题FAQ".
* [FA-practice] FlashAttention practitioner article (cf-1.com/news/4497868), sections
  "1.1 经典自注意力的那笔天价账单", "2.2 online softmax", "3.1 naive attention到flash
  kernel的替换路径".
* [FA-math17]   "大模型数学速成（17）：Flash Attention——不物化注意力矩阵", sections
  "一、标准 Attention 的痛点", "二、数学不变，变的是计算路径", "三、分块 + 在线 Softmax 直觉".

Arrays are laid out (batch, heads, seq, head_dim) as in [FA-practice] §1.1 and §3.1.
Every input is first converted to float64; every step is carried out in float64.
Nothing here blocks, fuses or reorders beyond what the definition states; the only
concession to size is that the query rows of one head may be processed in row
blocks, each of which still holds complete rows of S and P.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "attn_cross_head_fwd",
    "attn_cross_fwd_ref",
    "attn_gqa_bwd_ref",
    "kv_head_of",
    "merge_partials",
    "butterfly_pairs_visible",
    "butterfly_mask",
    "attn_masked_head_fwd",
    "attn_masked_head_bwd",
    "attn_rows_ref",
    "softmax_two_pass",
    "online_softmax_stats",
    "online_attention_row",
    "attn_head_fwd",
    "attn_head_bwd",
    "attn_fwd_ref",
    "attn_fwd_tiled_ref",
    "attn_bwd_ref",
]


# ----------------------------------------------------------------------------------
# softmax
# ----------------------------------------------------------------------------------
def softmax_two_pass(x):
    """Safe softmax along the last axis: subtract the row maximum, exponentiate,
    divide by the sum.

    [FA-chapter] "地基：流式 softmax": softmax exponentiates each score and divides by
    the total; subtracting the row maximum first keeps e^x from overflowing and
    cancels in the division, at the price of a first pass to find the maximum.
    [FA-practice] §2.2 gives the same three lines (m = max, l = sum exp(x - m),
    softmax = exp(x - m) / l).
    """
    x = np.asarray(x, dtype=np.float64)
    m = np.max(x, axis=-1, keepdims=True)
    e = np.exp(x - m)
    return e / np.sum(e, axis=-1, keepdims=True)


# ----------------------------------------------------------------------------------
# streaming (online) softmax -- used only to check the oracle's own algebra
# ----------------------------------------------------------------------------------
def _blocks(n, splits):
    cuts = [0] + sorted(int(s) for s in splits) + [n]
    return [(cuts[i], cuts[i + 1]) for i in range(len(cuts) - 1) if cuts[i + 1] > cuts[i]]


def online_softmax_stats(row, splits, form="updated_max"):
    """Run the streaming (m, l) recurrence over the blocks of ``row`` cut at ``splits``.

    Returns the list of (m, l) after each block; the final pair equals
    (max(row), sum(exp(row - max(row)))).

    form="updated_max"  -- [FA-chapter] "地基：流式 softmax" and the opening section: the
        new block's sum is taken against the *updated* running maximum, and only the
        running total is multiplied by e^{m_old - m_new}.  [FA-practice] §2.2 states
        the same update (alpha = exp(m1 - m2), l_new = alpha*l1 + sum(exp(x2 - m2))).
    form="block_local"  -- [FA-review] "方法细节": each block keeps its own maximum
        m~ and sum l~ = sum(exp(x - m~)); the merge is
        l_new = e^{m - m_new} l + e^{m~ - m_new} l~ with m_new = max(m, m~).
        [FA-math17] §三 works the two-block example in this shape.
    """
    row = np.asarray(row, dtype=np.float64)
    m = -np.inf
    l = 0.0
    out = []
    for lo, hi in _blocks(row.shape[0], splits):
        x = row[lo:hi]
        if form == "updated_max":
            m_new = max(m, float(np.max(x)))
            alpha = np.exp(m - m_new) if m != -np.inf else 0.0
            l = alpha * l + float(np.sum(np.exp(x - m_new)))
            m = m_new
        elif form == "block_local":
            mb = float(np.max(x))
            lb = float(np.sum(np.exp(x - mb)))
            m_new = max(m, mb)
            a_old = np.exp(m - m_new) if m != -np.inf else 0.0
            l = a_old * l + np.exp(mb - m_new) * lb
            m = m_new
        else:
            raise ValueError(f"unknown form {form!r}")
        out.append((m, l))
    return out


def online_attention_row(scores, values, splits):
    """One query row of attention by the streaming recurrence over key/value blocks.

    [FA-practice] §2.2: alpha = exp(m1 - m2); l_new = alpha*l1 + sum(exp(x2 - m2));
    acc_new = alpha*acc1 + exp(x2 - m2) @ V2; the output is acc/l at the end.
    [FA-chapter] "FlashAttention-2": the output is kept unnormalised and divided by l
    once at the end.  Returns (o, m, l).
    """
    s = np.asarray(scores, dtype=np.float64)
    v = np.asarray(values, dtype=np.float64)
    m = -np.inf
    l = 0.0
    acc = np.zeros(v.shape[1], dtype=np.float64)
    for lo, hi in _blocks(s.shape[0], splits):
        x = s[lo:hi]
        m_new = max(m, float(np.max(x)))
        alpha = np.exp(m - m_new) if m != -np.inf else 0.0
        e = np.exp(x - m_new)
        l = alpha * l + float(np.sum(e))
        acc = alpha * acc + e @ v[lo:hi]
        m = m_new
    return acc / l, m, l


# ----------------------------------------------------------------------------------
# the plain definition, one head
# ----------------------------------------------------------------------------------
def _scores(q, k, scale, causal, row0):
    """S = scale * Q K^T for query rows row0.. of one head, with the causal mask.

    [FA-math17] §一: S = Q K^T / sqrt(d).  [FA-practice] §3.1: scores = q @ k^T * scale.
    Causal ([FA-chapter] "FlashAttention-2": future tokens cannot be attended;
    [FA-math17] §五: lower-triangular visibility): key j is visible to query i iff
    j <= i, so S_ij = -inf for j > i.
    """
    s = scale * (q @ k.T)
    if causal:
        rows = np.arange(row0, row0 + q.shape[0])[:, None]
        cols = np.arange(k.shape[0])[None, :]
        s = np.where(cols > rows, -np.inf, s)
    return s


def _row_range(n, row_range):
    """The query rows [lo, hi) a call covers: all n rows, or the given range."""
    if row_range is None:
        return 0, n
    lo, hi = int(row_range[0]), int(row_range[1])
    if not 0 <= lo <= hi <= n:
        raise ValueError(f"row range {row_range} outside [0, {n}]")
    return lo, hi


def attn_head_fwd(q, k, v, scale, causal, row_block=None, return_sp=False, row_range=None):
    """Exact attention of one head: (O, LSE) or (O, LSE, S, P).

    S = scale*Q K^T (masked), m_i = max_j S_ij, E = exp(S - m), l_i = sum_j E_ij,
    P = E / l, O = P V, LSE_i = m_i + ln l_i (natural log, over the scaled scores).

    [FA-math17] §一/§二: O_i = sum_j P_ij V_j with P_ij = e^{S_ij} / sum_k e^{S_ik}.
    [FA-chapter] "地基：流式 softmax" for the max subtraction.  [FA-chapter]
    "FlashAttention——把整件事分块塞进 SRAM" and [FA-review] "方法细节": the forward
    keeps only O and the per-row statistics (m, l); LSE = m + ln l carries both.

    ``row_range=(lo, hi)`` computes only query rows lo..hi-1 (each row of O and LSE
    depends on its own row of S alone); the arrays returned then have hi - lo rows.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    lo, hi = _row_range(q.shape[0], row_range)
    n = hi - lo
    rb = max(n, 1) if row_block is None else int(row_block)
    o = np.empty((n, v.shape[1]), dtype=np.float64)
    lse = np.empty(n, dtype=np.float64)
    s_full = p_full = None
    if return_sp:
        s_full = np.empty((n, k.shape[0]), dtype=np.float64)
        p_full = np.empty((n, k.shape[0]), dtype=np.float64)
    for r0 in range(lo, hi, rb):
        r1 = min(hi, r0 + rb)
        s = _scores(q[r0:r1], k, scale, causal, r0)
        m = np.max(s, axis=1, keepdims=True)
        e = np.exp(s - m)
        l = np.sum(e, axis=1, keepdims=True)
        p = e / l
        o[r0 - lo:r1 - lo] = p @ v
        lse[r0 - lo:r1 - lo] = (m + np.log(l))[:, 0]
        if return_sp:
            s_full[r0 - lo:r1 - lo] = s
            p_full[r0 - lo:r1 - lo] = p
    if return_sp:
        return o, lse, s_full, p_full
    return o, lse


def attn_head_bwd(q, k, v, do, scale, causal, row_block=None, row_range=None):
    """Gradients of L = sum(dO * O) for one head: (dQ, dK, dV, D).

    The pages say only that the backward regenerates S and P from Q, K and the saved
    statistics instead of storing them ([FA-chapter] "FlashAttention——把整件事分块塞进
    SRAM", last paragraph; [FA-review] "方法细节" and FAQ).  The formulas are the
    derivative of the forward definition:

        dV = P^T dO,   dP = dO V^T,   D_i = sum_j P_ij dP_ij,
        dS = P o (dP - D),   dQ = scale * dS K,   dK = scale * dS^T Q.

    P is rebuilt here from the definition (not from any stored statistic).

    dK and dV are sums over the query rows i (dV_j = sum_i P_ij dO_i, dK_j = scale *
    sum_i dS_ij Q_i).  ``row_range=(lo, hi)`` takes only rows lo..hi-1: dQ and D are
    then those rows' (hi - lo rows), and dK, dV are those rows' contributions to the
    two sums, so the contributions of the parts of a partition of the rows add up to
    the whole head's dK and dV.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    lo, hi = _row_range(q.shape[0], row_range)
    n = hi - lo
    rb = max(n, 1) if row_block is None else int(row_block)
    dq = np.empty((n, q.shape[1]), dtype=np.float64)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dvec = np.empty(n, dtype=np.float64)
    for r0 in range(lo, hi, rb):
        r1 = min(hi, r0 + rb)
        s = _scores(q[r0:r1], k, scale, causal, r0)
        m = np.max(s, axis=1, keepdims=True)
        e = np.exp(s - m)
        p = e / np.sum(e, axis=1, keepdims=True)
        g = do[r0:r1]
        dv += p.T @ g
        dp = g @ v.T
        d_i = np.sum(p * dp, axis=1, keepdims=True)
        ds = p * (dp - d_i)
        dq[r0 - lo:r1 - lo] = scale * (ds @ k)
        dk += scale * (ds.T @ q[r0:r1])
        dvec[r0 - lo:r1 - lo] = d_i[:, 0]
    return dq, dk, dv, dvec


def attn_rows_ref(q_rows, rows, k, v, scale, causal, do_rows=None):
    """The plain definition for selected query rows of one head.

    q_rows: (R, d) query rows whose positions in the sequence are ``rows``; k, v: the
    whole head (N, d).  Returns (O_rows, LSE_rows) or, when ``do_rows`` is given,
    (O_rows, LSE_rows, dQ_rows, D_rows) with D_i = sum_j P_ij dP_ij and
    dQ_i = scale * sum_j P_ij (dP_ij - D_i) K_j -- the same formulas as
    ``attn_head_fwd`` / ``attn_head_bwd`` restricted to the given rows (each row of S,
    P, dP depends only on its own query row).
    """
    q = np.asarray(q_rows, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    rows = np.asarray(rows)
    s = scale * (q @ k.T)
    if causal:
        s = np.where(np.arange(k.shape[0])[None, :] > rows[:, None], -np.inf, s)
    m = np.max(s, axis=1, keepdims=True)
    e = np.exp(s - m)
    l = np.sum(e, axis=1, keepdims=True)
    p = e / l
    o = p @ v
    lse = (m + np.log(l))[:, 0]
    if do_rows is None:
        return o, lse
    g = np.asarray(do_rows, dtype=np.float64)
    dp = g @ v.T
    d_i = np.sum(p * dp, axis=1, keepdims=True)
    dq = scale * ((p * (dp - d_i)) @ k)
    return o, lse, dq, d_i[:, 0]


# ----------------------------------------------------------------------------------
# batched wrappers over (batch, heads)
# ----------------------------------------------------------------------------------
def _check4(*arrs):
    for a in arrs:
        if np.asarray(a).ndim != 4:
            raise ValueError("expected (batch, heads, seq, head_dim) arrays")


def attn_fwd_ref(q, k, v, scale, causal, row_block=None, heads=None):
    """Exact attention forward over (batch, heads, seq, head_dim) arrays.

    Returns (O, LSE) with O of shape (B, H, N, d) and LSE of shape (B, H, N), both
    float64.  ``heads`` optionally restricts the computation to a list of (b, h)
    pairs; the other entries of the result are NaN.
    """
    _check4(q, k, v)
    B, H, N, d = np.shape(q)
    o = np.full((B, H, N, np.shape(v)[3]), np.nan)
    lse = np.full((B, H, N), np.nan)
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in pairs:
        o[b, h], lse[b, h] = attn_head_fwd(q[b, h], k[b, h], v[b, h], scale, causal, row_block)
    return o, lse


def attn_bwd_ref(q, k, v, do, scale, causal, row_block=None, heads=None):
    """Exact attention backward over (batch, heads, seq, head_dim) arrays.

    Returns (dQ, dK, dV, D), float64; ``heads`` as in ``attn_fwd_ref``.
    """
    _check4(q, k, v, do)
    B, H, N, d = np.shape(q)
    dq = np.full(np.shape(q), np.nan)
    dk = np.full(np.shape(k), np.nan)
    dv = np.full(np.shape(v), np.nan)
    dvec = np.full((B, H, N), np.nan)
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in pairs:
        dq[b, h], dk[b, h], dv[b, h], dvec[b, h] = attn_head_bwd(
            q[b, h], k[b, h], v[b, h], do[b, h], scale, causal, row_block)
    return dq, dk, dv, dvec


def attn_fwd_tiled_ref(q, k, v, scale, causal, block_q, block_k):
    """Forward by the tiled streaming schedule, one head (N, d) arrays, float64.

    Used only to check the oracle's algebra: for each query block, stream the key
    blocks, update (m, l, acc) with the rescale e^{m_old - m_new}, divide by l at the
    end ([FA-chapter] "FlashAttention——把整件事分块塞进 SRAM" and "FlashAttention-2";
    [FA-math17] §三 and §四).  Returns (O, LSE).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n = q.shape[0]
    o = np.empty((n, v.shape[1]))
    lse = np.empty(n)
    for r0 in range(0, n, block_q):
        r1 = min(n, r0 + block_q)
        m = np.full(r1 - r0, -np.inf)
        l = np.zeros(r1 - r0)
        acc = np.zeros((r1 - r0, v.shape[1]))
        for c0 in range(0, k.shape[0], block_k):
            c1 = min(k.shape[0], c0 + block_k)
            s = scale * (q[r0:r1] @ k[c0:c1].T)
            if causal:
                rows = np.arange(r0, r1)[:, None]
                cols = np.arange(c0, c1)[None, :]
                s = np.where(cols > rows, -np.inf, s)
            m_new = np.maximum(m, np.max(s, axis=1))
            alpha = np.where(np.isneginf(m), 0.0, np.exp(m - np.where(np.isneginf(m_new), 0.0, m_new)))
            e = np.where(np.isneginf(s), 0.0, np.exp(s - np.where(np.isneginf(m_new), 0.0, m_new)[:, None]))
            l = alpha * l + np.sum(e, axis=1)
            acc = alpha[:, None] * acc + e @ v[c0:c1]
            m = m_new
        o[r0:r1] = acc / l[:, None]
        lse[r0:r1] = m + np.log(l)
    return o, lse


# ----------------------------------------------------------------------------------
# cross lengths (Nq != Nk), grouped key/value heads, split key ranges
# ----------------------------------------------------------------------------------
def _cross_scores(q, k, scale, causal):
    """S = scale * Q K^T for Nq query rows against Nk keys, causal bottom-right.

    With Nq != Nk the pages give no alignment; the reading taken here is the one under
    which the last query row is the newest token ([FA-practice] §3.1 describes
    decoding a new token against a key/value cache): key j is visible to query i
    iff j <= i + (Nk - Nq).  Nq = Nk gives the square mask of ``_scores``.
    """
    s = scale * (q @ k.T)
    if causal:
        nq, nk = q.shape[0], k.shape[0]
        rows = np.arange(nq)[:, None] + (nk - nq)
        cols = np.arange(nk)[None, :]
        s = np.where(cols > rows, -np.inf, s)
    return s


def attn_cross_head_fwd(q, k, v, scale, causal):
    """Exact attention of one head with Nq query rows and Nk keys: (O, LSE).

    The definition of ``attn_head_fwd`` with the bottom-right causal mask of
    ``_cross_scores``.  A row with no visible key (only when causal and Nk < Nq) has
    an empty softmax; the reading taken is O = 0 and LSE = -inf (the limit of a sum
    of no terms: l = 0, ln l = -inf).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    s = _cross_scores(q, k, scale, causal)
    o = np.zeros((q.shape[0], v.shape[1]))
    lse = np.full(q.shape[0], -np.inf)
    live = np.isfinite(s).any(axis=1)
    if live.any():
        sl = s[live]
        m = np.max(sl, axis=1, keepdims=True)
        e = np.exp(sl - m)
        l = np.sum(e, axis=1, keepdims=True)
        o[live] = (e / l) @ v
        lse[live] = (m + np.log(l))[:, 0]
    return o, lse


def kv_head_of(h, H, Hkv):
    """Key/value head read by query head h when H query heads share Hkv key/value
    heads (grouped-query attention): consecutive groups of G = H / Hkv query heads
    share one key/value head, h -> h // G.  The pages name grouped-query attention
    only as orthogonal to the tiling ("大模型数学速成（17）" §五); the grouping used is
    the usual contiguous one.  Hkv = H is ordinary multi-head attention.
    """
    if H % Hkv:
        raise ValueError("H must be a multiple of Hkv")
    return h // (H // Hkv)


def attn_cross_fwd_ref(q, k, v, scale, causal, heads=None):
    """Forward over q (B, H, Nq, d) and k, v (B, Hkv, Nk, d): (O, LSE), float64.

    Query head h reads key/value head ``kv_head_of(h, H, Hkv)``; each (b, h) is
    ``attn_cross_head_fwd``.  ``heads`` restricts the work to (b, h) pairs (others NaN).
    """
    _check4(q, k, v)
    B, H, Nq, _ = np.shape(q)
    Hkv = np.shape(k)[1]
    o = np.full((B, H, Nq, np.shape(v)[3]), np.nan)
    lse = np.full((B, H, Nq), np.nan)
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in pairs:
        hk = kv_head_of(h, H, Hkv)
        o[b, h], lse[b, h] = attn_cross_head_fwd(q[b, h], k[b, hk], v[b, hk], scale, causal)
    return o, lse


def attn_gqa_bwd_ref(q, k, v, do, scale, causal, row_block=None):
    """Backward with grouped key/value heads, square N: (dQ, dK, dV), float64.

    Every query head h is the ordinary attention of its own Q against key/value head
    kv_head_of(h); a key/value head's gradient is therefore the sum, over the query
    heads that read it, of the per-head gradients of ``attn_head_bwd``.
    """
    _check4(q, k, v, do)
    B, H, N, _ = np.shape(q)
    Hkv = np.shape(k)[1]
    dq = np.empty(np.shape(q))
    dk = np.zeros(np.shape(k))
    dv = np.zeros(np.shape(v))
    for b in range(B):
        for h in range(H):
            hk = kv_head_of(h, H, Hkv)
            gq, gk, gv, _ = attn_head_bwd(q[b, h], k[b, hk], v[b, hk], do[b, h], scale, causal, row_block)
            dq[b, h] = gq
            dk[b, hk] += gk
            dv[b, hk] += gv
    return dq, dk, dv


def merge_partials(o_parts, lse_parts):
    """Combine attention over disjoint key ranges into attention over their union.

    Part s holds O_s (rows x d, normalised over its own keys) and LSE_s; the union
    has LSE = ln sum_s e^{LSE_s} and O = sum_s e^{LSE_s - LSE} O_s.  This is the
    block-local merge of [FA-review] "方法细节" (l_new = e^{m-m_new} l + e^{m~-m_new} l~)
    with each part's (m, l) folded into LSE_s = m_s + ln l_s.  Parts with LSE_s = -inf
    (no visible key) contribute nothing; if every part is empty, O = 0, LSE = -inf.
    """
    o_parts = [np.asarray(o, dtype=np.float64) for o in o_parts]
    lse_parts = np.stack([np.asarray(x, dtype=np.float64) for x in lse_parts])   # (S, rows)
    m = np.max(lse_parts, axis=0)
    safe = np.where(np.isneginf(m), 0.0, m)
    w = np.where(np.isneginf(lse_parts), 0.0, np.exp(lse_parts - safe[None, :]))
    tot = np.sum(w, axis=0)
    lse = np.where(tot > 0, safe + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)
    o = np.zeros_like(o_parts[0])
    for s_, op in enumerate(o_parts):
        o += (w[s_] / np.where(tot > 0, tot, 1.0))[:, None] * op
    return o, lse


# ----------------------------------------------------------------------------------
# block-sparse attention with a fixed butterfly block pattern
# ----------------------------------------------------------------------------------
BUTTERFLY_BLOCK = 256


def butterfly_pairs_visible(p, q):
    """Block p of queries sees block q of keys in the butterfly pattern iff p == q or
    p and q differ in exactly one bit of their block index.

    [FA-review] "方法细节" names block-sparse FlashAttention with a fixed butterfly
    mask; the pages give neither the pattern's formula nor its block size.  The
    reading taken: the butterfly graph on block indices (an edge between indices that
    differ in one bit, plus the diagonal), with blocks of 256 rows and keys
    (``BUTTERFLY_BLOCK``).
    """
    x = int(p) ^ int(q)
    return x == 0 or (x & (x - 1)) == 0


def butterfly_mask(nq, nk, causal, block=BUTTERFLY_BLOCK):
    """Boolean (nq, nk) visibility matrix: butterfly blocks, and j <= i when causal."""
    bi = np.arange(nq)[:, None] // block
    bj = np.arange(nk)[None, :] // block
    x = bi ^ bj
    vis = (x & (x - 1)) == 0
    if causal:
        vis &= np.arange(nk)[None, :] <= np.arange(nq)[:, None]
    return vis


def attn_masked_head_fwd(q, k, v, scale, mask):
    """The definition of ``attn_head_fwd`` with an arbitrary boolean visibility mask
    (S_ij = -inf where the mask is False).  Rows with no visible key: O = 0, LSE = -inf."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    s = np.where(mask, scale * (q @ k.T), -np.inf)
    o = np.zeros((q.shape[0], v.shape[1]))
    lse = np.full(q.shape[0], -np.inf)
    live = mask.any(axis=1)
    if live.any():
        m = np.max(s[live], axis=1, keepdims=True)
        e = np.exp(s[live] - m)
        l = np.sum(e, axis=1, keepdims=True)
        o[live] = (e / l) @ v
        lse[live] = (m + np.log(l))[:, 0]
    return o, lse


def attn_masked_head_bwd(q, k, v, do, scale, mask):
    """Gradients of sum(dO * O) for ``attn_masked_head_fwd``: (dQ, dK, dV), the
    formulas of ``attn_head_bwd`` with P = 0 where the mask is False."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    s = np.where(mask, scale * (q @ k.T), -np.inf)
    p = np.zeros_like(s)
    live = mask.any(axis=1)
    m = np.max(s[live], axis=1, keepdims=True)
    e = np.exp(s[live] - m)
    p[live] = e / np.sum(e, axis=1, keepdims=True)
    dv = p.T @ do
    dp = do @ v.T
    d_i = np.sum(p * dp, axis=1, keepdims=True)
    ds = p * (dp - d_i)
    return scale * (ds @ k), scale * (ds.T @ q), dv
