"""Pins for the oracle's cross-length, grouped-head and split-key routines.  CPU only.

What pins them (none of these re-types the formula under test):
  * the printed two-block normaliser example ([1, 2 | 0, 3] -> m = 3, l ~ 1.553) read as
    a merge of two key ranges;
  * brute force with math.exp on tiny inputs;
  * reductions to the square-attention oracle, which has pins of its own: Nq = Nk, the
    last Nq rows of a square causal problem, a single query row, key/value heads
    repeated per group;
  * central finite differences for the grouped-head gradient.
A second group plants mistakes (top-left causal alignment, a merge that drops the
weights, a strided head map, a group gradient that is not summed) in copies of the
oracle and checks that a pin catches each.
"""

import math

import numpy as np
import pytest

import oracle
from oracle import attention as A
from tests import pins


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _qkv(r, nq, nk, d, scale_up=1.0):
    return (scale_up * r.standard_normal((nq, d)), scale_up * r.standard_normal((nk, d)),
            r.standard_normal((nk, d)))


# ------------------------------------------------------------ merge of key ranges
def check_merge_golden(merge):
    g = pins.read_golden("two_block_ell.txt")
    row = np.array(g["row"])
    cut = int(g["split"][0])
    parts = [row[:cut], row[cut:]]
    eye = np.eye(len(row))
    o_parts, lse_parts = [], []
    for lo, x in ((0, parts[0]), (cut, parts[1])):
        # attention of one query with scores x over keys lo.. whose values are unit rows
        lse = math.log(sum(math.exp(t) for t in x))
        p = np.array([math.exp(t - lse) for t in x])
        o_parts.append((p @ eye[lo:lo + len(x)])[None, :])
        lse_parts.append(np.array([lse]))
    o, lse = merge(o_parts, lse_parts)
    dec = int(g["decimals"][0])
    m2, l2 = g["m2"][0], g["l2"][0]
    assert round(math.exp(lse[0] - m2), dec) == l2           # the merged normaliser is l2 at m = 3
    direct = np.array([math.exp(t) for t in row])
    np.testing.assert_allclose(o[0], direct / direct.sum(), rtol=0, atol=1e-15)


def check_merge_random(merge):
    r = _rng(11)
    q, k, v = _qkv(r, 7, 50, 16)
    cuts = [0, 9, 10, 33, 50]
    o_parts, lse_parts = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        o_s, l_s = A.attn_cross_head_fwd(q, k[a:b], v[a:b], 0.3, False)
        o_parts.append(o_s)
        lse_parts.append(l_s)
    o, lse = merge(o_parts, lse_parts)
    o_ref, lse_ref = A.attn_head_fwd(q, k, v, 0.3, False) if q.shape[0] == k.shape[0] else \
        A.attn_cross_head_fwd(q, k, v, 0.3, False)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-13)


def check_merge_empty(merge):
    o1 = np.arange(6.0).reshape(2, 3)
    o, lse = merge([o1, np.ones((2, 3))], [np.array([0.5, -np.inf]), np.array([-np.inf, -np.inf])])
    np.testing.assert_array_equal(o[0], o1[0])
    assert lse[0] == 0.5
    assert np.all(o[1] == 0) and lse[1] == -np.inf


def test_merge_printed_example():
    check_merge_golden(A.merge_partials)


def test_merge_of_key_ranges_is_whole_attention():
    check_merge_random(A.merge_partials)


def test_merge_with_empty_parts():
    check_merge_empty(A.merge_partials)


# ------------------------------------------------------------ cross lengths
def check_single_query_sees_every_key(fwd):
    r = _rng(3)
    q, k, v = _qkv(r, 1, 37, 8)
    o_c, l_c = fwd(q, k, v, 0.4, True)
    # one query row, scores written out with math.exp
    s = [0.4 * float(q[0] @ k[j]) for j in range(37)]
    z = sum(math.exp(t) for t in s)
    o_bf = sum(math.exp(t) / z * v[j] for j, t in enumerate(s))
    np.testing.assert_allclose(o_c[0], o_bf, rtol=0, atol=1e-13)
    assert abs(l_c[0] - math.log(z)) < 1e-13


def check_tail_of_square(fwd):
    r = _rng(4)
    nk, nq = 40, 13
    qf, k, v = _qkv(r, nk, nk, 8)
    o_sq, l_sq = A.attn_head_fwd(qf, k, v, 0.35, True)
    o_c, l_c = fwd(qf[nk - nq:], k, v, 0.35, True)
    np.testing.assert_allclose(o_c, o_sq[nk - nq:], rtol=0, atol=1e-13)
    np.testing.assert_allclose(l_c, l_sq[nk - nq:], rtol=0, atol=1e-13)


def check_brute_force_tiny(fwd):
    r = _rng(5)
    nq, nk, d = 3, 5, 4
    q, k, v = _qkv(r, nq, nk, d)
    for causal in (False, True):
        o, lse = fwd(q, k, v, 0.5, causal)
        for i in range(nq):
            vis = [j for j in range(nk) if not causal or j <= i + (nk - nq)]
            s = {j: 0.5 * sum(q[i, c] * k[j, c] for c in range(d)) for j in vis}
            z = sum(math.exp(t) for t in s.values())
            for c in range(d):
                assert abs(o[i, c] - sum(math.exp(s[j]) / z * v[j, c] for j in vis)) < 1e-13
            assert abs(lse[i] - math.log(z)) < 1e-13


def check_fully_masked_rows(fwd):
    r = _rng(6)
    nq, nk = 9, 4
    q, k, v = _qkv(r, nq, nk, 8)
    o, lse = fwd(q, k, v, 0.5, True)
    dead = nq - nk                       # rows 0 .. dead-1 see no key
    assert np.all(o[:dead] == 0) and np.all(np.isneginf(lse[:dead]))
    o_sq, l_sq = A.attn_head_fwd(q[dead:], k, v, 0.5, True)   # the others: a square problem
    np.testing.assert_allclose(o[dead:], o_sq, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse[dead:], l_sq, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_cross_square_is_head_fwd(causal):
    r = _rng(7)
    q, k, v = _qkv(r, 30, 30, 16)
    o_c, l_c = A.attn_cross_head_fwd(q, k, v, 0.25, causal)
    o_h, l_h = A.attn_head_fwd(q, k, v, 0.25, causal)
    np.testing.assert_allclose(o_c, o_h, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l_c, l_h, rtol=0, atol=1e-13)


def test_cross_single_query_sees_every_key():
    check_single_query_sees_every_key(A.attn_cross_head_fwd)


def test_cross_bottom_right_is_tail_of_square():
    check_tail_of_square(A.attn_cross_head_fwd)


def test_cross_brute_force_tiny():
    check_brute_force_tiny(A.attn_cross_head_fwd)


def test_cross_fully_masked_rows():
    check_fully_masked_rows(A.attn_cross_head_fwd)


# ------------------------------------------------------------ grouped key/value heads
def check_head_map(kv_of):
    assert [kv_of(h, 8, 2) for h in range(8)] == [0, 0, 0, 0, 1, 1, 1, 1]
    assert [kv_of(h, 6, 6) for h in range(6)] == list(range(6))
    assert [kv_of(h, 4, 1) for h in range(4)] == [0, 0, 0, 0]


def check_gqa_fwd_is_repeated_mha(cross_ref):
    r = _rng(8)
    B, H, Hkv, N, d = 2, 6, 2, 20, 8
    q = r.standard_normal((B, H, N, d))
    k = r.standard_normal((B, Hkv, N, d))
    v = r.standard_normal((B, Hkv, N, d))
    rep = H // Hkv
    o_ref, l_ref = A.attn_fwd_ref(q, np.repeat(k, rep, axis=1), np.repeat(v, rep, axis=1), 0.3, True)
    o, lse = cross_ref(q, k, v, 0.3, True)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, l_ref, rtol=0, atol=1e-13)


def check_gqa_bwd_is_group_sum(gqa_bwd):
    r = _rng(9)
    B, H, Hkv, N, d = 1, 4, 2, 18, 8
    q = r.standard_normal((B, H, N, d))
    k = r.standard_normal((B, Hkv, N, d))
    v = r.standard_normal((B, Hkv, N, d))
    do = r.standard_normal((B, H, N, d))
    rep = H // Hkv
    dq_r, dk_r, dv_r, _ = A.attn_bwd_ref(q, np.repeat(k, rep, axis=1), np.repeat(v, rep, axis=1), do, 0.3, True)
    dq, dk, dv = gqa_bwd(q, k, v, do, 0.3, True)
    np.testing.assert_allclose(dq, dq_r, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, dk_r.reshape(B, Hkv, rep, N, d).sum(axis=2), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, dv_r.reshape(B, Hkv, rep, N, d).sum(axis=2), rtol=0, atol=1e-12)


def check_gqa_bwd_finite_differences(gqa_bwd):
    r = _rng(10)
    B, H, Hkv, N, d = 1, 4, 2, 6, 4
    q = r.standard_normal((B, H, N, d))
    k = r.standard_normal((B, Hkv, N, d))
    v = r.standard_normal((B, Hkv, N, d))
    do = r.standard_normal((B, H, N, d))

    def loss(kk, vv):
        o, _ = A.attn_cross_fwd_ref(q, kk, vv, 0.7, True)
        return float(np.sum(o * do))

    _, dk, dv = gqa_bwd(q, k, v, do, 0.7, True)
    eps = 1e-6
    for idx in [(0, 0, 1, 2), (0, 1, 5, 0), (0, 1, 3, 3)]:
        for arr, grad, is_k in ((k, dk, True), (v, dv, False)):
            p = arr.copy(); p[idx] += eps
            m = arr.copy(); m[idx] -= eps
            fd = (loss(p, v) - loss(m, v)) / (2 * eps) if is_k else (loss(k, p) - loss(k, m)) / (2 * eps)
            assert abs(fd - grad[idx]) < 1e-7


def test_head_map():
    check_head_map(A.kv_head_of)
    with pytest.raises(ValueError):
        A.kv_head_of(0, 6, 4)


def test_gqa_forward_is_repeated_mha():
    check_gqa_fwd_is_repeated_mha(A.attn_cross_fwd_ref)


def test_gqa_backward_is_group_sum():
    check_gqa_bwd_is_group_sum(A.attn_gqa_bwd_ref)


def test_gqa_backward_finite_differences():
    check_gqa_bwd_finite_differences(A.attn_gqa_bwd_ref)


def test_exports():
    for name in ("attn_cross_head_fwd", "attn_cross_fwd_ref", "attn_gqa_bwd_ref", "kv_head_of", "merge_partials"):
        assert getattr(oracle, name) is getattr(A, name)


# ------------------------------------------------------------ planted mistakes
def _top_left_cross(q, k, v, scale, causal):
    """attn_cross_head_fwd with the mask aligned top-left (j <= i) instead of bottom-right."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    s = scale * (q @ k.T)
    if causal:
        s = np.where(np.arange(k.shape[0])[None, :] > np.arange(q.shape[0])[:, None], -np.inf, s)
    live = np.isfinite(s).any(axis=1)
    o = np.zeros((q.shape[0], v.shape[1]))
    lse = np.full(q.shape[0], -np.inf)
    m = np.max(s[live], axis=1, keepdims=True)
    e = np.exp(s[live] - m)
    o[live] = (e / e.sum(axis=1, keepdims=True)) @ v
    lse[live] = (m + np.log(e.sum(axis=1, keepdims=True)))[:, 0]
    return o, lse


def _merge_unweighted(o_parts, lse_parts):
    """merge_partials that averages the parts instead of weighting them by e^{LSE_s}."""
    o = sum(np.asarray(x, dtype=np.float64) for x in o_parts) / len(o_parts)
    lse = np.log(np.sum(np.exp(np.stack(lse_parts)), axis=0))
    return o, lse


def _strided_head_map(h, H, Hkv):
    return h % Hkv


def _gqa_bwd_last_head_only(q, k, v, do, scale, causal):
    """attn_gqa_bwd_ref that overwrites instead of summing a key/value head's gradient."""
    B, H, N, _ = np.shape(q)
    Hkv = np.shape(k)[1]
    dq = np.empty(np.shape(q))
    dk = np.zeros(np.shape(k))
    dv = np.zeros(np.shape(v))
    for b in range(B):
        for h in range(H):
            hk = A.kv_head_of(h, H, Hkv)
            gq, gk, gv, _ = A.attn_head_bwd(q[b, h], k[b, hk], v[b, hk], do[b, h], scale, causal)
            dq[b, h], dk[b, hk], dv[b, hk] = gq, gk, gv
    return dq, dk, dv


def _fails(fn, *args):
    try:
        fn(*args)
    except AssertionError:
        return True
    return False


def test_planted_top_left_alignment_is_caught():
    assert _fails(check_single_query_sees_every_key, _top_left_cross)
    assert _fails(check_tail_of_square, _top_left_cross)


def test_planted_unweighted_merge_is_caught():
    assert _fails(check_merge_golden, _merge_unweighted)
    assert _fails(check_merge_random, _merge_unweighted)


def test_planted_strided_head_map_is_caught(monkeypatch):
    assert _fails(check_head_map, _strided_head_map)
    monkeypatch.setattr(A, "kv_head_of", _strided_head_map)
    assert _fails(check_gqa_fwd_is_repeated_mha, A.attn_cross_fwd_ref)


def test_planted_unsummed_group_gradient_is_caught():
    assert _fails(check_gqa_bwd_is_group_sum, _gqa_bwd_last_head_only)
    assert _fails(check_gqa_bwd_finite_differences, _gqa_bwd_last_head_only)
