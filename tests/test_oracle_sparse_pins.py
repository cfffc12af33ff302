"""Pins for the oracle's masked attention and butterfly block pattern.  CPU only.

  * the pattern on four and eight blocks written out by hand from its definition
    (indices that differ in one bit, plus the diagonal), and its symmetry;
  * an all-true mask reduces to the pinned dense oracle, the lower triangle to the
    pinned causal oracle, and a sequence inside one block to dense attention;
  * brute force with math.exp under a random mask, and central finite differences
    for the masked gradient;
  * planted mistakes (a pattern without the diagonal, one that also links indices two
    bits apart, a gradient that ignores the mask) are each caught.
"""

import math

import numpy as np
import pytest

from oracle import attention as A


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


FOUR = [[1, 1, 1, 0],
        [1, 1, 0, 1],
        [1, 0, 1, 1],
        [0, 1, 1, 1]]

EIGHT_ROW5 = [0, 1, 0, 0, 1, 1, 0, 1]   # 5 = 101b: sees 4 (100), 7 (111), 1 (001) and itself


def check_pattern(visible):
    for p in range(4):
        for q in range(4):
            assert int(bool(visible(p, q))) == FOUR[p][q], (p, q)
    assert [int(bool(visible(5, q))) for q in range(8)] == EIGHT_ROW5
    for p in range(16):
        for q in range(16):
            assert bool(visible(p, q)) == bool(visible(q, p))


def test_butterfly_pattern_by_hand():
    check_pattern(A.butterfly_pairs_visible)


def test_butterfly_mask_matches_pattern():
    blk = A.BUTTERFLY_BLOCK
    m = A.butterfly_mask(4 * blk, 4 * blk, False)
    for p in range(4):
        for q in range(4):
            sub = m[p * blk:(p + 1) * blk, q * blk:(q + 1) * blk]
            assert sub.all() if FOUR[p][q] else not sub.any()
    mc = A.butterfly_mask(4 * blk, 4 * blk, True)
    assert np.array_equal(mc, m & np.tri(4 * blk, dtype=bool))


@pytest.mark.parametrize("causal", [False, True])
def test_masked_reduces_to_dense_and_causal(causal):
    r = _rng(1)
    n, d = 40, 8
    q, k, v = r.standard_normal((n, d)), r.standard_normal((n, d)), r.standard_normal((n, d))
    mask = np.tri(n, dtype=bool) if causal else np.ones((n, n), dtype=bool)
    o, lse = A.attn_masked_head_fwd(q, k, v, 0.3, mask)
    o_ref, lse_ref = A.attn_head_fwd(q, k, v, 0.3, causal)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-13)
    g = A.attn_masked_head_bwd(q, k, v, r.standard_normal((n, d)), 0.3, mask)
    assert all(np.all(np.isfinite(x)) for x in g)


def test_butterfly_inside_one_block_is_dense():
    r = _rng(2)
    n = A.BUTTERFLY_BLOCK
    q, k, v = r.standard_normal((n, 8)), r.standard_normal((n, 8)), r.standard_normal((n, 8))
    o, lse = A.attn_masked_head_fwd(q, k, v, 0.2, A.butterfly_mask(n, n, False))
    o_ref, lse_ref = A.attn_head_fwd(q, k, v, 0.2, False)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-13)


def check_masked_brute_force(fwd):
    r = _rng(3)
    nq, nk, d = 4, 6, 3
    q, k, v = r.standard_normal((nq, d)), r.standard_normal((nk, d)), r.standard_normal((nk, d))
    mask = r.random((nq, nk)) < 0.5
    mask[2] = False                         # one row sees nothing
    mask[0, 0] = True
    o, lse = fwd(q, k, v, 0.7, mask)
    for i in range(nq):
        vis = [j for j in range(nk) if mask[i, j]]
        if not vis:
            assert np.all(o[i] == 0) and lse[i] == -np.inf
            continue
        s = {j: 0.7 * sum(q[i, c] * k[j, c] for c in range(d)) for j in vis}
        z = sum(math.exp(t) for t in s.values())
        for c in range(d):
            assert abs(o[i, c] - sum(math.exp(s[j]) / z * v[j, c] for j in vis)) < 1e-13
        assert abs(lse[i] - math.log(z)) < 1e-13


def test_masked_brute_force():
    check_masked_brute_force(A.attn_masked_head_fwd)


def check_masked_finite_differences(bwd):
    r = _rng(4)
    n, d = 7, 3
    q, k, v, do = (r.standard_normal((n, d)) for _ in range(4))
    mask = r.random((n, n)) < 0.6
    np.fill_diagonal(mask, True)
    dq, dk, dv = bwd(q, k, v, do, 0.9, mask)

    def loss(qq, kk, vv):
        return float(np.sum(A.attn_masked_head_fwd(qq, kk, vv, 0.9, mask)[0] * do))

    eps = 1e-6
    for arr, grad, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        for idx in [(0, 0), (3, 2), (6, 1)]:
            p, m = arr.copy(), arr.copy()
            p[idx] += eps
            m[idx] -= eps
            args_p = [q, k, v]
            args_m = [q, k, v]
            args_p[which], args_m[which] = p, m
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - grad[idx]) < 1e-7


def test_masked_finite_differences():
    check_masked_finite_differences(A.attn_masked_head_bwd)


# ------------------------------------------------------------ planted mistakes
def _no_diagonal(p, q):
    x = p ^ q
    return x != 0 and (x & (x - 1)) == 0


def _two_bits_too(p, q):
    return bin(p ^ q).count("1") <= 2


def _bwd_ignores_mask(q, k, v, do, scale, mask):
    dq, dk, dv, _ = A.attn_head_bwd(q, k, v, do, scale, False)
    return dq, dk, dv


def _fails(fn, *args):
    try:
        fn(*args)
    except AssertionError:
        return True
    return False


def test_planted_pattern_mistakes_are_caught():
    assert _fails(check_pattern, _no_diagonal)
    assert _fails(check_pattern, _two_bits_too)


def test_planted_unmasked_gradient_is_caught():
    assert _fails(check_masked_finite_differences, _bwd_ignores_mask)
