"""Pins for the fp64 oracle: printed worked examples, closed forms, invariants,
library routines, brute force and finite differences.  CPU only.

A second group plants mistakes in copies of the oracle (on the CPU) and checks that
at least one pin catches each: a dropped scale, a reversed causal mask, a transposed
product, a wrong log base, a sign error in dS and a missing max subtraction.
"""

import itertools

import numpy as np
import pytest

import oracle
from oracle import attention as A
from tests import pins


def _fwd(q, k, v, scale, causal):
    return A.attn_head_fwd(q, k, v, scale, causal)


def _fwd_sp(q, k, v, scale, causal):
    return A.attn_head_fwd(q, k, v, scale, causal, return_sp=True)


def _bwd(q, k, v, do, scale, causal):
    return A.attn_head_bwd(q, k, v, do, scale, causal)


# ------------------------------------------------------------ printed examples
def test_softmax_worked_example():
    g = pins.read_golden("softmax_2_1_3.txt")
    row = np.array(g["row"])
    p = oracle.softmax_two_pass(row)
    np.testing.assert_array_equal(np.round(p, int(g["softmax_decimals"][0])), g["softmax"])
    np.testing.assert_array_equal(np.round(np.exp(row), int(g["exp_decimals"][0])), g["exp"])
    assert round(float(np.exp(row).sum()), int(g["sum_decimals"][0])) == g["sum"][0]
    assert abs(p.sum() - 1.0) < 1e-15


@pytest.mark.parametrize("form", ["updated_max", "block_local"])
def test_two_block_ell_example(form):
    g = pins.read_golden("two_block_ell.txt")
    row = np.array(g["row"])
    (m1, l1), (m2, l2) = oracle.online_softmax_stats(row, [int(g["split"][0])], form=form)
    dec = int(g["decimals"][0])
    assert m1 == g["m1"][0] and m2 == g["m2"][0]
    assert round(l1, dec) == g["l1"][0]
    assert round(l2, dec) == g["l2"][0]
    direct = float(np.sum(np.exp(row - row.max())))
    assert abs(l2 - direct) < 1e-15


def test_rescale_factor_example():
    g = pins.read_golden("rescale_after_5.txt")
    first = np.array(g["first_block"])
    second = np.array(g["second_block"])
    row = np.concatenate([first, second])
    (m1, l1), (m2, l2) = oracle.online_softmax_stats(row, [len(first)])
    factor = np.exp(m1 - m2)
    assert round(float(factor), int(g["decimals"][0])) == g["factor"][0]
    assert abs(l2 - (factor * l1 + np.sum(np.exp(second - m2)))) < 1e-15
    # the running output is patched by the same factor
    v = np.arange(len(row) * 2, dtype=np.float64).reshape(len(row), 2)
    o, m, l = oracle.online_attention_row(row, v, [len(first)])
    e1 = np.exp(first - m1)
    acc1 = e1 @ v[: len(first)]
    acc2 = factor * acc1 + np.exp(second - m2) @ v[len(first):]
    np.testing.assert_allclose(o, acc2 / l2, rtol=1e-15, atol=0)


# ------------------------------------------------------------ brute force
@pytest.mark.parametrize("n", [1, 2, 3, 5, 8, 12])
def test_online_equals_two_pass_every_split(n):
    """Every one of the 2^(n-1) ways to cut a row into blocks gives the two-pass
    normaliser and output, in float64, to 1e-12 relative."""
    r = np.random.Generator(np.random.PCG64(100 + n))
    row = r.standard_normal(n) * 4
    v = r.standard_normal((n, 3))
    m_ref = row.max()
    l_ref = np.exp(row - m_ref).sum()
    o_ref = oracle.softmax_two_pass(row) @ v
    for mask in range(1 << max(n - 1, 0)):
        splits = [i + 1 for i in range(n - 1) if mask >> i & 1]
        for form in ("updated_max", "block_local"):
            m, l = oracle.online_softmax_stats(row, splits, form=form)[-1]
            assert m == m_ref
            assert abs(l - l_ref) <= 1e-12 * l_ref
        o, m, l = oracle.online_attention_row(row, v, splits)
        np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("bq,bk", [(1, 1), (4, 3), (16, 16), (5, 64)])
def test_tiled_schedule_equals_definition(causal, bq, bk):
    r = np.random.Generator(np.random.PCG64(7))
    n, d = 45, 6
    q, k, v = (r.standard_normal((n, d)) * 2 for _ in range(3))
    o, lse = A.attn_head_fwd(q, k, v, 0.5, causal)
    o2, lse2 = A.attn_fwd_tiled_ref(q, k, v, 0.5, causal, bq, bk)
    np.testing.assert_allclose(o2, o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, rtol=1e-13, atol=1e-13)


def test_row_blocking_is_exact():
    r = np.random.Generator(np.random.PCG64(8))
    n, d = 70, 5
    q, k, v, do = (r.standard_normal((n, d)) for _ in range(4))
    for causal in (False, True):
        o, lse = A.attn_head_fwd(q, k, v, 0.6, causal)
        o2, lse2 = A.attn_head_fwd(q, k, v, 0.6, causal, row_block=16)
        np.testing.assert_allclose(o2, o, rtol=1e-14, atol=1e-15)
        np.testing.assert_allclose(lse2, lse, rtol=1e-14, atol=1e-15)
        g = A.attn_head_bwd(q, k, v, do, 0.6, causal)
        g2 = A.attn_head_bwd(q, k, v, do, 0.6, causal, row_block=9)
        for a, b in zip(g, g2):
            np.testing.assert_allclose(b, a, rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------ closed forms etc.
def test_q_zero_uniform():
    pins.check_q_zero_uniform(_fwd)


def test_causal_row0_and_ones():
    pins.check_causal_row0_and_ones(_fwd)


def test_dominant_key_and_no_overflow():
    pins.check_dominant_key(_fwd)


def test_probability_matrix():
    pins.check_probabilities(_fwd_sp)


def test_against_scipy():
    pins.check_against_scipy(_fwd)


def test_permutations():
    pins.check_permutations(_fwd)


def test_backward_finite_differences():
    pins.check_finite_differences(_fwd, _bwd)


def test_backward_invariants():
    pins.check_backward_invariants(_fwd, _bwd)


def test_backward_q_zero_closed_form():
    pins.check_backward_closed_form_q_zero(_fwd, _bwd)


def test_batched_wrappers_match_heads():
    r = np.random.Generator(np.random.PCG64(9))
    B, H, N, d = 2, 3, 10, 4
    q, k, v, do = (r.standard_normal((B, H, N, d)) for _ in range(4))
    o, lse = oracle.attn_fwd_ref(q, k, v, 0.5, True)
    dq, dk, dv, dvec = oracle.attn_bwd_ref(q, k, v, do, 0.5, True)
    for b, h in itertools.product(range(B), range(H)):
        o1, l1 = A.attn_head_fwd(q[b, h], k[b, h], v[b, h], 0.5, True)
        np.testing.assert_array_equal(o[b, h], o1)
        np.testing.assert_array_equal(lse[b, h], l1)
        g = A.attn_head_bwd(q[b, h], k[b, h], v[b, h], do[b, h], 0.5, True)
        for x, y in zip((dq, dk, dv, dvec), g):
            np.testing.assert_array_equal(x[b, h], y)
    o_s, _ = oracle.attn_fwd_ref(q, k, v, 0.5, True, heads=[(1, 2)])
    assert np.isnan(o_s[0, 0]).all() and np.array_equal(o_s[1, 2], o[1, 2])


# ------------------------------------------------------------ planted mistakes
def _mut_fwd(kind):
    def fwd(q, k, v, scale, causal, return_sp=False):
        q = np.asarray(q, float)
        k = np.asarray(k, float)
        v = np.asarray(v, float)
        n = q.shape[0]
        sc = 1.0 if kind == "no_scale" else scale
        s = sc * (q @ k.T) if kind != "transposed" else sc * (k @ q.T)
        if causal:
            tri = np.triu_indices(n, 1) if kind != "mask_reversed" else np.tril_indices(n, -1)
            s[tri] = -np.inf
        m = s.max(1, keepdims=True) if kind != "no_max" else np.zeros((n, 1))
        with np.errstate(over="ignore", invalid="ignore"):   # the no_max mutant overflows on purpose
            e = np.exp(s - m)
            l = e.sum(1, keepdims=True)
            p = e / l
        o = p @ v
        lse = (m + (np.log2(l) if kind == "log2" else np.log(l)))[:, 0]
        return (o, lse, s, p) if return_sp else (o, lse)
    return fwd


def _mut_bwd(kind):
    def bwd(q, k, v, do, scale, causal):
        dq, dk, dv, dvec = A.attn_head_bwd(q, k, v, do, scale, causal)
        if kind == "ds_sign":
            # recompute with (D - dP) instead of (dP - D)
            s = scale * (q @ k.T)
            if causal:
                s[np.triu_indices(q.shape[0], 1)] = -np.inf
            p = np.exp(s - s.max(1, keepdims=True))
            p /= p.sum(1, keepdims=True)
            dp = do @ v.T
            ds = p * (dvec[:, None] - dp)
            dq = scale * ds @ k
            dk = scale * ds.T @ q
        elif kind == "dv_transposed":
            dv = dv[::-1].copy()
        elif kind == "dk_no_scale":
            dk = dk / scale
        return dq, dk, dv, dvec
    return bwd


def _fails(fn, *args):
    try:
        fn(*args)
    except AssertionError:
        return True
    return False


FWD_PINS = [pins.check_q_zero_uniform, pins.check_causal_row0_and_ones, pins.check_dominant_key,
            pins.check_against_scipy, pins.check_permutations]


@pytest.mark.parametrize("kind", ["no_scale", "mask_reversed", "transposed", "log2", "no_max"])
def test_planted_forward_mistake_is_caught(kind):
    fwd = _mut_fwd(kind)
    caught = [p.__name__ for p in FWD_PINS if _fails(p, fwd)]
    caught += ["probabilities"] if _fails(pins.check_probabilities, lambda *a: fwd(*a, return_sp=True)) else []
    assert caught, f"no pin caught the planted mistake {kind!r}"


@pytest.mark.parametrize("kind", ["ds_sign", "dv_transposed", "dk_no_scale"])
def test_planted_backward_mistake_is_caught(kind):
    bwd = _mut_bwd(kind)
    caught = _fails(pins.check_finite_differences, _fwd, bwd) or _fails(pins.check_backward_invariants, _fwd, bwd)
    assert caught, f"no pin caught the planted mistake {kind!r}"


def test_real_oracle_passes_every_mutation_harness():
    # the harness itself must not fail the unmutated oracle
    for p in FWD_PINS:
        p(_fwd)
    pins.check_probabilities(_fwd_sp)


@pytest.mark.parametrize("causal", [False, True])
def test_row_subset_matches_whole_head(causal):
    """attn_rows_ref on scattered rows equals the whole-head forward and the dQ, D of
    the whole-head backward on those rows."""
    r = np.random.Generator(np.random.PCG64(21))
    n, d = 57, 6
    q, k, v, do = (r.standard_normal((n, d)) for _ in range(4))
    o, lse = A.attn_head_fwd(q, k, v, 0.45, causal)
    dq, dk, dv, dvec = A.attn_head_bwd(q, k, v, do, 0.45, causal)
    rows = np.array([0, 3, 17, 31, 56])
    o_r, lse_r, dq_r, d_r = oracle.attn_rows_ref(q[rows], rows, k, v, 0.45, causal, do[rows])
    np.testing.assert_allclose(o_r, o[rows], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse_r, lse[rows], rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(dq_r, dq[rows], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(d_r, dvec[rows], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_row_ranges_partition_the_head(causal):
    """Forward rows and backward contributions over a partition of the query rows
    (ragged parts, an empty part, blocks that straddle the cuts) add up to the
    whole head: O and LSE rows, dQ and D rows match, and the parts' dK and dV
    contributions sum to the whole head's dK and dV.  A range whose causal mask
    were taken from the range's own first row instead of its place in the
    sequence would fail the causal case."""
    r = np.random.Generator(np.random.PCG64(22))
    n, d = 70, 5
    q, k, v, do = (r.standard_normal((n, d)) for _ in range(4))
    o, lse = A.attn_head_fwd(q, k, v, 0.6, causal)
    dq, dk, dv, dvec = A.attn_head_bwd(q, k, v, do, 0.6, causal)
    dk_sum, dv_sum = np.zeros_like(dk), np.zeros_like(dv)
    for lo, hi in [(0, 13), (13, 13), (13, 50), (50, 70)]:
        o_p, lse_p = A.attn_head_fwd(q, k, v, 0.6, causal, row_block=8, row_range=(lo, hi))
        assert o_p.shape == (hi - lo, d) and lse_p.shape == (hi - lo,)
        np.testing.assert_allclose(o_p, o[lo:hi], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(lse_p, lse[lo:hi], rtol=1e-14, atol=1e-14)
        dq_p, dk_p, dv_p, d_p = A.attn_head_bwd(q, k, v, do, 0.6, causal, row_block=8, row_range=(lo, hi))
        np.testing.assert_allclose(dq_p, dq[lo:hi], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(d_p, dvec[lo:hi], rtol=1e-12, atol=1e-13)
        dk_sum += dk_p
        dv_sum += dv_p
    np.testing.assert_allclose(dk_sum, dk, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dv_sum, dv, rtol=1e-12, atol=1e-13)
    with pytest.raises(ValueError):
        A.attn_head_fwd(q, k, v, 0.6, causal, row_range=(5, 71))
