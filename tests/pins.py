"""Pin checks for the attention oracle, written so that a mutated oracle can be fed in.

Each ``check_*`` takes the oracle's per-head forward (and, where needed, backward)
callable and raises AssertionError when the result contradicts what the pages or
the mathematics fix.  ``tests/test_oracle_pins.py`` runs them against the real
oracle (all must pass) and against deliberately broken copies (each must fail).
"""

from __future__ import annotations

import itertools
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = [float(x) for x in vals]
    return out


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


# ---------------------------------------------------------------- forward pins
def check_q_zero_uniform(fwd, n=37, d=5, seed=11):
    """Q = 0 makes every visible score equal, so P is uniform over the visible keys:
    non-causal O = mean(V), LSE = ln N; causal O_i = mean(V_0..i), LSE_i = ln(i+1)."""
    r = _rng(seed)
    q = np.zeros((n, d))
    k = r.standard_normal((n, d))
    v = r.standard_normal((n, d))
    o, lse = fwd(q, k, v, 0.37, False)[:2]
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(0), o.shape), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.full(n, np.log(n)), rtol=0, atol=1e-12)
    o, lse = fwd(q, k, v, 0.37, True)[:2]
    prefix_mean = np.cumsum(v, axis=0) / np.arange(1, n + 1)[:, None]
    np.testing.assert_allclose(o, prefix_mean, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.log(np.arange(1, n + 1)), rtol=0, atol=1e-12)


def check_causal_row0_and_ones(fwd, n=19, d=7, seed=12):
    """Causal row 0 sees only key 0: O_0 = V_0 and LSE_0 = scale * q_0.k_0.
    V = all ones gives O = 1 everywhere (rows of P sum to one)."""
    r = _rng(seed)
    q, k, v = (r.standard_normal((n, d)) for _ in range(3))
    scale = 0.29
    o, lse = fwd(q, k, v, scale, True)[:2]
    np.testing.assert_allclose(o[0], v[0], rtol=0, atol=1e-13)
    assert abs(lse[0] - scale * float(q[0] @ k[0])) < 1e-12
    for causal in (False, True):
        o1, _ = fwd(q, k, np.ones((n, d)), scale, causal)[:2]
        np.testing.assert_allclose(o1, np.ones((n, d)), rtol=0, atol=1e-13)


def check_dominant_key(fwd, n=23, d=6, seed=13):
    """One key whose score exceeds the others by a wide margin takes all the weight:
    O ~= V_j and LSE ~= S_ij.  The scores are >= 100 and must not overflow
    (e^89 already exceeds float32).  The scores here are ~800, past float64's own
    overflow point (e^709), so only max subtraction keeps the result finite."""
    r = _rng(seed)
    k = r.standard_normal((n, d)) * 0.01
    j = 9
    k[j] = 0.0
    k[j, 0] = 1.0
    q = np.zeros((n, d))
    q[:, 0] = 800.0
    v = r.standard_normal((n, d))
    o, lse = fwd(q, k, v, 1.0, False)[:2]
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    np.testing.assert_allclose(o, np.broadcast_to(v[j], o.shape), rtol=0, atol=1e-9)
    np.testing.assert_allclose(lse, np.full(n, 800.0), rtol=0, atol=1e-6)


def check_probabilities(fwd_sp, n=29, d=8, seed=14):
    """Rows of P sum to one, 0 <= P <= 1, and causal P_ij = 0 for j > i."""
    r = _rng(seed)
    q, k, v = (r.standard_normal((n, d)) for _ in range(3))
    for causal in (False, True):
        _, _, s, p = fwd_sp(q, k, v, 0.5, causal)
        np.testing.assert_allclose(p.sum(1), np.ones(n), rtol=0, atol=1e-13)
        assert np.all(p >= 0) and np.all(p <= 1)
        if causal:
            assert np.all(p[np.triu_indices(n, 1)] == 0)
            assert np.all(np.isneginf(s[np.triu_indices(n, 1)]))


def check_against_scipy(fwd, n=41, d=9, seed=15):
    """Library pin: P from scipy.special.softmax, LSE from scipy.special.logsumexp of
    the scaled scores (a different implementation of the same definition)."""
    from scipy.special import logsumexp, softmax
    r = _rng(seed)
    q, k, v = (r.standard_normal((n, d)) for _ in range(3))
    scale = d ** -0.5
    for causal in (False, True):
        s = scale * np.einsum("id,jd->ij", q, k)
        if causal:
            s[np.triu_indices(n, 1)] = -np.inf
        o, lse = fwd(q, k, v, scale, causal)[:2]
        np.testing.assert_allclose(lse, logsumexp(s, axis=1), rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(o, softmax(s, axis=1) @ v, rtol=1e-12, atol=1e-13)


def check_permutations(fwd, n=31, d=6, seed=16):
    """Non-causal attention is invariant under a joint permutation of the K and V rows
    and equivariant under a permutation of the Q rows."""
    r = _rng(seed)
    q, k, v = (r.standard_normal((n, d)) for _ in range(3))
    o, lse = fwd(q, k, v, 0.4, False)[:2]
    pk = r.permutation(n)
    o2, lse2 = fwd(q, k[pk], v[pk], 0.4, False)[:2]
    np.testing.assert_allclose(o2, o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, rtol=1e-13, atol=1e-13)
    pq = r.permutation(n)
    o3, lse3 = fwd(q[pq], k, v, 0.4, False)[:2]
    np.testing.assert_allclose(o3, o[pq], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse3, lse[pq], rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- backward pins
def _loss(fwd, q, k, v, do, scale, causal):
    o = fwd(q, k, v, scale, causal)[0]
    return float(np.sum(do * o))


def check_finite_differences(fwd, bwd, n=7, d=3, seed=17, h=1e-6, rtol=1e-7):
    """Backward against central finite differences of L = sum(dO * O) in float64."""
    r = _rng(seed)
    q, k, v, do = (r.standard_normal((n, d)) for _ in range(4))
    scale = 0.71
    for causal in (False, True):
        dq, dk, dv = bwd(q, k, v, do, scale, causal)[:3]
        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            num = np.empty_like(x)
            for idx in itertools.product(range(n), range(d)):
                xp = x.copy()
                xm = x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p = {"q": q, "k": k, "v": v}
                args_m = {"q": q, "k": k, "v": v}
                args_p[name] = xp
                args_m[name] = xm
                num[idx] = (_loss(fwd, args_p["q"], args_p["k"], args_p["v"], do, scale, causal)
                            - _loss(fwd, args_m["q"], args_m["k"], args_m["v"], do, scale, causal)) / (2 * h)
            err = np.linalg.norm(num - g) / max(np.linalg.norm(g), 1e-300)
            assert err <= rtol, f"d{name} causal={causal}: rel err {err:.3e}"


def check_backward_invariants(fwd, bwd, n=33, d=8, seed=18):
    """sum_j dS_ij = 0 for every row, hence sum_j dK_j = 0 per head;
    D_i = dO_i . O_i; sum_j dV_j = sum_i dO_i (rows of P sum to one)."""
    r = _rng(seed)
    q, k, v, do = (r.standard_normal((n, d)) for _ in range(4))
    for causal in (False, True):
        o = fwd(q, k, v, 0.3, causal)[0]
        dq, dk, dv, dvec = bwd(q, k, v, do, 0.3, causal)
        np.testing.assert_allclose(dk.sum(0), np.zeros(d), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dvec, np.sum(do * o, axis=1), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dv.sum(0), do.sum(0), rtol=1e-12, atol=1e-12)


def check_backward_closed_form_q_zero(fwd, bwd, n=12, d=4, seed=19):
    """Non-causal, Q = 0: P = 1/N everywhere, so dV_j = mean_i... = (1/N) sum_i dO_i
    for every key j, and dQ_i = scale * sum_j P_ij (dP_ij - D_i) K_j with
    dP = dO V^T, D_i = mean_j dP_ij."""
    r = _rng(seed)
    q = np.zeros((n, d))
    k, v, do = (r.standard_normal((n, d)) for _ in range(3))
    dq, dk, dv, _ = bwd(q, k, v, do, 0.8, False)
    np.testing.assert_allclose(dv, np.broadcast_to(do.sum(0) / n, dv.shape), rtol=0, atol=1e-12)
    dp = do @ v.T
    expect_dq = 0.8 * ((dp - dp.mean(1, keepdims=True)) / n) @ k
    np.testing.assert_allclose(dq, expect_dq, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, np.zeros_like(dk), rtol=0, atol=1e-12)
