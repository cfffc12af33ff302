"""The pooled oracle jobs used by the full-size GPU parity tests reproduce the
whole-head oracle: forward rows concatenated over ranges of query rows, and the dK, dV
contributions of the ranges summed.  CPU only (spawned worker processes)."""

import numpy as np
import pytest

import oracle
from exact_tiled_attention_27_gb300.inputs import make_case
from tests import oracle_jobs


def test_row_ranges_cover_rows_once():
    for n, parts in [(1, 1), (5, 8), (300, 3), (65536, 8), (1000, 7)]:
        rs = oracle_jobs.row_ranges(n, parts)
        assert rs[0][0] == 0 and rs[-1][1] == n and len(rs) <= parts
        assert all(a[1] == b[0] for a, b in zip(rs, rs[1:]))
        assert all(hi > lo for lo, hi in rs)


@pytest.mark.parametrize("causal", [False, True])
def test_pooled_head_equals_whole_head(causal):
    case = make_case(2, 2, 300, 64, "bf16", causal, workload_index=95, mult=3.0)
    jobs = oracle_jobs.HeadJobs(case, 1, 0, parts=3, row_block=64, with_bwd=True)
    o, lse, pv_abs = jobs.forward()
    dq, dk, dv = jobs.backward()
    f = lambda n: case.f64(n)[1, 0]  # noqa: E731
    o_ref, lse_ref = oracle.attn_head_fwd(f("q"), f("k"), f("v"), case.scale, causal)
    dq_ref, dk_ref, dv_ref, _ = oracle.attn_head_bwd(f("q"), f("k"), f("v"), f("do"), case.scale, causal)
    np.testing.assert_allclose(o, o_ref, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-13, atol=1e-13)
    pv_ref, _ = oracle.attn_head_fwd(f("q"), f("k"), np.abs(f("v")), case.scale, causal)
    np.testing.assert_allclose(pv_abs, pv_ref, rtol=1e-13, atol=1e-13)
    assert np.all(pv_abs >= np.abs(o) - 1e-12)   # |P V| <= P |V|
    for a, b in [(dq, dq_ref), (dk, dk_ref), (dv, dv_ref)]:
        np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-12)
