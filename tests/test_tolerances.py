"""The O tolerance of the GPU parity tests (tests/gpu_util.py), checked on the CPU:
the P-rounding term bounds what rounding P to 16 bits before P.V does to O, and the
check catches a planted error."""

import numpy as np
import pytest

import oracle
from exact_tiled_attention_27_gb300.inputs import bits_to_f64, f64_to_bits, make_case
from tests import gpu_util as G


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("mult", [1.0, 3.0])
def test_p_rounding_term_bounds_16bit_p(dtype, mult):
    """O computed with P rounded to the 16-bit type and divided by the sum of the
    rounded P stays within 2u/(1-u) ((P|V|) + |O|) of the exact O, element by element."""
    case = make_case(1, 2, 384, 64, dtype, True, workload_index=96, mult=mult)
    for h in range(2):
        q, k, v = (case.f64(n)[0, h] for n in ("q", "k", "v"))
        o, lse, s, p = oracle.attn_head_fwd(q, k, v, case.scale, True, return_sp=True)
        pv_abs, _ = oracle.attn_head_fwd(q, k, np.abs(v), case.scale, True)
        # any common factor of a row cancels: round the row scaled by its largest entry
        e = p / p.max(axis=1, keepdims=True)
        e16 = bits_to_f64(f64_to_bits(e, dtype), dtype)   # via float32: one more rounding of 2^-24
        o16 = (e16 @ v) / e16.sum(axis=1, keepdims=True)
        u = G.unit_roundoff(dtype) + 2.0 ** -23
        bound = 2 * u / (1 - u) * (pv_abs + np.abs(o))
        assert np.all(np.abs(o16 - o) <= bound + 1e-12)
        # and the term is not vacuous: it is within a small factor of the largest effect
        assert np.max(np.abs(o16 - o)) > 0


def test_check_forward_catches_a_planted_error():
    case = make_case(1, 1, 200, 64, "bf16", False, workload_index=97)
    q, k, v = (case.f64(n)[0, 0] for n in ("q", "k", "v"))
    o, lse = oracle.attn_head_fwd(q, k, v, case.scale, False)
    pv_abs, _ = oracle.attn_head_fwd(q, k, np.abs(v), case.scale, False)
    o16 = bits_to_f64(f64_to_bits(o, "bf16"), "bf16")
    G.check_forward(o16, lse, o, lse, "rounded exact O", "bf16", pv_abs)
    bad = o16.copy()
    bad[17, 5] += 0.05
    with pytest.raises(AssertionError):
        G.check_forward(bad, lse, o, lse, "planted 0.05", "bf16", pv_abs)
    with pytest.raises(AssertionError):
        G.check_forward(o16, lse + 2e-3, o, lse, "planted lse", "bf16", pv_abs)


def test_half_ulp_matches_the_grids():
    x = np.array([1.0, 1.5, 2.0, 3.99, 8.0, 15.0, 0.3])
    np.testing.assert_array_equal(G.half_ulp(x, "bf16"), [2.0 ** -8, 2.0 ** -8, 2.0 ** -7, 2.0 ** -7, 2.0 ** -5,
                                                          2.0 ** -5, 2.0 ** -10])
    np.testing.assert_array_equal(G.half_ulp(x, "fp16"), [2.0 ** -11, 2.0 ** -11, 2.0 ** -10, 2.0 ** -10,
                                                          2.0 ** -8, 2.0 ** -8, 2.0 ** -13])
    # rounding to the grid moves a value by at most half an ulp
    r = np.random.Generator(np.random.PCG64(5)).standard_normal(10000) * 4
    for dt in ("bf16", "fp16"):
        rr = bits_to_f64(f64_to_bits(r, dt), dt)
        assert np.all(np.abs(rr - r) <= G.half_ulp(r, dt) * (1 + 2.0 ** -20))
