"""Helpers shared by the GPU tests: upload seeded 16-bit bits, read results back as
float64, the comparison metrics, and the tolerances the parity tests enforce.

Tolerances (stated for the 16-bit inputs against the float64 oracle):
  O:            element by element |err| <= max(2e-2, r) + ulp(O_ref)/2, and
                ||err||_2 / ||ref||_2 <= 5e-3, where
                * ulp(x) is the spacing of the output's 16-bit grid at |x| (2^(e-7) for
                  bf16 and 2^(e-10) for fp16 when 2^e <= |x| < 2^(e+1)): O is returned in
                  the 16-bit type, and even the exact O rounded to nearest errs by up to
                  half of that spacing (0.031 in bf16 at |O| in [8, 16), which the inputs
                  scaled by 3 reach);
                * r is the most that rounding the probabilities to the 16-bit type before
                  the P.V product can move O (production kernels multiply 16-bit tiles):
                  with p_j -> p_j (1 + d_j), |d_j| <= u (unit roundoff, 2^-8 for bf16,
                  2^-11 for fp16) and O divided by the sum of the rounded p, O_i moves by
                  sum_j w_ij (d_j - dbar)(V_j - O_i) / (1 + dbar), at most
                  r_ic = 2u/(1-u) * sum_j P_ij |V_jc - O_ic| <= 2u/(1-u) ((P|V|)_ic + |O_ic|).
                  The right-hand side is what the tests use (P|V| is the oracle run with
                  |V| as the values).  For unit-scale inputs r stays below 2e-2, so the
                  stated bound holds as stated; with inputs scaled by 3 a row whose weight
                  is spread over keys with large |V| can reach r > 2e-2.
                When P|V| is not supplied, r is taken as 0 (the stated 2e-2).
  lse:          max |err| <= 1e-3
  dQ, dK, dV:   ||err||_2 / ||ref||_2 <= 1e-2

FP8 forward (against exact attention on the de-quantised inputs, so that only what the
kernel adds is measured): P is rounded to E4M3 before P.V.  Round-to-nearest with a
3-bit mantissa errs by at most 2^-4 of a value and, over a binade, by 2^-4/sqrt(3)
root-mean-square at most; with independent errors over many keys O's relative L2
error is at most that RMS (0.036), and in the worst case, every error aligned, one
row of O is off by 2^-4 max|V|.  Hence:
  O:            max |err| <= 2^-4 * max|V| + 1e-2  and  relL2 <= 4e-2
  lse:          max |err| <= 1e-3 (it uses the unrounded P)
"""

import numpy as np

O_MAXABS = 2e-2
O_RELL2 = 5e-3
LSE_ABS = 1e-3
GRAD_RELL2 = 1e-2
FP8_O_RELL2 = 4e-2
FP8_O_MAXABS_PER_V = 2.0 ** -4
FP8_O_MAXABS_EXTRA = 1e-2


def torch_dtype(dtype):
    import torch
    return torch.bfloat16 if dtype == "bf16" else torch.float16


def to_device(bits, dtype):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch_dtype(dtype)).cuda()


def to_f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def maxabs(a, b):
    return float(np.max(np.abs(a - b))) if a.size else 0.0


def rel_l2(a, ref):
    den = float(np.linalg.norm(ref))
    num = float(np.linalg.norm(a - ref))
    return num / den if den > 0 else num


def half_ulp(x, dtype):
    """Half the spacing of the 16-bit grid (bf16: 8 significant bits, fp16: 11) at |x|,
    element by element; for |x| in [2^e, 2^(e+1)) that is 2^(e-8) or 2^(e-11).  fp16's
    subnormal spacing 2^-24 is the floor."""
    bits = 8 if dtype == "bf16" else 11
    _, ex = np.frexp(np.abs(np.asarray(x, dtype=np.float64)))   # |x| = m 2^ex, m in [0.5, 1)
    h = np.ldexp(1.0, ex - 1 - bits)
    return np.maximum(h, 2.0 ** -25) if dtype == "fp16" else h


def unit_roundoff(dtype):
    return 2.0 ** -8 if dtype == "bf16" else 2.0 ** -11


def p_rounding_bound(o_ref, pv_abs, dtype):
    """Most that rounding P to the 16-bit type can move each element of O:
    2u/(1-u) ((P|V|) + |O|) (module docstring)."""
    u = unit_roundoff(dtype)
    return 2.0 * u / (1.0 - u) * (np.asarray(pv_abs) + np.abs(o_ref))


def check_forward(o, lse, o_ref, lse_ref, label="", dtype="bf16", pv_abs=None):
    """O element by element within max(2e-2, r) + half an ulp of the 16-bit output
    grid, O's relative L2 error, and lse's absolute error (bounds in the module
    docstring).  `pv_abs` = P|V| from the oracle enables the P-rounding term r."""
    ma, rl, la = maxabs(o, o_ref), rel_l2(o, o_ref), maxabs(lse, lse_ref)
    allow = O_MAXABS if pv_abs is None else np.maximum(O_MAXABS, p_rounding_bound(o_ref, pv_abs, dtype))
    over = np.abs(o - o_ref) - half_ulp(o_ref, dtype) - allow
    worst = float(np.max(over)) if o.size else -1.0
    excess = float(np.max(np.abs(o - o_ref) - half_ulp(o_ref, dtype))) if o.size else 0.0
    msg = (f"{label} O maxabs={ma:.3e} (beyond half an ulp of the {dtype} grid: {excess:.3e}; "
           f"margin to the bound {-worst:.3e}) relL2={rl:.3e} lse abs={la:.3e}")
    print(msg)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), msg
    assert worst <= 0.0 and rl <= O_RELL2 and la <= LSE_ABS, msg
    return ma, rl, la


def check_backward(grads, refs, label=""):
    errs = [rel_l2(g, r) for g, r in zip(grads, refs)]
    msg = f"{label} relL2 dQ={errs[0]:.3e} dK={errs[1]:.3e} dV={errs[2]:.3e}"
    print(msg)
    for g in grads:
        assert np.all(np.isfinite(g)), msg
    assert max(errs) <= GRAD_RELL2, msg
    return errs


def check_forward_fp8(o, lse, o_ref, lse_ref, vmax, label=""):
    ma, rl, la = maxabs(o, o_ref), rel_l2(o, o_ref), maxabs(lse, lse_ref)
    bound = FP8_O_MAXABS_PER_V * vmax + FP8_O_MAXABS_EXTRA
    msg = f"{label} O maxabs={ma:.3e} (bound {bound:.2e}) relL2={rl:.3e} lse abs={la:.3e}"
    print(msg)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), msg
    assert ma <= bound and rl <= FP8_O_RELL2 and la <= LSE_ABS, msg
    return ma, rl, la
