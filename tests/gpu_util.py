"""Helpers shared by the GPU tests: upload seeded 16-bit bits, read results back as
float64, the comparison metrics, and the tolerances the parity tests enforce.

Tolerances (stated for the 16-bit inputs against the float64 oracle):
  O:            max |err| <= 2e-2 * mult and ||err||_2 / ||ref||_2 <= 5e-3, where mult
                is the factor the Gaussian inputs were multiplied by (1 for unit-scale
                data, 3 for the "x3" sweep).  O is a convex combination of V rows, so its
                magnitude -- and the spacing of the 16-bit grid it is rounded to --
                grows with mult; at mult = 3 the exact O rounded to bf16 already errs by
                up to 0.031 > 2e-2.
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


def check_forward(o, lse, o_ref, lse_ref, label="", mult=1.0):
    ma, rl, la = maxabs(o, o_ref), rel_l2(o, o_ref), maxabs(lse, lse_ref)
    msg = f"{label} O maxabs={ma:.3e} (bound {O_MAXABS * mult:.1e}) relL2={rl:.3e} lse abs={la:.3e}"
    print(msg)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), msg
    assert ma <= O_MAXABS * mult and rl <= O_RELL2 and la <= LSE_ABS, msg
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
