"""GPU parity of the FP8 path against the oracle (oracle/fp8.py).

  * fa_quantize_fp8: codes and scales bit for bit equal to the oracle's block
    quantization of the same 16-bit inputs -- per block and per tensor, with and
    without the rotation of Q and K, row-major and in the transposed V^T layout
    (whose padding keys must read +0);
  * fa_fwd_fp8: O and lse against exact attention on the de-quantised inputs, the
    inputs quantized by the oracle (tolerances of tests/gpu_util.py, derived from the
    E4M3 rounding of P): several tiles, ragged tails, causal and not, d = 64 and 128,
    bf16 and fp16 output;
  * the error study of the FP8 section: O error against exact attention on the
    original 16-bit inputs, for an outlier channel in Q and K (block scales with and
    without the rotation) and for an isolated outlier (one scale per tensor against
    one per block).  The rotation and the block scales must each cut the error.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from oracle import fp8 as F  # noqa: E402
from exact_tiled_attention_27_gb300 import build, forward_fp8, fp8_vt_cols, last_kernel_status, quantize_fp8  # noqa: E402
from exact_tiled_attention_27_gb300.inputs import (  # noqa: E402
    bits_to_f64, make_case, random_signs, with_outlier_channel, with_outlier_entry)
from tests import gpu_util as G  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()


def _vt_layout(codes):
    """(B, H, N, d) codes -> the (B, H, d, Nt) V^T layout with +0 padding."""
    B, H, N, d = codes.shape
    out = np.zeros((B, H, d, fp8_vt_cols(N)), dtype=np.uint8)
    out[:, :, :, :N] = np.swapaxes(codes, 2, 3)
    return out


QUANT_CASES = [
    # B, H, N, d, dtype, per_tensor, rotate, transpose
    (2, 3, 300, 64, "bf16", False, False, False),
    (1, 2, 1000, 128, "fp16", False, True, False),
    (1, 2, 777, 64, "bf16", True, False, True),
    (2, 1, 129, 128, "bf16", False, False, True),
    (1, 1, 5000, 64, "fp16", True, True, False),
    (1, 2, 64, 64, "bf16", False, True, True),
    (1, 1, 1, 128, "bf16", False, True, False),
]


@pytest.mark.parametrize("B,H,N,d,dtype,per_tensor,rotate,transpose", QUANT_CASES)
def test_quantizer_matches_oracle_bit_for_bit(B, H, N, d, dtype, per_tensor, rotate, transpose):
    c = make_case(B, H, N, d, dtype, False, workload_index=230, length_index=N + d)
    x = G.to_device(c.q, dtype)
    signs = random_signs(d, 2300 + d) if rotate else None
    codes, scales = quantize_fp8(x, per_tensor=per_tensor, signs=None if signs is None else torch.from_numpy(signs).cuda(),
                                 transpose=transpose)
    torch.cuda.synchronize()
    ref_codes, ref_scales = F.quantize_blocks(bits_to_f64(c.q, dtype), per_tensor=per_tensor, signs=signs)
    assert np.array_equal(scales.cpu().numpy(), ref_scales)
    want = _vt_layout(ref_codes) if transpose else ref_codes
    got = codes.cpu().numpy()
    assert got.shape == want.shape
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} codes differ, first at {bad[:3].tolist()}"


FWD_CASES = [
    # B, H, N, d, out dtype, causal, rotate
    (1, 2, 256, 64, "bf16", False, False),
    (2, 2, 1000, 64, "bf16", True, True),
    (1, 2, 777, 128, "fp16", True, False),
    (1, 1, 2048, 128, "bf16", False, True),
    (1, 3, 130, 64, "bf16", True, False),
    (1, 2, 4096, 64, "fp16", True, False),
    (1, 1, 100, 128, "bf16", False, False),
    (2, 2, 1, 64, "bf16", True, True),         # one key: the V^T rows are padded from 1 to 16 bytes
    (1, 2, 17, 128, "fp16", False, False),     # V^T row stride 32 bytes, 15 of them padding
]


@pytest.mark.parametrize("B,H,N,d,dtype,causal,rotate", FWD_CASES)
def test_fp8_forward_matches_oracle(B, H, N, d, dtype, causal, rotate):
    c = make_case(B, H, N, d, "bf16", causal, workload_index=231, length_index=N + d)
    signs = random_signs(d, 2310 + d) if rotate else None
    cq, sq = F.quantize_blocks(bits_to_f64(c.q, "bf16"), signs=signs)
    ck, sk = F.quantize_blocks(bits_to_f64(c.k, "bf16"), signs=signs)
    cv, sv = F.quantize_blocks(bits_to_f64(c.v, "bf16"))
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    o, lse = forward_fp8(dev(cq), dev(ck), dev(_vt_layout(cv)), dev(sq), dev(sk), dev(sv), scale=c.scale,
                         causal=causal, out_dtype=G.torch_dtype(dtype))
    torch.cuda.synchronize()
    assert last_kernel_status() == 0
    o_ref, lse_ref = F.attn_fp8_ref(cq, sq, ck, sk, cv, sv, c.scale, causal)
    vmax = float(np.abs(F.dequantize_blocks(cv, sv)).max())
    G.check_forward_fp8(G.to_f64(o), G.to_f64(lse), o_ref, lse_ref, vmax, f"fp8 B{B} H{H} N{N} d{d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
def test_rows_dominated_by_one_key_return_its_value(d):
    """K = Q with large entries: every causal row's own key outweighs the others by
    e^40 or more, so O_i = V_i.  The dominant weight's E4M3 rounding (up to 2^-4) must
    not reach O: the kernel divides by the weight P.V actually used."""
    N = 640
    c = make_case(1, 2, N, d, "bf16", True, workload_index=234, length_index=d)
    q64 = bits_to_f64(c.q, "bf16") * 5.0
    cq, sq = F.quantize_blocks(q64)
    cv, sv = F.quantize_blocks(bits_to_f64(c.v, "bf16"))
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    o, lse = forward_fp8(dev(cq), dev(cq), dev(_vt_layout(cv)), dev(sq), dev(sq), dev(sv), causal=True)
    torch.cuda.synchronize()
    assert last_kernel_status() == 0
    o_ref, lse_ref = F.attn_fp8_ref(cq, sq, cq, sq, cv, sv, d ** -0.5, True)
    v_deq = F.dequantize_blocks(cv, sv)
    assert np.abs(o_ref - v_deq).max() < 1e-12          # the reference is V itself
    err = np.abs(G.to_f64(o) - o_ref)
    assert np.all(err <= 2.0 ** -8 * np.abs(o_ref) + 1e-6), f"max err {err.max():.3e}"
    assert G.maxabs(G.to_f64(lse), lse_ref) <= G.LSE_ABS


def _fp8_error(q_bits, k_bits, v_bits, scale, causal, per_tensor, signs):
    """relL2 of the FP8 path's O (GPU quantizer + FP8 forward) against exact attention
    on the original 16-bit inputs."""
    q, k, v = (G.to_device(b, "bf16") for b in (q_bits, k_bits, v_bits))
    sg = None if signs is None else torch.from_numpy(signs).cuda()
    q8, sq = quantize_fp8(q, per_tensor=per_tensor, signs=sg)
    k8, sk = quantize_fp8(k, per_tensor=per_tensor, signs=sg)
    vt8, sv = quantize_fp8(v, per_tensor=per_tensor, transpose=True)
    o, _ = forward_fp8(q8, k8, vt8, sq, sk, sv, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert last_kernel_status() == 0
    o_ex, _ = oracle.attn_fwd_ref(*(bits_to_f64(b, "bf16") for b in (q_bits, k_bits, v_bits)), scale, causal)
    return G.rel_l2(G.to_f64(o), o_ex)


def test_error_study_outliers():
    B, H, N, d = 1, 2, 1024, 64
    signs = random_signs(d, 2320)
    print("\nFP8 O relL2 vs exact attention on the 16-bit inputs")
    print("outlier channel x F in Q and K (scale 1/sqrt(d-1+F^4)): F, per tensor, per block, per block + rotation")
    errs = {}
    for Fm in (1, 8, 32, 128):
        c = make_case(B, H, N, d, "bf16", True, workload_index=232, length_index=Fm)
        q = with_outlier_channel(c.q, "bf16", 3, Fm)
        k = with_outlier_channel(c.k, "bf16", 3, Fm)
        sc = 1.0 / np.sqrt(d - 1 + Fm ** 4)
        e = [_fp8_error(q, k, c.v, sc, True, True, None), _fp8_error(q, k, c.v, sc, True, False, None),
             _fp8_error(q, k, c.v, sc, True, False, signs)]
        errs[Fm] = e
        print(f"  {Fm:4d}  {e[0]:.4f}  {e[1]:.4f}  {e[2]:.4f}")
    print("isolated outlier (one entry of Q, K and V set to A): A, per tensor, per block")
    iso = {}
    for A in (1e2, 1e4, 1e5):
        c = make_case(B, H, N, d, "bf16", True, workload_index=233, length_index=int(np.log10(A)))
        q = with_outlier_entry(c.q, "bf16", (0, 0, 5, 7), A)
        k = with_outlier_entry(c.k, "bf16", (0, 1, 700, 2), A)
        v = with_outlier_entry(c.v, "bf16", (0, 0, 900, 1), A)
        e = [_fp8_error(q, k, v, c.scale, True, True, None), _fp8_error(q, k, v, c.scale, True, False, None)]
        iso[A] = e
        print(f"  {A:8.0e}  {e[0]:.4f}  {e[1]:.4f}")
    # without outliers the three agree; with them the rotation and the block scales
    # each cut the error
    assert max(errs[1]) < 0.08
    assert errs[128][2] < 0.6 * errs[128][1] and errs[128][1] < errs[128][0]
    assert iso[1e5][0] > 2 * iso[1e5][1]
