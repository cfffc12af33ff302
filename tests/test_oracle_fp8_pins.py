"""Pins for the oracle's FP8 reference (oracle/fp8.py).  CPU only.

  * the E4M3 format: the page's two printed facts (256 bit patterns, largest value
    448), values written out by hand from the bit layout, agreement with PyTorch's
    float8_e4m3fn conversion (a library routine), ties to even and saturation;
  * the rotation: the Sylvester matrix written out at order 4, orthogonality, the
    page's statement that the rotation changes no dot product, and the float32
    butterflies against the float64 matrix product;
  * block quantization: exactly representable blocks round-trip exactly, the error
    bound of one E4M3 rounding, a block's largest magnitude maps to 448, and the page's
    claims that an outlier spoils only its own block under block scales while a single
    tensor scale collapses the small values onto a few levels, and that the rotation
    cuts the error an outlier causes;
  * the FP8 attention reference equals the pinned dense oracle on exactly
    representable inputs, and attention is unchanged by rotating Q and K before any
    rounding;
  * planted mistakes (ties away from zero, no saturation, signs applied after the
    transform, a swapped butterfly, a per-tensor scale in block mode) are each caught.
"""

import numpy as np
import pytest

import oracle
from oracle import fp8 as F
from tests.pins import read_golden


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


# ---------------------------------------------------------------- the E4M3 format
def test_page_facts_bit_patterns_and_max():
    g = read_golden("e4m3_format.txt")
    codes = np.arange(256, dtype=np.uint8)
    vals = F.e4m3_decode(codes)
    assert len(codes) == int(g["bit_patterns"][0])
    assert np.nanmax(vals) == float(g["max_value"][0]) == F.E4M3_MAX
    assert np.nanmin(vals) == -F.E4M3_MAX
    assert np.isnan(vals).sum() == 2           # S.1111.111, no infinities
    assert np.isfinite(vals[~np.isnan(vals)]).all()


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x38, 1.0), (0x39, 1.125), (0x3F, 1.875), (0x40, 2.0),
    (0x08, 2.0 ** -6), (0x07, 7 / 8 * 2.0 ** -6), (0x01, 2.0 ** -9),
    (0x7E, 448.0), (0x7D, 416.0), (0xB8, -1.0), (0xFE, -448.0), (0x80, -0.0),
])
def test_decode_by_hand(code, value):
    assert F.e4m3_decode(np.uint8(code)) == value


def _check_encoder(enc):
    # ties: 1.0625 lies halfway between 1.0 (mantissa 0) and 1.125 (mantissa 1);
    # 1.1875 halfway between 1.125 and 1.25 (mantissa 2); 2^-10 halfway between 0 and 2^-9
    assert enc(np.float32(1.0625)) == 0x38
    assert enc(np.float32(1.1875)) == 0x3A
    assert enc(np.float32(2.0 ** -10)) == 0x00
    assert enc(np.float32(3 * 2.0 ** -10)) == 0x02
    assert enc(np.float32(-1.0625)) == 0xB8
    # saturation and signed zero
    assert enc(np.float32(1000.0)) == 0x7E and enc(np.float32(-1e6)) == 0xFE
    assert enc(np.float32(460.0)) == 0x7E
    assert enc(np.float32(-0.0)) == 0x80 and enc(np.float32(-1e-6)) == 0x80


def test_encode_ties_and_saturation():
    _check_encoder(F.e4m3_encode)


def test_encode_matches_library_conversion():
    torch = pytest.importorskip("torch")
    r = _rng(3)
    x = np.concatenate([r.standard_normal(200000) * 40, r.standard_normal(50000) * 0.01,
                        F.e4m3_values()[:-1] + np.diff(F.e4m3_values()) / 2,   # every midpoint
                        -F.e4m3_values()]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(F.e4m3_encode(x), ref)


def test_round_trip_and_monotone():
    v = F.e4m3_values()
    assert np.all(np.diff(v) > 0)
    assert np.array_equal(F.e4m3_encode(v), np.arange(127, dtype=np.uint8))
    assert np.array_equal(F.e4m3_decode(F.e4m3_encode(-v[1:])), -v[1:])


def test_planted_encoder_mistakes_are_caught():
    vals = F.e4m3_values()

    def ties_away(x):
        a = min(abs(float(x)), 448.0)
        i = int(np.argmin(np.abs(vals - a) - 1e-12 * vals))   # prefers the larger on ties
        return i | (0x80 if np.signbit(x) else 0)

    def no_saturation(x):
        if abs(float(x)) > 448:
            return 0x7F
        return int(F.e4m3_encode(x))

    for enc in (ties_away, no_saturation):
        with pytest.raises(AssertionError):
            _check_encoder(enc)


# ---------------------------------------------------------------- the rotation
def test_hadamard_order_four_by_hand():
    H4 = [[1, 1, 1, 1], [1, -1, 1, -1], [1, 1, -1, -1], [1, -1, -1, 1]]
    assert np.array_equal(F.hadamard(4), np.array(H4, dtype=float))
    for d in (2, 8, 64, 128):
        H = F.hadamard(d)
        assert np.array_equal(H @ H.T, d * np.eye(d))


def _signs(d, seed=5):
    return np.where(_rng(seed).random(d) < 0.5, -1.0, 1.0)


@pytest.mark.parametrize("d", [64, 128])
def test_rotation_is_orthogonal_and_keeps_dot_products(d):
    r = _rng(d)
    q = r.standard_normal((50, d))
    k = r.standard_normal((60, d))
    s = _signs(d)
    qr, kr = F.rotate_exact(q, s), F.rotate_exact(k, s)
    assert np.allclose(np.linalg.norm(qr, axis=1), np.linalg.norm(q, axis=1), rtol=1e-13)
    assert np.allclose(qr @ kr.T, q @ k.T, rtol=0, atol=1e-12)     # "the dot product is unchanged"
    R = F.rotate_exact(np.eye(d), s)
    assert np.allclose(R @ R.T, np.eye(d), atol=1e-14)


@pytest.mark.parametrize("d", [64, 128])
def test_fp32_butterflies_match_the_matrix(d):
    x = _rng(d + 1).standard_normal((300, d)).astype(np.float32)
    s = _signs(d, 9)
    got = F.rotate_fp32(x, s).astype(np.float64)
    ref = F.rotate_exact(x.astype(np.float64), s)
    err = np.abs(got - ref).max() / np.abs(ref).max()
    assert err < 4e-7 * np.log2(d)


def test_planted_rotation_mistakes_are_caught():
    d = 64
    x = _rng(7).standard_normal((20, d))
    s = _signs(d, 4)
    ref = F.rotate_exact(x, s)
    signs_after = (x @ F.hadamard(d)) * s / np.sqrt(d)
    assert not np.allclose(signs_after, ref, atol=1e-3)
    swapped = x * s
    h = 1
    while h < d:   # butterfly with (a - b, a + b): a wrong transform
        z = swapped.reshape(x.shape[0], d // (2 * h), 2, h)
        a, b = z[:, :, 0, :].copy(), z[:, :, 1, :].copy()
        z[:, :, 0, :], z[:, :, 1, :] = a - b, a + b
        swapped = z.reshape(x.shape[0], d)
        h *= 2
    assert not np.allclose(swapped / np.sqrt(d), ref, atol=1e-3)


# ---------------------------------------------------------------- block quantization
def test_exactly_representable_blocks_round_trip():
    r = _rng(11)
    B, H, N, d = 1, 2, 300, 64
    codes = r.integers(0, 0x7F, size=(B, H, N, d)).astype(np.uint8) | np.where(r.random((B, H, N, d)) < 0.5, 0x80, 0).astype(np.uint8)
    nb = 3
    codes[:, :, ::128, 0] = 0x7E                       # every block holds +-448
    pw = 2.0 ** r.integers(-6, 3, size=(B, H, nb))     # power-of-two scales
    x = F.e4m3_decode(codes) * np.repeat(pw, 128, axis=2)[:, :, :N, None]
    c2, s2 = F.quantize_blocks(x)
    assert np.array_equal(s2, pw.astype(np.float32))
    assert np.array_equal(F.dequantize_blocks(c2, s2), np.where(codes == 0x80, 0.0, x))


def test_rounding_error_bound_and_block_max():
    r = _rng(12)
    x = (r.standard_normal((2, 3, 400, 64)) * np.exp(r.standard_normal((2, 3, 400, 1)))).astype(np.float32)
    codes, scales = F.quantize_blocks(x)
    deq = F.dequantize_blocks(codes, scales)
    s_rows = np.repeat(scales.astype(np.float64), 128, axis=2)[:, :, :400, None]
    bound = np.maximum(2.0 ** -4 * np.abs(x), 2.0 ** -10 * s_rows) * (1 + 1e-6)
    assert np.all(np.abs(deq - x) <= bound)
    for j in range(scales.shape[2]):
        blk = codes[:, :, j * 128:(j + 1) * 128, :]
        assert np.all(np.abs(F.e4m3_decode(blk)).max(axis=(2, 3)) == 448.0)


def _planted_outlier(seed=13, big=1e5):
    # E4M3 keeps its relative precision over 2^17 of range, so a single tensor scale
    # only collapses the N(0,1) values onto few levels once the outlier is about 2^14
    # times larger than them (they then fall into the subnormals)
    x = _rng(seed).standard_normal((1, 1, 512, 64)).astype(np.float32)
    y = x.copy()
    y[0, 0, 5, 7] = big          # block 0 only
    return x, y


def test_outlier_spoils_only_its_own_block():
    x, y = _planted_outlier()
    cx, sx = F.quantize_blocks(x)
    cy, sy = F.quantize_blocks(y)
    assert sy[0, 0, 0] > 100 * sx[0, 0, 0]
    assert np.array_equal(cx[:, :, 128:], cy[:, :, 128:]) and np.array_equal(sx[:, :, 1:], sy[:, :, 1:])
    # with one scale for the tensor, the small values of another block collapse onto a
    # few levels
    ct, st = F.quantize_blocks(y, per_tensor=True)
    assert np.all(st == st[0, 0, 0])
    levels_block = len(np.unique(cy[0, 0, 128:256]))
    levels_tensor = len(np.unique(ct[0, 0, 128:256]))
    assert levels_tensor < levels_block / 4
    err_block = np.abs(F.dequantize_blocks(cy, sy) - y)[0, 0, 128:].mean()
    err_tensor = np.abs(F.dequantize_blocks(ct, st) - y)[0, 0, 128:].mean()
    assert err_tensor > 3 * err_block


def test_planted_per_tensor_scale_in_block_mode_is_caught():
    x, y = _planted_outlier()
    cy, sy = F.quantize_blocks(y)
    wrong = np.broadcast_to(sy.max(axis=2, keepdims=True), sy.shape)
    assert not np.array_equal(wrong, sy)


def test_rotation_cuts_the_outlier_error_of_qk():
    r = _rng(14)
    d = 64
    q = r.standard_normal((1, 1, 128, d)).astype(np.float32)
    k = r.standard_normal((1, 1, 128, d)).astype(np.float32)
    q[0, 0, :, 3] *= 40.0        # one outlier channel, as in real activations
    k[0, 0, :, 3] *= 40.0
    s = _signs(d, 2)
    exact = q[0, 0].astype(np.float64) @ k[0, 0].astype(np.float64).T

    def err(signs):
        cq, sq = F.quantize_blocks(q, signs=signs)
        ck, sk = F.quantize_blocks(k, signs=signs)
        got = F.dequantize_blocks(cq, sq)[0, 0] @ F.dequantize_blocks(ck, sk)[0, 0].T
        return np.linalg.norm(got - exact) / np.linalg.norm(exact)

    assert err(s) < 0.5 * err(None)


# ---------------------------------------------------------------- FP8 attention reference
def test_fp8_reference_on_representable_inputs_is_the_dense_oracle():
    r = _rng(15)
    B, H, N, d = 1, 2, 200, 64
    mk = lambda: r.integers(0, 0x7F, size=(B, H, N, d)).astype(np.uint8) | np.where(  # noqa: E731
        r.random((B, H, N, d)) < 0.5, 0x80, 0).astype(np.uint8)
    cq, ck, cv = mk(), mk(), mk()
    sq = np.full((B, H, 2), 2.0 ** -8, np.float32)
    sk = np.full((B, H, 2), 2.0 ** -7, np.float32)
    sv = np.full((B, H, 2), 2.0 ** -9, np.float32)
    for causal in (False, True):
        o, lse = F.attn_fp8_ref(cq, sq, ck, sk, cv, sv, 0.125, causal)
        o2, lse2 = oracle.attn_fwd_ref(F.e4m3_decode(cq) / 256, F.e4m3_decode(ck) / 128, F.e4m3_decode(cv) / 512,
                                       0.125, causal)
        assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def test_attention_is_unchanged_by_rotating_q_and_k():
    r = _rng(16)
    q, k, v = (r.standard_normal((1, 2, 96, 64)) for _ in range(3))
    s = _signs(64, 8)
    for causal in (False, True):
        o1, l1 = oracle.attn_fwd_ref(q, k, v, 0.125, causal)
        o2, l2 = oracle.attn_fwd_ref(F.rotate_exact(q, s), F.rotate_exact(k, s), v, 0.125, causal)
        assert np.abs(o1 - o2).max() < 1e-12 and np.abs(l1 - l2).max() < 1e-12
