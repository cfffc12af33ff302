"""Reference of the FP8 (E4M3) forward: the E4M3 number format, block quantization,
the fixed random rotation of Q and K, and exact attention on the de-quantised inputs.

TEST INFRASTRUCTURE ONLY (see the package docstring): nothing on the product path
imports this module, and this module imports nothing from the product path.

Source: [FA-chapter] "Flash Attention" (mlx.void.app), section "FlashAttention-3——重叠与
低精度".  That section fixes the facts used here:

* an fp8 number in the E4M3 format has 256 bit patterns and a largest value of 448;
* everything depends on the scale that maps the data onto that grid; one scale for a
  whole tensor lets a single outlier stretch the grid so that the small values collapse
  onto a few levels;
* block quantization gives every small block its own scale, so an outlier spoils only
  its own block;
* incoherent processing multiplies Q and K by one fixed random rotation before rounding,
  spreading an outlier's energy over every dimension; before any rounding the rotation
  changes no dot product, after rounding nothing is preserved exactly.

Where the section leaves a step open, the plainest reading is taken (each is listed
with the design notes):

* E4M3 is the sign / 4-bit exponent (bias 7) / 3-bit mantissa format whose largest
  finite value is 448 = 1.75 * 2^8: exponent field 15 with mantissa 7 is the only NaN
  pattern, there are no infinities, exponent field 0 holds the subnormals m/8 * 2^-6.
  Rounding is to nearest, ties to the even mantissa, saturating at +-448.
* A block is 128 consecutive rows (query rows for Q, keys for K and V) of one
  (batch, head), all d columns: the tile the kernel works on.  Its scale is
  amax / 448, so the block's largest magnitude maps onto the format's largest value.
* The rotation is the randomized Hadamard transform R = diag(s) H / sqrt(d): H is the
  Sylvester-Hadamard matrix and s a fixed vector of random signs (Ailon and Chazelle's
  fast Johnson-Lindenstrauss construction).  A row x becomes x R.  R is orthogonal, so
  (q R) . (k R) = q . k.
* The quantized values are decided in float32, the precision of the kernel that makes
  them: the rotation is the Walsh-Hadamard transform computed by the radix-2
  butterflies in the order h = 1, 2, 4, ... in float32, scale = fl32(amax / 448),
  inv = fl32(1 / scale), code = E4M3(fl32(x * inv)).
"""

from __future__ import annotations

import numpy as np

from .attention import attn_fwd_ref

__all__ = [
    "E4M3_MAX",
    "QUANT_BLOCK",
    "e4m3_values",
    "e4m3_decode",
    "e4m3_encode",
    "hadamard",
    "rotate_exact",
    "rotate_fp32",
    "quantize_blocks",
    "dequantize_blocks",
    "attn_fp8_ref",
]

E4M3_MAX = 448.0
QUANT_BLOCK = 128


# ----------------------------------------------------------------------------------
# the E4M3 format
# ----------------------------------------------------------------------------------
def e4m3_decode(codes):
    """Value (float64) of each 8-bit E4M3 code: sign bit 7, exponent bits 6..3 with bias
    7, mantissa bits 2..0.  Exponent field 0 is subnormal (m/8 * 2^-6); the pattern
    S.1111.111 is NaN; there is no infinity."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((e == 15) & ((c & 7) == 7), np.nan, mag)
    return sign * mag


def e4m3_values():
    """The finite non-negative E4M3 values, by code 0x00 .. 0x7E (increasing)."""
    return e4m3_decode(np.arange(0x7F, dtype=np.uint8))


_POS = None


def e4m3_encode(x):
    """E4M3 code of each value of x: round to nearest, ties to the code with the even
    mantissa, magnitudes beyond 448 saturate to 448, the sign is kept (also for zero).
    The comparison is exact: x is taken as given (float32 or float64) and every E4M3
    value is exact in float64."""
    global _POS
    if _POS is None:
        _POS = e4m3_values()
    x = np.asarray(x, dtype=np.float64)
    if np.isnan(x).any():
        raise ValueError("e4m3_encode: NaN input")
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.searchsorted(_POS, a, side="left")          # first value >= a
    hi = np.minimum(hi, len(_POS) - 1)
    lo = np.maximum(hi - 1, 0)
    d_hi = _POS[hi] - a
    d_lo = a - _POS[lo]
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((hi & 1) == 0) & (hi != lo))
    code = np.where(pick_hi, hi, lo)
    code = np.where(_POS[hi] == a, hi, code)            # exact hits
    return (code | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)


# ----------------------------------------------------------------------------------
# the fixed random rotation of Q and K
# ----------------------------------------------------------------------------------
def hadamard(d):
    """Sylvester-Hadamard matrix of order d (a power of two): H[i, j] = (-1)^popcount(i & j)."""
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    i = np.arange(d)
    bits = np.bitwise_and.outer(i, i)
    pop = np.zeros_like(bits)
    while bits.any():
        pop += bits & 1
        bits >>= 1
    return np.where(pop & 1, -1.0, 1.0)


def rotate_exact(x, signs):
    """x R with R = diag(signs) H / sqrt(d), in float64 (the rotation as mathematics)."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    return (x * np.asarray(signs, dtype=np.float64)) @ hadamard(d) / np.sqrt(d)


def rotate_fp32(x, signs):
    """The same rotation evaluated in float32 by the in-place Walsh-Hadamard butterflies
    (pairs (i, i + h) -> (a + b, a - b) for h = 1, 2, 4, ..., d/2), then one multiply by
    fl32(1/sqrt(d)).  This is the order in which the quantizing kernel rounds, so the
    float32 result -- and the code it rounds to -- is the kernel's, bit for bit."""
    z = np.asarray(x, dtype=np.float32) * np.asarray(signs, dtype=np.float32)
    d = z.shape[-1]
    z = z.copy()
    h = 1
    while h < d:
        z = z.reshape(z.shape[:-1] + (d // (2 * h), 2, h))
        a = z[..., 0, :].copy()
        b = z[..., 1, :].copy()
        z[..., 0, :] = a + b
        z[..., 1, :] = a - b
        z = z.reshape(z.shape[:-3] + (d,))
        h *= 2
    return z * np.float32(1.0 / np.sqrt(d))


# ----------------------------------------------------------------------------------
# block quantization
# ----------------------------------------------------------------------------------
def quantize_blocks(x, per_tensor=False, signs=None, block=QUANT_BLOCK):
    """E4M3 codes and float32 scales of x (B, H, N, d), one scale per `block` rows of
    one (batch, head) -- or, with per_tensor, one scale for the whole head written to
    every block.  With `signs`, rows are first rotated (rotate_fp32).

    Returns (codes uint8 (B, H, N, d), scales float32 (B, H, ceil(N / block))).  The
    value represented is codes * scale of the code's block."""
    y = np.asarray(x, dtype=np.float32)
    if signs is not None:
        y = rotate_fp32(y, signs)
    B, H, N, d = y.shape
    nb = (N + block - 1) // block
    amax = np.zeros((B, H, nb), dtype=np.float32)
    for j in range(nb):
        amax[:, :, j] = np.abs(y[:, :, j * block:(j + 1) * block, :]).max(axis=(2, 3))
    if per_tensor:
        amax = np.broadcast_to(amax.max(axis=2, keepdims=True), amax.shape).copy()
    scales = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    inv = (np.float32(1.0) / scales).astype(np.float32)
    inv_rows = np.repeat(inv, block, axis=2)[:, :, :N, None]
    return e4m3_encode((y * inv_rows).astype(np.float32)), scales


def dequantize_blocks(codes, scales, block=QUANT_BLOCK):
    """float64 values codes * scale (the scale of each row's block)."""
    N = codes.shape[2]
    s = np.repeat(np.asarray(scales, dtype=np.float64), block, axis=2)[:, :, :N, None]
    return e4m3_decode(codes) * s


def attn_fp8_ref(q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, scale, causal, heads=None):
    """The FP8 forward's reference: exact attention (the plain definition, float64) on
    the de-quantised inputs.  Whatever the kernel adds beyond this -- the rounding of P to
    E4M3 before P.V, float32 accumulation -- is measured against it."""
    q = dequantize_blocks(q_codes, q_scales)
    k = dequantize_blocks(k_codes, k_scales)
    v = dequantize_blocks(v_codes, v_scales)
    return attn_fwd_ref(q, k, v, scale, causal, heads=heads)
