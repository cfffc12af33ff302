"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds no attention arithmetic: it draws i.i.d. Gaussian numbers from a
seeded numpy PCG64 stream, rounds them to a 16-bit float format (round to nearest,
ties to even) and hands out the 16-bit bit patterns.  The same bits are uploaded to
the GPU and widened exactly to float64 for the oracle, so both sides see identical
operands.

Seed rule: seed = 1000*workload_index + 10*length_index + {q: 0, k: 1, v: 2, do: 3}.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

TENSOR_OFFSET = {"q": 0, "k": 1, "v": 2, "do": 3}

DTYPES = ("bf16", "fp16")


def seed_for(workload_index: int, length_index: int, tensor: str) -> int:
    return 1000 * int(workload_index) + 10 * int(length_index) + TENSOR_OFFSET[tensor]


def _round_f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest, ties to even (finite input)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def gaussian_bits(shape, seed: int, dtype: str = "bf16", mult: float = 1.0) -> np.ndarray:
    """i.i.d. N(0,1) * mult drawn in float32 from PCG64(seed), rounded to ``dtype``.

    Returns a uint16 array of the 16-bit patterns.
    """
    if dtype not in DTYPES:
        raise ValueError(f"dtype must be one of {DTYPES}")
    rng = np.random.Generator(np.random.PCG64(int(seed)))
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if mult != 1.0:
        x *= np.float32(mult)
    if dtype == "bf16":
        return _round_f32_to_bf16_bits(x)
    return x.astype(np.float16).view(np.uint16)


def bits_to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of 16-bit patterns to float64."""
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    if dtype == "fp16":
        return bits.view(np.float16).astype(np.float64)
    raise ValueError(f"dtype must be one of {DTYPES}")


def f64_to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values to 16-bit patterns (via float32), for hand-built inputs."""
    x32 = np.asarray(x, dtype=np.float32)
    if dtype == "bf16":
        return _round_f32_to_bf16_bits(x32)
    return x32.astype(np.float16).view(np.uint16)


@dataclass
class Case:
    """One synthetic attention problem: 16-bit bit patterns of shape (B, H, N, d)."""
    B: int
    H: int
    N: int
    d: int
    dtype: str
    causal: bool
    scale: float
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    do: np.ndarray | None

    def f64(self, name: str) -> np.ndarray:
        return bits_to_f64(getattr(self, name), self.dtype)


def make_case(B, H, N, d, dtype="bf16", causal=False, scale=None, workload_index=0,
              length_index=0, mult=1.0, with_do=True) -> Case:
    """Seeded Q, K, V (x ``mult``) and dO (unscaled) for one problem."""
    shape = (int(B), int(H), int(N), int(d))
    scale = float(d) ** -0.5 if scale is None else float(scale)
    q = gaussian_bits(shape, seed_for(workload_index, length_index, "q"), dtype, mult)
    k = gaussian_bits(shape, seed_for(workload_index, length_index, "k"), dtype, mult)
    v = gaussian_bits(shape, seed_for(workload_index, length_index, "v"), dtype, mult)
    do = gaussian_bits(shape, seed_for(workload_index, length_index, "do"), dtype) if with_do else None
    return Case(int(B), int(H), int(N), int(d), dtype, bool(causal), scale, q, k, v, do)


@dataclass
class CrossCase:
    B: int
    H: int
    Hkv: int
    Nq: int
    Nk: int
    d: int
    dtype: str
    causal: bool
    scale: float
    q: np.ndarray    # (B, H, Nq, d) 16-bit bits
    k: np.ndarray    # (B, Hkv, Nk, d)
    v: np.ndarray    # (B, Hkv, Nk, d)
    do: np.ndarray   # (B, H, Nq, d) or None


def make_cross_case(B, H, Hkv, Nq, Nk, d, dtype="bf16", causal=False, scale=None, workload_index=0,
                    length_index=0, mult=1.0, with_do=True) -> CrossCase:
    """Seeded Q (B, H, Nq, d), K and V (B, Hkv, Nk, d) (x ``mult``) and dO (unscaled)."""
    scale = float(d) ** -0.5 if scale is None else float(scale)
    qs, ks = (int(B), int(H), int(Nq), int(d)), (int(B), int(Hkv), int(Nk), int(d))
    q = gaussian_bits(qs, seed_for(workload_index, length_index, "q"), dtype, mult)
    k = gaussian_bits(ks, seed_for(workload_index, length_index, "k"), dtype, mult)
    v = gaussian_bits(ks, seed_for(workload_index, length_index, "v"), dtype, mult)
    do = gaussian_bits(qs, seed_for(workload_index, length_index, "do"), dtype) if with_do else None
    return CrossCase(int(B), int(H), int(Hkv), int(Nq), int(Nk), int(d), dtype, bool(causal), scale, q, k, v, do)


# The workloads, as (name, B, H, N, d, dtype, causal, backward, mult).  The sweep
# entries keep B*N = 65536 tokens.
WORKLOADS = {
    "c1_tiny": dict(B=1, H=1, N=256, d=64, dtype="bf16", causal=False, backward=False, mult=1.0, index=1),
    "c2_gpt2s": dict(B=8, H=12, N=1024, d=64, dtype="bf16", causal=True, backward=True, mult=1.0, index=2),
    "c3_prefill": dict(B=1, H=8, N=4096, d=64, dtype="bf16", causal=True, backward=False, mult=1.0, index=3),
    "c4a_long": dict(B=4, H=16, N=8192, d=64, dtype="fp16", causal=True, backward=True, mult=1.0, index=4),
    "c4b_long_d128": dict(B=4, H=8, N=8192, d=128, dtype="fp16", causal=True, backward=True, mult=1.0, index=4,
                          length_index=1),
}
SWEEP_N = (512, 1024, 2048, 4096, 8192, 16384, 32768, 65536)
for _i, _n in enumerate(SWEEP_N):
    for _c in (True, False):
        WORKLOADS[f"c5_n{_n}_{'causal' if _c else 'full'}"] = dict(
            B=65536 // _n, H=16, N=_n, d=64, dtype="bf16", causal=_c, backward=True, mult=3.0,
            index=5, length_index=_i)


# Workloads of the cross-length, grouped-head and decode entry points (fa_fwd_cross,
# fa_bwd_gqa, fa_decode): prefill and chunked prefill with grouped key/value heads,
# and decoding one new token against a key/value cache.
EXTRA_WORKLOADS = {
    "x1_gqa_prefill": dict(kind="cross", B=2, H=32, Hkv=8, Nq=8192, Nk=8192, d=128, dtype="bf16", causal=True,
                           backward=True, index=20),
    "x2_chunked_prefill": dict(kind="cross", B=4, H=32, Hkv=8, Nq=2048, Nk=16384, d=128, dtype="bf16", causal=True,
                               backward=False, index=21),
    "x3_decode_gqa": dict(kind="decode", B=8, H=32, Hkv=8, Nq=1, Nk=32768, d=128, dtype="bf16", causal=True,
                          backward=False, index=22),
    "x4_decode_mha": dict(kind="decode", B=16, H=32, Hkv=32, Nq=1, Nk=8192, d=128, dtype="bf16", causal=True,
                          backward=False, index=23),
    # block-sparse (butterfly) training step at long sequence length
    "x5_butterfly_64k": dict(kind="sparse", B=1, H=16, Hkv=16, Nq=65536, Nk=65536, d=64, dtype="bf16",
                             causal=False, backward=True, index=24),
    # FP8 (E4M3) forward at the shapes of the 16-bit c4a / c4b workloads: Q and K rotated
    # and block-quantized, V block-quantized into the transposed layout
    "x6_fp8_c4a": dict(kind="fp8", B=4, H=16, Hkv=16, Nq=8192, Nk=8192, d=64, dtype="bf16", causal=True,
                       backward=False, index=25),
    "x7_fp8_c4b": dict(kind="fp8", B=4, H=8, Hkv=8, Nq=8192, Nk=8192, d=128, dtype="bf16", causal=True,
                       backward=False, index=26),
}


def extra_case(name: str) -> CrossCase:
    w = EXTRA_WORKLOADS[name]
    return make_cross_case(w["B"], w["H"], w["Hkv"], w["Nq"], w["Nk"], w["d"], w["dtype"], w["causal"],
                           workload_index=w["index"], with_do=w["backward"])


def workload_case(name: str, with_do=None) -> Case:
    w = WORKLOADS[name]
    wd = w["backward"] if with_do is None else with_do
    return make_case(w["B"], w["H"], w["N"], w["d"], w["dtype"], w["causal"], None,
                     w["index"], w.get("length_index", 0), w["mult"], wd)


def random_signs(d: int, seed: int) -> np.ndarray:
    """d random signs (+1.0 / -1.0, float32) from PCG64(seed): the random draw of the
    fixed rotation that multiplies Q and K before FP8 rounding.  Drawn here and passed
    to both sides as an input."""
    rng = np.random.Generator(np.random.PCG64(int(seed)))
    return np.where(rng.random(int(d)) < 0.5, -1.0, 1.0).astype(np.float32)


def with_outlier_channel(bits: np.ndarray, dtype: str, channel: int, factor: float) -> np.ndarray:
    """The same 16-bit values with column `channel` multiplied by `factor` (rounded back
    to `dtype`): the outlier channel of the FP8 error study."""
    x = bits_to_f64(bits, dtype)
    x[..., channel] *= factor
    return f64_to_bits(x, dtype)


def with_outlier_entry(bits: np.ndarray, dtype: str, index: tuple, value: float) -> np.ndarray:
    """The same 16-bit values with one entry set to `value`: an isolated outlier."""
    x = bits_to_f64(bits, dtype)
    x[index] = value
    return f64_to_bits(x, dtype)
