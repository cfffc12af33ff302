"""Boundary tests that need no GPU: the library builds, loads, exports every entry
point include/fa.h declares, and rejects invalid arguments before touching a device."""

import ctypes
import os
import re

import pytest

from exact_tiled_attention_27_gb300 import binding, build
from exact_tiled_attention_27_gb300.inputs import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s+(fa_\w+)\s*\(", text, flags=re.M)


def test_header_declares_expected_entry_points():
    names = set(declared_functions())
    assert {"fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_strerror", "fa_get_last_kernel_status"} <= names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in fa.h but not exported"


def test_status_enum_matches_binding():
    text = open(HEADER).read()
    for name, code in re.findall(r"(FA_(?:OK|ERR_\w+))\s*=\s*(\d+)", text):
        assert binding.STATUS[int(code)] == name


def test_strerror_covers_every_code(lib):
    for code in binding.STATUS:
        s = lib.fa_strerror(code).decode()
        assert s and s != "unknown status"
    assert lib.fa_strerror(12345).decode() == "unknown status"


P = ctypes.c_void_p(0x10000)      # a 16-byte aligned stand-in; never dereferenced on error paths
PM = ctypes.c_void_p(0x10008)     # misaligned
NULL = ctypes.c_void_p(0)


def fwd(lib, q=P, k=P, v=P, o=P, lse=P, B=1, H=1, N=128, d=64, scale=0.125, causal=0, dtype=0):
    return lib.fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, NULL)


def bwd(lib, ws=P, ws_bytes=None, q=P, B=1, H=1, N=128, d=64, scale=0.125, dtype=0, dq=P):
    if ws_bytes is None:
        ws_bytes = lib.fa_bwd_workspace_size(B, H, N, d) if B > 0 and H > 0 and N > 0 else 0
    return lib.fa_bwd(q, P, P, P, P, P, dq, P, P, ws, ws_bytes, B, H, N, d, scale, 0, dtype, NULL)


def test_forward_validation_codes(lib):
    C = binding.STATUS_CODE
    assert fwd(lib, dtype=2) == C["FA_ERR_DTYPE"]
    assert fwd(lib, d=32) == C["FA_ERR_UNSUPPORTED_D"]
    assert fwd(lib, d=96) == C["FA_ERR_UNSUPPORTED_D"]
    assert fwd(lib, B=0) == C["FA_ERR_SHAPE"]
    assert fwd(lib, H=-1) == C["FA_ERR_SHAPE"]
    assert fwd(lib, N=0) == C["FA_ERR_SHAPE"]
    assert fwd(lib, B=1 << 16, H=1 << 16) == C["FA_ERR_SHAPE"]
    assert fwd(lib, scale=0.0) == C["FA_ERR_SCALE"]
    assert fwd(lib, scale=-1.0) == C["FA_ERR_SCALE"]
    assert fwd(lib, scale=float("nan")) == C["FA_ERR_SCALE"]
    assert fwd(lib, scale=float("inf")) == C["FA_ERR_SCALE"]
    assert fwd(lib, q=NULL) == C["FA_ERR_NULL"]
    assert fwd(lib, lse=NULL) == C["FA_ERR_NULL"]
    assert fwd(lib, k=PM) == C["FA_ERR_ALIGN"]
    assert fwd(lib, o=PM) == C["FA_ERR_ALIGN"]


def test_size_limits_are_pinned(lib):
    """The size limits: B*H <= 2^30 heads and B*H*N < 2^31 rows per tensor.  A call at
    the limit passes the shape check (it then stops at the null pointer, before any
    device work); one row more is FA_ERR_SHAPE.  Any call that fits in device memory
    is inside these limits: 2^31 rows of Q and of O alone take 512 GiB at d = 64."""
    C = binding.STATUS_CODE
    for B, H, N in [(1, 2, (1 << 30) - 1), (1 << 10, 1 << 10, (1 << 11) - 1), (1, 1 << 30, 1)]:
        assert fwd(lib, q=NULL, B=B, H=H, N=N) == C["FA_ERR_NULL"]
        assert bwd(lib, q=NULL, ws=P, ws_bytes=1 << 62, B=B, H=H, N=N) == C["FA_ERR_NULL"]
    for B, H, N in [(1, 2, 1 << 30), (1 << 10, 1 << 10, 1 << 11), (1, (1 << 30) + 1, 1), (2, 1 << 30, 1)]:
        assert fwd(lib, q=NULL, B=B, H=H, N=N) == C["FA_ERR_SHAPE"]
        assert lib.fa_bwd_workspace_size(B, H, N, 64) == 0


def fwd_cross(lib, q=P, k=P, B=1, H=4, Hkv=2, Nq=3, Nk=300, d=64, scale=0.125, causal=1, dtype=0):
    return lib.fa_fwd_cross(q, k, P, P, P, B, H, Hkv, Nq, Nk, d, scale, causal, dtype, NULL)


def test_forward_cross_validation_codes(lib):
    C = binding.STATUS_CODE
    assert fwd_cross(lib, Hkv=3) == C["FA_ERR_SHAPE"]          # 3 does not divide 4
    assert fwd_cross(lib, Hkv=0) == C["FA_ERR_SHAPE"]
    assert fwd_cross(lib, Hkv=8) == C["FA_ERR_SHAPE"]          # more key/value heads than query heads
    assert fwd_cross(lib, Nq=0) == C["FA_ERR_SHAPE"]
    assert fwd_cross(lib, Nk=0) == C["FA_ERR_SHAPE"]
    assert fwd_cross(lib, d=80) == C["FA_ERR_UNSUPPORTED_D"]
    assert fwd_cross(lib, dtype=5) == C["FA_ERR_DTYPE"]
    assert fwd_cross(lib, scale=0.0) == C["FA_ERR_SCALE"]
    assert fwd_cross(lib, q=NULL) == C["FA_ERR_NULL"]
    assert fwd_cross(lib, k=PM) == C["FA_ERR_ALIGN"]


def test_backward_gqa_validation_codes(lib):
    C = binding.STATUS_CODE
    need = lib.fa_bwd_workspace_size(1, 4, 128, 64)

    def call(H=4, Hkv=2, N=128, ws_bytes=need):
        return lib.fa_bwd_gqa(P, P, P, P, P, P, P, P, P, P, ws_bytes, 1, H, Hkv, N, 64, 0.125, 1, 0, NULL)

    assert call(Hkv=3) == C["FA_ERR_SHAPE"]
    assert call(Hkv=0) == C["FA_ERR_SHAPE"]
    assert call(Hkv=8) == C["FA_ERR_SHAPE"]
    assert call(N=0) == C["FA_ERR_SHAPE"]
    assert call(ws_bytes=need - 1) == C["FA_ERR_WORKSPACE"]


def test_fp8_entry_points_validate(lib):
    C = binding.STATUS_CODE
    assert [lib.fa_fp8_vt_cols(n) for n in (0, 1, 16, 17, 1000)] == [0, 16, 16, 32, 1008]

    def quant(x=P, x8=P, scales=P, B=1, H=1, N=128, d=64, dtype=0, signs=NULL):
        return lib.fa_quantize_fp8(x, x8, scales, B, H, N, d, dtype, signs, 0, 0, NULL)

    assert quant(x=NULL) == C["FA_ERR_NULL"]
    assert quant(scales=NULL) == C["FA_ERR_NULL"]
    assert quant(d=80) == C["FA_ERR_UNSUPPORTED_D"]
    assert quant(dtype=3) == C["FA_ERR_DTYPE"]
    assert quant(N=0) == C["FA_ERR_SHAPE"]
    assert quant(x8=PM) == C["FA_ERR_ALIGN"]
    assert quant(signs=ctypes.c_void_p(0x10002)) == C["FA_ERR_ALIGN"]

    def f8(q=P, vt=P, ks=P, o=P, B=1, H=1, N=128, d=64, scale=0.125, dtype=0):
        return lib.fa_fwd_fp8(q, P, vt, P, ks, P, o, P, B, H, N, d, scale, 1, dtype, NULL)

    assert f8(q=NULL) == C["FA_ERR_NULL"]
    assert f8(ks=NULL) == C["FA_ERR_NULL"]
    assert f8(vt=PM) == C["FA_ERR_ALIGN"]
    assert f8(ks=ctypes.c_void_p(0x10002)) == C["FA_ERR_ALIGN"]
    assert f8(d=32) == C["FA_ERR_UNSUPPORTED_D"]
    assert f8(dtype=2) == C["FA_ERR_DTYPE"]
    assert f8(scale=0.0) == C["FA_ERR_SCALE"]
    assert f8(B=0) == C["FA_ERR_SHAPE"]


def test_decode_validation_and_workspace(lib):
    C = binding.STATUS_CODE

    def call(H=8, Hkv=2, Nq=1, Nk=4096, d=64, ws=P, ws_bytes=None, scale=0.125, B=1):
        if ws_bytes is None:
            ws_bytes = lib.fa_decode_workspace_size(B, H, Hkv, Nq, Nk, d)
        return lib.fa_decode(P, P, P, P, P, ws, ws_bytes, B, H, Hkv, Nq, Nk, d, scale, 1, 0, NULL)

    assert call(Hkv=3) == C["FA_ERR_SHAPE"]
    assert call(H=16, Hkv=1) == C["FA_ERR_SHAPE"]              # 16 rows per key/value head > 8
    assert call(Nq=3) == C["FA_ERR_SHAPE"]                     # 4 x 3 rows > 8
    assert call(Nk=0) == C["FA_ERR_SHAPE"]
    assert call(d=96) == C["FA_ERR_UNSUPPORTED_D"]
    assert call(scale=float("nan")) == C["FA_ERR_SCALE"]
    assert call(B=65536, H=8, Hkv=1) == C["FA_ERR_SHAPE"]     # one grid row per key/value head: <= 65535
    assert lib.fa_decode_workspace_size(65536, 8, 1, 1, 4096, 64) == 0
    assert call(ws=NULL) == C["FA_ERR_WORKSPACE"]
    assert call(ws_bytes=1) == C["FA_ERR_WORKSPACE"]
    # ranges of >= 256 keys, at most 128: per range B*Hkv*M rows of d float32 + one lse
    for H, Hkv, Nq, Nk, d in [(8, 2, 1, 4096, 64), (4, 4, 2, 100000, 128), (32, 4, 1, 300, 64)]:
        M = (H // Hkv) * Nq
        smax = min(128, max(1, Nk // 256))
        up = lambda x: (x + 255) // 256 * 256
        expect = 0 if smax == 1 else up(smax * Hkv * M * d * 4) + up(smax * Hkv * M * 4)
        assert lib.fa_decode_workspace_size(1, H, Hkv, Nq, Nk, d) == expect
    assert lib.fa_decode_workspace_size(1, 8, 2, 1, 255, 64) == 0     # one range: no workspace
    assert lib.fa_decode_workspace_size(1, 8, 3, 1, 4096, 64) == 0    # invalid grouping


def test_butterfly_blocks_match_brute_force(lib):
    """The key blocks each butterfly query pair visits (host utility of the library)."""
    buf = (ctypes.c_int * 64)()
    for nblocks in (1, 2, 3, 7, 8, 16, 33, 64):
        npairs = (nblocks + 1) // 2
        for pair in range(npairs):
            for direction in (-1, 0, 1):
                want = []
                for p2 in range(npairs):
                    x = pair ^ p2
                    if (x & (x - 1)) == 0 and (direction == 0 or (p2 <= pair if direction < 0 else p2 >= pair)):
                        want += [b for b in (2 * p2, 2 * p2 + 1) if b < nblocks]
                n = lib.fa_butterfly_blocks(nblocks, pair, direction, buf, 64)
                assert n == len(want) and list(buf[:n]) == want, (nblocks, pair, direction)
    assert lib.fa_butterfly_blocks(0, 0, 0, buf, 64) == -1
    assert lib.fa_butterfly_blocks(8, 4, 0, buf, 64) == -1     # pair out of range
    assert lib.fa_butterfly_blocks(8, 0, 2, buf, 64) == -1


def test_sparse_validation_codes(lib):
    C = binding.STATUS_CODE
    assert lib.fa_fwd_sparse(P, P, P, P, P, 1, 1, 512, 64, 0.125, 0, 2, 0, NULL) == C["FA_ERR_PATTERN"]
    assert lib.fa_fwd_sparse(P, P, P, P, P, 1, 1, 0, 64, 0.125, 0, 1, 0, NULL) == C["FA_ERR_SHAPE"]
    need = lib.fa_bwd_workspace_size(1, 1, 512, 64)
    assert lib.fa_bwd_sparse(P, P, P, P, P, P, P, P, P, P, need, 1, 1, 512, 64, 0.125, 0, 0, 0, NULL) == \
        C["FA_ERR_PATTERN"]
    assert lib.fa_bwd_sparse(P, P, P, P, P, P, P, P, P, NULL, need, 1, 1, 512, 64, 0.125, 0, 1, 0, NULL) == \
        C["FA_ERR_WORKSPACE"]


def test_backward_validation_codes(lib):
    C = binding.STATUS_CODE
    assert bwd(lib, dtype=7) == C["FA_ERR_DTYPE"]
    assert bwd(lib, d=256) == C["FA_ERR_UNSUPPORTED_D"]
    assert bwd(lib, N=0) == C["FA_ERR_SHAPE"]
    assert bwd(lib, scale=float("nan")) == C["FA_ERR_SCALE"]
    assert bwd(lib, q=NULL) == C["FA_ERR_NULL"]
    assert bwd(lib, dq=PM) == C["FA_ERR_ALIGN"]
    assert bwd(lib, ws=NULL) == C["FA_ERR_WORKSPACE"]
    need = lib.fa_bwd_workspace_size(1, 1, 128, 64)
    assert bwd(lib, ws_bytes=need - 1) == C["FA_ERR_WORKSPACE"]
    assert bwd(lib, ws=ctypes.c_void_p(0x10010)) == C["FA_ERR_WORKSPACE"]   # not 256-byte aligned


def test_valid_arguments_without_gpu_report_no_device(lib):
    """On a machine with no CUDA device the call gets past validation and stops at
    the device check, with nothing launched."""
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("a GPU is present")
    except ImportError:
        pass
    assert fwd(lib) == binding.STATUS_CODE["FA_ERR_NO_DEVICE"]
    assert fwd_cross(lib) == binding.STATUS_CODE["FA_ERR_NO_DEVICE"]
    assert bwd(lib) == binding.STATUS_CODE["FA_ERR_NO_DEVICE"]
    assert lib.fa_get_last_kernel_status(NULL) == binding.STATUS_CODE["FA_ERR_NO_DEVICE"]


@pytest.mark.parametrize("B,H,N,d", [(1, 1, 1, 64), (2, 3, 129, 128), (8, 12, 1024, 64), (4, 16, 8192, 64)])
def test_workspace_size_formula(lib, B, H, N, d):
    npad = (N + 127) // 128 * 128

    def up(x):
        return (x + 255) // 256 * 256

    # tile counter, one 4 KB statistics tile per 128-row query block, float32 dQ accumulator
    expect = 256 + up(B * H * (npad // 128) * 4096) + up(B * H * N * d * 4)
    assert lib.fa_bwd_workspace_size(B, H, N, d) == expect
    assert lib.fa_bwd_workspace_size(0, H, N, d) == 0
    assert lib.fa_bwd_workspace_size(B, H, N, 80) == 0


def test_workloads_table_matches_the_stated_shapes():
    assert WORKLOADS["c2_gpt2s"]["B"] * WORKLOADS["c2_gpt2s"]["H"] == 96
    for name, w in WORKLOADS.items():
        if name.startswith("c5_"):
            assert w["B"] * w["N"] == 65536 and w["mult"] == 3.0


def test_noalloc_validates_like_fa_bwd_and_checks_its_limit(lib):
    """fa_bwd_noalloc reports fa_bwd's validation errors, refuses sizes beyond its
    built-in scratch array, and without a GPU stops at the device check."""
    C = binding.STATUS_CODE

    def call(B=1, H=1, N=128, d=64, dtype=0, q=P, scale=0.125):
        return lib.fa_bwd_noalloc(q, P, P, P, P, P, P, P, P, B, H, N, d, scale, 0, dtype, NULL)

    assert call(dtype=3) == C["FA_ERR_DTYPE"]
    assert call(d=48) == C["FA_ERR_UNSUPPORTED_D"]
    assert call(q=NULL) == C["FA_ERR_NULL"]
    assert call(q=PM) == C["FA_ERR_ALIGN"]
    assert call(scale=-2.0) == C["FA_ERR_SCALE"]
    assert call(B=2, H=16, N=4096) == C["FA_ERR_SCRATCH_LIMIT"]
    assert lib.fa_bwd_workspace_size(2, 16, 4096, 64) > lib.fa_bwd_noalloc_max_scratch() == 32 << 20
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except ImportError:
        has_gpu = False
    if not has_gpu:
        assert call() == C["FA_ERR_NO_DEVICE"]


def test_no_cpu_fallback():
    """The product path has no CPU route: a missing library raises, and host tensors are
    refused before any compute."""
    torch = pytest.importorskip("torch")
    with pytest.raises(RuntimeError, match="not found"):
        binding.load_library(os.path.join(ROOT, "no_such_dir", "libfa_gb300.so"))
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.forward(q, q, q)
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.backward(q, q, q, q, q, torch.zeros(1, 1, 128))
