"""Python binding of the C ABI in include/fa.h: argument marshalling only.

Every step of the attention computation runs in the CUDA kernels of
``lib/libfa_gb300.so``; this module checks torch tensors, passes their device
pointers and the current CUDA stream to the library, and turns status codes into
exceptions.  There is no fallback: if the library is missing or the device is not an
sm_100-family GPU, the call raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "lib", "libfa_gb300.so")

FA_BF16, FA_FP16 = 0, 1
STATUS = {
    0: "FA_OK", 1: "FA_ERR_NULL", 2: "FA_ERR_SHAPE", 3: "FA_ERR_UNSUPPORTED_D", 4: "FA_ERR_DTYPE",
    5: "FA_ERR_ALIGN", 6: "FA_ERR_WORKSPACE", 7: "FA_ERR_LAUNCH", 8: "FA_ERR_DEVICE_TIMEOUT",
    9: "FA_ERR_NO_DEVICE", 10: "FA_ERR_SCALE", 11: "FA_ERR_SCRATCH_LIMIT", 12: "FA_ERR_PATTERN",
}
STATUS_CODE = {v: k for k, v in STATUS.items()}

_lib = None
_lock = threading.Lock()


class FaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({strerror(status)})")


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"CUDA library not found at {p}; build it with "
                "`python -m exact_tiled_attention_27_gb300.build`")
        lib = ctypes.CDLL(p)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
        lib.fa_fwd.restype = i
        lib.fa_fwd_sparse.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, i, vp]
        lib.fa_fwd_sparse.restype = i
        lib.fa_bwd_sparse.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, f, i, i, i, vp]
        lib.fa_bwd_sparse.restype = i
        lib.fa_butterfly_blocks.argtypes = [i, i, i, ctypes.POINTER(ctypes.c_int), i]
        lib.fa_butterfly_blocks.restype = i
        lib.fa_fwd_cross.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp]
        lib.fa_fwd_cross.restype = i
        lib.fa_bwd_workspace_size.argtypes = [i, i, i, i]
        lib.fa_bwd_workspace_size.restype = sz
        lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, f, i, i, vp]
        lib.fa_bwd.restype = i
        for name in ("fa_bwd_preprocess", "fa_bwd_dkdv", "fa_bwd_dq_convert"):
            fn = getattr(lib, name)
            fn.argtypes = lib.fa_bwd.argtypes
            fn.restype = i
        lib.fa_decode_workspace_size.argtypes = [i, i, i, i, i, i]
        lib.fa_decode_workspace_size.restype = sz
        lib.fa_decode.argtypes = [vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, i, f, i, i, vp]
        lib.fa_decode.restype = i
        lib.fa_bwd_gqa.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, f, i, i, vp]
        lib.fa_bwd_gqa.restype = i
        lib.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
        lib.fa_bwd_noalloc.restype = i
        lib.fa_bwd_noalloc_max_scratch.argtypes = []
        lib.fa_bwd_noalloc_max_scratch.restype = sz
        lib.fa_fp8_vt_cols.argtypes = [i]
        lib.fa_fp8_vt_cols.restype = i
        lib.fa_quantize_fp8.argtypes = [vp, vp, vp, i, i, i, i, i, vp, i, i, vp]
        lib.fa_quantize_fp8.restype = i
        lib.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
        lib.fa_fwd_fp8.restype = i
        lib.fa_strerror.argtypes = [i]
        lib.fa_strerror.restype = ctypes.c_char_p
        lib.fa_get_last_kernel_status.argtypes = [vp]
        lib.fa_get_last_kernel_status.restype = i
        lib.fa_device_sm_count.argtypes = []
        lib.fa_device_sm_count.restype = i
        lib.fa_debug_wait_timeout.argtypes = [ctypes.c_uint, vp]
        lib.fa_debug_wait_timeout.restype = i
        if path is None:
            _lib = lib
        return lib


def strerror(status: int) -> str:
    try:
        return load_library().fa_strerror(int(status)).decode()
    except Exception:  # library missing: still give the symbolic name
        return STATUS.get(int(status), "unknown")


# ----------------------------------------------------------------------------- torch glue
def _torch():
    import torch
    return torch


def _dtype_code(t):
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return FA_BF16
    if t.dtype == torch.float16:
        return FA_FP16
    raise TypeError(f"expected bfloat16 or float16 tensors, got {t.dtype}")


def _check_bhnd(name, t, shape, dtype):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (batch, heads, seq, head_dim)")


def _stream_handle(stream=None):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def workspace_size(B, H, N, d) -> int:
    return int(load_library().fa_bwd_workspace_size(B, H, N, d))


PATTERNS = {"butterfly": 1}


def forward(q, k, v, scale=None, causal=False, out=None, lse=None, stream=None, pattern=None):
    """Exact attention forward.  q, k, v: (B, H, N, d) bf16/fp16 CUDA tensors.

    Returns (o, lse): o like q, lse float32 (B, H, N), natural-log row log-sum-exp
    of scale * q k^T.  ``scale`` defaults to d ** -0.5.  Runs on the current stream.
    ``pattern="butterfly"`` restricts attention to the butterfly block pattern
    (fa_fwd_sparse).
    """
    torch = _torch()
    B, H, N, d = q.shape
    _check_bhnd("q", q, (B, H, N, d), q.dtype)
    _check_bhnd("k", k, (B, H, N, d), q.dtype)
    _check_bhnd("v", v, (B, H, N, d), q.dtype)
    scale = float(d) ** -0.5 if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check_bhnd("out", out, (B, H, N, d), q.dtype)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 (B, H, N) tensor")
    if pattern is not None:
        st = load_library().fa_fwd_sparse(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d, scale,
                                          1 if causal else 0, PATTERNS[pattern], _dtype_code(q),
                                          _stream_handle(stream))
        if st != 0:
            raise FaError(st, "fa_fwd_sparse")
        return out, lse
    st = load_library().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d, scale,
                               1 if causal else 0, _dtype_code(q), _stream_handle(stream))
    if st != 0:
        raise FaError(st, "fa_fwd")
    return out, lse


def forward_cross(q, k, v, scale=None, causal=False, out=None, lse=None, stream=None):
    """Forward with Nq != Nk and grouped key/value heads.  q: (B, H, Nq, d); k, v:
    (B, Hkv, Nk, d) with Hkv dividing H.  The causal mask is aligned bottom-right
    (query i sees key j iff j <= i + Nk - Nq).  Returns (o, lse) like ``forward``.
    """
    torch = _torch()
    B, H, Nq, d = q.shape
    Hkv, Nk = int(k.shape[1]), int(k.shape[2])
    _check_bhnd("q", q, (B, H, Nq, d), q.dtype)
    _check_bhnd("k", k, (B, Hkv, Nk, d), q.dtype)
    _check_bhnd("v", v, (B, Hkv, Nk, d), q.dtype)
    scale = float(d) ** -0.5 if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    _check_bhnd("out", out, (B, H, Nq, d), q.dtype)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, Nq) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 (B, H, Nq) tensor")
    st = load_library().fa_fwd_cross(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Hkv, Nq, Nk, d,
                                     scale, 1 if causal else 0, _dtype_code(q), _stream_handle(stream))
    if st != 0:
        raise FaError(st, "fa_fwd_cross")
    return out, lse


def decode(q, k, v, scale=None, causal=True, out=None, lse=None, workspace=None, stream=None):
    """Split-key decode for a few query rows: q (B, H, Nq, d), k, v (B, Hkv, Nk, d)
    with (H / Hkv) * Nq <= 8.  Same result as ``forward_cross``; returns (o, lse).
    ``workspace`` (optional) is a CUDA uint8 tensor of at least
    ``decode_workspace_size(...)`` bytes."""
    torch = _torch()
    B, H, Nq, d = q.shape
    Hkv, Nk = int(k.shape[1]), int(k.shape[2])
    _check_bhnd("q", q, (B, H, Nq, d), q.dtype)
    _check_bhnd("k", k, (B, Hkv, Nk, d), q.dtype)
    _check_bhnd("v", v, (B, Hkv, Nk, d), q.dtype)
    scale = float(d) ** -0.5 if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    _check_bhnd("out", out, (B, H, Nq, d), q.dtype)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, Nq) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 (B, H, Nq) tensor")
    lib = load_library()
    need = int(lib.fa_decode_workspace_size(B, H, Hkv, Nq, Nk, d))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = _ptr(workspace) if workspace is not None else ctypes.c_void_p(0)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib.fa_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), ws_ptr, ws_bytes, B, H, Hkv, Nq, Nk, d,
                       scale, 1 if causal else 0, _dtype_code(q), _stream_handle(stream))
    if st != 0:
        raise FaError(st, "fa_decode")
    return out, lse


def decode_workspace_size(B, H, Hkv, Nq, Nk, d) -> int:
    return int(load_library().fa_decode_workspace_size(B, H, Hkv, Nq, Nk, d))


def backward(q, k, v, o, do, lse, scale=None, causal=False, dq=None, dk=None, dv=None, workspace=None,
             stream=None, stage=None, pattern=None):
    """Exact attention backward.  Returns (dq, dk, dv): dq like q, dk and dv like k.

    k and v may have fewer heads than q (grouped key/value heads, Hkv dividing H);
    dk and dv then sum over the query heads of each group.  ``workspace`` (optional)
    is a CUDA uint8 tensor of at least workspace_size(B,H,N,d) bytes; one is allocated
    through torch when it is not given.  ``stage`` runs one of the three launches of
    the backward ("preprocess", "dkdv", "dq_convert"; Hkv = H only); calling the three
    in order with the same workspace equals the default (all three).
    """
    torch = _torch()
    B, H, N, d = q.shape
    Hkv = int(k.shape[1])
    for name, t in (("q", q), ("o", o), ("do", do)):
        _check_bhnd(name, t, (B, H, N, d), q.dtype)
    for name, t in (("k", k), ("v", v)):
        _check_bhnd(name, t, (B, Hkv, N, d), q.dtype)
    if Hkv != H and stage is not None:
        raise ValueError("the single-stage calls take Hkv == H")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 (B, H, N) tensor")
    scale = float(d) ** -0.5 if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check_bhnd("dq", dq, (B, H, N, d), q.dtype)
    for name, t in (("dk", dk), ("dv", dv)):
        _check_bhnd(name, t, (B, Hkv, N, d), q.dtype)
    need = workspace_size(B, H, N, d)
    fn_name = {None: "fa_bwd", "preprocess": "fa_bwd_preprocess", "dkdv": "fa_bwd_dkdv",
               "dq_convert": "fa_bwd_dq_convert"}[stage]
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace too small: need {need} bytes")
    if pattern is not None:
        if Hkv != H or stage is not None:
            raise ValueError("the block pattern takes Hkv == H and the whole backward")
        st = load_library().fa_bwd_sparse(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                                          _ptr(dk), _ptr(dv), _ptr(workspace), need, B, H, N, d, scale,
                                          1 if causal else 0, PATTERNS[pattern], _dtype_code(q),
                                          _stream_handle(stream))
        if st != 0:
            raise FaError(st, "fa_bwd_sparse")
        return dq, dk, dv
    if Hkv != H:
        fn_name = "fa_bwd_gqa"
        st = load_library().fa_bwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk),
                                       _ptr(dv), _ptr(workspace), need, B, H, Hkv, N, d, scale, 1 if causal else 0,
                                       _dtype_code(q), _stream_handle(stream))
        if st != 0:
            raise FaError(st, fn_name)
        return dq, dk, dv
    fn = getattr(load_library(), fn_name)
    st = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
            _ptr(workspace), need, B, H, N, d, scale, 1 if causal else 0, _dtype_code(q), _stream_handle(stream))
    if st != 0:
        raise FaError(st, fn_name)
    return dq, dk, dv


def last_kernel_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status."""
    return int(load_library().fa_get_last_kernel_status(_stream_handle(stream)))


def device_sm_count() -> int:
    return int(load_library().fa_device_sm_count())


def debug_wait_timeout(limit_us: int, stream=None) -> int:
    return int(load_library().fa_debug_wait_timeout(int(limit_us), _stream_handle(stream)))


# ----------------------------------------------------------------------------- FP8 forward
def fp8_vt_cols(N) -> int:
    """Row length Nt (bytes) of the transposed V codes: N rounded up to 16."""
    return (int(N) + 15) // 16 * 16


def quantize_fp8(x, per_tensor=False, signs=None, transpose=False, stream=None):
    """E4M3 codes and per-128-row-block float32 scales of x (B, H, N, d) bf16/fp16
    (fa_quantize_fp8).  ``signs``: optional (d,) float32 CUDA tensor of +-1 -- rows are
    then rotated by diag(signs) H / sqrt(d) first (use the same signs for q and k).
    ``transpose=True`` gives the (B, H, d, Nt) V^T layout ``forward_fp8`` reads.

    Returns (codes uint8, scales float32 (B, H, ceil(N/128)))."""
    torch = _torch()
    B, H, N, d = x.shape
    _check_bhnd("x", x, (B, H, N, d), x.dtype)
    nb = (N + 127) // 128
    codes = torch.empty((B, H, d, fp8_vt_cols(N)) if transpose else (B, H, N, d), dtype=torch.uint8,
                        device=x.device)
    scales = torch.empty((B, H, nb), dtype=torch.float32, device=x.device)
    sp = None
    if signs is not None:
        if not signs.is_cuda or signs.dtype != torch.float32 or tuple(signs.shape) != (d,) or not signs.is_contiguous():
            raise ValueError("signs must be a contiguous float32 CUDA tensor of shape (d,)")
        sp = _ptr(signs)
    st = load_library().fa_quantize_fp8(_ptr(x), _ptr(codes), _ptr(scales), B, H, N, d, _dtype_code(x), sp,
                                        1 if per_tensor else 0, 1 if transpose else 0, _stream_handle(stream))
    if st != 0:
        raise FaError(st, "fa_quantize_fp8")
    return codes, scales


def forward_fp8(q8, k8, vt8, q_scale, k_scale, v_scale, scale=None, causal=False, out_dtype=None, out=None,
                lse=None, stream=None):
    """FP8 forward (fa_fwd_fp8): q8, k8 (B, H, N, d) and vt8 (B, H, d, Nt) uint8 E4M3 codes
    with (B, H, ceil(N/128)) float32 block scales, as made by ``quantize_fp8``.  ``scale``
    defaults to d ** -0.5.  Returns (o, lse): o (B, H, N, d) in ``out_dtype`` (bfloat16 by
    default), lse float32 (B, H, N)."""
    torch = _torch()
    B, H, N, d = q8.shape
    nb = (N + 127) // 128
    out_dtype = torch.bfloat16 if out_dtype is None else out_dtype
    _check_bhnd("q8", q8, (B, H, N, d), torch.uint8)
    _check_bhnd("k8", k8, (B, H, N, d), torch.uint8)
    _check_bhnd("vt8", vt8, (B, H, d, fp8_vt_cols(N)), torch.uint8)
    for name, t in (("q_scale", q_scale), ("k_scale", k_scale), ("v_scale", v_scale)):
        _check_bhnd(name, t, (B, H, nb), torch.float32)
    scale = float(d) ** -0.5 if scale is None else float(scale)
    if out is None:
        out = torch.empty((B, H, N, d), dtype=out_dtype, device=q8.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    _check_bhnd("out", out, (B, H, N, d), out_dtype)
    _check_bhnd("lse", lse, (B, H, N), torch.float32)
    st = load_library().fa_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(vt8), _ptr(q_scale), _ptr(k_scale), _ptr(v_scale),
                                   _ptr(out), _ptr(lse), B, H, N, d, scale, 1 if causal else 0, _dtype_code(out),
                                   _stream_handle(stream))
    if st != 0:
        raise FaError(st, "fa_fwd_fp8")
    return out, lse
