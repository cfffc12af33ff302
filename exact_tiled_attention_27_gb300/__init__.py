"""Exact tiled attention for GB300 (sm_103a).

O = softmax(scale * Q K^T) V computed tile by tile with the streaming softmax rescale
(the score matrix never reaches device memory), plus the backward pass that
recomputes P on chip.  The computation lives in the CUDA library built from
``csrc/`` (C ABI in ``include/fa.h``); this package is the thin Python binding.

    from exact_tiled_attention_27_gb300 import forward, backward
    o, lse = forward(q, k, v, causal=True)
    dq, dk, dv = backward(q, k, v, o, do, lse, causal=True)
"""

from .binding import (  # noqa: F401
    FA_BF16,
    FA_FP16,
    STATUS,
    STATUS_CODE,
    FaError,
    backward,
    debug_wait_timeout,
    decode,
    decode_workspace_size,
    device_sm_count,
    forward,
    forward_cross,
    forward_fp8,
    fp8_vt_cols,
    quantize_fp8,
    last_kernel_status,
    load_library,
    strerror,
    workspace_size,
)
