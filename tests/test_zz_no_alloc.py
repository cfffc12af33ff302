"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Callers such as a plugin host that only hands over the tensors to work on, or code
running under a caching allocator that already owns the device's memory, cannot
provide fa_bwd's workspace.  fa_bwd_noalloc keeps its scratch in a fixed array inside
the library instead.  These tests call it through the C ABI and check its dq, dk, dv
against fa_bwd's (the entry point with a caller workspace) on two calls in a row --
the second call reuses the array exactly as the first left it -- within the gradient
tolerance of the other parity tests.

This file is collected last on purpose, so that a run that stops at the first
failure has already run every other test; it also passes when run on its own.
"""

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from exact_tiled_attention_27_gb300 import binding, build, forward  # noqa: E402
from exact_tiled_attention_27_gb300.inputs import make_case  # noqa: E402
from tests import gpu_util as G  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    return binding.load_library()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("B,H,N,d,dtype,causal", [(2, 3, 300, 64, "bf16", True), (1, 4, 257, 128, "fp16", False)])
def test_noalloc_matches_workspace_backward_twice(lib, B, H, N, d, dtype, causal):
    case = make_case(B, H, N, d, dtype, causal, workload_index=95, length_index=d // 64)
    q, k, v, do = (G.to_device(getattr(case, n), dtype) for n in ("q", "k", "v", "do"))
    o, lse = forward(q, k, v, scale=case.scale, causal=causal)
    code = binding.FA_BF16 if dtype == "bf16" else binding.FA_FP16
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    c = 1 if causal else 0

    # the existing entry point, with a workspace the caller allocated
    ref = [torch.empty_like(q) for _ in range(3)]
    ws_bytes = lib.fa_bwd_workspace_size(B, H, N, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    st = lib.fa_bwd(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(ref[0]), _p(ref[1]), _p(ref[2]), _p(ws),
                    ws_bytes, B, H, N, d, case.scale, c, code, stream)
    assert st == 0, binding.strerror(st)
    torch.cuda.synchronize()
    ref64 = [G.to_f64(t) for t in ref]

    for call in range(2):
        out = [torch.full_like(q, float("nan")) for _ in range(3)]
        st = lib.fa_bwd_noalloc(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(out[0]), _p(out[1]), _p(out[2]),
                                B, H, N, d, case.scale, c, code, stream)
        assert st == 0, binding.strerror(st)
        assert binding.last_kernel_status() == 0
        got = [G.to_f64(t) for t in out]
        for name, g, r in zip(("dq", "dk", "dv"), got, ref64):
            assert np.all(np.isfinite(g)), f"call {call}: {name} not finite"
            err = G.rel_l2(g, r)
            print(f"call {call} {name}: relL2 vs fa_bwd = {err:.2e}")
            assert err <= G.GRAD_RELL2, f"call {call}: {name} relL2 {err:.3e}"
        # dk and dv involve no atomics: they must be identical to fa_bwd's
        assert np.array_equal(got[1], ref64[1]) and np.array_equal(got[2], ref64[2])


def test_noalloc_rejects_sizes_beyond_its_array(lib):
    """A problem whose scratch exceeds the built-in array is refused before any launch,
    and the output buffers are left untouched."""
    B, H, N, d = 2, 16, 4096, 64            # needs ~34 MB > 32 MiB
    assert lib.fa_bwd_workspace_size(B, H, N, d) > lib.fa_bwd_noalloc_max_scratch()
    t = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((B, H, N), dtype=torch.float32, device="cuda")
    outs = [torch.full_like(t, 7.0) for _ in range(3)]
    st = lib.fa_bwd_noalloc(_p(t), _p(t), _p(t), _p(t), _p(t), _p(lse), _p(outs[0]), _p(outs[1]), _p(outs[2]),
                            B, H, N, d, 0.125, 1, binding.FA_BF16,
                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == binding.STATUS_CODE["FA_ERR_SCRATCH_LIMIT"]
    torch.cuda.synchronize()
    for x in outs:
        assert bool(torch.all(x == 7.0))
