"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle on the
same seeded 16-bit inputs, element by element.

Small shapes cover tile boundaries and ragged tails (N in {1, 17, 127, 128, 129, 255,
256, 383}), both head sizes, both 16-bit types, causal on and off, and inputs scaled
by 3 (frequent moves of the running maximum).  The workload shapes follow in
test_gpu_workloads.py.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from exact_tiled_attention_27_gb300 import backward, build, forward  # noqa: E402
from exact_tiled_attention_27_gb300.inputs import make_case  # noqa: E402
from tests import gpu_util as G  # noqa: E402

pytestmark = pytest.mark.gpu

SMALL_N = [1, 17, 127, 128, 129, 255, 256, 383]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()


def run_and_check(case, with_bwd=True, label=""):
    q, k, v = (G.to_device(getattr(case, n), case.dtype) for n in ("q", "k", "v"))
    o, lse = forward(q, k, v, scale=case.scale, causal=case.causal)
    torch.cuda.synchronize()
    q64, k64, v64 = case.f64("q"), case.f64("k"), case.f64("v")
    o_ref, lse_ref = oracle.attn_fwd_ref(q64, k64, v64, case.scale, case.causal)
    pv_abs, _ = oracle.attn_fwd_ref(q64, k64, np.abs(v64), case.scale, case.causal)
    G.check_forward(G.to_f64(o), G.to_f64(lse), o_ref, lse_ref, label, case.dtype, pv_abs)
    if not with_bwd:
        return
    do = G.to_device(case.do, case.dtype)
    dq, dk, dv = backward(q, k, v, o, do, lse, scale=case.scale, causal=case.causal)
    torch.cuda.synchronize()
    refs = oracle.attn_bwd_ref(q64, k64, v64, case.f64("do"), case.scale, case.causal)[:3]
    G.check_backward([G.to_f64(x) for x in (dq, dk, dv)], refs, label)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", SMALL_N)
def test_small_shapes(N, d, causal, dtype):
    case = make_case(1, 2, N, d, dtype, causal, workload_index=90, length_index=N % 97)
    run_and_check(case, True, f"N={N} d={d} causal={causal} {dtype}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [129, 383, 640])
def test_scaled_inputs_move_the_maximum(N, d, causal):
    """Inputs x3: logits with std ~9 move the running maximum often."""
    case = make_case(2, 2, N, d, "bf16", causal, workload_index=91, length_index=N % 89, mult=3.0)
    run_and_check(case, True, f"x3 N={N} d={d} causal={causal}")


@pytest.mark.parametrize("scale", [0.01, 0.3, 1.0])
def test_explicit_scale(scale):
    case = make_case(1, 3, 200, 64, "bf16", True, scale=scale, workload_index=92)
    run_and_check(case, True, f"scale={scale}")


def test_many_heads_persistent_loop():
    """More tiles than SMs: every CTA walks several tiles of the persistent loop."""
    case = make_case(3, 40, 300, 64, "bf16", True, workload_index=93)
    run_and_check(case, True, "B=3 H=40 N=300")


def test_large_logits_do_not_overflow():
    """Scores of several hundred: the running maximum keeps exp finite."""
    case = make_case(1, 2, 256, 64, "fp16", False, scale=4.0, workload_index=94, mult=3.0)
    run_and_check(case, False, "scale=4 x3")


@pytest.mark.parametrize("N,causal,dtype", [(3001, False, "bf16"), (6001, True, "fp16")])
def test_long_tiles_wide_dq_staging(N, causal, dtype):
    """d = 64 with 24 or more query blocks per key tile: the backward stages dQ in
    32-column chunks (one per warp) instead of 16-column ones; ragged last block."""
    case = make_case(1, 2, N, 64, dtype, causal, workload_index=95, length_index=N % 83)
    run_and_check(case, True, f"wide dQ N={N} causal={causal} {dtype}")
