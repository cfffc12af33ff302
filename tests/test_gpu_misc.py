"""GPU checks beyond element-wise parity: the bounded-wait timeout path, bitwise
repeatability of the forward, guard bands around every output, and invariance of
non-causal attention under a joint permutation of the key/value rows."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from exact_tiled_attention_27_gb300 import (STATUS_CODE, backward, build, debug_wait_timeout,  # noqa: E402
                                            forward, last_kernel_status)
from exact_tiled_attention_27_gb300.inputs import make_case  # noqa: E402
from tests import gpu_util as G  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()


def test_bounded_wait_reports_timeout_and_context_survives():
    """A kernel waits on an mbarrier nobody arrives on, with a 2 ms bound: it gives up,
    records the timeout and returns; the next launches run normally."""
    assert last_kernel_status() == 0
    assert debug_wait_timeout(2000) == 0
    assert last_kernel_status() == STATUS_CODE["FA_ERR_DEVICE_TIMEOUT"]
    assert last_kernel_status() == 0          # reading clears the word
    case = make_case(1, 1, 130, 64, "bf16", True, workload_index=96)
    q, k, v = (G.to_device(getattr(case, n), "bf16") for n in ("q", "k", "v"))
    o, lse = forward(q, k, v, causal=True)
    assert last_kernel_status() == 0
    assert bool(torch.isfinite(o.float()).all())


@pytest.mark.parametrize("d", [64, 128])
def test_forward_is_bitwise_repeatable(d):
    case = make_case(2, 4, 777, d, "bf16", True, workload_index=97)
    q, k, v = (G.to_device(getattr(case, n), "bf16") for n in ("q", "k", "v"))
    o1, l1 = forward(q, k, v, causal=True)
    o2, l2 = forward(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def _banded(shape, dtype, fill):
    """A view of `shape` inside a larger buffer with 4 KiB sentinel bands on each side."""
    n = int(np.prod(shape))
    per = 4096 // torch.tensor([], dtype=dtype).element_size()
    buf = torch.full((n + 2 * per,), fill, dtype=dtype, device="cuda")
    return buf, buf[per:per + n].view(shape), per


@pytest.mark.parametrize("d", [64, 128])
def test_outputs_stay_inside_their_buffers(d):
    B, H, N = 1, 3, 201
    case = make_case(B, H, N, d, "bf16", True, workload_index=98)
    q, k, v, do = (G.to_device(getattr(case, n), "bf16") for n in ("q", "k", "v", "do"))
    o_buf, o, o_per = _banded((B, H, N, d), torch.bfloat16, 3.0)
    l_buf, lse, l_per = _banded((B, H, N), torch.float32, 5.0)
    forward(q, k, v, causal=True, out=o, lse=lse)
    outs = [_banded((B, H, N, d), torch.bfloat16, 9.0) for _ in range(3)]
    backward(q, k, v, o, do, lse, causal=True, dq=outs[0][1], dk=outs[1][1], dv=outs[2][1])
    torch.cuda.synchronize()
    assert last_kernel_status() == 0
    for buf, fill, per in [(o_buf, 3.0, o_per), (l_buf, 5.0, l_per)] + [(b, 9.0, p) for b, _, p in outs]:
        assert bool((buf[:per] == fill).all()) and bool((buf[-per:] == fill).all())


def test_noncausal_invariant_under_joint_kv_permutation():
    case = make_case(1, 2, 300, 64, "fp16", False, workload_index=99)
    q, k, v = (G.to_device(getattr(case, n), "fp16") for n in ("q", "k", "v"))
    perm = torch.randperm(300, generator=torch.Generator().manual_seed(5)).cuda()
    o1, l1 = forward(q, k, v)
    o2, l2 = forward(q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous())
    torch.cuda.synchronize()
    d_o = (o1.float() - o2.float()).abs().max().item()
    d_l = (l1 - l2).abs().max().item()
    print(f"max |dO| {d_o:.2e}, max |dlse| {d_l:.2e}")
    assert d_o <= 2e-2 and d_l <= 1e-3
