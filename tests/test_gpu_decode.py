"""GPU parity of fa_decode (split-key decode, CUDA cores) against the float64 oracle:
one to eight query rows per key/value head, grouped heads, one key range and many,
the bottom-right causal mask with several new tokens, and rows that see no key.
Tolerances are those of tests/gpu_util.py."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from exact_tiled_attention_27_gb300 import build, decode, decode_workspace_size, forward_cross  # noqa: E402
from exact_tiled_attention_27_gb300 import last_kernel_status  # noqa: E402
from exact_tiled_attention_27_gb300.inputs import bits_to_f64, make_cross_case  # noqa: E402
from tests import gpu_util as G  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()


CASES = [
    # B, H, Hkv, Nq, Nk, d, dtype, causal
    (1, 4, 4, 1, 100, 64, "fp16", True),       # one row per head, one key range
    (2, 8, 2, 1, 5000, 128, "bf16", True),     # 4 rows per key/value head, many ranges
    (2, 32, 4, 1, 3000, 64, "bf16", True),     # 8 rows per key/value head
    (1, 2, 2, 3, 777, 64, "bf16", True),       # three new tokens: the mask matters
    (1, 2, 1, 4, 20000, 128, "fp16", True),    # 8 rows, 78 ranges
    (1, 1, 1, 8, 5, 64, "bf16", True),         # Nk < Nq: three rows see no key
    (3, 6, 3, 2, 1111, 64, "fp16", False),
    # d = 128 runs the TMA-fed kernel: partial stages, the mask, rows that see no key,
    # ranges of many stages
    (1, 4, 4, 1, 100, 128, "fp16", True),
    (1, 2, 2, 3, 777, 128, "bf16", True),
    (1, 1, 1, 8, 5, 128, "bf16", True),
    (3, 6, 3, 2, 1111, 128, "fp16", False),
    (2, 8, 8, 1, 40000, 128, "bf16", True),
]


@pytest.mark.parametrize("B,H,Hkv,Nq,Nk,d,dtype,causal", CASES)
def test_decode_matches_oracle(B, H, Hkv, Nq, Nk, d, dtype, causal):
    c = make_cross_case(B, H, Hkv, Nq, Nk, d, dtype, causal, workload_index=210, length_index=Nk + 13 * Nq)
    q, k, v = (G.to_device(getattr(c, n), dtype) for n in ("q", "k", "v"))
    o, lse = decode(q, k, v, scale=c.scale, causal=causal)
    torch.cuda.synchronize()
    assert last_kernel_status() == 0
    o, lse = G.to_f64(o), G.to_f64(lse)
    o_ref, lse_ref = oracle.attn_cross_fwd_ref(bits_to_f64(c.q, dtype), bits_to_f64(c.k, dtype),
                                               bits_to_f64(c.v, dtype), c.scale, causal)
    dead = np.isneginf(lse_ref)
    if dead.any():
        assert np.all(np.isneginf(lse[dead])) and np.all(o[dead] == 0.0)
    live = ~dead
    G.check_forward(o[live], lse[live], o_ref[live], lse_ref[live], f"decode B{B} H{H}/{Hkv} {Nq}x{Nk} d{d}", dtype)


@pytest.mark.parametrize("d", [64, 128])
def test_decode_agrees_with_tile_forward_and_is_repeatable(d):
    c = make_cross_case(4, 16, 2, 1, 9000, d, "bf16", True, workload_index=211)
    q, k, v = (G.to_device(getattr(c, n), "bf16") for n in ("q", "k", "v"))
    ws = torch.empty(decode_workspace_size(4, 16, 2, 1, 9000, d), dtype=torch.uint8, device="cuda")
    o1, l1 = decode(q, k, v, causal=True, workspace=ws)
    o2, l2 = decode(q, k, v, causal=True, workspace=ws)
    o3, l3 = forward_cross(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert (o1.float() - o3.float()).abs().max().item() <= 2e-2
    assert (l1 - l3).abs().max().item() <= 1e-3
