"""GPU parity of fa_fwd_cross: Nq != Nk (causal mask aligned bottom-right), grouped
key/value heads, and rows that see no key, against the float64 oracle on the same
seeded 16-bit inputs (every head, every row).  Tolerances are those of tests/gpu_util.py;
rows with no visible key must be exactly O = 0 and lse = -inf."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from exact_tiled_attention_27_gb300 import backward, build, forward, forward_cross, last_kernel_status  # noqa: E402
from exact_tiled_attention_27_gb300.inputs import bits_to_f64, make_case, make_cross_case  # noqa: E402
from tests import gpu_util as G  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()


CASES = [
    # B, H, Hkv, Nq, Nk, d, dtype, causal
    (1, 2, 2, 77, 300, 64, "bf16", True),      # fewer queries than keys, ragged both
    (1, 2, 2, 300, 77, 64, "bf16", True),      # more queries than keys: 223 rows see no key
    (1, 2, 2, 300, 77, 64, "bf16", False),
    (2, 4, 1, 128, 640, 128, "fp16", True),    # one key/value head for four query heads
    (1, 8, 2, 513, 1000, 64, "bf16", False),   # grouped heads, non-causal
    (2, 6, 3, 200, 450, 64, "fp16", True),     # grouped heads, causal
    (1, 3, 3, 1, 1000, 64, "bf16", True),      # a single query row against 1000 keys
    (1, 4, 2, 5, 129, 128, "bf16", True),
    (1, 2, 1, 1000, 3, 64, "bf16", True),      # 997 rows see no key
]


def _run_cross(c):
    q = G.to_device(c.q, c.dtype)
    k = G.to_device(c.k, c.dtype)
    v = G.to_device(c.v, c.dtype)
    o, lse = forward_cross(q, k, v, scale=c.scale, causal=c.causal)
    torch.cuda.synchronize()
    assert last_kernel_status() == 0
    return G.to_f64(o), G.to_f64(lse)


@pytest.mark.parametrize("B,H,Hkv,Nq,Nk,d,dtype,causal", CASES)
def test_cross_matches_oracle(B, H, Hkv, Nq, Nk, d, dtype, causal):
    c = make_cross_case(B, H, Hkv, Nq, Nk, d, dtype, causal, workload_index=200, length_index=Nq * 7 + Nk)
    o, lse = _run_cross(c)
    o_ref, lse_ref = oracle.attn_cross_fwd_ref(bits_to_f64(c.q, dtype), bits_to_f64(c.k, dtype),
                                               bits_to_f64(c.v, dtype), c.scale, causal)
    dead = np.isneginf(lse_ref)
    if dead.any():
        assert np.all(np.isneginf(lse[dead])), "rows with no visible key must have lse = -inf"
        assert np.all(o[dead] == 0.0), "rows with no visible key must have O = 0"
    live = ~dead
    G.check_forward(o[live], lse[live], o_ref[live], lse_ref[live], f"cross B{B} H{H}/{Hkv} {Nq}x{Nk} d{d}", dtype)


@pytest.mark.parametrize("causal", [True, False])
def test_square_cross_is_bitwise_fwd(causal):
    c = make_case(2, 3, 333, 64, "bf16", causal, workload_index=201)
    q, k, v = (G.to_device(getattr(c, n), "bf16") for n in ("q", "k", "v"))
    o1, l1 = forward(q, k, v, causal=causal)
    o2, l2 = forward_cross(q, k, v, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_grouped_heads_equal_repeated_heads():
    """Hkv < H gives bitwise the result of fa_fwd on K/V heads repeated per group."""
    c = make_cross_case(2, 8, 2, 384, 384, 64, "bf16", True, workload_index=202)
    q = G.to_device(c.q, "bf16")
    k = G.to_device(c.k, "bf16")
    v = G.to_device(c.v, "bf16")
    o1, l1 = forward_cross(q, k, v, causal=True)
    o2, l2 = forward(q, k.repeat_interleave(4, dim=1).contiguous(), v.repeat_interleave(4, dim=1).contiguous(),
                     causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


GQA_BWD_CASES = [
    # B, H, Hkv, N, d, dtype, causal
    (1, 4, 2, 300, 64, "bf16", True),
    (2, 6, 3, 256, 64, "fp16", False),
    (1, 8, 1, 200, 128, "bf16", True),
    (1, 4, 4, 129, 128, "fp16", True),    # Hkv = H: the same call takes the ordinary path
]


@pytest.mark.parametrize("B,H,Hkv,N,d,dtype,causal", GQA_BWD_CASES)
def test_grouped_backward_matches_oracle(B, H, Hkv, N, d, dtype, causal):
    c = make_cross_case(B, H, Hkv, N, N, d, dtype, causal, workload_index=203, length_index=N + H)
    q, k, v, do = (G.to_device(getattr(c, n), dtype) for n in ("q", "k", "v", "do"))
    o, lse = forward_cross(q, k, v, scale=c.scale, causal=causal)
    dq, dk, dv = backward(q, k, v, o, do, lse, scale=c.scale, causal=causal)
    torch.cuda.synchronize()
    assert last_kernel_status() == 0
    q64, k64, v64, do64 = (bits_to_f64(getattr(c, n), dtype) for n in ("q", "k", "v", "do"))
    refs = oracle.attn_gqa_bwd_ref(q64, k64, v64, do64, c.scale, causal)
    for b in range(B):
        for hk in range(Hkv):
            G.check_backward([np.zeros(1), G.to_f64(dk[b, hk]), G.to_f64(dv[b, hk])],
                             [np.zeros(1), refs[1][b, hk], refs[2][b, hk]], f"gqa dK/dV ({b},{hk})")
        for h in range(H):
            err = G.rel_l2(G.to_f64(dq[b, h]), refs[0][b, h])
            assert err <= G.GRAD_RELL2, f"dQ ({b},{h}) relL2 {err:.3e}"
