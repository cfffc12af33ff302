"""GPU parity of the butterfly block-sparse forward and backward (fa_fwd_sparse,
fa_bwd_sparse) against the float64 oracle's masked attention on the same seeded inputs:
whole heads, several pair counts (powers of two and not), ragged N, causal and not.
Tolerances are those of tests/gpu_util.py."""

import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from exact_tiled_attention_27_gb300 import backward, build, forward, last_kernel_status  # noqa: E402
from exact_tiled_attention_27_gb300.inputs import bits_to_f64, make_case  # noqa: E402
from tests import gpu_util as G  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()


CASES = [
    # B, H, N, d, dtype, causal
    (1, 2, 1024, 64, "bf16", False),     # 4 pairs
    (1, 2, 1024, 64, "bf16", True),
    (1, 2, 2048, 128, "fp16", True),     # 8 pairs
    (2, 1, 1500, 64, "bf16", False),     # 12 blocks (6 pairs, not a power of two), ragged tail
    (1, 1, 1700, 128, "bf16", True),     # 14 blocks, ragged tail
    (1, 1, 1300, 64, "fp16", True),      # 11 blocks: the last pair holds one block
    (1, 3, 200, 64, "bf16", True),       # a single pair: dense
]


@pytest.mark.parametrize("B,H,N,d,dtype,causal", CASES)
def test_butterfly_matches_oracle(B, H, N, d, dtype, causal):
    c = make_case(B, H, N, d, dtype, causal, workload_index=220, length_index=N + d)
    q, k, v, do = (G.to_device(getattr(c, n), dtype) for n in ("q", "k", "v", "do"))
    o, lse = forward(q, k, v, scale=c.scale, causal=causal, pattern="butterfly")
    dq, dk, dv = backward(q, k, v, o, do, lse, scale=c.scale, causal=causal, pattern="butterfly")
    torch.cuda.synchronize()
    assert last_kernel_status() == 0
    mask = oracle.butterfly_mask(N, N, causal)
    for b in range(B):
        for h in range(H):
            f = lambda name: bits_to_f64(getattr(c, name)[b, h], dtype)  # noqa: E731
            o_ref, lse_ref = oracle.attn_masked_head_fwd(f("q"), f("k"), f("v"), c.scale, mask)
            G.check_forward(G.to_f64(o[b, h]), G.to_f64(lse[b, h]), o_ref, lse_ref, f"butterfly N{N} ({b},{h})", dtype)
            refs = oracle.attn_masked_head_bwd(f("q"), f("k"), f("v"), f("do"), c.scale, mask)
            G.check_backward([G.to_f64(x[b, h]) for x in (dq, dk, dv)], refs, f"butterfly N{N} ({b},{h})")


def test_single_pair_is_dense():
    """With at most 256 keys the pattern is one block: the sparse and the dense kernels
    both give the dense causal result.  (They need not agree bit for bit: a launch this
    small runs the dense forward with each query block's keys split between the two
    sub-tiles and merged.)"""
    c = make_case(1, 4, 250, 64, "bf16", True, workload_index=221)
    q, k, v = (G.to_device(getattr(c, n), "bf16") for n in ("q", "k", "v"))
    o1, l1 = forward(q, k, v, causal=True, pattern="butterfly")
    o2, l2 = forward(q, k, v, causal=True)
    torch.cuda.synchronize()
    for h in range(4):
        f = lambda name: bits_to_f64(getattr(c, name)[0, h], "bf16")  # noqa: E731
        o_ref, lse_ref = oracle.attn_head_fwd(f("q"), f("k"), f("v"), c.scale, True)
        for o, lse, label in ((o1, l1, "butterfly"), (o2, l2, "dense")):
            G.check_forward(G.to_f64(o[0, h]), G.to_f64(lse[0, h]), o_ref, lse_ref, f"{label} N250 head {h}", "bf16")
