"""GPU parity at the workloads' full sizes, through the same entry points and launch
configuration that bench.py times (fa_fwd, then the three launches of fa_bwd).

Every tensor is computed in full on the GPU.  The float64 oracle then checks:
  * whole (b, h) heads -- all of them for the smallest workload, seeded samples
    (always including the first and last head) where a head is cheap enough;
  * at sequence lengths where a whole head is too costly in float64, seeded sampled
    query rows (O, lse, dQ are row-local) in two heads, plus two identities that hold
    exactly for every head at any size: sum_j dK_j = 0 (the rows of dS sum to zero)
    and sum_j dV_j = sum_i dO_i (the rows of P sum to one), checked in every head to
    the gradient tolerance relative to the head's Frobenius norm.
Tolerances are those of tests/gpu_util.py.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from exact_tiled_attention_27_gb300 import backward, build, forward  # noqa: E402
from exact_tiled_attention_27_gb300.inputs import SWEEP_N, WORKLOADS, bits_to_f64, workload_case  # noqa: E402
from tests import gpu_util as G  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()


def _run(case, with_bwd):
    q, k, v = (G.to_device(getattr(case, n), case.dtype) for n in ("q", "k", "v"))
    o, lse = forward(q, k, v, scale=case.scale, causal=case.causal)
    grads = None
    if with_bwd:
        do = G.to_device(case.do, case.dtype)
        grads = backward(q, k, v, o, do, lse, scale=case.scale, causal=case.causal)
    torch.cuda.synchronize()
    return o, lse, grads


def _heads(B, H, count, seed):
    pairs = {(0, 0), (B - 1, H - 1)}
    r = np.random.Generator(np.random.PCG64(seed))
    while len(pairs) < min(count, B * H):
        pairs.add((int(r.integers(B)), int(r.integers(H))))
    return sorted(pairs)


def _f64(case, name, b, h, rows=None):
    bits = getattr(case, name)[b, h]
    return bits_to_f64(bits if rows is None else bits[rows], case.dtype)


def _check_heads(case, o, lse, grads, heads, mult, label, row_block=None):
    for b, h in heads:
        q64, k64, v64 = _f64(case, "q", b, h), _f64(case, "k", b, h), _f64(case, "v", b, h)
        o_ref, lse_ref = oracle.attn_head_fwd(q64, k64, v64, case.scale, case.causal, row_block)
        G.check_forward(G.to_f64(o[b, h]), G.to_f64(lse[b, h]), o_ref, lse_ref, f"{label} head ({b},{h})", mult)
        if grads is not None:
            refs = oracle.attn_head_bwd(q64, k64, v64, _f64(case, "do", b, h), case.scale, case.causal, row_block)
            G.check_backward([G.to_f64(g[b, h]) for g in grads], refs[:3], f"{label} head ({b},{h})")


def _check_rows(case, o, lse, grads, heads, nrows, mult, label):
    r = np.random.Generator(np.random.PCG64(case.N))
    for b, h in heads:
        rows = np.unique(np.concatenate([[0, case.N - 1], r.integers(0, case.N, nrows)]))
        k64, v64 = _f64(case, "k", b, h), _f64(case, "v", b, h)
        q_rows = _f64(case, "q", b, h, rows)
        if grads is None:
            o_ref, lse_ref = oracle.attn_rows_ref(q_rows, rows, k64, v64, case.scale, case.causal)
        else:
            o_ref, lse_ref, dq_ref, _ = oracle.attn_rows_ref(q_rows, rows, k64, v64, case.scale, case.causal,
                                                              _f64(case, "do", b, h, rows))
        idx = torch.as_tensor(rows, device=o.device)
        G.check_forward(G.to_f64(o[b, h].index_select(0, idx)), G.to_f64(lse[b, h].index_select(0, idx)), o_ref,
                        lse_ref, f"{label} rows of head ({b},{h})", mult)
        if grads is not None:
            dq = G.to_f64(grads[0][b, h].index_select(0, idx))
            err = G.rel_l2(dq, dq_ref)
            print(f"{label} rows of head ({b},{h}): dQ relL2 {err:.3e}")
            assert err <= G.GRAD_RELL2


def _check_identities(case, grads, label):
    """sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i in every head (float32 sums on the GPU)."""
    dq, dk, dv = grads
    do = G.to_device(case.do, case.dtype).float()
    dk32, dv32 = dk.float(), dv.float()
    sum_dk = dk32.sum(dim=2)
    res_dv = dv32.sum(dim=2) - do.sum(dim=2)
    norm_dk = dk32.pow(2).sum(dim=(2, 3)).sqrt()
    norm_dv = dv32.pow(2).sum(dim=(2, 3)).sqrt()
    r_dk = (sum_dk.pow(2).sum(-1).sqrt() / norm_dk).max().item()
    r_dv = (res_dv.pow(2).sum(-1).sqrt() / norm_dv).max().item()
    print(f"{label}: max over heads |sum dK|/|dK| = {r_dk:.3e}, |sum dV - sum dO|/|dV| = {r_dv:.3e}")
    assert r_dk <= G.GRAD_RELL2 and r_dv <= G.GRAD_RELL2
    assert bool(torch.isfinite(dq).all())


def test_tiny_workload_full_oracle():
    case = workload_case("c1_tiny")
    o, lse, _ = _run(case, False)
    _check_heads(case, o, lse, None, [(0, 0)], 1.0, "c1")


def test_gpt2_small_workload():
    """B=8 H=12 N=1024 d=64 bf16 causal, forward and backward: eight whole heads."""
    case = workload_case("c2_gpt2s")
    o, lse, grads = _run(case, True)
    _check_heads(case, o, lse, grads, _heads(8, 12, 8, 2), 1.0, "c2")
    _check_identities(case, grads, "c2")


def test_prefill_workload():
    """B=1 H=8 N=4096 d=64 bf16 causal, forward: two whole heads."""
    case = workload_case("c3_prefill")
    o, lse, _ = _run(case, False)
    _check_heads(case, o, lse, None, _heads(1, 8, 2, 3), 1.0, "c3")


@pytest.mark.parametrize("name", ["c4a_long", "c4b_long_d128"])
def test_long_context_workloads(name):
    """B=4 N=8192 fp16 causal, forward and backward: one whole head, sampled rows of two
    more, identities in every head."""
    case = workload_case(name)
    o, lse, grads = _run(case, True)
    heads = _heads(case.B, case.H, 3, 4)
    _check_heads(case, o, lse, grads, heads[:1], 1.0, name, row_block=1024)
    _check_rows(case, o, lse, grads, heads[1:], 48, 1.0, name)
    _check_identities(case, grads, name)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("N", SWEEP_N)
def test_sequence_sweep(N, causal):
    """B*N = 65536 tokens, H=16, d=64, bf16 inputs x3, forward and backward."""
    name = f"c5_n{N}_{'causal' if causal else 'full'}"
    w = WORKLOADS[name]
    case = workload_case(name)
    o, lse, grads = _run(case, True)
    heads = _heads(case.B, case.H, 2, 5 + N)
    if N <= 8192:
        _check_heads(case, o, lse, grads, heads[:1], w["mult"], name, row_block=1024)
    _check_rows(case, o, lse, grads, heads, 32, w["mult"], name)
    _check_identities(case, grads, name)
