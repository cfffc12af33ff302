"""GPU parity at the workloads' full sizes, through the same entry points and launch
configuration that bench.py times (fa_fwd, then the three launches of fa_bwd).

Every tensor is computed in full on the GPU.  The float64 oracle then checks whole
(b, h) heads element by element -- O, lse, dQ, dK and dV:
  * every head of the smallest workload, eight heads of the GPT-2-small shape and two
    of the 4096-token prefill;
  * four heads (the first, the last and two seeded ones) of each long-context workload
    and of every sequence-sweep length up to 8192;
  * two heads (the first and the last) at sweep lengths 16384, 32768 and 65536.
Heads are independent, so each sampled head is a complete check of the kernels on
that head.  On top, two identities that hold exactly in every head at any size are
checked in all heads: sum_j dK_j = 0 (the rows of dS sum to zero) and
sum_j dV_j = sum_i dO_i (the rows of P sum to one).

The oracle's heads at 8192 tokens and beyond run in a pool of CPU processes
(tests/oracle_jobs.py), split into ranges of query rows, while the GPU runs the next
workload.  Tolerances are those of tests/gpu_util.py.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from exact_tiled_attention_27_gb300 import backward, build, forward  # noqa: E402
from exact_tiled_attention_27_gb300.inputs import SWEEP_N, WORKLOADS, bits_to_f64, workload_case  # noqa: E402
from tests import gpu_util as G  # noqa: E402
from tests import oracle_jobs  # noqa: E402

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


def _f64(case, name, b, h):
    return bits_to_f64(getattr(case, name)[b, h], case.dtype)


def _check_heads_inline(case, o, lse, grads, heads, label):
    """Whole heads against the oracle, computed here (small workloads)."""
    for b, h in heads:
        q64, k64, v64 = _f64(case, "q", b, h), _f64(case, "k", b, h), _f64(case, "v", b, h)
        o_ref, lse_ref = oracle.attn_head_fwd(q64, k64, v64, case.scale, case.causal)
        pv_abs, _ = oracle.attn_head_fwd(q64, k64, np.abs(v64), case.scale, case.causal)
        G.check_forward(G.to_f64(o[b, h]), G.to_f64(lse[b, h]), o_ref, lse_ref, f"{label} head ({b},{h})",
                        case.dtype, pv_abs)
        if grads is not None:
            refs = oracle.attn_head_bwd(q64, k64, v64, _f64(case, "do", b, h), case.scale, case.causal)
            G.check_backward([G.to_f64(g[b, h]) for g in grads], refs[:3], f"{label} head ({b},{h})")


def _identities(case, grads):
    """max over heads of |sum_j dK_j| / |dK| and |sum_j dV_j - sum_i dO_i| / |dV|
    (float32 sums on the GPU)."""
    dq, dk, dv = grads
    do = G.to_device(case.do, case.dtype).float()
    dk32, dv32 = dk.float(), dv.float()
    res_dk = dk32.sum(dim=2)
    res_dv = dv32.sum(dim=2) - do.sum(dim=2)
    norm_dk = dk32.pow(2).sum(dim=(2, 3)).sqrt()
    norm_dv = dv32.pow(2).sum(dim=(2, 3)).sqrt()
    r_dk = (res_dk.pow(2).sum(-1).sqrt() / norm_dk).max().item()
    r_dv = (res_dv.pow(2).sum(-1).sqrt() / norm_dv).max().item()
    return r_dk, r_dv, bool(torch.isfinite(dq).all())


def _assert_identities(ident, label):
    r_dk, r_dv, dq_finite = ident
    print(f"{label}: every head |sum dK|/|dK| <= {r_dk:.3e}, |sum dV - sum dO|/|dV| <= {r_dv:.3e}")
    assert r_dk <= G.GRAD_RELL2 and r_dv <= G.GRAD_RELL2 and dq_finite


class PooledRun:
    """One workload: its GPU results on the sampled heads (float32 on the host), the
    oracle's jobs for those heads, and the identities over every head."""

    def __init__(self, name, heads, parts, row_block):
        w = WORKLOADS[name]
        case = workload_case(name)
        self.name, self.dtype, self.heads = name, case.dtype, heads
        self.jobs = {bh: oracle_jobs.HeadJobs(case, *bh, parts, row_block, w["backward"]) for bh in heads}
        o, lse, grads = _run(case, w["backward"])
        host = lambda t: t.float().cpu().numpy()  # noqa: E731
        self.gpu = {}
        for b, h in heads:
            g = [host(x[b, h]) for x in grads] if grads is not None else None
            self.gpu[(b, h)] = (host(o[b, h]), host(lse[b, h]), g)
        self.ident = _identities(case, grads) if grads is not None else None
        del o, lse, grads, case
        torch.cuda.empty_cache()

    def check(self):
        for bh in self.heads:
            label = f"{self.name} head {bh}"
            o, lse, g = self.gpu[bh]
            o_ref, lse_ref, pv_abs = self.jobs[bh].forward()
            G.check_forward(o.astype(np.float64), lse.astype(np.float64), o_ref, lse_ref, label, self.dtype, pv_abs)
            if g is not None:
                G.check_backward([x.astype(np.float64) for x in g], self.jobs[bh].backward(), label)
        if self.ident is not None:
            _assert_identities(self.ident, self.name)


def _parts(N):
    """Ranges of query rows per oracle head: about 8192 rows each."""
    return max(1, N // 8192)


def _row_block(N):
    return None if N <= 2048 else (1024 if N <= 8192 else 256)


def test_tiny_workload_full_oracle():
    case = workload_case("c1_tiny")
    o, lse, _ = _run(case, False)
    _check_heads_inline(case, o, lse, None, [(0, 0)], "c1")


def test_gpt2_small_workload():
    """B=8 H=12 N=1024 d=64 bf16 causal, forward and backward: eight whole heads."""
    case = workload_case("c2_gpt2s")
    o, lse, grads = _run(case, True)
    _check_heads_inline(case, o, lse, grads, _heads(8, 12, 8, 2), "c2")
    _assert_identities(_identities(case, grads), "c2")


def test_prefill_workload():
    """B=1 H=8 N=4096 d=64 bf16 causal, forward: two whole heads."""
    case = workload_case("c3_prefill")
    o, lse, _ = _run(case, False)
    _check_heads_inline(case, o, lse, None, _heads(1, 8, 2, 3), "c3")


@pytest.mark.parametrize("name", ["c4a_long", "c4b_long_d128"])
def test_long_context_workloads(name):
    """B=4 N=8192 fp16 causal, forward and backward: four whole heads, identities in
    every head."""
    w = WORKLOADS[name]
    PooledRun(name, _heads(w["B"], w["H"], 4, 4), _parts(w["N"]), _row_block(w["N"])).check()


def _sweep_name(N, causal):
    return f"c5_n{N}_{'causal' if causal else 'full'}"


@pytest.fixture(scope="module")
def sweep_runs():
    """Every sweep workload run on the GPU once, longest first, with its oracle jobs
    submitted before its GPU run so that the pool works while the GPU runs the rest."""
    runs = {}
    for N in sorted(SWEEP_N, reverse=True):
        for causal in (True, False):
            name = _sweep_name(N, causal)
            w = WORKLOADS[name]
            count = 4 if N <= 8192 else 2
            heads = _heads(w["B"], w["H"], count, 5 + N)
            runs[name] = PooledRun(name, heads, _parts(N), _row_block(N))
    return runs


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("N", SWEEP_N)
def test_sequence_sweep(sweep_runs, N, causal):
    """B*N = 65536 tokens, H=16, d=64, bf16 inputs x3, forward and backward: whole
    heads (four up to 8192 tokens, two beyond) element by element against the oracle."""
    sweep_runs[_sweep_name(N, causal)].check()
