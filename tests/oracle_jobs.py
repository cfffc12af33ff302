"""Float64 oracle jobs for the full-size GPU parity tests, run in a pool of CPU
processes so that the oracle's work spreads over the host cores and overlaps the GPU
runs.

A whole head at 65536 tokens costs the oracle several minutes on one core, so each
head is cut into ranges of query rows: the forward rows of a range are exactly the
whole head's rows, and the backward's dK and dV of the head are the sums of the
ranges' contributions (``oracle.attn_head_bwd`` with ``row_range``, pinned in
tests/test_oracle_pins.py).  The pool uses the "spawn" start method (safe after CUDA
has been initialised in the test process) and one BLAS thread per worker.

Test infrastructure only; nothing on the product path imports this module.  numpy is
imported only inside the job functions, after the worker's initializer has fixed the
BLAS thread count.
"""

from __future__ import annotations

import concurrent.futures as cf
import multiprocessing as mp
import os

_POOL = None


def _init_worker():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"


def pool():
    """The shared pool (created on first use): one process per host core but one."""
    global _POOL
    if _POOL is None:
        workers = max(1, (os.cpu_count() or 2) - 1)
        _POOL = cf.ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("spawn"),
                                       initializer=_init_worker)
    return _POOL


def shutdown():
    global _POOL
    if _POOL is not None:
        _POOL.shutdown(wait=True, cancel_futures=True)
        _POOL = None


def head_fwd(q_bits, k_bits, v_bits, dtype, scale, causal, row_block, row_range):
    """(O, LSE, P|V|) of query rows row_range of one head, from its 16-bit inputs;
    P|V| (the oracle run with |V| as the values) sizes the P-rounding term of the O
    tolerance."""
    import numpy as np

    import oracle
    from exact_tiled_attention_27_gb300.inputs import bits_to_f64
    q, k, v = (bits_to_f64(x, dtype) for x in (q_bits, k_bits, v_bits))
    o, lse = oracle.attn_head_fwd(q, k, v, scale, causal, row_block, row_range=row_range)
    pv_abs, _ = oracle.attn_head_fwd(q, k, np.abs(v), scale, causal, row_block, row_range=row_range)
    return o, lse, pv_abs


def head_bwd(q_bits, k_bits, v_bits, do_bits, dtype, scale, causal, row_block, row_range):
    """(dQ rows, dK contribution, dV contribution) of query rows row_range of one head."""
    import oracle
    from exact_tiled_attention_27_gb300.inputs import bits_to_f64
    q, k, v, do = (bits_to_f64(x, dtype) for x in (q_bits, k_bits, v_bits, do_bits))
    dq, dk, dv, _ = oracle.attn_head_bwd(q, k, v, do, scale, causal, row_block, row_range=row_range)
    return dq, dk, dv


def row_ranges(n, parts):
    """`parts` contiguous ranges covering rows 0..n-1 (the last may be shorter)."""
    step = -(-n // parts)
    return [(lo, min(n, lo + step)) for lo in range(0, n, step)]


class HeadJobs:
    """The oracle's forward and backward of one (b, h) head, submitted to the pool in
    `parts` ranges of query rows."""

    def __init__(self, case, b, h, parts, row_block, with_bwd):
        ex = pool()
        q, k, v = (getattr(case, n)[b, h].copy() for n in ("q", "k", "v"))
        do = case.do[b, h].copy() if with_bwd else None
        self.ranges = row_ranges(case.N, parts)
        args = (case.dtype, case.scale, case.causal, row_block)
        self.fwd = [ex.submit(head_fwd, q, k, v, *args, r) for r in self.ranges]
        self.bwd = [ex.submit(head_bwd, q, k, v, do, *args, r) for r in self.ranges] if with_bwd else None

    def forward(self):
        """(O, LSE, P|V|) of the whole head."""
        import numpy as np
        parts = [f.result() for f in self.fwd]
        return tuple(np.concatenate([p[i] for p in parts]) for i in range(3))

    def backward(self):
        import numpy as np
        parts = [f.result() for f in self.bwd]
        dq = np.concatenate([p[0] for p in parts])
        dk = sum(p[1] for p in parts)
        dv = sum(p[2] for p in parts)
        return dq, dk, dv
