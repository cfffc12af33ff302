"""The multi-GPU mode of bench.py is "replicas only": every rank runs the whole
workload on its own GPU, with no collective on the data path; ranks meet only to
take the maximum step time, and the whole-job value is world * work / that time.
This host-side logic is tested here with world_size-2 gloo process groups on CPU."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [1.0 + rank, 0.25 * (rank + 1), 3.0 - rank]   # step, fwd, bwd ms on this rank
        reduced = bench.reduce_step_times(mine)
        out[rank] = reduced
    finally:
        dist.destroy_process_group()


def test_step_times_take_the_max_over_two_ranks():
    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert out[0] == out[1] == [2.0, 0.5, 3.0]


def test_single_process_times_pass_through():
    assert not dist.is_initialized()
    assert bench.reduce_step_times([1.5, 0.5, 1.0]) == [1.5, 0.5, 1.0]


def test_job_throughput_scales_with_replicas():
    f = 14 * 8 * 12 * 1024 * 1024 * 64 / 2          # one causal fwd+bwd step of the GPT-2-small workload
    one = bench.job_throughput(1, f, 0.1)
    assert one == pytest.approx(f / 1e-4 / 1e12)
    assert bench.job_throughput(4, f, 0.1) == pytest.approx(4 * one)
    assert bench.job_throughput(2, f, 0.2) == pytest.approx(one)   # weak scaling: slowest rank sets the pace


def test_cross_visible_pairs_closed_forms():
    """FLOP count of the cross-length workloads: (query, key) pairs under the
    bottom-right causal mask."""
    import bench
    for n in (1, 7, 128, 1000):
        assert bench.cross_visible_pairs(n, n, True) == n * (n + 1) // 2       # the square triangle
        assert bench.cross_visible_pairs(n, n, False) == n * n
    assert bench.cross_visible_pairs(1, 500, True) == 500                       # one new token sees the cache
    assert bench.cross_visible_pairs(10, 4, True) == sum(range(1, 5))          # six rows see nothing
    nq, nk = 300, 1000
    assert bench.cross_visible_pairs(nq, nk, True) == nq * (nk - nq) + nq * (nq + 1) // 2


def test_butterfly_visible_pairs_counts():
    """FLOP count of the block-sparse workload against the oracle's own mask."""
    import bench
    import numpy as np
    from oracle import attention as A
    for n, causal in ((256, False), (1000, False), (1000, True), (1300, True), (2048, False)):
        want = int(A.butterfly_mask(n, n, causal).sum())
        assert bench.butterfly_visible_pairs(n, causal) == want, (n, causal)
    assert bench.butterfly_visible_pairs(256, True) == 256 * 257 // 2
    # 2^15 keys = 128 blocks of 256: each links 1 + log2(128) = 8 of them
    assert np.isclose(bench.butterfly_visible_pairs(1 << 15, False) / (1 << 30), 8 / 128)
