"""Host-side argument handling of bench.py that must act before numpy loads."""

import bench


def test_cpu_threads_is_read_from_either_form():
    assert bench._cpu_threads_arg(["--workload", "c2_gpt2s", "--cpu-threads", "4"]) == "4"
    assert bench._cpu_threads_arg(["--cpu-threads=1", "--steps", "3"]) == "1"
    assert bench._cpu_threads_arg(["--steps", "3"]) is None
    assert bench._cpu_threads_arg(["--cpu-threads"]) is None       # argparse reports the missing value


def test_oracle_threads_defaults_to_every_core(monkeypatch):
    import os
    monkeypatch.setattr(bench, "CPU_THREADS", None)
    assert bench.oracle_threads() == os.cpu_count()
    monkeypatch.setattr(bench, "CPU_THREADS", "3")
    assert bench.oracle_threads() == 3


def test_visible_pairs_of_row_ranges_add_up():
    for N in (1, 7, 128, 1000):
        for causal in (False, True):
            cuts = sorted({0, N, N // 3, N // 2})
            total = sum(bench.visible_pairs(N, causal, lo, hi) for lo, hi in zip(cuts, cuts[1:]))
            assert total == (N * (N + 1) // 2 if causal else N * N)
    assert bench.visible_pairs(10, True, 0, 1) == 1 and bench.visible_pairs(10, True, 9, 10) == 10


def test_oracle_sample_is_bounded_and_counts_work():
    w = bench.WORKLOADS["c1_tiny"]
    n, rows, el, tf = bench.oracle_sample(w, 0.0, max_samples=2)
    assert n == 1 and rows == w["N"] and el > 0 and tf > 0
    assert "whole (b,h) heads" in bench.sample_text(w, n, rows, el)


def test_step_brackets_alternate_whole_steps_and_per_launch_steps():
    plan = bench.step_brackets(20, 4)
    assert plan.count(True) == 10 and plan.count(False) == 10
    assert plan[0] is False and plan[1] is True
    assert bench.step_brackets(1, 4) == [True]                    # one step: per-launch times and the step
    assert bench.step_brackets(5, 1) == [True] * 5                # a forward-only step is one launch
    assert bench.step_brackets(3, 4) == [False, True, False]
