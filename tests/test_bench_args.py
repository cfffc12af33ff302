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
