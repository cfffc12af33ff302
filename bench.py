#!/usr/bin/env python
"""Attention throughput on GB300: TFLOPS of the forward and of forward+backward.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--e2e-steps E] [--cpu-seconds S] [--cpu-threads T]

A step is one forward (fa_fwd) and one backward (the three launches of fa_bwd) over
one batch of seeded synthetic inputs already resident in device memory.  Between
timed steps a 256 MiB buffer is written to flush the 129 MB L2; the flush is outside
the CUDA-event brackets.  FLOPs follow the usual convention: forward 4*B*H*N^2*d,
backward 10*B*H*N^2*d, both halved under the causal mask.

Prints one JSON line (rank 0).  With --impl reference the float64 CPU oracle is timed
instead, on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _cpu_threads_arg(argv):
    """The --cpu-threads value, read before numpy is first imported: the BLAS library
    fixes its thread pool when it loads."""
    for i, a in enumerate(argv):
        if a == "--cpu-threads" and i + 1 < len(argv):
            return argv[i + 1]
        if a.startswith("--cpu-threads="):
            return a.split("=", 1)[1]
    return None


CPU_THREADS = _cpu_threads_arg(sys.argv[1:])
if CPU_THREADS is not None:
    for _var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[_var] = CPU_THREADS

from exact_tiled_attention_27_gb300.inputs import EXTRA_WORKLOADS, WORKLOADS, extra_case, workload_case  # noqa: E402

METRIC = "attention TFLOPS fwd and fwd+bwd (bf16, causal/non) and % of GB300 BF16 tensor peak"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "c5_n65536_causal"
FALLBACK_PEAK_TFLOPS = 1900.0
FALLBACK_SUSTAINED_TFLOPS = 1700.0


def flops(w, which):
    B, H, N, d = w["B"], w["H"], w["N"], w["d"]
    base = B * H * N * N * d
    f = {"fwd": 4 * base, "bwd": 10 * base, "fwd_bwd": 14 * base}[which]
    return f / 2 if w["causal"] else f


def reduce_step_times(times, device=None):
    """Max over ranks of per-rank step times (ms): the job is as slow as its slowest
    replica.  Works with any initialised process group (nccl on GPUs, gloo on CPU);
    returns the input unchanged when there is no process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(times)
    t = torch.tensor(list(times), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def step_brackets(steps, launches):
    """Event bracketing of the timed steps: True for a step with an event after every
    launch (the per-kernel times), False for one with events at its two ends only (the
    step time).  The two alternate; a one-launch step, or a single timed step, serves both."""
    return [launches == 1 or steps == 1 or i % 2 == 1 for i in range(steps)]


def job_throughput(world, flops_per_step, ms_per_step):
    """Whole-job TFLOP/s of `world` replicas that each do `flops_per_step` per step and
    take (at most, over ranks) `ms_per_step`."""
    return world * flops_per_step / (ms_per_step * 1e-3) / 1e12


def describe(name, w):
    parts = f"B={w['B']} H={w['H']} N={w['N']} d={w['d']} {w['dtype']} {'causal' if w['causal'] else 'non-causal'}"
    mult = f" inputs x{w['mult']:g}" if w["mult"] != 1.0 else ""
    return f"{name}: {parts}{mult} {'fwd+bwd' if w['backward'] else 'fwd'}"


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["bf16_tflops"]), float(j.get("bf16_tflops_sustained", j["bf16_tflops"])), "measured"
    return FALLBACK_PEAK_TFLOPS, FALLBACK_SUSTAINED_TFLOPS, "fallback"


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t is not None:
            self.t.join(timeout=5)
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------- our arm
def run_ours(args, w, rank, world, local_rank):
    import numpy as np
    import torch

    from exact_tiled_attention_27_gb300 import build as fa_build
    from exact_tiled_attention_27_gb300 import binding as fa

    fa_build.build()
    lib = fa.load_library()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    sh = fa._stream_handle(stream)
    case = workload_case(args.workload)
    tdt = torch.bfloat16 if w["dtype"] == "bf16" else torch.float16
    dcode = fa.FA_BF16 if w["dtype"] == "bf16" else fa.FA_FP16
    B, H, N, d = w["B"], w["H"], w["N"], w["d"]
    causal = 1 if w["causal"] else 0
    scale = case.scale

    def host(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(tdt).pin_memory()

    h_in = [host(case.q), host(case.k), host(case.v)] + ([host(case.do)] if w["backward"] else [])
    d_in = [t.to(dev) for t in h_in]
    q, k, v = d_in[:3]
    do = d_in[3] if w["backward"] else None
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3)) if w["backward"] else (None, None, None)
    ws_bytes = fa.workspace_size(B, H, N, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    P = fa._ptr

    def call(st, what):
        if st != 0:
            raise fa.FaError(st, what)

    def fwd():
        call(lib.fa_fwd(P(q), P(k), P(v), P(o), P(lse), B, H, N, d, scale, causal, dcode, sh), "fa_fwd")

    bwd_args = None
    if w["backward"]:
        bwd_args = lambda: (P(q), P(k), P(v), P(o), P(do), P(lse), P(dq), P(dk), P(dv), P(ws), ws_bytes,  # noqa: E731
                            B, H, N, d, scale, causal, dcode, sh)

    stages = []
    if w["backward"]:
        stages = [lib.fa_bwd_preprocess, lib.fa_bwd_dkdv, lib.fa_bwd_dq_convert]

    n_ev = 2 + len(stages)
    launches_per_step = 1 + len(stages)

    def step(evs=None, per_launch=True):
        # per_launch: an event after every launch (the launches then run one after
        # another); otherwise events at the step's two ends only, so that each launch's
        # set-up overlaps the previous kernel's tail as it does in a training loop
        if evs:
            evs[0].record(stream)
        fwd()
        if evs and per_launch:
            evs[1].record(stream)
        for i, fn in enumerate(stages):
            call(fn(*bwd_args()), fn.__name__)
            if evs and per_launch:
                evs[2 + i].record(stream)
        if evs and not per_launch:
            evs[1].record(stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if fa.last_kernel_status() != 0:
        raise RuntimeError("a kernel reported a pipeline timeout during warm-up")

    # The timed steps alternate: even steps are bracketed by two events (the step time),
    # odd steps carry an event after every launch (the per-kernel times of the roofline).
    # A forward-only step has one launch, so every step serves both.
    per_launch = step_brackets(args.steps, launches_per_step)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev if pl else 2)] for pl in per_launch]
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.2)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        step(ev[i], per_launch[i])
    torch.cuda.synchronize()
    wall1 = time.perf_counter()
    if world > 1:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    status = fa.last_kernel_status()
    if status != 0:
        raise RuntimeError(f"a kernel reported {fa.STATUS.get(status)} in the timed region")

    # medians over the timed steps: each launch's event time (steps with per-launch
    # events) and the whole step (steps bracketed at their ends only)
    seg = [[ev[i][j].elapsed_time(ev[i][j + 1]) for j in range(n_ev - 1)]
           for i in range(args.steps) if per_launch[i]]
    t_fwd = statistics.median(s[0] for s in seg)
    t_stage = [statistics.median(s[1 + j] for s in seg) for j in range(len(stages))]
    t_bwd = sum(t_stage)
    whole = [ev[i][0].elapsed_time(ev[i][-1]) for i in range(args.steps) if not per_launch[i] or not stages]
    t_serial = t_fwd + t_bwd
    t_step = statistics.median(whole) if whole else t_serial
    n_whole, n_per = len(whole), len(seg)
    if world > 1:
        t_step, t_fwd, t_bwd = reduce_step_times([t_step, t_fwd, t_bwd], device=dev)

    f_fwd = flops(w, "fwd")
    f_bwd = flops(w, "bwd") if w["backward"] else 0.0
    f_step = f_fwd + f_bwd
    value = job_throughput(world, f_step, t_step)
    peak_burst, peak_sus, peak_src = measured_peaks()

    # ---------------------------------------------------------------- end to end (host buffers)
    e2e = None
    if args.e2e_steps > 0:
        # Every step uploads its inputs from pinned host memory and reads all of its
        # outputs back, as a training loop's data path does.  The steps are pipelined on
        # three streams with double-buffered device tensors: step i+1's upload and step
        # i-1's read-back run while step i computes (the copy engines are full duplex).
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        h_out = [[torch.empty_like(o, device="cpu").pin_memory(), torch.empty_like(lse, device="cpu").pin_memory()]
                 + ([torch.empty_like(q, device="cpu").pin_memory() for _ in range(3)] if w["backward"] else [])
                 for _ in range(2)]
        dbuf_in = [d_in, [torch.empty_like(t) for t in d_in]]
        dbuf_out = [[o, lse] + ([dq, dk, dv] if w["backward"] else []),
                    [torch.empty_like(o), torch.empty_like(lse)]
                    + ([torch.empty_like(q) for _ in range(3)] if w["backward"] else [])]
        h2d = sum(t.numel() * t.element_size() for t in h_in)
        d2h = sum(t.numel() * t.element_size() for t in h_out[0])
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        for e in ev_comp + ev_out:
            e.record(stream)
        sh_c = fa._stream_handle(stream)

        def compute(b):
            qi, ki, vi = dbuf_in[b][:3]
            oo, ll = dbuf_out[b][:2]
            call(lib.fa_fwd(P(qi), P(ki), P(vi), P(oo), P(ll), B, H, N, d, scale, causal, dcode, sh_c), "fa_fwd")
            if w["backward"]:
                gq, gk, gv = dbuf_out[b][2:]
                for fn in stages:
                    call(fn(P(qi), P(ki), P(vi), P(oo), P(dbuf_in[b][3]), P(ll), P(gq), P(gk), P(gv), P(ws), ws_bytes,
                            B, H, N, d, scale, causal, dcode, sh_c), fn.__name__)

        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        total = args.e2e_steps + 2
        for it in range(total):
            b = it % 2
            if it == 2:
                # the two untimed steps fill both buffer sets; the timed window opens on an
                # idle GPU with step 2's upload, so it holds exactly e2e_steps uploads,
                # computes and read-backs (overlapped with one another) and nothing else
                torch.cuda.synchronize()
                e0.record(s_in)
            with torch.cuda.stream(s_in):          # upload step it (after step it-2 used the buffer)
                s_in.wait_event(ev_comp[b])
                for hsrc, ddst in zip(h_in, dbuf_in[b]):
                    ddst.copy_(hsrc, non_blocking=True)
                ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])            # compute step it (after step it-2's outputs were read)
            stream.wait_event(ev_out[b])
            compute(b)
            ev_comp[b].record(stream)
            with torch.cuda.stream(s_out):         # read back step it
                s_out.wait_event(ev_comp[b])
                for dsrc, hdst in zip(dbuf_out[b], h_out[b]):
                    hdst.copy_(dsrc, non_blocking=True)
                ev_out[b].record(s_out)
        e1.record(s_out)
        torch.cuda.synchronize()
        t_e2e = e0.elapsed_time(e1) / args.e2e_steps
        e2e = {"value": round(world * f_step / (t_e2e * 1e-3) / 1e12, 3), "unit": UNIT,
               "ms_per_step": round(t_e2e, 4), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "pipelining": "step i+1 upload and step i-1 read-back overlap step i's kernels (3 streams, "
                             "double-buffered device tensors)"}

    # dominant kernel: the dK/dV kernel when there is a backward, else the forward.
    # Each launch is bracketed alone by CUDA events, so the denominator is the burst
    # (not the power-capped sustained) measured bf16 peak.
    if w["backward"]:
        dom_name, dom_t, dom_f = "bwd_kv_kernel", t_stage[1], f_bwd
    else:
        dom_name, dom_t, dom_f = "fwd_kernel", t_fwd, f_fwd
    achieved = dom_f / (dom_t * 1e-3) / 1e12
    fwd_tf = f_fwd / (t_fwd * 1e-3) / 1e12
    roofline = {"bound": "tensor", "kernel": dom_name, "achieved": round(achieved, 2), "peak": peak_burst,
                "unit": UNIT, "frac": round(achieved / peak_burst, 4),
                "peak_source": f"{peak_src} bf16 cuBLAS burst (each launch timed alone by CUDA events)",
                "fwd_kernel": {"achieved": round(fwd_tf, 2), "frac": round(fwd_tf / peak_burst, 4)},
                "traffic": traffic_for(dom_name, args.workload)}
    if w["backward"]:
        bwd_tf = f_bwd / (t_bwd * 1e-3) / 1e12
        roofline["bwd_kv_kernel"] = {"achieved": round(achieved, 2), "frac": round(achieved / peak_burst, 4)}
        roofline["bwd_three_launches"] = {"achieved": round(bwd_tf, 2), "frac": round(bwd_tf / peak_burst, 4)}
    result = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w["dtype"], "data": "synthetic (seeded i.i.d. N(0,1) 16-bit inputs)",
        "config": {"workload": describe(args.workload, w), "B": B, "H": H, "N": N, "d": d, "causal": bool(causal),
                   "l2": "flushed between steps by a 256 MiB write outside the timed brackets",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "tflops": {"fwd": round(f_fwd / (t_fwd * 1e-3) / 1e12, 2),
                   "bwd": round(f_bwd / (t_bwd * 1e-3) / 1e12, 2) if w["backward"] else None,
                   "fwd_bwd": round(f_step / (t_step * 1e-3) / 1e12, 2)},
        "pct_of_peak": {"fwd": round(100 * f_fwd / (t_fwd * 1e-3) / 1e12 / peak_burst, 2),
                        "bwd": round(100 * f_bwd / (t_bwd * 1e-3) / 1e12 / peak_burst, 2) if w["backward"] else None,
                        "fwd_bwd": round(100 * f_step / (t_step * 1e-3) / 1e12 / peak_burst, 2),
                        "peak": f"{peak_burst} TFLOP/s dense bf16 ({peak_src}, burst)"},
        "ms": {"fwd": round(t_fwd, 5), "bwd": round(t_bwd, 5),
               "bwd_stages": [round(x, 5) for x in t_stage], "launches_one_by_one": round(t_serial, 5)},
        "timing": (f"ms_per_step: median of {n_whole} timed steps with events at their two ends only; "
                   f"ms, tflops.fwd/bwd and roofline: medians of {n_per} timed steps with an event after "
                   "every launch, which serialises the launches" if stages else
                   f"median of {n_whole} timed steps, one launch each"),
        "roofline": roofline,
        "gpu_launches": launches_per_step * args.steps,
        "wall_s_timed": round(wall1 - wall0, 3),
    }
    if clk:
        result["clocks"] = clk
    if e2e:
        result["e2e"] = e2e
    return result


# ---------------------------------------------------------------------------- extra workloads
def cross_visible_pairs(Nq, Nk, causal):
    """(query row, key) pairs that take part: all of them, or under the bottom-right
    causal mask sum_i clamp(i + Nk - Nq + 1, 0, Nk)."""
    if not causal:
        return Nq * Nk
    return sum(min(Nk, max(0, i + Nk - Nq + 1)) for i in range(Nq))


def butterfly_visible_pairs(N, causal, block=128):
    """(query row, key) pairs inside the butterfly pattern (256-row blocks = pairs of
    128-row tiles linked when equal or one bit apart), with key <= query when causal."""
    nb = (N + block - 1) // block
    npairs = (nb + 1) // 2
    total = 0
    for i in range(nb):
        rows = min(N, (i + 1) * block) - i * block
        for kb in range(nb):
            x = (i // 2) ^ (kb // 2)
            if kb // 2 >= npairs or (x & (x - 1)) != 0:
                continue
            k0, k1 = kb * block, min(N, (kb + 1) * block)
            if not causal:
                total += rows * (k1 - k0)
            else:
                for r in range(i * block, i * block + rows):
                    total += max(0, min(k1, r + 1) - k0)
    return total


def run_extra(args, w, local_rank):
    """Time one of the cross-length / grouped-head / decode workloads (single GPU).

    cross: a step is fa_fwd_cross (+ fa_bwd_gqa when the workload has a backward);
           TFLOP/s with 4*d (forward) and 10*d (backward) flops per visible
           (query row, key) pair and query head.
    decode: a step is fa_decode; GB/s of the bytes the method must move (K and V once,
           Q, O and lse), against the measured copy bandwidth.
    """
    import numpy as np
    import torch

    from exact_tiled_attention_27_gb300 import build as fa_build
    from exact_tiled_attention_27_gb300 import binding as fa

    fa_build.build()
    lib = fa.load_library()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    sh = fa._stream_handle(stream)
    c = extra_case(args.workload)
    tdt = torch.bfloat16 if w["dtype"] == "bf16" else torch.float16
    dcode = fa.FA_BF16 if w["dtype"] == "bf16" else fa.FA_FP16
    B, H, Hkv, Nq, Nk, d = w["B"], w["H"], w["Hkv"], w["Nq"], w["Nk"], w["d"]
    causal = 1 if w["causal"] else 0
    up = lambda bits: torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(tdt).to(dev)  # noqa: E731
    q, k, v = up(c.q), up(c.k), up(c.v)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
    P = fa._ptr
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def call(st, what):
        if st != 0:
            raise fa.FaError(st, what)

    launches = 1
    dense_step = None
    if w["kind"] == "sparse":
        do = up(c.do)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws_bytes = fa.workspace_size(B, H, Nq, d)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        launches = 4

        def step():
            call(lib.fa_fwd_sparse(P(q), P(k), P(v), P(o), P(lse), B, H, Nq, d, c.scale, causal, 1, dcode, sh),
                 "fa_fwd_sparse")
            call(lib.fa_bwd_sparse(P(q), P(k), P(v), P(o), P(do), P(lse), P(dq), P(dk), P(dv), P(ws), ws_bytes, B, H,
                                   Nq, d, c.scale, causal, 1, dcode, sh), "fa_bwd_sparse")

        def dense_step():
            call(lib.fa_fwd(P(q), P(k), P(v), P(o), P(lse), B, H, Nq, d, c.scale, causal, dcode, sh), "fa_fwd")
            call(lib.fa_bwd(P(q), P(k), P(v), P(o), P(do), P(lse), P(dq), P(dk), P(dv), P(ws), ws_bytes, B, H, Nq, d,
                            c.scale, causal, dcode, sh), "fa_bwd")
    elif w["kind"] == "fp8":
        from exact_tiled_attention_27_gb300.inputs import random_signs
        signs = torch.from_numpy(random_signs(d, 1000 * w["index"] + 7)).to(dev)
        nb = (Nq + 127) // 128
        q8 = torch.empty((B, H, Nq, d), dtype=torch.uint8, device=dev)
        k8 = torch.empty_like(q8)
        vt8 = torch.empty((B, H, d, lib.fa_fp8_vt_cols(Nq)), dtype=torch.uint8, device=dev)
        sq, sk, sv = (torch.empty((B, H, nb), dtype=torch.float32, device=dev) for _ in range(3))

        def quantize():
            call(lib.fa_quantize_fp8(P(q), P(q8), P(sq), B, H, Nq, d, dcode, P(signs), 0, 0, sh), "fa_quantize_fp8")
            call(lib.fa_quantize_fp8(P(k), P(k8), P(sk), B, H, Nq, d, dcode, P(signs), 0, 0, sh), "fa_quantize_fp8")
            call(lib.fa_quantize_fp8(P(v), P(vt8), P(sv), B, H, Nq, d, dcode, None, 0, 1, sh), "fa_quantize_fp8")

        quantize()

        def step():
            call(lib.fa_fwd_fp8(P(q8), P(k8), P(vt8), P(sq), P(sk), P(sv), P(o), P(lse), B, H, Nq, d, c.scale,
                                causal, dcode, sh), "fa_fwd_fp8")

        def dense_step():   # the 16-bit forward on the same (unquantized) inputs
            call(lib.fa_fwd(P(q), P(k), P(v), P(o), P(lse), B, H, Nq, d, c.scale, causal, dcode, sh), "fa_fwd")
    elif w["kind"] == "decode":
        ws_bytes = int(lib.fa_decode_workspace_size(B, H, Hkv, Nq, Nk, d))
        ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
        launches = 2 if ws_bytes > 0 else 1

        def step():
            call(lib.fa_decode(P(q), P(k), P(v), P(o), P(lse), P(ws), ws_bytes, B, H, Hkv, Nq, Nk, d, c.scale,
                               causal, dcode, sh), "fa_decode")
    else:
        do = up(c.do) if w["backward"] else None
        if w["backward"]:
            dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
            ws_bytes = fa.workspace_size(B, H, Nq, d)
            ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
            launches = 4

        def step():
            call(lib.fa_fwd_cross(P(q), P(k), P(v), P(o), P(lse), B, H, Hkv, Nq, Nk, d, c.scale, causal, dcode, sh),
                 "fa_fwd_cross")
            if w["backward"]:
                call(lib.fa_bwd_gqa(P(q), P(k), P(v), P(o), P(do), P(lse), P(dq), P(dk), P(dv), P(ws), ws_bytes, B,
                                    H, Hkv, Nq, d, c.scale, causal, dcode, sh), "fa_bwd_gqa")

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.2)
    for e0, e1 in ev:
        flush.zero_()
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    status = fa.last_kernel_status()
    if status != 0:
        raise RuntimeError(f"a kernel reported {fa.STATUS.get(status)} in the timed region")
    t = statistics.median(e0.elapsed_time(e1) for e0, e1 in ev)   # ms per step
    t_dense = None
    if dense_step is not None:   # the same step with the dense kernels, for the speed-up
        for _ in range(args.warmup):
            flush.zero_()
            dense_step()
        ts = []
        for e0, e1 in ev:
            flush.zero_()
            e0.record(stream)
            dense_step()
            e1.record(stream)
        torch.cuda.synchronize()
        t_dense = statistics.median(e0.elapsed_time(e1) for e0, e1 in ev)
    t_quant = None
    if w["kind"] == "fp8":   # the three quantizing calls, timed the same way
        for _ in range(args.warmup):
            flush.zero_()
            quantize()
        for e0, e1 in ev:
            flush.zero_()
            e0.record(stream)
            quantize()
            e1.record(stream)
        torch.cuda.synchronize()
        t_quant = statistics.median(e0.elapsed_time(e1) for e0, e1 in ev)
    cfg = {"workload": f"{args.workload}: B={B} H={H} Hkv={Hkv} Nq={Nq} Nk={Nk} d={d} {w['dtype']} "
                       f"{'causal (bottom-right)' if causal else 'non-causal'}"
                       f"{' fwd+bwd' if w['backward'] else ''}",
           "l2": "flushed between steps by a 256 MiB write outside the timed brackets", "parallelism": "single GPU"}
    res = {"n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t, 5),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w["dtype"],
           "data": "synthetic (seeded i.i.d. N(0,1) 16-bit inputs)", "config": cfg,
           "gpu_launches": launches * args.steps}
    if w["kind"] == "sparse":
        pairs = H * B * butterfly_visible_pairs(Nq, bool(causal))
        f = pairs * d * 14
        tf = f / (t * 1e-3) / 1e12
        peak_burst, peak_sus, src = measured_peaks()
        res.update({"metric": "block-sparse attention TFLOPS over the pattern's (query, key) pairs "
                              "(fa_fwd_sparse + fa_bwd_sparse)",
                    "value": round(tf, 2), "unit": UNIT,
                    "speedup_vs_dense": round(t_dense / t, 3), "dense_ms_per_step": round(t_dense, 5),
                    "pattern_density": round(pairs / (H * B * (Nq * Nq if not causal else Nq * (Nq + 1) / 2)), 5),
                    "roofline": {"bound": "tensor", "kernel": "fwd_kernel + bwd_kv_kernel", "achieved": round(tf, 2),
                                 "peak": peak_burst, "unit": UNIT, "frac": round(tf / peak_burst, 4),
                                 "peak_source": f"{src} bf16 cuBLAS burst", "traffic": None}})
    elif w["kind"] == "fp8":
        pairs = H * B * cross_visible_pairs(Nq, Nk, bool(causal))
        f = pairs * d * 4
        tf = f / (t * 1e-3) / 1e12
        peak_burst, peak_sus, src = measured_peaks()
        # no measured FP8 peak: the measured bf16 one times the nominal dense ratio 4.5 / 2.25
        p8_burst = 2 * peak_burst
        res["dtype"] = "e4m3"
        res["config"]["workload"] = (f"{args.workload}: B={B} H={H} N={Nq} d={d} E4M3 Q/K/V, 128-row block scales, "
                                     f"Q and K rotated, {'causal' if causal else 'non-causal'} forward, "
                                     f"{w['dtype']} O")
        res.update({"metric": "FP8 attention forward TFLOPS (fa_fwd_fp8, 4*d flops per visible (query, key) pair)",
                    "value": round(tf, 2), "unit": UNIT,
                    "bf16_forward_ms": round(t_dense, 5), "speedup_vs_bf16_forward": round(t_dense / t, 3),
                    "quantize_ms": round(t_quant, 5),
                    "with_quantize_tflops": round(f / ((t + t_quant) * 1e-3) / 1e12, 2),
                    "roofline": {"bound": "tensor", "kernel": "fwd_fp8_kernel", "achieved": round(tf, 2),
                                 "peak": p8_burst, "unit": UNIT, "frac": round(tf / p8_burst, 4),
                                 "peak_source": f"{src} bf16 cuBLAS burst x 2 (nominal fp8/bf16 dense ratio)",
                                 "traffic": traffic_for("fwd_fp8_kernel", args.workload)}})
    elif w["kind"] == "decode":
        nbytes = 2 * B * Hkv * Nk * d * 2 + 2 * B * H * Nq * d * 2 + B * H * Nq * 4
        gbs = nbytes / (t * 1e-3) / 1e9
        dec_kernel = "decode_split_kernel"
        hbm, src = 6800.0, "fallback"
        pk = os.path.join(ROOT, "MEASURED_PEAKS.json")
        if os.path.exists(pk):
            with open(pk) as f:
                hbm, src = float(json.load(f)["hbm_gbs"]), "measured"
        res.update({"metric": "decode: bytes of K, V, Q, O and lse moved per second", "value": round(gbs, 1),
                    "unit": "GB/s",
                    "roofline": {"bound": "hbm", "kernel": dec_kernel, "achieved": round(gbs, 1),
                                 "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 4),
                                 "peak_source": f"{src} copy bandwidth",
                                 "traffic": traffic_for(dec_kernel, args.workload)}})
    else:
        pairs = H * B * cross_visible_pairs(Nq, Nk, bool(causal))
        f = pairs * d * (4 + (10 if w["backward"] else 0))
        tf = f / (t * 1e-3) / 1e12
        peak_burst, peak_sus, src = measured_peaks()
        res.update({"metric": "attention TFLOPS (fa_fwd_cross" + (" + fa_bwd_gqa)" if w["backward"] else ")"),
                    "value": round(tf, 2), "unit": UNIT,
                    "roofline": {"bound": "tensor", "kernel": "fwd_kernel" + (" + bwd_kv_kernel" if w["backward"]
                                                                             else ""),
                                 "achieved": round(tf, 2), "peak": peak_burst, "unit": UNIT,
                                 "frac": round(tf / peak_burst, 4),
                                 "peak_source": f"{src} bf16 cuBLAS burst", "traffic": None}})
    if clk:
        res["clocks"] = clk
    return res


KERNEL_SOURCE = {"fwd_kernel": "fwd.cu", "bwd_kv_kernel": "bwd.cu", "decode_split_kernel": "decode.cu",
                 "fwd_fp8_kernel": "fwd_fp8.cu"}


def source_sha256(kernel):
    import hashlib
    path = os.path.join(ROOT, "exact_tiled_attention_27_gb300", "csrc", KERNEL_SOURCE[kernel])
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def traffic_for(kernel, workload):
    """DRAM bytes per launch from a committed ncu capture, or None when there is none or
    the kernel's source has changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        with open(p) as f:
            j = json.load(f)
        entry = j.get(f"{kernel}:{workload}")
        if not entry or entry.get("source_sha256") != source_sha256(kernel):
            return None
        return entry.get("bytes_per_launch")
    except (OSError, ValueError, KeyError):
        return None


# ---------------------------------------------------------------------------- oracle arm
SAMPLE_SCORES = 1 << 23   # score-matrix entries per oracle sample (rows x keys)


def visible_pairs(N, causal, lo, hi):
    """(query row, key) pairs of query rows lo..hi-1 that the mask lets through."""
    if not causal:
        return (hi - lo) * N
    return (lo + 1 + hi) * (hi - lo) // 2


def oracle_sample(w, seconds, max_samples=None):
    """Time the float64 oracle on a bounded sample of the workload until `seconds`
    have passed (at least one sample).  A sample is one range of consecutive query
    rows of one (b, h) head -- the whole head when it has at most SAMPLE_SCORES score
    entries -- forward and, where the workload has one, backward
    (oracle.attn_head_fwd / attn_head_bwd with row_range).  Successive samples visit
    the heads in turn and move through the sequence, so that under the causal mask
    short and long rows are both taken.  The rate counts the method's flops of the
    rows done: 4*d (forward) and 10*d (backward) per visible (query row, key) pair.
    Returns (samples, rows per sample, seconds, TFLOP/s)."""
    import oracle
    from exact_tiled_attention_27_gb300.inputs import bits_to_f64
    case = workload_case_cached(w)
    B, H, N, d = w["B"], w["H"], w["N"], w["d"]
    rows = max(1, min(N, SAMPLE_SCORES // N))
    nranges = -(-N // rows)
    rb = 1024 if rows > 1024 else None
    per_pair = 4 * d + (10 * d if w["backward"] else 0)
    done, work, el = 0, 0, 0.0
    t0 = time.perf_counter()
    while True:
        bh = done % (B * H)
        b, h = divmod(bh, H)
        lo = ((done * 7919) % nranges) * rows   # a stride prime to typical range counts
        hi = min(N, lo + rows)
        f = lambda name: bits_to_f64(getattr(case, name)[b, h], case.dtype)  # noqa: E731
        q64, k64, v64 = f("q"), f("k"), f("v")
        do64 = f("do") if w["backward"] else None
        t1 = time.perf_counter()
        oracle.attn_head_fwd(q64, k64, v64, case.scale, w["causal"], rb, row_range=(lo, hi))
        if w["backward"]:
            oracle.attn_head_bwd(q64, k64, v64, do64, case.scale, w["causal"], rb, row_range=(lo, hi))
        el += time.perf_counter() - t1
        work += per_pair * visible_pairs(N, w["causal"], lo, hi)
        done += 1
        if time.perf_counter() - t0 >= seconds or (max_samples and done >= max_samples):
            break
    return done, rows, el, work / el / 1e12


def sample_text(w, n, rows, el):
    what = "forward+backward" if w["backward"] else "forward"
    unit = "whole (b,h) heads" if rows >= w["N"] else f"ranges of {rows} query rows x all {w['N']} keys"
    return (f"{n} {unit} ({what}, float64 numpy, heads taken in turn, rows spread over the sequence; "
            f"workload has {w['B'] * w['H']} heads of {w['N']} rows), {el:.1f} s")


def oracle_threads():
    """Threads the oracle's BLAS calls run on: --cpu-threads, else every host core."""
    return int(CPU_THREADS) if CPU_THREADS is not None else os.cpu_count()


_CASE_CACHE = {}


def workload_case_cached(w):
    key = id(w)
    if key not in _CASE_CACHE:
        name = [n for n, x in WORKLOADS.items() if x is w][0]
        _CASE_CACHE[key] = workload_case(name)
    return _CASE_CACHE[key]


def run_reference(args, w):
    # warm-up and timed steps, each one bounded sample of the workload
    for _ in range(args.warmup):
        oracle_sample(w, 0.0, max_samples=1)
    vals, n_total, el_total, rows = [], 0, 0.0, 0
    for _ in range(args.steps):
        n, rows, el, tf = oracle_sample(w, args.cpu_seconds / max(args.steps, 1))
        vals.append(tf)
        n_total += n
        el_total += el
    value = statistics.median(vals)
    cores = oracle_threads()
    sample = f"over {args.steps} steps: " + sample_text(w, n_total, rows, el_total)
    return {"metric": METRIC, "value": round(value, 6), "unit": UNIT, "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * el_total / max(args.steps, 1), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded i.i.d. N(0,1) 16-bit inputs widened to float64)",
            "config": {"workload": describe(args.workload, w)},
            "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS) + sorted(EXTRA_WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="wall-clock budget of the oracle's CPU-baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-threads", type=int, default=None,
                    help="BLAS threads of the oracle (default: every host core)")
    args = ap.parse_args()
    if args.cpu_threads is not None and args.cpu_threads < 1:
        ap.error("--cpu-threads must be >= 1")
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.workload in EXTRA_WORKLOADS:
        if args.impl == "reference" or world > 1:
            ap.error("the extra workloads time this library on one GPU only")
        print(json.dumps(run_extra(args, EXTRA_WORKLOADS[args.workload], local_rank)))
        return 0
    w = WORKLOADS[args.workload]

    if args.impl == "reference":
        if rank != 0:
            return 0
        steps = max(1, min(args.steps, 20))
        args.steps = steps
        print(json.dumps(run_reference(args, w)))
        return 0

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    result = run_ours(args, w, rank, world, local_rank)
    if rank == 0 and not args.no_cpu_baseline:
        n, rows, el, tf = oracle_sample(w, args.cpu_seconds)
        result["cpu_baseline"] = {"value": round(tf, 6), "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
                                  "sample": sample_text(w, n, rows, el)}
    if rank == 0:
        print(json.dumps(result))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
