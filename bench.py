#!/usr/bin/env python
"""Benchmark of the exact-attention hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input,
three calls of the library:
  1. causal prefill, GPT-2 shape: B=8, h=12, T=1024, d=64, bf16,
  2. causal prefill, very long: B=1, h=12, T=16384, d=64, fp16, inputs x0.5
     (the largest prefill workload), and
  3. decode against a KV cache: B=32, h=12, T_q=1, T_kv=16384, d=64, bf16
     (split-KV kernel + exact merge kernel).
The two prefills run on the tensor cores; the decode streams the cache.

Metric: the step's roofline time divided by its measured time, in percent.
The roofline time of a call is max(FLOPs / tensor peak, bytes / HBM peak)
with the algorithmic FLOPs (4*d per visible query-key pair, causal pairs
counted) and bytes (Q, K, V read once, O and lse written once); the peaks
are the measured ones in MEASURED_PEAKS.json. `value` is whole-job
throughput in units of one GB300's roofline: 100 * N * t_roof / t_step,
so at N=1 it is the percentage of the roofline reached. Each call's own
fraction is in `calls`, and every workload (the seven runs) is measured on
its own, with an L2 flush between launches, in `runs`.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the float64 CPU oracle (the only other program that
computes this path) on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

# the oracle leg uses numpy BLAS on every host core; say so explicitly
_CORES = os.cpu_count() or 1
os.environ.setdefault("OPENBLAS_NUM_THREADS", str(_CORES))
os.environ.setdefault("OMP_NUM_THREADS", str(_CORES))

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "causal prefill attention TFLOP/s + decode KV GB/s, as % of GB300 roofline"
UNIT = "% of one GB300 roofline (whole job)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
_CSRC = os.path.join(ROOT, "exact_io_aware_attn_gb300", "csrc")
# the sources each traffic entry's kernels are built from
KERNEL_SOURCES = {
    "decode": [os.path.join(_CSRC, "decode_sm103.cu"), os.path.join(_CSRC, "merge_sm103.cuh")],
    "prefill": [os.path.join(_CSRC, "prefill_sm103.cu")],
    "prefill_very_long": [os.path.join(_CSRC, "prefill_sm103.cu")],
}
# repeats of the step after the timed K steps: >= 3 repeats of >= 20 steps
REPEATS = 3
REPEAT_MIN_STEPS = 20
# per-workload timing: launches per repeat, repeats, warm-up launches
RUN_LAUNCHES, RUN_REPEATS, RUN_WARMUP = 20, 3, 3
L2_FLUSH_BYTES = 256 << 20      # twice the 129 MB L2


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return dict(FALLBACK_PEAKS, source="fallback")


def source_sha(paths):
    h = hashlib.sha256()
    for path in paths:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_traffic(kind):
    """DRAM bytes per launch from a committed ncu capture, or None if the
    kernel source changed since the counters were taken."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        t = json.load(f).get(kind)
    if not t or t.get("source_sha") != source_sha(KERNEL_SOURCES[kind]):
        return None
    return float(t["dram_bytes_per_launch"])


# ----------------------------------------------------------------- work model
def step_calls():
    """The step's calls: (key, workload, traffic key)."""
    from exact_io_aware_attn_gb300.inputs import DECODE, GPT2_PREFILL, VERY_LONG
    return [("prefill_gpt2", GPT2_PREFILL, "prefill"),
            ("prefill_very_long", VERY_LONG, "prefill_very_long"),
            ("decode", DECODE, "decode")]


def work_of(w, peaks):
    """Algorithmic FLOPs and bytes of one call of workload w, its roofline
    time and which roof binds."""
    from exact_io_aware_attn_gb300 import cost
    fl = cost.flops(w.B, w.h, w.T_q, w.T_kv, w.d, w.causal)
    by = cost.min_bytes(w.B, w.h, w.T_q, w.T_kv, w.d, h_kv=w.kv_heads)
    t_tc = fl / (peaks["bf16_tflops"] * 1e12)
    t_bw = by / (peaks["hbm_gbs"] * 1e9)
    return {"flops": fl, "bytes": by, "t_roof": max(t_tc, t_bw),
            "bound": "tensor" if t_tc >= t_bw else "hbm"}


def config_block():
    calls = step_calls()
    return {
        "workload": " + ".join(w.name for _, w, _ in calls),
        **{key: w.describe() for key, w, _ in calls},
        "l2": "inputs larger than L2: each step streams the 1.61 GB KV cache, which also "
              "evicts the prefill inputs (38 MB and 75 MB) before the next step; the per-workload "
              "runs flush L2 before every timed launch (a 256 MB write, then a 256 MB read)",
        "data": "synthetic N(0,1) from torch CPU generator seed 0, q then k then v "
                "(x0.5 for the very long prefill)",
    }


# ----------------------------------------------------------------- distributed
def dist_init(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device=None):
    """Maximum of a float over all ranks (timing only; no data-path exchange)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- CPU oracle
_INPUTS = {}


def cached_inputs(w, one_head=False):
    """make_workload(w) (CPU tensors), kept for reuse: drawing the decode
    cache takes seconds. one_head: a single head of w's shape and
    distribution (B = h = 1, same seed), for the oracle's row samples."""
    import dataclasses

    from exact_io_aware_attn_gb300.inputs import make_workload
    key = (w.name, one_head)
    if key not in _INPUTS:
        _INPUTS[key] = make_workload(dataclasses.replace(w, B=1, h=1, h_kv=0) if one_head else w)
    return _INPUTS[key]


def oracle_sample(w, n_rows):
    """Time the float64 oracle on n_rows query rows of workload w. Prefill:
    the last n_rows rows of one head of w's shape and distribution (a causal
    row sees as many keys as in the full problem). Decode: n_rows whole
    (b, h) rows of the workload itself. Returns (seconds, rows, rows of the
    whole call). The oracle forms each row's whole score vector, so its cost
    per row does not depend on the mask: whole-call time = seconds * total /
    rows."""
    import numpy as np

    import oracle
    if w.T_q == 1:
        q, k, v = cached_inputs(w)
        n_rows = max(1, min(n_rows, w.B * w.h))
        t0 = time.perf_counter()
        for i in range(n_rows):
            b, h = divmod(i, w.h)
            oracle.standard_attention(q[b, h].double().numpy(), k[b, h].double().numpy(),
                                      v[b, h].double().numpy(), scale=w.scale, causal=False)
        return time.perf_counter() - t0, n_rows, w.B * w.h
    q, k, v = cached_inputs(w, one_head=True)
    n_rows = max(1, min(n_rows, w.T_q))
    rows = np.arange(w.T_q - n_rows, w.T_q)
    qn, kn, vn = q[0, 0].double().numpy(), k[0, 0].double().numpy(), v[0, 0].double().numpy()
    t0 = time.perf_counter()
    oracle.standard_attention(qn, kn, vn, scale=w.scale, causal=w.causal, rows=rows)
    return time.perf_counter() - t0, n_rows, w.B * w.h * w.T_q


def describe_sample(w, n):
    blas = f"float64 numpy, BLAS threads {os.environ['OPENBLAS_NUM_THREADS']}"
    if w.T_q == 1:
        return f"{n} of {w.B * w.h} (b, h) decode rows, {blas}"
    return (f"the last {n} query rows of one head of the same shape and distribution "
            f"(of {w.B * w.h * w.T_q} rows in the call), {blas}")


# oracle rows per workload for its timing (a second or so each), by T_q
ORACLE_SAMPLE_ROWS = {1: 48, 256: 256, 1024: 1024, 4096: 512, 8192: 256, 16384: 128}


def oracle_estimate(w):
    """(seconds for the whole call, sample description) for the float64 oracle."""
    secs, n, total = oracle_sample(w, ORACLE_SAMPLE_ROWS.get(w.T_q, 256))
    return secs * total / n, describe_sample(w, n) + "; whole-call time scaled from the sample"


def cpu_baseline(peaks, oracle_times):
    """The oracle on the host cores for the whole step, from per-call row
    samples (oracle_times: key -> (seconds per whole call, sample))."""
    calls = step_calls()
    t_roof = sum(work_of(w, peaks)["t_roof"] for _, w, _ in calls)
    secs = sum(oracle_times[key][0] for key, _, _ in calls)
    return {"value": 100.0 * t_roof / secs, "unit": UNIT, "cores": _CORES, "kind": "oracle",
            "sample": "; ".join(f"{key}: {oracle_times[key][1]}" for key, _, _ in calls),
            "seconds_per_step": secs}


# ----------------------------------------------------------------- reference arm
def run_reference(args):
    """The oracle, as it stands, on the host cores: each step is a bounded
    sample of the step's three calls (query rows of the prefills, whole
    decode rows), sized so that warm-up + timed steps take a minute or two."""
    rank, world, _ = dist_init(args.gpus)
    if rank != 0:
        return 0
    peaks = load_peaks()
    calls = step_calls()
    # calibration: seconds per sampled row of each call, on samples of the
    # size the steps use at most (the oracle's matrices grow with the rows)
    per_row = {}
    for key, w, _ in calls:
        oracle_sample(w, 4)                                   # first touch
        secs, n, total = oracle_sample(w, max(1, ORACLE_SAMPLE_ROWS.get(w.T_q, 256) // 4))
        per_row[key] = (secs / n, total)
    budget = 90.0 / max(1, args.steps + args.warmup)        # seconds per step
    share = budget / len(calls)
    rows = {key: int(max(1, min(total, ORACLE_SAMPLE_ROWS.get(w.T_q, 256),
                                share // max(per_row[key][0], 1e-6))))
            for key, w, _ in calls}

    def one_step():
        """Seconds the oracle would take for the whole step: each call's
        sampled rows timed and scaled to all of its rows."""
        t = 0.0
        for key, w, _ in calls:
            secs, n, total = oracle_sample(w, rows[key])
            rows[key] = n
            t += secs * total / n
        return t

    for _ in range(args.warmup):
        one_step()
    tot = sum(one_step() for _ in range(args.steps))
    per_step_s = tot / max(1, args.steps)
    roof = sum(work_of(w, peaks)["t_roof"] for _, w, _ in calls)
    value = 100.0 * roof / per_step_s
    sample = ("each step: " + "; ".join(f"{key}: {describe_sample(w, rows[key])}"
                                        for key, w, _ in calls)
              + "; each call's time scaled from its sampled rows to the whole call")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_block(),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": _CORES, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------- our arm
def time_launches(call, stream, flush=None, n=RUN_LAUNCHES, reps=RUN_REPEATS, warmup=RUN_WARMUP):
    """Per-launch CUDA-event times (ms) of `call` on `stream`: `reps` repeats
    of `n` launches, each launch bracketed by its own events with an L2
    flush before it (outside the events). Returns the mean of each repeat."""
    import torch
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    means = []
    for _ in range(reps):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        for a, b in ev:
            if flush is not None:
                flush()
            a.record(stream)
            call()
            b.record(stream)
        torch.cuda.synchronize()
        means.append(sum(a.elapsed_time(b) for a, b in ev) / n)
    return means


def measure_runs(dev, stream, peaks, with_oracle):
    """Every workload on its own: kernel, time per call, throughput and
    fractions of the two roofs, and the oracle's time for the same call."""
    import torch

    from exact_io_aware_attn_gb300 import _lib
    from exact_io_aware_attn_gb300.inputs import WORKLOADS
    flush_w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_out = torch.empty((), dtype=torch.float32, device=dev)

    def flush():
        # write a buffer twice the size of L2 (evicts the inputs), then read
        # another one (evicts the written lines, so no write-back of them
        # lands inside the timed launch)
        flush_w.zero_()
        torch.sum(flush_r, dim=0, out=flush_out)
    runs = {}
    for w in WORKLOADS:
        q, k, v = (t.to(dev) for t in cached_inputs(w))
        o = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)

        def call():
            _lib.attn_fwd(q, k, v, causal=w.causal, out=o, lse=lse, stream=stream)
        means = time_launches(call, stream, flush=flush)
        st, word = _lib.get_device_error()
        if st != _lib.ATTN_OK:
            raise SystemExit(f"device status {st} ({word:#x}) in workload {w.name}")
        ms = statistics.median(means)
        wk = work_of(w, peaks)
        tflops = wk["flops"] / (ms * 1e-3) / 1e12
        gbs = wk["bytes"] / (ms * 1e-3) / 1e9
        entry = {
            "kernel": _lib.last_kernel_name(), "us_per_call": ms * 1e3,
            "repeats_us": [m * 1e3 for m in means],
            "spread_pct": 100.0 * (max(means) - min(means)) / ms,
            "tflops": tflops, "gbs": gbs,
            "frac_tensor_peak": tflops / peaks["bf16_tflops"],
            "frac_tensor_peak_sustained": tflops / peaks["bf16_tflops_sustained"],
            "frac_hbm_peak": gbs / peaks["hbm_gbs"],
            "bound": wk["bound"], "frac_of_roofline": wk["t_roof"] / (ms * 1e-3),
            "flops": wk["flops"], "bytes": wk["bytes"],
        }
        if with_oracle:
            secs, sample = oracle_estimate(w)
            entry["oracle_s_per_call"] = secs
            entry["oracle_sample"] = sample
        runs[w.name] = entry
        del q, k, v, o, lse
    del flush_w, flush_r, flush_out
    torch.cuda.empty_cache()
    return runs


def run_ours(args):
    import torch

    from exact_io_aware_attn_gb300 import _lib, build as build_mod

    rank, world, local = dist_init(args.gpus)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (there is no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    build_mod.build()
    peaks = load_peaks()
    calls = step_calls()
    works = {key: work_of(w, peaks) for key, w, _ in calls}

    inputs_cpu = {key: cached_inputs(w) for key, w, _ in calls}
    dev_in = {key: [t.to(dev) for t in grp] for key, grp in inputs_cpu.items()}
    outs = {key: (torch.empty_like(q), torch.empty(q.shape[:3], dtype=torch.float32, device=dev))
            for key, (q, _, _) in dev_in.items()}
    causal = {key: w.causal for key, w, _ in calls}
    stream = torch.cuda.current_stream(dev)

    def launch(key):
        q, k, v = dev_in[key]
        o, lse = outs[key]
        _lib.attn_fwd(q, k, v, causal=causal[key], out=o, lse=lse, stream=stream)

    def step():
        for key, _, _ in calls:
            launch(key)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    st, word = _lib.get_device_error()
    if st != _lib.ATTN_OK:
        raise SystemExit(f"device status {st} ({word:#x}) after warm-up")
    kernels = {}
    for key, _, _ in calls:
        launch(key)
        kernels[key] = _lib.last_kernel_name()
    launches_per_step = sum(2 if "+" in name else 1 for name in kernels.values())
    torch.cuda.synchronize()

    K = args.steps
    n_calls = len(calls)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_calls + 1)] for _ in range(K)]
    with ClockSampler(local) as clocks:
        barrier(world)
        torch.cuda.synchronize()
        for i in range(K):
            ev[i][0].record(stream)
            for c, (key, _, _) in enumerate(calls):
                launch(key)
                ev[i][c + 1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        # repeats: >= 3 back-to-back loops of >= 20 steps each, after the
        # timed K steps (whatever K is)
        rep_steps = max(REPEAT_MIN_STEPS, K)
        rep_ev = []
        for _ in range(REPEATS):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(rep_steps):
                step()
            b.record(stream)
            rep_ev.append((a, b))
        torch.cuda.synchronize()
    st, word = _lib.get_device_error()
    if st != _lib.ATTN_OK:
        raise SystemExit(f"device status {st} ({word:#x}) in the timed region")
    total_ms = ev[0][0].elapsed_time(ev[K - 1][n_calls])
    call_ms = {key: sum(e[c].elapsed_time(e[c + 1]) for e in ev) / K
               for c, (key, _, _) in enumerate(calls)}
    step_ms = max_over_ranks(total_ms / K, world, dev)
    rep_ms = [a.elapsed_time(b) / rep_steps for a, b in rep_ev]
    repeats = {"n": REPEATS, "steps_each": rep_steps,
               "ms_per_step": rep_ms, "ms_per_step_median": statistics.median(rep_ms),
               "spread_pct": 100.0 * (max(rep_ms) - min(rep_ms)) / statistics.median(rep_ms)}

    # end to end through the public API with host buffers: pinned H2D of the
    # step's inputs, the three calls, D2H of every output, every step
    host_in = {key: [t.pin_memory() for t in grp] for key, grp in inputs_cpu.items()}
    host_out = {key: (torch.empty(o.shape, dtype=o.dtype).pin_memory(),
                      torch.empty(lse.shape, dtype=torch.float32).pin_memory())
                for key, (o, lse) in outs.items()}
    h2d = sum(t.numel() * t.element_size() for grp in host_in.values() for t in grp)
    d2h = sum(t.numel() * t.element_size() for pair in host_out.values() for t in pair)
    # the C-ABI host-buffer entry: it copies the inputs in, runs the same
    # kernels on its device region, and copies o and lse out, in stream order
    bufs = {}
    for key, grp in host_in.items():
        B_, h_, T_q_, d_ = grp[0].shape
        nbytes = _lib.host_buffer_bytes(B_, h_, grp[1].shape[1], T_q_, grp[1].shape[2], d_)
        bufs[key] = torch.empty(nbytes, dtype=torch.uint8, device=dev)

    def e2e_step():
        for key, _, _ in calls:
            o_h, lse_h = host_out[key]
            _lib.attn_fwd_host(*host_in[key], causal=causal[key], out=o_h, lse=lse_h,
                               device_buffer=bufs[key], stream=stream, synchronize=False)

    e2e_steps = min(K, 20)
    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3 / e2e_steps, world, dev)
    del bufs, host_in, host_out
    del dev_in, outs
    torch.cuda.empty_cache()

    if rank != 0:
        return 0

    with_oracle = world == 1 and not args.no_cpu_baseline
    runs = measure_runs(dev, stream, peaks, with_oracle) if not args.no_runs else None

    roof_step = sum(wk["t_roof"] for wk in works.values())
    value = 100.0 * world * roof_step / (step_ms * 1e-3)
    e2e_value = 100.0 * world * roof_step / (e2e_ms * 1e-3)
    peak_note = "of measured" if peaks["source"] == "measured" else "of fallback"
    call_lines = {}
    for key, w, tkey in calls:
        wk, ms = works[key], call_ms[key]
        tflops = wk["flops"] / (ms * 1e-3) / 1e12
        gbs = wk["bytes"] / (ms * 1e-3) / 1e9
        call_lines[key] = {
            "workload": w.name, "kernel": kernels[key], "bound": wk["bound"],
            "ms_per_launch": ms, "tflops": tflops, "gbs": gbs,
            "frac_tensor_peak": tflops / peaks["bf16_tflops"],
            "frac_hbm_peak": gbs / peaks["hbm_gbs"],
            "frac_of_roofline": wk["t_roof"] / (ms * 1e-3),
            "share_of_step": ms / (total_ms / K),
            "algorithmic_flops_per_launch": wk["flops"],
            "algorithmic_bytes_per_launch": wk["bytes"],
            "traffic": load_traffic(tkey),
        }
    # the dominant kernel: the call with the largest share of the step
    dom = max(call_lines, key=lambda key: call_lines[key]["ms_per_launch"])
    dl = call_lines[dom]
    if dl["bound"] == "tensor":
        roofline = {"bound": "tensor", "achieved": dl["tflops"], "peak": peaks["bf16_tflops"],
                    "unit": "TFLOP/s", "frac": dl["tflops"] / peaks["bf16_tflops"]}
    else:
        roofline = {"bound": "hbm", "achieved": dl["gbs"], "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": dl["gbs"] / peaks["hbm_gbs"]}
    roofline.update({"traffic": dl["traffic"], "kernel": f"{dom}: {dl['kernel']}",
                     "peak_kind": peak_note + " (burst)",
                     "algorithmic_flops_per_launch": dl["algorithmic_flops_per_launch"],
                     "algorithmic_bytes_per_launch": dl["algorithmic_bytes_per_launch"],
                     "ms_per_launch": dl["ms_per_launch"]})
    dec = call_lines["decode"]
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16+f16", "data": "synthetic",
        "config": config_block(),
        "parallelism": "replicas only" if world > 1 else "single GPU",
        "roofline": roofline,
        "roofline_decode": {"bound": "hbm", "achieved": dec["gbs"], "peak": peaks["hbm_gbs"],
                            "unit": "GB/s", "frac": dec["gbs"] / peaks["hbm_gbs"],
                            "traffic": dec["traffic"], "kernel": dec["kernel"],
                            "peak_kind": peak_note},
        "calls": call_lines,
        "clocks": clocks.summary(),
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": e2e_steps},
        "gpu_launches": launches_per_step * K,
        "gpu_launches_note": f"{launches_per_step} per step (two prefill kernels, the decode's "
                             "split and merge kernels) x K timed steps",
        "repeats": repeats,
        # device memory the library needs beyond the caller's inputs and
        # outputs: the decode's split partials (stream-ordered, per call); the
        # prefills need none (the T x T scores never exist)
        "extra_device_bytes": {"prefill_gpt2": 0, "prefill_very_long": 0,
                               "decode": _lib.workspace_bytes(
                                   calls[2][1].B, calls[2][1].h, calls[2][1].T_q,
                                   calls[2][1].T_kv, calls[2][1].d, 0)},
        "peaks": {k: peaks[k] for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained",
                                        "source")},
        "runs": runs,
    }
    if with_oracle and runs is not None:
        by_name = {r: runs[r] for r in runs}
        oracle_times = {key: (by_name[w.name]["oracle_s_per_call"],
                              by_name[w.name]["oracle_sample"]) for key, w, _ in calls}
        line["cpu_baseline"] = cpu_baseline(peaks, oracle_times)
    print(json.dumps(line), flush=True)
    return 0


def run_kernel_case(args):
    """Profiling mode: one call of the step (--kernel-case prefill|decode), or
    any named workload (--kernel-case NAME, see inputs.WORKLOADS), repeated
    --steps times after --warmup calls; prints one JSON line with the mean
    time per call and its throughput, no benchmark line. --case-batch
    overrides B for small ncu captures."""
    import dataclasses

    import torch

    from exact_io_aware_attn_gb300 import _lib, build as build_mod, cost
    from exact_io_aware_attn_gb300.inputs import (DECODE, EXTRA_WORKLOADS, GPT2_PREFILL,
                                                  WORKLOADS, make_workload)

    build_mod.build()
    named = {w.name: w for w in WORKLOADS + EXTRA_WORKLOADS}
    w = {"prefill": GPT2_PREFILL, "decode": DECODE}.get(args.kernel_case) or named[args.kernel_case]
    if args.case_batch:
        w = dataclasses.replace(w, B=args.case_batch)
    q, k, v = (t.cuda() for t in make_workload(w))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    if w.kv_heads != w.h:
        def call():
            _lib.attn_fwd_gqa(q, k, v, causal=w.causal, out=o, lse=lse)
    else:
        def call():
            _lib.attn_fwd(q, k, v, causal=w.causal, out=o, lse=lse)
    if args.splits is not None:
        # prefill with an explicit key-partition count (1 = unsplit)
        ws = torch.empty(max(16, _lib.splitkv_workspace_bytes(w.B, w.h, w.T_q, w.T_kv, w.d,
                                                             args.splits)),
                         dtype=torch.uint8, device=q.device)

        def call():
            _lib.attn_fwd_splitkv(q, k, v, causal=w.causal, out=o, lse=lse,
                                  num_splits=args.splits, workspace=ws)
    paged_bytes = None
    if args.page_size:
        # the decode workload's cache laid out in pages, in a seeded random
        # order; lengths full, or (--var-len) uniform in [T/4, T]
        if w.T_q != 1:
            raise SystemExit("--page-size needs a decode workload (T_q = 1)")
        ps = args.page_size
        gen = torch.Generator().manual_seed(w.seed + 11)
        lens = torch.full((w.B,), w.T_kv, dtype=torch.int32)
        if args.var_len:
            lens = torch.randint(w.T_kv // 4, w.T_kv + 1, (w.B,), generator=gen, dtype=torch.int32)
        max_pages = -(-w.T_kv // ps)
        num_pages = w.B * max_pages
        perm = torch.randperm(num_pages, generator=gen)
        table = perm.reshape(w.B, max_pages).to(torch.int32)
        kp = torch.empty((num_pages, w.kv_heads, ps, w.d), dtype=k.dtype, device=k.device)
        vp = torch.empty_like(kp)
        pages_of = k.view(w.B, w.kv_heads, max_pages, ps, w.d).permute(0, 2, 1, 3, 4)
        kp[table.long().flatten().to(k.device)] = pages_of.reshape(num_pages, w.kv_heads, ps, w.d)
        pages_of = v.view(w.B, w.kv_heads, max_pages, ps, w.d).permute(0, 2, 1, 3, 4)
        vp[table.long().flatten().to(k.device)] = pages_of.reshape(num_pages, w.kv_heads, ps, w.d)
        del k, v
        qd = q[:, :, 0].contiguous()
        od = torch.empty_like(qd)
        lsed = torch.empty((w.B, w.h), dtype=torch.float32, device=q.device)
        table_d, lens_d = table.to(q.device), lens.to(q.device)
        paged_bytes = (2 * int(lens.sum()) * w.kv_heads * w.d * 2 + 2 * w.B * w.h * w.d * 2
                       + w.B * w.h * 4)

        def call():
            _lib.attn_fwd_paged_decode(qd, kp, vp, table_d, lens_d, out=od, lse=lsed)
    if args.backward:
        from exact_io_aware_attn_gb300.inputs import make_dout
        call()
        dout = make_dout(w.B, w.h, w.T_q, w.d, w.dtype, w.seed, device=q.device)
        grads = [torch.empty_like(t) for t in (q, k, v)]
        ws = torch.empty(_lib.bwd_workspace_bytes(w.B, w.h, w.T_q, w.T_kv, w.d), dtype=torch.uint8,
                         device=q.device)

        def call():
            _lib.attn_bwd(q, k, v, o, lse, dout, causal=w.causal, dq=grads[0], dk=grads[1],
                          dv=grads[2], workspace=ws)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        call()
    b.record()
    torch.cuda.synchronize()
    st, word = _lib.get_device_error()
    if st != _lib.ATTN_OK:
        raise SystemExit(f"device status {st} ({word:#x})")
    sec = a.elapsed_time(b) / max(1, args.steps) * 1e-3
    if args.backward:
        fl = cost.bwd_flops(w.B, w.h, w.T_q, w.T_kv, w.d, w.causal)
        by = cost.bwd_min_bytes(w.B, w.h, w.T_q, w.T_kv, w.d, h_kv=w.kv_heads)
    elif paged_bytes is not None:
        fl = cost.flops(w.B, w.h, w.T_q, w.T_kv, w.d, w.causal)
        by = paged_bytes
    else:
        fl = cost.flops(w.B, w.h, w.T_q, w.T_kv, w.d, w.causal)
        by = cost.min_bytes(w.B, w.h, w.T_q, w.T_kv, w.d, h_kv=w.kv_heads)
    peaks = load_peaks()
    kind = "backward" if args.backward else (
        f"paged decode, page {args.page_size}" + (", variable lengths" if args.var_len else "")
        if args.page_size else "forward")
    print(json.dumps({"workload": w.name, "pass": kind,
                      "B": w.B, "kernel": _lib.last_kernel_name(),
                      "us_per_call": sec * 1e6, "tflops": fl / sec / 1e12,
                      "gbs": by / sec / 1e9,
                      "frac_tensor_peak": fl / sec / 1e12 / peaks["bf16_tflops"],
                      "frac_hbm_peak": by / sec / 1e9 / peaks["hbm_gbs"]}), flush=True)
    return 0


def run_naive_table(args):
    """The pages' comparison on GB300: causal attention of B=1, h=12, d=64,
    fp16 heads at T = 512 ... 16384, the IO-aware forward (attn_fwd) beside
    the materialising baseline (attn_fwd_naive, which writes the T x T score
    and probability matrices to device memory). Per T: CUDA-event time per
    call (L2 flushed before each launch), and the device bytes each call
    needs beyond its inputs (outputs plus library workspace). Prints one
    JSON line."""
    import torch

    from exact_io_aware_attn_gb300 import _lib, build as build_mod
    from exact_io_aware_attn_gb300.inputs import F16, make_qkv

    build_mod.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    flush_w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_out = torch.empty((), dtype=torch.float32, device=dev)

    def flush():
        flush_w.zero_()
        torch.sum(flush_r, dim=0, out=flush_out)

    B, h, d = 1, 12, 64
    rows = []
    for T in (512, 1024, 2048, 4096, 8192, 16384):
        q, k, v = (t.to(dev) for t in make_qkv(B, h, T, T, d, F16, 1.0, 0))
        o = torch.empty_like(q)
        lse = torch.empty((B, h, T), dtype=torch.float32, device=dev)
        out_bytes = o.numel() * 2 + lse.numel() * 4
        io_ws = _lib.splitkv_workspace_bytes(B, h, T, T, d, 0)

        def io_call():
            _lib.attn_fwd(q, k, v, causal=True, out=o, lse=lse, stream=stream)
        io_ms = statistics.median(time_launches(io_call, stream, flush=flush))
        io_name = _lib.last_kernel_name()
        o_io = o.clone()
        nb = _lib.naive_workspace_bytes(B, h, T, T)
        ws = torch.empty(nb, dtype=torch.uint8, device=dev)

        def naive_call():
            _lib.attn_fwd_naive(q, k, v, causal=True, out=o, lse=lse, workspace=ws, stream=stream)
        naive_ms = statistics.median(time_launches(naive_call, stream, flush=flush, n=10))
        st, word = _lib.get_device_error()
        if st != _lib.ATTN_OK:
            raise SystemExit(f"device status {st} ({word:#x}) at T={T}")
        diff = float((o.float() - o_io.float()).abs().max())
        rows.append({"T": T, "io_aware_kernel": io_name, "io_aware_us": io_ms * 1e3,
                     "naive_kernel": _lib.last_kernel_name(), "naive_us": naive_ms * 1e3,
                     "speedup": naive_ms / io_ms,
                     "io_aware_bytes_beyond_inputs": out_bytes + io_ws,
                     "naive_bytes_beyond_inputs": out_bytes + nb,
                     "memory_ratio": (out_bytes + nb) / (out_bytes + io_ws),
                     "max_abs_diff_o": diff})
        del q, k, v, o, lse, ws, o_io
        torch.cuda.empty_cache()
    by_t = {r["T"]: r for r in rows}
    print(json.dumps({"table": "io_aware_vs_naive", "B": B, "h": h, "d": d, "dtype": "f16",
                      "causal": True, "rows": rows,
                      "speedup_at_8192": by_t[8192]["speedup"],
                      "memory_ratio_at_16384": by_t[16384]["memory_ratio"]}), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[1])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-runs", action="store_true",
                    help="skip the per-workload measurements (and with them the oracle timing)")
    ap.add_argument("--kernel-case", metavar="prefill|decode|WORKLOAD",
                    help="profiling mode: run only this call of the step, or a named workload")
    ap.add_argument("--case-batch", type=int, default=None,
                    help="batch size override for --kernel-case")
    ap.add_argument("--backward", action="store_true",
                    help="with --kernel-case: time the backward pass (attn_bwd) instead")
    ap.add_argument("--page-size", type=int, default=0,
                    help="with a decode --kernel-case: lay the cache out in pages of this many "
                         "rows (random page order) and time attn_fwd_paged_decode")
    ap.add_argument("--splits", type=int, default=None,
                    help="with a prefill --kernel-case: attn_fwd_splitkv with this many key "
                         "partitions (1 = unsplit; 0 = the library's choice)")
    ap.add_argument("--naive-table", action="store_true",
                    help="time the IO-aware forward beside the materialising baseline at "
                         "T = 512 ... 16384 (B 1, h 12, d 64, fp16, causal)")
    ap.add_argument("--var-len", action="store_true",
                    help="with --page-size: sequence lengths uniform in [T/4, T]")
    args = ap.parse_args(argv)
    if args.naive_table:
        return run_naive_table(args)
    if args.kernel_case:
        return run_kernel_case(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
