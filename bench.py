#!/usr/bin/env python
"""Benchmark of the exact-attention hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input:
  1. causal prefill, GPT-2 shape: B=8, h=12, T=1024, d=64, bf16 (tensor-core
     kernel), and
  2. decode against a KV cache: B=32, h=12, T_q=1, T_kv=16384, d=64, bf16
     (split-KV kernel + exact merge kernel).

Metric: the step's roofline time divided by its measured time, in percent.
The roofline time of a kernel is max(FLOPs / tensor peak, bytes / HBM peak)
with the algorithmic FLOPs (4*d per visible query-key pair, causal pairs
counted) and bytes (Q, K, V read once, O and lse written once); the peaks
are the measured ones in MEASURED_PEAKS.json. `value` is whole-job
throughput in units of one GB300's roofline: 100 * N * t_roof / t_step,
so at N=1 it is the percentage of the roofline reached.

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
KERNEL_SOURCES = {
    "decode": os.path.join(ROOT, "exact_io_aware_attn_gb300", "csrc", "decode_sm103.cu"),
    "prefill": os.path.join(ROOT, "exact_io_aware_attn_gb300", "csrc", "prefill_sm103.cu"),
}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return dict(FALLBACK_PEAKS, source="fallback")


def source_sha(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


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
def step_work():
    from exact_io_aware_attn_gb300 import cost
    from exact_io_aware_attn_gb300.inputs import DECODE, GPT2_PREFILL
    p, d = GPT2_PREFILL, DECODE
    return {
        "prefill_flops": cost.flops(p.B, p.h, p.T_q, p.T_kv, p.d, p.causal),
        "prefill_bytes": cost.min_bytes(p.B, p.h, p.T_q, p.T_kv, p.d),
        "decode_flops": cost.flops(d.B, d.h, d.T_q, d.T_kv, d.d, d.causal),
        "decode_bytes": cost.min_bytes(d.B, d.h, d.T_q, d.T_kv, d.d),
    }


def roofline_times(work, peaks):
    tc = peaks["bf16_tflops"] * 1e12
    bw = peaks["hbm_gbs"] * 1e9
    tp = max(work["prefill_flops"] / tc, work["prefill_bytes"] / bw)
    td = max(work["decode_flops"] / tc, work["decode_bytes"] / bw)
    return tp, td


def config_block():
    from exact_io_aware_attn_gb300.inputs import DECODE, GPT2_PREFILL
    return {
        "workload": "gpt2_causal_prefill_B8_h12_T1024_d64_bf16 + decode_B32_h12_Tkv16384_d64_bf16",
        "prefill": GPT2_PREFILL.describe(),
        "decode": DECODE.describe(),
        "l2": "inputs larger than L2: each step streams the 1.61 GB KV cache, which also "
              "evicts the 38 MB of prefill inputs before the next step",
        "data": "synthetic N(0,1) from torch CPU generator seed 0, q then k then v",
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
def oracle_step_sample(inputs_cpu, n_prefill_heads, n_decode_rows):
    """Time the float64 oracle on a bounded sample of one step. Returns
    (seconds, fraction of the prefill heads, fraction of the decode rows)."""
    import oracle
    from exact_io_aware_attn_gb300.inputs import DECODE, GPT2_PREFILL
    (pq, pk, pv), (dq, dk, dv) = inputs_cpu
    scale = 0.125
    t0 = time.perf_counter()
    done = 0
    for b in range(GPT2_PREFILL.B):
        for h in range(GPT2_PREFILL.h):
            if done == n_prefill_heads:
                break
            oracle.standard_attention(pq[b, h].double().numpy(), pk[b, h].double().numpy(),
                                      pv[b, h].double().numpy(), scale=scale, causal=True)
            done += 1
    rows = 0
    for b in range(DECODE.B):
        for h in range(DECODE.h):
            if rows == n_decode_rows:
                break
            oracle.standard_attention(dq[b, h].double().numpy(), dk[b, h].double().numpy(),
                                      dv[b, h].double().numpy(), scale=scale, causal=False)
            rows += 1
    dt = time.perf_counter() - t0
    return dt, done / (GPT2_PREFILL.B * GPT2_PREFILL.h), rows / (DECODE.B * DECODE.h)


def make_inputs_cpu():
    from exact_io_aware_attn_gb300.inputs import DECODE, GPT2_PREFILL, make_workload
    return make_workload(GPT2_PREFILL), make_workload(DECODE)


def cpu_baseline(inputs_cpu, peaks, prefill_heads=96, decode_rows=384):
    work = step_work()
    tp, td = roofline_times(work, peaks)
    secs, fp, fd = oracle_step_sample(inputs_cpu, prefill_heads, decode_rows)
    value = 100.0 * (fp * tp + fd * td) / secs
    return {"value": value, "unit": UNIT, "cores": _CORES, "kind": "oracle",
            "sample": f"{prefill_heads} of 96 prefill heads and {decode_rows} of 384 decode rows "
                      f"of one step, float64 numpy (BLAS threads {os.environ['OPENBLAS_NUM_THREADS']})",
            "seconds": secs}


# ----------------------------------------------------------------- reference arm
def run_reference(args):
    """The oracle, as it stands, on the host cores: each step is a bounded
    sample of the step's work (whole prefill heads and whole decode rows),
    sized so that warm-up + timed steps take about a minute and a half."""
    rank, world, _ = dist_init(args.gpus)
    if rank != 0:
        return 0
    peaks = load_peaks()
    inputs_cpu = make_inputs_cpu()
    unit_s, _, _ = oracle_step_sample(inputs_cpu, 1, 1)        # calibration unit
    per_step = 90.0 / max(1, args.steps + args.warmup)
    units = int(max(1, min(8, per_step // max(unit_s, 1e-6))))
    heads, rows = units, units
    for _ in range(args.warmup):
        oracle_step_sample(inputs_cpu, heads, rows)
    tot, fp, fd = 0.0, 0.0, 0.0
    for _ in range(args.steps):
        secs, fp, fd = oracle_step_sample(inputs_cpu, heads, rows)
        tot += secs
    work = step_work()
    tp, td = roofline_times(work, peaks)
    per_step_s = tot / max(1, args.steps)
    value = 100.0 * (fp * tp + fd * td) / per_step_s
    sample = (f"each step: {heads} of 96 prefill heads and {rows} of 384 decode rows, "
              f"float64 numpy (BLAS threads {os.environ['OPENBLAS_NUM_THREADS']})")
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
def run_ours(args):
    import torch

    from exact_io_aware_attn_gb300 import _lib, build as build_mod
    from exact_io_aware_attn_gb300.inputs import DECODE, GPT2_PREFILL

    rank, world, local = dist_init(args.gpus)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (there is no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    build_mod.build()
    peaks = load_peaks()
    work = step_work()
    tp_roof, td_roof = roofline_times(work, peaks)

    inputs_cpu = make_inputs_cpu()
    (pq, pk, pv), (dq, dk, dv) = [[t.to(dev) for t in grp] for grp in inputs_cpu]
    po = torch.empty_like(pq)
    plse = torch.empty(pq.shape[:3], dtype=torch.float32, device=dev)
    do = torch.empty_like(dq)
    dlse = torch.empty(dq.shape[:3], dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        _lib.attn_fwd(pq, pk, pv, causal=True, out=po, lse=plse)
        _lib.attn_fwd(dq, dk, dv, causal=False, out=do, lse=dlse)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    st, word = _lib.get_device_error()
    if st != _lib.ATTN_OK:
        raise SystemExit(f"device status {st} ({word:#x}) after warm-up")
    kernels = {"prefill": None, "decode": None}
    _lib.attn_fwd(pq, pk, pv, causal=True, out=po, lse=plse)
    kernels["prefill"] = _lib.last_kernel_name()
    _lib.attn_fwd(dq, dk, dv, causal=False, out=do, lse=dlse)
    kernels["decode"] = _lib.last_kernel_name()
    splits = _lib.decode_num_splits(DECODE.B, DECODE.h, DECODE.T_kv, DECODE.d)

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    with ClockSampler(local) as clocks:
        barrier(world)
        torch.cuda.synchronize()
        for i in range(K):
            ev[i][0].record(stream)
            _lib.attn_fwd(pq, pk, pv, causal=True, out=po, lse=plse)
            ev[i][1].record(stream)
            _lib.attn_fwd(dq, dk, dv, causal=False, out=do, lse=dlse)
            ev[i][2].record(stream)
        torch.cuda.synchronize()
        barrier(world)
    st, word = _lib.get_device_error()
    if st != _lib.ATTN_OK:
        raise SystemExit(f"device status {st} ({word:#x}) in the timed region")
    total_ms = ev[0][0].elapsed_time(ev[K - 1][2])
    pre_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / K
    dec_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / K
    step_ms = max_over_ranks(total_ms / K, world, dev)
    # the K steps as 5 back-to-back repeats (>= 20 steps each at the default K):
    # median and spread of the per-repeat step time
    R = 5 if K >= 5 else 1
    per = K // R
    rep_ms = [ev[r * per][0].elapsed_time(ev[r * per + per - 1][2]) / per for r in range(R)]
    repeats = {"n": R, "steps_each": per, "ms_per_step_median": statistics.median(rep_ms),
               "spread_pct": 100.0 * (max(rep_ms) - min(rep_ms)) / statistics.median(rep_ms)}

    # end to end through the public API with host buffers: pinned H2D of the
    # step's inputs, the two calls, D2H of both outputs, every step
    host_in = [[t.pin_memory() for t in grp] for grp in inputs_cpu]
    host_out = [torch.empty(po.shape, dtype=po.dtype).pin_memory(),
                torch.empty(plse.shape, dtype=torch.float32).pin_memory(),
                torch.empty(do.shape, dtype=do.dtype).pin_memory(),
                torch.empty(dlse.shape, dtype=torch.float32).pin_memory()]
    h2d = sum(t.numel() * t.element_size() for grp in host_in for t in grp)
    d2h = sum(t.numel() * t.element_size() for t in host_out)

    # the C-ABI host-buffer entry: it copies the inputs in, runs the same
    # kernels on its device region, and copies o and lse out, in stream order
    bufs = []
    for grp in host_in:
        B_, h_, T_q_, d_ = grp[0].shape
        nbytes = _lib.host_buffer_bytes(B_, h_, grp[1].shape[1], T_q_, grp[1].shape[2], d_)
        bufs.append(torch.empty(nbytes, dtype=torch.uint8, device=dev))

    def e2e_step():
        _lib.attn_fwd_host(*host_in[0], causal=True, out=host_out[0], lse=host_out[1],
                           device_buffer=bufs[0], stream=stream, synchronize=False)
        _lib.attn_fwd_host(*host_in[1], causal=False, out=host_out[2], lse=host_out[3],
                           device_buffer=bufs[1], stream=stream, synchronize=False)

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

    if rank != 0:
        return 0

    roof_step = tp_roof + td_roof
    value = 100.0 * world * roof_step / (step_ms * 1e-3)
    e2e_value = 100.0 * world * roof_step / (e2e_ms * 1e-3)
    dec_gbs = work["decode_bytes"] / (dec_ms * 1e-3) / 1e9
    pre_tflops = work["prefill_flops"] / (pre_ms * 1e-3) / 1e12
    pre_gbs = work["prefill_bytes"] / (pre_ms * 1e-3) / 1e9
    peak_note = "of measured" if peaks["source"] == "measured" else "of fallback"
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_block(),
        "parallelism": "replicas only" if world > 1 else "single GPU",
        "kernels": kernels, "decode_splits": splits,
        "roofline": {"bound": "hbm", "kernel": "decode (split + merge)", "achieved": dec_gbs,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": dec_gbs / peaks["hbm_gbs"],
                     "traffic": load_traffic("decode"), "peak_kind": peak_note,
                     "algorithmic_bytes_per_launch": work["decode_bytes"],
                     "ms_per_launch": dec_ms},
        "roofline_prefill": {
            "bound": "hbm" if work["prefill_flops"] / work["prefill_bytes"] <
                     peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9) else "tensor",
            "kernel": kernels["prefill"], "achieved_tflops": pre_tflops,
            "tensor_peak_tflops": peaks["bf16_tflops"],
            "frac_of_tensor_peak": pre_tflops / peaks["bf16_tflops"],
            "achieved_gbs": pre_gbs, "frac_of_roofline": tp_roof / (pre_ms * 1e-3),
            "traffic": load_traffic("prefill"), "peak_kind": peak_note,
            "algorithmic_flops_per_launch": work["prefill_flops"],
            "algorithmic_bytes_per_launch": work["prefill_bytes"], "ms_per_launch": pre_ms},
        "clocks": clocks.summary(),
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": e2e_steps},
        "gpu_launches": 3 * K,
        "repeats": repeats,
        # device memory the library needs beyond the caller's inputs and
        # outputs: the decode's split partials (stream-ordered, per call); the
        # prefill needs none (the T x T scores never exist)
        "extra_device_bytes": {"prefill": 0, "decode": _lib.workspace_bytes(
            DECODE.B, DECODE.h, DECODE.T_q, DECODE.T_kv, DECODE.d, 0)},
        "peaks": {k: peaks[k] for k in ("hbm_gbs", "bf16_tflops", "source")},
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inputs_cpu, peaks)
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


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[1])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
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
    ap.add_argument("--var-len", action="store_true",
                    help="with --page-size: sequence lengths uniform in [T/4, T]")
    args = ap.parse_args(argv)
    if args.kernel_case:
        return run_kernel_case(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
