#!/usr/bin/env python3
"""Benchmark of the packed variable-length attention forward on one GB300.

One step = one call of the whole path (plan kernel + fused attention kernel)
over one batch of synthetic input resident in HBM.  The headline workload is
the largest one that fits one GPU: one sequence L=65556, 16 heads, head_dim
72 (attention_forward shape-table row #8).  The line also carries a second
full record for L=16742, 32 heads, head_dim 128 (row #9) under "records",
and every workload's microseconds (median, p10, p90), TFLOP/s and SM clock
under "shapes".  Metric: TFLOP/s with FLOPs = 4 * sum(L_q * L_k) * H * D
(true head_dim).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) the ranks split the heads of the workload (strong
scaling: the whole job is one call's worth of work): rank r computes its
contiguous block of heads in place with attn_varlen_fwd_heads, with no
collective on the data path; the slowest rank sets the time and rank 0
prints the JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from workloads import (C1, C2, C3, C4, C5, CHUNK_CONFIGS, CONFIGS, D256, EXTRA_CONFIGS,  # noqa: E402
                       PAGED_CONFIGS, make_inputs, make_paged_inputs, sample_rows)

ALL_WORKLOADS = {**CONFIGS, **EXTRA_CONFIGS}

HEADLINE = C4
SECOND = C3  # the other full record (the dense head_dim-128 shape)
METRIC = "varlen attn fwd TFLOP/s (4*sum(L^2)*H*D)"
PAGE_TPROD_TFLOPS = {  # the page's T_Prod converted with the same FLOP count
    C1.name: 2.0, C2.name: 80.5, C3.name: 123.1, C4.name: 83.3}
L2_FLUSH_BYTES = 256 << 20
NOMINAL_BF16_TFLOPS = 2250.0  # GB300 dense bf16, nominal (context; the roofline uses the measured peak)
GRAPH_CALLS = 20              # calls per CUDA-graph replay for the launch-bound workload


# The sources that build, plan and launch the attention kernels (the paged
# decode and chunked delta-rule kernels live in translation units of their own
# and cannot change them).
ATTN_KERNEL_SOURCES = ("attn_varlen_api.cu", "attn_varlen_internal.h", "attn_varlen_kernels.cu",
                       "attn_varlen_device.cuh", "attn_varlen_d256.cu", "ptx.cuh")


def kernel_source_sha() -> str:
    import hashlib
    csrc = os.path.join(ROOT, "variable_length_prefill_gb300", "csrc")
    h = hashlib.sha256()
    for n in ATTN_KERNEL_SOURCES:
        h.update(n.encode())
        with open(os.path.join(csrc, n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(workload_name: str):
    """DRAM bytes of one fwd launch from the committed ncu summary, or None
    when the kernel sources changed since that capture."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("csrc_sha256") != kernel_source_sha():
        return None
    return d.get("traffic_bytes", {}).get(workload_name)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"bf16_tflops": d["bf16_tflops"], "bf16_tflops_sustained": d.get("bf16_tflops_sustained"),
                "hbm_gbs": d["hbm_gbs"], "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock/throttle sampling while the timed regions run.

    Every sample carries nvidia-smi's timestamp, so one sampler can cover
    several timed legs: ``window(t0, t1)`` summarises the samples taken
    between two ``time.time()`` readings."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"attn_varlen_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def samples(self):
        """[(epoch seconds or None, sm MHz, max MHz, set of active reasons)]"""
        import datetime
        out = []
        if self.proc is None or not os.path.exists(self.path):
            return out
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    sm, smax = float(parts[2]), float(parts[3])
                except ValueError:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    ts = None
                reasons = {n for n, v in zip(self.REASONS, parts[6:10]) if v.lower() == "active"}
                out.append((ts, sm, smax, reasons))
        return out

    def summary(self, t0: float | None = None, t1: float | None = None):
        """Median SM clock under load, max clock, p10/p90 and throttle reasons
        of the samples in [t0, t1] (all samples without a window)."""
        smp = self.samples()
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        if t0 is not None:
            smp = [x for x in smp if x[0] is not None and t0 <= x[0] <= t1]
        if not smp:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        mx = smp[-1][2]
        sms = [x[1] for x in smp]
        busy = sorted(s for s in sms if s > 0.3 * mx) or sorted(sms)
        reasons = set().union(*(x[3] for x in smp))
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": mx,
                "sm_mhz_p10": busy[len(busy) // 10], "sm_mhz_p90": busy[(9 * len(busy)) // 10],
                "reasons": sorted(reasons), "samples": len(smp)}


def cpu_oracle_rate(w, max_seconds=12.0, nthreads=0, x=None):
    """Oracle throughput on a bounded, seeded sample of rows of workload w
    (``x``: its inputs, when already drawn)."""
    import oracle
    x = make_inputs(w) if x is None else x
    rows_all = sample_rows(w, 4096, seed_offset=2000)
    cu = x["cu_q"]
    # rows of one head, all keys of their sequence: time a growing sample
    n = 64
    t_used, done_rows, done_flops = 0.0, 0, 0.0
    lk = np.diff(x["cu_k"])
    seq_of = np.searchsorted(cu, rows_all[:, 0], side="right") - 1
    start = 0
    while t_used < max_seconds and start < rows_all.shape[0]:
        rows = rows_all[start:start + n]
        t0 = time.perf_counter()
        oracle.attn_rows(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"], rows, nthreads=nthreads)
        t_used += time.perf_counter() - t0
        done_rows += rows.shape[0]
        done_flops += float(np.sum(4.0 * lk[seq_of[start:start + n]] * w.head_dim))
        start += n
        n = min(n * 2, 4096)
    return {"rows": done_rows, "seconds": t_used, "tflops": done_flops / t_used / 1e12,
            "rows_per_s": done_rows / t_used, "cores": oracle.max_threads(nthreads)}


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle, timed on the host cores.

    Each step is a bounded sample of the headline workload (rows of it, all
    keys each), sized so that warm-up plus timed steps take about a minute."""
    if rank != 0:
        return
    w = ALL_WORKLOADS[args.workload] if args.workload else HEADLINE
    x = make_inputs(w)
    per_step = min(5.0, max(0.2, 60.0 / max(args.steps + args.warmup, 1)))
    for _ in range(args.warmup):
        cpu_oracle_rate(w, max_seconds=per_step, x=x)
    runs = [cpu_oracle_rate(w, max_seconds=per_step, x=x) for _ in range(args.steps)]
    flops = sum(r["tflops"] * r["seconds"] for r in runs)
    secs = sum(r["seconds"] for r in runs)
    val = flops / secs if secs > 0 else 0.0
    rows = sum(r["rows"] for r in runs)
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": secs / max(args.steps, 1) * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, world),
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": runs[0]["cores"] if runs else None,
                             "kind": "oracle",
                             "sample": f"{rows} seeded (token, head) rows of {w.name}, all keys "
                                       f"each, {per_step:.1f} s per step"},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def max_over_ranks(x: float, device) -> float:
    """Largest value of x over all ranks (the slowest rank sets the time)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_throughput(job_flops_per_step: float, steps: int, seconds: float) -> float:
    """TFLOP/s of all ranks together: ``job_flops_per_step`` is the work all
    ranks do in one step together (the ranks split one workload's heads),
    timed by the slowest rank."""
    return job_flops_per_step * steps / seconds / 1e12


class L2Flush:
    """Run before each timed call: write a buffer larger than L2, then read
    it back.  Measured on GB300: after the write alone a 276-token call
    timed the same as with no flush at all (19.4 against 19.0 us; with the
    read-back 26.6 us), so the write did not evict a small working set from
    L2, and it left dirty lines that an HBM-bound call (paged decode row #0:
    34.8 against 28.7 us) wrote back inside its own timed region.  After
    the read-back L2 holds clean lines of the buffer only."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
        self.acc = torch.zeros((), dtype=torch.int64, device=dev)

    def __call__(self):
        import torch
        self.w.fill_(1)
        torch.sum(self.w, dim=0, dtype=torch.int64, out=self.acc)


L2_NOTE = "flushed before every step (256 MiB written, then read back)"


# GPU-side spin before each timed call (outside the timed region), so the
# host has queued the call's launches before its start event: a short call
# is then timed on the device alone, without host enqueue gaps.
SPIN_CYCLES = 200_000


def time_calls(fn, steps, flush_buf, stream):
    import torch
    durs = []
    for _ in range(steps):
        if flush_buf is not None:
            flush_buf()
        torch.cuda._sleep(SPIN_CYCLES)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        durs.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in durs]


def graph_us_per_call(fn, stream) -> float:
    """Microseconds per call of `fn` replayed GRAPH_CALLS times from one
    captured CUDA graph (launch overhead amortised); L2 stays warm."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(GRAPH_CALLS):
            fn()
    g.replay()
    torch.cuda.synchronize()
    reps = []
    for _ in range(5):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        reps.append(a.elapsed_time(b) * 1e3 / GRAPH_CALLS)
    return statistics.median(reps)


def run_profile_chunk(args):
    """Only the chunked delta-rule output on one of the page's shapes: warm-up
    and timed calls with L2 flushed before each, for runs under a profiler."""
    import torch

    import variable_length_prefill_gb300 as vlp
    dev = torch.device("cuda", 0)
    vlp.load()
    cw = CHUNK_CONFIGS[args.profile_chunk]
    gen = torch.Generator(device=dev).manual_seed(cw.seed)
    B, T, Hq, Hv = cw.batch_size, cw.token_count, cw.num_q_heads, cw.num_v_heads
    rnd = lambda *sh: (torch.randn(*sh, device=dev, generator=gen) * 0.02).to(torch.bfloat16)  # noqa: E731
    q, k, v = rnd(B, T, Hq, 128), rnd(B, T, Hq, 128), rnd(B, T, Hv, 128)
    h = rnd(B, cw.num_chunks, Hv, 128, 128)
    g = -torch.rand(B, T, Hv, device=dev, generator=gen)
    out = torch.empty(B, T, Hv, 128, dtype=torch.bfloat16, device=dev)
    flush = L2Flush(dev)
    fn = lambda: vlp.chunk_delta_rule_output(q, k, v, h, g, out=out)  # noqa: E731
    for _ in range(args.warmup):
        fn()
    durs = time_calls(fn, args.steps, flush, torch.cuda.current_stream(dev))
    vlp.check()
    us = statistics.median(durs) * 1e3
    print(json.dumps({"profile": True, "workload": "chunk_o_" + cw.name, "steps": args.steps,
                      "us_median": round(us, 2),
                      "gbs_algorithmic": round(cw.algorithmic_bytes() / (us * 1e-6) / 1e9, 1)}),
          flush=True)


def run_profile_paged(args):
    """Only paged decode on one of the page's shapes: warm-up and timed calls
    with L2 flushed before each, for runs under a profiler."""
    import numpy as np
    import torch

    import variable_length_prefill_gb300 as vlp
    dev = torch.device("cuda", 0)
    vlp.load()
    pw = PAGED_CONFIGS[args.profile_paged]
    xs = make_paged_inputs(pw)
    tdt = torch.bfloat16 if pw.dtype == "bf16" else torch.float16
    t = {n: torch.from_numpy(xs[n].view(np.int16)).view(tdt).to(dev)
         for n in ("query", "k_cache", "v_cache")}
    tables = torch.from_numpy(xs["block_tables"]).to(dev)
    lens = torch.from_numpy(xs["seq_lens"]).to(dev)
    out = torch.empty_like(t["query"])
    flush = L2Flush(dev)
    fn = lambda: vlp.paged_attn_decode(t["query"], t["k_cache"], t["v_cache"], tables, lens,  # noqa: E731
                                       out=out)
    for _ in range(args.warmup):
        fn()
    durs = time_calls(fn, args.steps, flush, torch.cuda.current_stream(dev))
    vlp.check()
    us = statistics.median(durs) * 1e3
    print(json.dumps({"profile": True, "workload": "paged_" + pw.name, "steps": args.steps,
                      "us_median": round(us, 2),
                      "gbs_algorithmic": round(pw.algorithmic_bytes() / (us * 1e-6) / 1e9, 1)}),
          flush=True)


def workload_config(w, world: int = 1) -> dict:
    """The JSON line's config for workload w (both arms print the same)."""
    return {"workload": w.name, "seq_lens": list(w.seq_lens_q), "num_heads": w.num_heads,
            "head_dim": w.head_dim, "l2": L2_NOTE,
            "parallelism": f"heads split over {world} GPU(s)"}


def percentiles_us(durs_ms) -> dict:
    """Median, p10 and p90 of CUDA-event durations (ms) in microseconds."""
    d = sorted(durs_ms)
    return {"us": round(statistics.median(d) * 1e3, 2), "us_p10": round(d[len(d) // 10] * 1e3, 2),
            "us_p90": round(d[(9 * len(d)) // 10] * 1e3, 2), "calls": len(d)}


def timed_leg(fn, min_calls, flush_buf, stream, min_seconds=0.25):
    """CUDA-event durations (ms) of at least ``min_calls`` calls, repeated
    until the leg also spans ``min_seconds`` of wall time (so the clock
    sampler sees it), with its (start, end) wall-clock times."""
    import torch
    t0 = time.time()
    durs = []
    while True:
        durs += time_calls(fn, min_calls, flush_buf, stream)
        if time.time() - t0 >= min_seconds:
            break
    torch.cuda.synchronize()
    return durs, (t0, time.time())


def clock_entry(c: dict) -> dict:
    return {"sm_mhz": c.get("sm_mhz"), "sm_mhz_p10": c.get("sm_mhz_p10"),
            "sm_mhz_p90": c.get("sm_mhz_p90"), "reasons": c.get("reasons"),
            "samples": c.get("samples")}


def roofline_block(w, per_call_tflops, peaks, kernel):
    return {"bound": "tensor", "achieved": round(per_call_tflops, 2),
            "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": round(per_call_tflops / peaks["bf16_tflops"], 4),
            "frac_of_nominal_2250": round(per_call_tflops / NOMINAL_BF16_TFLOPS, 4),
            "traffic": measured_traffic(w.name),
            "algorithmic_bytes": w.algorithmic_bytes(),
            "peak_source": peaks["source"] + " bf16 burst",
            "kernel": kernel}


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import variable_length_prefill_gb300 as vlp
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    vlp.load()
    peaks = load_peaks()
    stream = torch.cuda.current_stream(dev)

    def device_inputs(w):
        x = make_inputs(w)
        t = {n: torch.from_numpy(x[n].view(np.int16)).view(torch.bfloat16).to(dev)
             for n in ("q", "k", "v")}
        return x, t, torch.from_numpy(x["cu_q"]).to(dev), torch.from_numpy(x["cu_k"]).to(dev)

    def kernel_name(w):
        return (f"attn_varlen_fwd_kernel<{w.head_dim}> (+ plan kernel in the timed call)")

    flush = L2Flush(dev)
    w = ALL_WORKLOADS[args.workload] if args.workload else HEADLINE
    x, t, cu_q, cu_k = device_inputs(w)
    out = torch.empty_like(t["q"])
    # this rank's heads (all of them on one GPU)
    shard = vlp.head_shard(w.num_heads, rank, world) if world > 1 else None
    step = lambda: vlp.attn_varlen_fwd(t["q"], t["k"], t["v"], cu_q, cu_k, out=out,  # noqa: E731
                                       heads=shard)
    for _ in range(args.warmup):
        step()
    vlp.check()

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clocks:
        durs = time_calls(step, args.steps, flush, stream)
    vlp.check()
    if args.profile:
        # kernels only (for profiler runs): no end-to-end leg, shapes or CPU baseline
        if rank == 0:
            print(json.dumps({"profile": True, "workload": w.name, "steps": args.steps,
                              "ms_per_step": sum(durs) / args.steps}), flush=True)
        return
    t_sum = max_over_ranks(sum(durs) / 1e3, dev)  # seconds of device time over the K steps
    flops = w.flops()  # the whole job's work per step (all ranks together)
    value = whole_job_throughput(flops, args.steps, t_sum)
    ms_per_step = t_sum / args.steps * 1e3
    per_call_tflops = flops / world / (t_sum / args.steps) / 1e12  # one GPU's kernel rate

    # End to end through the public API with host buffers (pinned): every
    # step copies its inputs host -> device, runs the call and copies the
    # output back.  Two buffer sets let step i+1's input copies and step i-1's
    # output copy run on copy streams while step i computes; each step still
    # moves all of its bytes inside the timed region.  The serial form (copy,
    # compute, copy on one stream) is reported beside it.
    host = {n: torch.from_numpy(x[n].view(np.int16)).pin_memory() for n in ("q", "k", "v")}
    hcu_q = torch.from_numpy(x["cu_q"]).pin_memory()
    hcu_k = torch.from_numpy(x["cu_k"]).pin_memory()
    houts = [torch.empty(host["q"].shape, dtype=torch.int16).pin_memory() for _ in range(2)]
    bufs = [{"q": torch.empty_like(t["q"]), "k": torch.empty_like(t["k"]),
             "v": torch.empty_like(t["v"]), "cq": torch.empty_like(cu_q), "ck": torch.empty_like(cu_k),
             "out": torch.empty_like(t["q"])} for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host.values()) + 2 * hcu_q.numel() * 4
    d2h = houts[0].numel() * 2
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def copy_in(b):
        b["q"].view(torch.int16).copy_(host["q"], non_blocking=True)
        b["k"].view(torch.int16).copy_(host["k"], non_blocking=True)
        b["v"].view(torch.int16).copy_(host["v"], non_blocking=True)
        b["cq"].copy_(hcu_q, non_blocking=True)
        b["ck"].copy_(hcu_k, non_blocking=True)

    def run_e2e_pipelined(n):
        """n steps; returns seconds from the first input copy to the last output copy."""
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_comp = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        start.record(s_in)
        s_out.wait_event(start)
        stream.wait_event(start)
        for i in range(n):
            b, ho = bufs[i % 2], houts[i % 2]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_comp[i - 2])  # step i-2 has read this buffer set
                copy_in(b)
                ev_in[i].record(s_in)
            stream.wait_event(ev_in[i])
            if i >= 2:
                stream.wait_event(ev_out[i - 2])  # step i-2's output has been copied out
            vlp.attn_varlen_fwd(b["q"], b["k"], b["v"], b["cq"], b["ck"], out=b["out"],
                                heads=shard, stream=stream)
            ev_comp[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[i])
                ho.copy_(b["out"].view(torch.int16), non_blocking=True)
                ev_out[i].record(s_out)
        end.record(s_out)
        torch.cuda.synchronize()
        return start.elapsed_time(end) / 1e3

    def e2e_serial_step():
        b = bufs[0]
        copy_in(b)
        vlp.attn_varlen_fwd(b["q"], b["k"], b["v"], b["cq"], b["ck"], out=b["out"], heads=shard)
        houts[0].copy_(b["out"].view(torch.int16), non_blocking=True)

    e2e_steps = max(3, min(args.steps, 20))
    run_e2e_pipelined(2)
    e2e_value = whole_job_throughput(flops, e2e_steps,
                                     max_over_ranks(run_e2e_pipelined(e2e_steps), dev))
    for _ in range(2):
        e2e_serial_step()
    torch.cuda.synchronize()
    e2e_durs = time_calls(e2e_serial_step, e2e_steps, None, stream)
    e2e_serial = whole_job_throughput(flops, e2e_steps, max_over_ranks(sum(e2e_durs) / 1e3, dev))
    del bufs, host, houts

    # The second full record and every workload once more, under one clock
    # sampler: microseconds per call (median, p10, p90) with L2 flushed
    # before each call (cold) and without (warm), the SM clock of each leg,
    # and cycles per call (us x MHz) to separate clock drift from cache
    # effects; for the launch-bound C1 also the time per call inside a
    # replayed CUDA graph.
    records, shapes = {}, {}
    if not args.headline_only:
        with ClockSampler(local_rank) as sampler:
            if w is not SECOND:
                xs, ts, cq, ck = device_inputs(SECOND)
                os_ = torch.empty_like(ts["q"])
                fn = lambda: vlp.attn_varlen_fwd(ts["q"], ts["k"], ts["v"], cq, ck, out=os_)  # noqa: E731
                for _ in range(3):
                    fn()
                d2, win = timed_leg(fn, max(args.steps, 20), flush, stream)
                vlp.check()
                t2 = max_over_ranks(statistics.median(d2) / 1e3, dev)
                tf2 = SECOND.flops() / t2 / 1e12
                records[SECOND.name] = {
                    "metric": METRIC, "value": round(tf2 * world, 3), "unit": "TFLOP/s",
                    "ms_per_step": round(t2 * 1e3, 4), **percentiles_us(d2),
                    "config": workload_config(SECOND),
                    "roofline": roofline_block(SECOND, tf2, peaks, kernel_name(SECOND)),
                    "clocks": clock_entry(sampler.summary(*win))}
                del ts, os_
            for ws in (C1, C2, C3, C4, C5, D256):
                xs, ts, cq, ck = device_inputs(ws)
                os_ = torch.empty_like(ts["q"])
                fn = lambda: vlp.attn_varlen_fwd(ts["q"], ts["k"], ts["v"], cq, ck, out=os_)  # noqa: E731
                for _ in range(3):
                    fn()
                n = 10 if ws is C4 else 20
                cold, win_c = timed_leg(fn, n, flush, stream)
                warm, win_w = timed_leg(fn, n, None, stream)
                pc, pw = percentiles_us(cold), percentiles_us(warm)
                cc, cw_ = clock_entry(sampler.summary(*win_c)), clock_entry(sampler.summary(*win_w))
                tf = ws.flops() / (pc["us"] * 1e-6) / 1e12
                entry = {**pc, "tflops": round(tf, 2),
                         "pct_bf16_peak": round(100.0 * tf / peaks["bf16_tflops"], 2),
                         "pct_nominal_2250": round(100.0 * tf / NOMINAL_BF16_TFLOPS, 2),
                         "gbs_algorithmic": round(ws.algorithmic_bytes() / (pc["us"] * 1e-6) / 1e9, 1),
                         "page_tprod_tflops": PAGE_TPROD_TFLOPS.get(ws.name),
                         "clocks": cc,
                         "kcycles": round(pc["us"] * cc["sm_mhz"] / 1e3, 1) if cc["sm_mhz"] else None,
                         "warm_l2": {**pw, "clocks": cw_,
                                     "kcycles": round(pw["us"] * cw_["sm_mhz"] / 1e3, 1)
                                     if cw_["sm_mhz"] else None}}
                if ws is C1:
                    entry["us_per_call_in_graph"] = round(graph_us_per_call(fn, stream), 2)
                shapes[ws.name] = entry
                del ts, os_
            vlp.check()
            # the causal variant of the same workloads (FLOPs of the visible pairs)
            for ws in (C2, C3, C5, D256):
                xs, ts, cq, ck = device_inputs(ws)
                os_ = torch.empty_like(ts["q"])
                fn = lambda: vlp.attn_varlen_fwd(ts["q"], ts["k"], ts["v"], cq, ck, out=os_,  # noqa: E731
                                                 causal=True)
                for _ in range(3):
                    fn()
                d, win = timed_leg(fn, 10, flush, stream)
                pc = percentiles_us(d)
                vis = sum(int(np.clip(np.arange(a) + 1 + b - a, 0, b).sum())
                          for a, b in zip(ws.seq_lens_q, ws.lens_k) if a > 0 and b > 0)
                shapes[ws.name + "_causal"] = {
                    **pc, "tflops": round(4.0 * vis * ws.num_heads * ws.head_dim /
                                          (pc["us"] * 1e-6) / 1e12, 2),
                    "clocks": clock_entry(sampler.summary(*win))}
                del ts, os_
            # paged single-query decode: the page's shape table, HBM-bound
            for name, pw in PAGED_CONFIGS.items():
                xs = make_paged_inputs(pw)
                tdt = torch.bfloat16 if pw.dtype == "bf16" else torch.float16
                pt = {n: torch.from_numpy(xs[n].view(np.int16)).view(tdt).to(dev)
                      for n in ("query", "k_cache", "v_cache")}
                tb = torch.from_numpy(xs["block_tables"]).to(dev)
                ln = torch.from_numpy(xs["seq_lens"]).to(dev)
                po = torch.empty_like(pt["query"])
                fn = lambda: vlp.paged_attn_decode(pt["query"], pt["k_cache"], pt["v_cache"],  # noqa: E731
                                                   tb, ln, out=po)
                for _ in range(3):
                    fn()
                d, win = timed_leg(fn, 20, flush, stream, min_seconds=0.1)
                pc = percentiles_us(d)
                gbs = pw.algorithmic_bytes() / (pc["us"] * 1e-6) / 1e9
                shapes["paged_" + pw.name] = {
                    **pc, "gbs_algorithmic": round(gbs, 1),
                    "pct_hbm": round(100.0 * gbs / peaks["hbm_gbs"], 2),
                    "clocks": clock_entry(sampler.summary(*win))}
            vlp.check()
            # chunked gated delta-rule output: the page's shape table, HBM-bound;
            # inputs drawn on the device with the test recipe's distributions
            for name, cw in CHUNK_CONFIGS.items():
                gen = torch.Generator(device=dev).manual_seed(cw.seed)
                B, T, Hq, Hv = cw.batch_size, cw.token_count, cw.num_q_heads, cw.num_v_heads
                rnd = lambda *sh: (torch.randn(*sh, device=dev, generator=gen) * 0.02).to(torch.bfloat16)  # noqa: E731
                cq_, ck_, cv_ = rnd(B, T, Hq, 128), rnd(B, T, Hq, 128), rnd(B, T, Hv, 128)
                ch_ = rnd(B, cw.num_chunks, Hv, 128, 128)
                cg_ = -torch.rand(B, T, Hv, device=dev, generator=gen)
                co_ = torch.empty(B, T, Hv, 128, dtype=torch.bfloat16, device=dev)
                fn = lambda: vlp.chunk_delta_rule_output(cq_, ck_, cv_, ch_, cg_, out=co_)  # noqa: E731
                for _ in range(3):
                    fn()
                d, win = timed_leg(fn, 20, flush, stream, min_seconds=0.1)
                pc = percentiles_us(d)
                gbs = cw.algorithmic_bytes() / (pc["us"] * 1e-6) / 1e9
                shapes["chunk_o_" + cw.name] = {
                    **pc, "gbs_algorithmic": round(gbs, 1),
                    "pct_hbm": round(100.0 * gbs / peaks["hbm_gbs"], 2),
                    "clocks": clock_entry(sampler.summary(*win))}
                del cq_, ck_, cv_, ch_, cg_, co_
            vlp.check()

    if rank != 0:
        return
    cpu = cpu_oracle_rate(w, max_seconds=args.cpu_seconds, x=x)
    cpu1 = cpu_oracle_rate(w, max_seconds=min(4.0, args.cpu_seconds), nthreads=1, x=x)
    tprod = PAGE_TPROD_TFLOPS.get(w.name)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "strong",
        # the page's T_Prod for this workload (other, unnamed hardware): context
        "vs_baseline": round(value / tprod, 3) if tprod else None,
        "dtype": "bf16", "data": "synthetic",
        "config": workload_config(w, world),
        **{k: v for k, v in percentiles_us(durs).items() if k != "us"},
        "roofline": roofline_block(w, per_call_tflops, peaks, kernel_name(w)),
        "cpu_baseline": {"value": cpu["tflops"], "unit": "TFLOP/s", "cores": cpu["cores"],
                         "kind": "oracle", "rows_per_s": cpu["rows_per_s"],
                         "rows_per_s_1_thread": cpu1["rows_per_s"],
                         "sample": f"{cpu['rows']} seeded (token, head) rows of {w.name}, "
                                   f"all keys each, {cpu['seconds']:.1f} s"},
        "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "form": "inputs of step i+1 and the output of step i-1 copied on two copy "
                        "streams while step i computes (two buffer sets)",
                "serial_value": round(e2e_serial, 3)},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks.summary(),
        "records": records,
        "shapes": shapes,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--headline-only", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--workload", choices=sorted(ALL_WORKLOADS), default=None,
                    help="time this workload instead of the headline one")
    ap.add_argument("--profile", action="store_true",
                    help="warm-up and timed steps only, for runs under a profiler")
    ap.add_argument("--profile-chunk", choices=sorted(CHUNK_CONFIGS), default=None,
                    help="time only the chunked delta-rule output on this shape (profiler runs)")
    ap.add_argument("--profile-paged", choices=sorted(PAGED_CONFIGS), default=None,
                    help="time only paged decode on this shape (profiler runs)")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.profile_chunk:
        run_profile_chunk(args)
        return
    if args.profile_paged:
        run_profile_paged(args)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
