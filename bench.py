"""Benchmark of the GB300 fused attention backward (one JSON line on rank 0).

A step is one whole backward pass -- preprocess, main kernel, postprocess --
over the workload the headline metric is quoted on: B=2, Hq=32, Hkv=8 (GQA),
Sq=Sk=8192, D=128, bf16, causal (seeded synthetic inputs; O and LSE from the
library's forward, outside the timed region).  The inputs of a step (Q, K, V,
O, dO: about 470 MB) are larger than the 129 MB L2, so no flush is needed
between steps.  --workload picks another of the five workloads (varlen
included); one whose inputs are under 256 MB has a 256 MB buffer written
between timed steps, outside the per-step events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

value  : TFLOPS over all ranks, FLOP = 10*B*Hq*Sq*Sk*D / 2 (causal), device
         time from CUDA events with inputs resident in HBM
e2e    : the same metric through fa_bwd with host (pinned) buffers: each step
         copies its inputs in and its outputs (dQ, dK, dV) out; copies and
         compute of consecutive steps overlap on separate streams
roofline: the main kernel (a dense contraction, tensor-bound) against the
         measured dense bf16 peak
cpu_baseline: the fp64 CPU oracle, as it stands, on a bounded sample (a causal
         prefix of one kv-head group), timed on this host's cores
--impl reference: the same metric for the oracle alone (the reference arm).

Multi-GPU (torchrun, N>1): independent replicas of the workload, one per GPU,
no collective on the data path ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attn-bwd TFLOPS/GPU (10·B·H·Sq·Sk·D, causal halved) and % of bf16 tensor peak"
UNIT = "TFLOPS"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return dict(bf16=d["bf16_tflops"], bf16_sustained=d.get("bf16_tflops_sustained"),
                    hbm=d["hbm_gbs"], source="measured")
    return dict(bf16=1900.0, bf16_sustained=1700.0, hbm=6800.0, source="fallback")


def clock_log_path(name):
    """Where the clock sampler writes its raw CSV: $FA_BENCH_LOG_DIR if set,
    else the system temporary directory (the JSON line carries the summary)."""
    import tempfile
    d = os.environ.get("FA_BENCH_LOG_DIR") or tempfile.gettempdir()
    return os.path.join(d, "%s.%d.csv" % (name, os.getpid()))


def max_over_ranks(x, device):
    """The largest value of x over all ranks of the process group (x itself
    without one): the job's time is that of its slowest rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flop_per_rank, world_size, ms_per_step):
    """Whole-job TFLOPS: the work of every rank over the slowest rank's time."""
    return flop_per_rank * world_size / (ms_per_step * 1e-3) / 1e12


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi clocks / throttle reasons, sampled every 10 ms from start()
    (before the warm-up, since the tool takes a while to come up) to stop();
    stop(window) keeps the samples whose timestamps fall inside the host-clock
    window of the timed region."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, path: str):
        self.path = path
        self.proc = None
        try:
            self.fh = open(path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-i", str(device_index), "-lms", "10"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    @staticmethod
    def _seconds(stamp):
        import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(stamp, fmt).timestamp()
            except ValueError:
                pass
        return None

    def stop(self, window=None):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append((self._seconds(parts[0]), float(parts[2]), float(parts[3]),
                             [n for n, v in zip(names, parts[6:10]) if v.lower() == "active"]))
            except ValueError:
                continue
        scope = "whole run"
        if window is not None:
            inside = [r for r in rows if r[0] is not None and window[0] <= r[0] <= window[1]]
            if inside:
                rows, scope = inside, "timed region"
        if not rows:
            return None
        sm = [r[1] for r in rows]
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(r[2] for r in rows),
                "reasons": sorted({n for r in rows for n in r[3]}), "samples": len(rows),
                "scope": scope}


def cpu_baseline(w, inputs_cpu, prefix: int):
    """Times the oracle's backward on a causal prefix of one kv-head group.

    Sample: batch 0, kv head 0 with its G query heads, positions [0, prefix);
    the oracle recomputes its own fp64 forward.  Returns (TFLOPS, seconds, cores)."""
    import numpy as np

    import oracle
    from attention_backward_preprocess_gb300.workloads import bwd_flops
    G = w.Hq // w.Hkv
    q = inputs_cpu["q"][:1, :prefix, :G].double().numpy()
    k = inputs_cpu["k"][:1, :prefix, :1].double().numpy()
    v = inputs_cpu["v"][:1, :prefix, :1].double().numpy()
    do = inputs_cpu["dout"][:1, :prefix, :G].double().numpy()
    sub = w.with_(B=1, Sq=prefix, Sk=prefix, Hq=G, Hkv=1, varlen=None)
    cores = oracle.max_threads()
    t0 = time.perf_counter()
    oracle.backward(q, k, v, do, w.softmax_scale, w.causal)
    dt = time.perf_counter() - t0
    tflops = bwd_flops(sub) / dt / 1e12
    return tflops, dt, cores, ("oracle fp64 backward (own forward) on seeded inputs shaped like "
                               "%s: 1 kv head with its %d query heads, %d positions, %s "
                               "(%.3g algorithmic FLOP)" % (w.name, G, prefix,
                                                            "causal" if w.causal else "full",
                                                            bwd_flops(sub)))


def run_reference(args, w):
    """The reference arm: the CPU oracle as it stands, on a bounded sample per step."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import torch

    from attention_backward_preprocess_gb300.workloads import generate
    x = generate(w.with_(B=1, Sq=args.ref_prefix, Sk=args.ref_prefix, varlen=None), "cpu")
    times, vals = [], []
    for i in range(args.warmup + args.steps):
        tf, dt, cores, sample = cpu_baseline(w, x, args.ref_prefix)
        if i >= args.warmup:
            times.append(dt)
            vals.append(tf)
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, torch.Generator)",
        "config": config_of(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def config_of(w, lengths=None, flushed=False):
    c = {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq, "Sk": w.Sk,
         "D": w.D, "causal": w.causal, "deterministic": w.deterministic,
         **({} if w.Dv is None else {"Dv": w.Dv}),
         "l2": ("L2 written over (256 MB) between timed steps" if flushed
                else "inputs larger than L2 (no flush)"),
         "parallelism": "replicas"}
    if lengths is not None:
        c["varlen_lengths"] = list(lengths)
    return c


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=None)
    ap.add_argument("--cpu-prefix", type=int, default=8192)
    ap.add_argument("--ref-prefix", type=int, default=1024)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    # extension runs (fa_fwd_ext / fa_bwd_ext; not the headline line)
    ap.add_argument("--window", default=None, help="LEFT,RIGHT local window (-1: unbounded)")
    ap.add_argument("--alibi", action="store_true", help="ALiBi slopes 2^(-8 h / Hq)")
    ap.add_argument("--bias", action="store_true",
                    help="elementwise bias [B, Hq, Sq, Sk] and its gradient dBias")
    ap.add_argument("--dropout", type=float, default=0.0, help="dropout probability")
    ap.add_argument("--dropout-mask", action="store_true",
                    help="with --dropout: the forward stores the keep flags, the backward reads them")
    ap.add_argument("--head-dim", type=int, default=None,
                    help="query / key head dim other than the workload's (up to 256)")
    ap.add_argument("--head-dim-v", type=int, default=None,
                    help="value head dim other than the query / key one (one fa_bwd call per step)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    from attention_backward_preprocess_gb300.workloads import BENCH_WORKLOAD, WORKLOADS
    w = WORKLOADS[args.workload or BENCH_WORKLOAD]
    if args.head_dim or args.head_dim_v:
        D = args.head_dim or w.D
        Dv = args.head_dim_v if args.head_dim_v and args.head_dim_v != D else None
        w = w.with_(name="%s_dqk%d%s" % (w.name, D, "" if Dv is None else "_dv%d" % Dv), D=D, Dv=Dv,
                    scale=w.softmax_scale if w.scale is not None else None)
    if args.impl == "reference":
        return run_reference(args, w)
    if args.window or args.alibi or args.bias or args.dropout > 0:
        return run_ext(args, w)

    import torch

    import attention_backward_preprocess_gb300 as fa
    from attention_backward_preprocess_gb300.workloads import bwd_flops, generate

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    fa.lib()

    x = generate(w, dev)
    q, k, v, do = x["q"], x["k"], x["v"], x["dout"]
    varlen = w.varlen is not None
    # varlen: packed [total, H, D] tensors and cu_seqlens (main also launches the
    # kernel that builds the work-unit list from them)
    vl = dict(cu_seqlens_q=x["cu_q"], cu_seqlens_k=x["cu_k"], max_seqlen_q=x["max_len"],
              max_seqlen_k=x["max_len"]) if varlen else {}
    o, lse = fa.fa_fwd(q, k, v, causal=w.causal, softmax_scale=w.softmax_scale, **vl)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    Sq = x["max_len"] if varlen else w.Sq
    nbytes = fa.workspace_bytes(w.B, Sq, Sq if varlen else w.Sk, w.Hq, w.Hkv, w.D,
                                varlen=varlen, deterministic=w.deterministic)
    work = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    flops = bwd_flops(w, x.get("lengths"))
    stream = torch.cuda.current_stream()
    kw = dict(causal=w.causal, softmax_scale=w.softmax_scale, deterministic=w.deterministic,
              dq=dq, dk=dk, dv=dv, **vl)
    if varlen:
        # the packed row counts, known here: no call reads cu_seqlens[B] back
        # (which would synchronise the stream every call)
        kw["totals"] = (sum(x["lengths"]), sum(x["lengths"]))
    # a step reads Q, K, V, O, dO; below twice the 129 MB L2 the L2 is written
    # over between timed steps (outside the per-step events)
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v, o, do))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if in_bytes < (256 << 20) else None

    def step():
        if w.Dv is not None:
            # the stage calls carry no value head dim: one whole call per step
            e1.record(stream)
            fa.fa_bwd(q, k, v, o, do, lse, workspace=work, **kw)
            e2.record(stream)
            return
        fa.fa_bwd_stages(q, k, v, o, do, lse, work, stages=("pre",), **kw)
        e1.record(stream)
        fa.fa_bwd_stages(q, k, v, o, do, lse, work, stages=("main",), **kw)
        e2.record(stream)
        fa.fa_bwd_stages(q, k, v, o, do, lse, work, stages=("post",), **kw)

    e1 = torch.cuda.Event(enable_timing=True)
    e2 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev.index, clock_log_path("bench_clocks"))
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert fa.device_status(work) == fa.FA_OK

    def barrier():
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier()
    t_host0 = time.time()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        a, b_, c, d = ev[i]
        e1, e2 = b_, c
        if flush is not None:
            flush.fill_(i & 255)
        a.record(stream)
        step()
        d.record(stream)
    end.record(stream)
    barrier()
    clk = clocks.stop((t_host0, time.time()))
    total_ms = start.elapsed_time(end)
    if flush is not None:   # steps only, without the L2 overwrite between them
        total_ms = sum(ev[i][0].elapsed_time(ev[i][3]) for i in range(args.steps))
    pre_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps)]
    main_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(args.steps)]
    post_ms = [ev[i][2].elapsed_time(ev[i][3]) for i in range(args.steps)]
    status = fa.device_status(work)
    total_ms = max_over_ranks(total_ms, dev)
    ms_per_step = total_ms / args.steps
    value = job_throughput(flops, ws, ms_per_step)

    # ---------------------------------------------------------------- e2e
    e2e = None
    if not args.no_e2e:
        host = {n: t.cpu().pin_memory() for n, t in (("q", q), ("k", k), ("v", v), ("o", o),
                                                   ("dout", do), ("lse", lse))}
        if varlen:
            host["cu_q"] = x["cu_q"].cpu().pin_memory()
            host["cu_k"] = x["cu_k"].cpu().pin_memory()
        # Steps overlap as in a training loop that prefetches: the inputs of step
        # i are copied in (own stream) while step i-1 computes, and the results
        # of step i-1 are read back (own stream) while step i computes.  Two
        # sets of device buffers alternate; every step still copies all of its
        # inputs in and all of its results out.
        dev_in = [{n: torch.empty_like(t, device=dev) for n, t in host.items()} for _ in range(2)]
        dev_out = [[torch.empty_like(t) for t in (q, k, v)] for _ in range(2)]
        outs_h = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (q, k, v)]
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = sum(t.numel() * t.element_size() for t in outs_h)
        e2e_steps = max(3, min(args.steps, 10))
        h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of set b copied in
        ev_used = [torch.cuda.Event() for _ in range(2)]   # the step on set b computed
        ev_out = [torch.cuda.Event() for _ in range(2)]    # results of set b read back

        def e2e_step(i):
            b = i % 2
            with torch.cuda.stream(h2d_s):
                h2d_s.wait_event(ev_used[b])
                for n in host:
                    dev_in[b][n].copy_(host[n], non_blocking=True)
                ev_in[b].record(h2d_s)
            stream.wait_event(ev_in[b])
            stream.wait_event(ev_out[b])
            di = dev_in[b]
            evl = dict(cu_seqlens_q=di["cu_q"], cu_seqlens_k=di["cu_k"],
                       max_seqlen_q=x["max_len"], max_seqlen_k=x["max_len"],
                       totals=kw["totals"]) if varlen else {}
            gq, gk, gv = fa.fa_bwd(di["q"], di["k"], di["v"], di["o"], di["dout"], di["lse"],
                                   causal=w.causal, softmax_scale=w.softmax_scale,
                                   deterministic=w.deterministic, dq=dev_out[b][0],
                                   dk=dev_out[b][1], dv=dev_out[b][2], **evl)
            ev_used[b].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(ev_used[b])
                for hbuf, g in zip(outs_h, (gq, gk, gv)):
                    hbuf.copy_(g, non_blocking=True)
                ev_out[b].record(d2h_s)

        for i in range(2):
            e2e_step(i)
        barrier()
        s2 = torch.cuda.Event(enable_timing=True)
        t2 = torch.cuda.Event(enable_timing=True)
        s2.record(stream)
        h2d_s.wait_stream(stream)
        for i in range(e2e_steps):
            e2e_step(i)
        stream.wait_stream(d2h_s)
        t2.record(stream)
        barrier()
        e2e_ms = max_over_ranks(s2.elapsed_time(t2) / e2e_steps, dev)
        e2e = {"value": job_throughput(flops, ws, e2e_ms), "unit": UNIT,
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": e2e_steps}

    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return 0

    pk = peaks()
    main_avg = statistics.mean(main_ms)
    achieved = flops / (main_avg * 1e-3) / 1e12
    tokens_q = q.shape[0] if varlen else w.B * w.Sq
    elems_q = tokens_q * w.Hq * w.D
    elems_o = tokens_q * w.Hq * w.value_dim
    rows = tokens_q * w.Hq
    pre_bytes = 2 * elems_o * 2 + rows * 4 * 2 + rows * 4 + elems_q * 4    # O, dO in; LSE in; Dv, LSE2 out; dQaccum zero
    post_bytes = elems_q * 4 + elems_q * 2
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "main_kernel_traffic.json")
    if os.path.exists(tpath):
        t = json.load(open(tpath))
        if t.get("workload") == w.name and t.get("kernel_source_hash") == source_hash():
            traffic = t.get("dram_bytes_per_launch")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "fp16",
        "data": "synthetic (seeded N(0,1), torch.Generator on device)",
        "config": config_of(w, x.get("lengths"), flush is not None),
        "pct_of_bf16_peak": 100.0 * value / ws / pk["bf16"],
        "roofline": {"kernel": "bwd_main_kernel" if (w.D <= 128 and w.Dv is None) else "bwd_wide_kernel",
                     "bound": "tensor", "achieved": achieved,
                     "peak": pk["bf16"], "unit": "TFLOP/s", "frac": achieved / pk["bf16"],
                     "traffic": traffic,
                     "peak_note": "%s dense bf16 burst (bf16_tflops); sustained %s" % (
                         pk["source"], pk["bf16_sustained"]),
                     "algorithmic_flop_per_launch": flops},
        "kernels_ms": ({"preprocess": statistics.mean(pre_ms), "main": main_avg,
                        "postprocess": statistics.mean(post_ms)} if w.Dv is None
                       else {"whole_call": main_avg}),
        "kernels_gbs": ({"preprocess": pre_bytes / (statistics.mean(pre_ms) * 1e-3) / 1e9,
                         "postprocess": post_bytes / (statistics.mean(post_ms) * 1e-3) / 1e9,
                         "hbm_peak": pk["hbm"]} if w.Dv is None else None),
        # preprocess, main, postprocess (+ the varlen work-unit scheduler)
        "gpu_launches": (4 if varlen else 3) * args.steps,
        "device_status": status,
        "e2e": e2e,
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        xs = generate(w.with_(B=1, Sq=args.cpu_prefix, Sk=args.cpu_prefix, varlen=None), "cpu")
        tf, dt, cores, sample = cpu_baseline(w, xs, args.cpu_prefix)
        line["cpu_baseline"] = {"value": tf, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "seconds": dt, "sample": sample}
    print(json.dumps(line))
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def visible_pairs(lq, lk, causal, wl, wr):
    """(query, key) pairs of one head that the mask leaves visible: key j is
    visible to query i iff i + d - wl <= j <= i + d + wr, d = lk - lq (-1:
    unbounded side), and j <= i + d when causal."""
    import numpy as np
    i = np.arange(lq, dtype=np.int64) + (lk - lq)
    hi = np.full(lq, lk - 1) if wr < 0 else np.minimum(lk - 1, i + wr)
    if causal:
        hi = np.minimum(hi, i)
    lo = np.zeros(lq, dtype=np.int64) if wl < 0 else np.maximum(0, i - wl)
    return int(np.maximum(hi - lo + 1, 0).sum())


def run_ext(args, w):
    """Times fa_fwd_ext and fa_bwd_ext (one call: preprocess, main, postprocess)
    on workload w with the requested extensions; one GPU, one JSON line.  The
    FLOP counts are over the visible pairs: 4 D (forward) and 10 D (backward)
    per pair."""
    import torch

    import attention_backward_preprocess_gb300 as fa
    from attention_backward_preprocess_gb300.workloads import generate

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fa.lib()
    x = generate(w, dev)
    q, k, v, do = x["q"], x["k"], x["v"], x["dout"]
    varlen = w.varlen is not None
    vl = dict(cu_seqlens_q=x["cu_q"], cu_seqlens_k=x["cu_k"], max_seqlen_q=x["max_len"],
              max_seqlen_k=x["max_len"],
              totals=(sum(x["lengths"]), sum(x["lengths"]))) if varlen else {}
    wl, wr = (int(t) for t in args.window.split(",")) if args.window else (-1, -1)
    ext = {}
    if args.window:
        ext["window"] = (wl, wr)
    if args.alibi:
        ext["alibi_slopes"] = torch.tensor([2.0 ** (-8.0 * (h + 1) / w.Hq) for h in range(w.Hq)],
                                           dtype=torch.float32, device=dev)
    dbias = None
    if args.bias:
        if varlen:
            raise SystemExit("--bias: dense workloads only")
        g = torch.Generator(device=dev).manual_seed(7)
        ext["bias"] = torch.randn((w.B, w.Hq, w.Sq, w.Sk), generator=g, device=dev).to(q.dtype)
        dbias = torch.empty_like(ext["bias"])
    if args.dropout > 0:
        ext["dropout"] = (args.dropout, 0x5EED, 0)
        if args.dropout_mask:
            # the forward writes the keep flags, the backward reads them
            mask = torch.empty(fa.dropout_mask_shape(q, k, vl.get("cu_seqlens_q"),
                                                     vl.get("max_seqlen_k")),
                               dtype=torch.int32, device=dev)
            ext["dropout"] = (args.dropout, 0x5EED, 0, mask)
    lengths = x.get("lengths") or [w.Sq] * w.B
    pairs = sum(visible_pairs(L, L if varlen else w.Sk, w.causal, wl, wr) for L in lengths) * w.Hq
    fl_fwd, fl_bwd = 4.0 * w.D * pairs, 10.0 * w.D * pairs
    o, lse = fa.fa_fwd(q, k, v, causal=w.causal, softmax_scale=w.softmax_scale, **vl, **ext)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    Sq = x["max_len"] if varlen else w.Sq
    work = torch.empty(fa.workspace_bytes(w.B, Sq, Sq if varlen else w.Sk, w.Hq, w.Hkv, w.D,
                                          varlen=varlen, deterministic=w.deterministic),
                       dtype=torch.uint8, device=dev)
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v, o, do))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if in_bytes < (256 << 20) else None
    stream = torch.cuda.current_stream()

    def fwd():
        fa.fa_fwd(q, k, v, causal=w.causal, softmax_scale=w.softmax_scale, **vl, **ext)

    def bwd():
        fa.fa_bwd(q, k, v, o, do, lse, causal=w.causal, softmax_scale=w.softmax_scale,
                  deterministic=w.deterministic, dq=dq, dk=dk, dv=dv, workspace=work, dbias=dbias,
                  **vl, **ext)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        for a, b in ev:
            if flush is not None:
                flush.fill_(1)
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ev)

    clocks = ClockSampler(dev.index, clock_log_path("bench_ext_clocks"))
    f_ms = timed(fwd)
    b_ms = timed(bwd)
    clk = clocks.stop()
    status = fa.device_status(work)
    fstatus = fa.device_status()
    pk = peaks()
    exts = {k_: (list(v_[:3]) if k_ in ("window", "dropout") else True) for k_, v_ in ext.items()}
    if len(ext.get("dropout", ())) > 3:
        exts["dropout_mask"] = "stored by the forward, read by the backward"
    if dbias is not None:
        exts["dbias"] = True
    line = {
        "metric": "attention-backward TFLOPS with extensions (visible pairs)",
        "value": fl_bwd / (b_ms * 1e-3) / 1e12, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": b_ms, "higher_is_better": True,
        "dtype": "bf16" if w.dtype == "bf16" else "fp16", "data": "synthetic",
        "config": dict(config_of(w, x.get("lengths"), flush is not None), extensions=exts,
                       visible_pairs=pairs),
        "pct_of_bf16_peak": 100.0 * fl_bwd / (b_ms * 1e-3) / 1e12 / pk["bf16"],
        "forward": {"ms": f_ms, "tflops": fl_fwd / (f_ms * 1e-3) / 1e12,
                    "pct_of_bf16_peak": 100.0 * fl_fwd / (f_ms * 1e-3) / 1e12 / pk["bf16"]},
        "device_status": [status, fstatus], "clocks": clk,
    }
    print(json.dumps(line))
    return 0


def code_text(text):
    """C++ source without comments and whitespace: what the compiler sees of it
    (a comment edit leaves the kernel, and its counters, unchanged)."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return re.sub(r"\s+", "", text)


def source_hash(read=None):
    import hashlib
    h = hashlib.sha256()
    for f in ("fa_bwd_main.cu", "fa_bwd_units.cuh", "fa_device.cuh", "fa_params.h"):
        path = os.path.join("attention_backward_preprocess_gb300", "csrc", f)
        text = read(path) if read else open(os.path.join(ROOT, path)).read()
        h.update(code_text(text).encode())
    return h.hexdigest()[:16]


if __name__ == "__main__":
    sys.exit(main())
