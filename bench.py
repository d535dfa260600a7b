"""Benchmark of the sink-attention hot path on GB300.

One step = one pass of the decode path over the long-context workload (8
sequences x 131072 cached tokens, 64 query / 8 KV heads, head_dim 64, page size
16, seeded random page permutation): sink_attn_decode with 32 splits (the sink
in split 0 only), then sink_attn_merge.  Headline metric: algorithmic decode
bytes per second (KV cache + q + out + lse + page table), with the decode
kernel's fraction of the measured HBM copy bandwidth.  The same JSON line
carries the causal prefill (4 x 8192 tokens, 64/8 heads) in TFLOP/s against the
measured dense bf16 peak, the ragged mixed batch, the 64 x 4096 paged decode,
small-batch decode in a CUDA graph, the tiny prefill and the kernels around
attention.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle on bounded samples of the same
workload (every host core).  For N > 1 (torchrun) every rank runs its own
replica on its own GPU; nothing is exchanged but the timing.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

# The CPU baseline runs the oracle on one thread per core, each with one BLAS thread,
# so that the number of cores it uses is exact.
os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("OMP_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "sink-attn prefill TFLOP/s & decode KV GB/s on 1 GB300, % of roofline"
DECODE = workloads.WORKLOADS["paged_decode"]
PREFILL = workloads.WORKLOADS["causal_prefill"]
LONG = workloads.WORKLOADS["long_decode"]
LONG_WORKLOAD = "long_decode: 8 x 131072 cached tokens, 64/8 heads, d 64, page 16, 32 splits + merge"
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal (context for the measured-copy fraction)
# kernel sources whose hash keys the recorded DRAM traffic (profiles/traffic.txt)
DECODE_SOURCES = ("decode.cu", "ptx.cuh", "internal.h", "rope_math.cuh")
PREFILL_SOURCES = ("prefill.cu", "ptx.cuh", "internal.h", "rope_math.cuh")
ROPE_SOURCES = ("rope.cu", "rope_args.h", "internal.h", "ptx.cuh", "rope_math.cuh")


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return dict(hbm=p["hbm_gbs"], bf16=p["bf16_tflops"], bf16_sust=p["bf16_tflops_sustained"],
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sust=1700.0, source="fallback")


def recorded_traffic(kernel, sources):
    """DRAM bytes per full-size launch from profiles/traffic.txt, or None when the
    kernel sources changed after the capture (or nothing was recorded)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    h = hashlib.sha256()
    for f in sources:
        h.update(open(os.path.join(ROOT, "attention_softmax_sinks_gb300", "csrc", f), "rb").read())
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        kv = dict(item.split("=", 1) for item in line.split())
        if kv.get("kernel") == kernel and kv.get("source_sha") == h.hexdigest()[:16]:
            return int(kv["bytes_per_launch"])
    return None


def max_over_ranks(x, world):
    """Largest value of x over all ranks (the job time is the slowest rank's)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank_step, world, ms_per_step):
    """Whole-job GB/s: every rank processes its own replica in the (max) step time."""
    return bytes_per_rank_step * world / (ms_per_step * 1e-3) / 1e9


def decode_bytes(batch, kv_len, hq, hkv, d, max_pages):
    """Algorithmic bytes of one decode step: KV read once, q, out, lse, page table, lens, sinks."""
    kv = batch * kv_len * hkv * d * 2 * 2
    return kv + batch * hq * d * 2 * 2 + batch * hq * 4 + batch * max_pages * 4 + batch * 4 + hq * 4


def prefill_flops(batch, seqlen, hq, d):
    pairs = seqlen * (seqlen + 1) // 2
    return 4.0 * hq * d * pairs * batch


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"], samples=0)
        time.sleep(0.1)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), reasons=parts[4:9]))
            except ValueError:
                continue
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        if not rows:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["no samples"], samples=0)
        loaded = [r for r in rows if r["sm"] > 0.5 * r["smax"]] or rows
        seen = set()
        for r in loaded:
            for n, v in zip(names[1:], r["reasons"][1:]):
                if v.lower() == "active":
                    seen.add(n)
        return dict(sm_mhz=statistics.median(r["sm"] for r in loaded),
                    sm_max_mhz=max(r["smax"] for r in rows), reasons=sorted(seen),
                    samples=len(loaded))


# ----------------------------------------------------------------------------- our arm
def to_dev(x, torch, device):
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(x).to(device)


def run_ours(args, rank, world, device):
    import torch
    import attention_softmax_sinks_gb300 as sa
    from attention_softmax_sinks_gb300 import _build

    _build.build()
    sa.load_library()
    torch.cuda.set_device(device)
    pk = peaks()
    cfg = LONG
    b, kvl, hq, hkv, d, s = cfg["batch"], cfg["kv_len"], cfg["hq"], cfg["hkv"], cfg["d"], cfg["num_splits"]
    host = workloads.make_decode(cfg["seed"], [kvl] * b, hq, hkv, d, cfg["page_size"], cfg["sink_std"])
    names = ("q", "k_pages", "v_pages", "page_table", "kv_lens", "sinks")
    dev = {n: to_dev(host[n], torch, device) for n in names}
    part_o = torch.empty((b, s, hq, d), dtype=torch.float32, device=device)
    part_l = torch.empty((b, s, hq), dtype=torch.float32, device=device)
    out = torch.empty((b, hq, d), dtype=torch.bfloat16, device=device)
    lse = torch.empty((b, hq), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    max_pages = host["page_table"].shape[1]
    alg_bytes = decode_bytes(b, kvl, hq, hkv, d, max_pages)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        sa.sink_attn_decode(dev["q"], dev["k_pages"], dev["v_pages"], dev["page_table"], dev["kv_lens"],
                            dev["sinks"], cfg["sm_scale"], num_splits=s, out=part_o, lse=part_l, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        sa.sink_attn_merge(part_o, part_l, out=out, lse=lse, stream=stream)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(device)

    for _ in range(args.warmup):
        step()
    barrier()
    clocks = ClockSampler(device.index if device.index is not None else 0)
    clocks.start()
    # one timed pass: events at both ends of the K steps and around every decode launch,
    # so the decode kernel's time and the step time come from the same launches
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier()
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    barrier()
    clk = clocks.stop()
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), world)
    ms_per_step = total_ms / args.steps
    dec_ms = sum(e0.elapsed_time(e1) for e0, e1 in evs) / args.steps
    value = job_throughput(alg_bytes, world, ms_per_step)
    achieved = alg_bytes / (dec_ms * 1e-3) / 1e9
    status = sa.sink_attn_device_status(True)

    # ---- end to end through the public API: pinned host inputs in, result out
    def pin(x):
        x = np.ascontiguousarray(x)
        t = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16) if x.dtype == np.uint16 else torch.from_numpy(x)
        return t.pin_memory()

    pinned = {n: pin(host[n]) for n in names}
    h_out = torch.empty((b, hq, d), dtype=torch.bfloat16).pin_memory()
    h_lse = torch.empty((b, hq), dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in pinned.values())
    d2h = h_out.numel() * h_out.element_size() + h_lse.numel() * h_lse.element_size()
    e2e_steps = max(3, min(10, args.steps))

    def e2e_step():
        for n in names:
            dev[n].copy_(pinned[n], non_blocking=True)
        step()
        h_out.copy_(out, non_blocking=True)
        h_lse.copy_(lse, non_blocking=True)

    e2e_step()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world)
    del pinned, dev, part_o, part_l
    torch.cuda.empty_cache()

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded N(0,1) bf16 q/k/v, N(0,1) fp32 sinks, permuted pages",
        "config": {"workload": LONG_WORKLOAD,
                   "batch": b, "kv_len": kvl, "num_splits": s,
                   "l2": "inputs > L2 (2 GiB KV per step)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "algorithmic_bytes_per_step": alg_bytes},
        "e2e": {"value": round(job_throughput(alg_bytes, world, e2e_ms), 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": 2 * args.steps,
        "clocks": {k: clk[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
        "device_status": status,
    }
    roofline = {"bound": "hbm", "kernel": "sink_decode_kernel", "achieved": round(achieved, 1),
                "peak": pk["hbm"], "unit": "GB/s", "frac": round(achieved / pk["hbm"], 4),
                "peak_source": pk["source"] + " copy",
                "frac_of_nominal_hbm": round(achieved / NOMINAL_HBM_GBS, 4),
                "traffic": recorded_traffic("sink_decode_kernel_long", DECODE_SOURCES),
                "kernel_ms": round(dec_ms, 5)}
    if not args.no_prefill:
        around = bench_around_attention(args, sa, torch, device, pk)
        around["linear"] = bench_linear(args, sa, torch, device, pk)
        line["around"] = around
        line["fused_qkv_prefill"] = bench_fused_qkv(args, sa, torch, device, pk)
        line["tiny_prefill"] = bench_tiny_prefill(args, sa, torch, device, pk)
        line["small_batch_decode"] = bench_graph_decode(args, sa, torch, device, pk, 32, DECODE["kv_len"], 7)
        line["long_single_decode"] = bench_graph_decode(args, sa, torch, device, pk, 8, LONG["kv_len"], 3)
        line["paged_decode"] = bench_paged_decode(args, sa, torch, device, pk)
        line["mixed"] = bench_mixed(args, sa, torch, device, pk)
        line["prefill"] = bench_prefill(args, sa, torch, device, pk)
    line["roofline"] = roofline
    return line, host


def bench_paged_decode(args, sa, torch, device, pk):
    """Paged decode: 64 sequences x 4096 cached tokens (512 MiB of KV, larger than L2),
    64/8 heads, the library's split count, decode then merge; one pass timed at its ends,
    one with events around each decode launch."""
    cfg = DECODE
    b, kvl, hq, hkv, d = cfg["batch"], cfg["kv_len"], cfg["hq"], cfg["hkv"], cfg["d"]
    host = workloads.make_decode(cfg["seed"], [kvl] * b, hq, hkv, d, cfg["page_size"], cfg["sink_std"])
    dv = {n: to_dev(host[n], torch, device) for n in ("q", "k_pages", "v_pages", "page_table", "kv_lens", "sinks")}
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    s = sa.sink_attn_decode_splits(b, hkv, kvl, cfg["page_size"], sms)
    po = torch.empty((b, s, hq, d), dtype=torch.float32, device=device)
    pl = torch.empty((b, s, hq), dtype=torch.float32, device=device)
    out = torch.empty((b, hq, d), dtype=torch.bfloat16, device=device)
    lse = torch.empty((b, hq), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        if s > 1:
            sa.sink_attn_decode(dv["q"], dv["k_pages"], dv["v_pages"], dv["page_table"], dv["kv_lens"],
                                dv["sinks"], cfg["sm_scale"], num_splits=s, out=po, lse=pl, stream=stream)
        else:
            sa.sink_attn_decode(dv["q"], dv["k_pages"], dv["v_pages"], dv["page_table"], dv["kv_lens"],
                                dv["sinks"], cfg["sm_scale"], num_splits=1, out=out, lse=lse, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        if s > 1:
            sa.sink_attn_merge(po, pl, out=out, lse=lse, stream=stream)

    for _ in range(5):
        step()
    reps = max(10, min(100, args.steps))
    torch.cuda.synchronize(device)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(reps):
        step()
    t1.record(stream)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for e in evs:
        step(e)
    torch.cuda.synchronize(device)
    step_ms = t0.elapsed_time(t1) / reps
    dec_ms = sum(a.elapsed_time(c) for a, c in evs) / reps
    nbytes = decode_bytes(b, kvl, hq, hkv, d, dv["page_table"].shape[1])
    del dv
    torch.cuda.empty_cache()
    ach = nbytes / (dec_ms * 1e-3) / 1e9
    return {"workload": "64 x 4096 tokens", "num_splits": s, "step_us": round(step_ms * 1e3, 2),
            "value": round(nbytes / (step_ms * 1e-3) / 1e9, 1), "unit": "GB/s", "kernel": "sink_decode_kernel",
            "kernel_us": round(dec_ms * 1e3, 2), "achieved": round(ach, 1), "peak": pk["hbm"],
            "frac": round(ach / pk["hbm"], 4), "frac_of_nominal_hbm": round(ach / NOMINAL_HBM_GBS, 4),
            "traffic": recorded_traffic("sink_decode_kernel", DECODE_SOURCES),
            "gpu_launches": (2 if s > 1 else 1) * (2 * reps + 5)}


def bench_mixed(args, sa, torch, device, pk):
    """Ragged mixed batch: 32 sequences, KV log-uniform in [1, 32768], half decode rows
    (q_len 1) and half prefill chunks (q_len 128..2048), one sink_attn_prefill_paged call."""
    cfg = workloads.WORKLOADS["ragged_mixed"]
    q_lens, kv_lens = workloads.ragged_mixed_lengths(cfg["seed"] + 2, cfg["num_seqs"], cfg["max_kv"])
    host = workloads.make_mixed(cfg["seed"], q_lens, kv_lens, cfg["hq"], cfg["hkv"], cfg["d"],
                                cfg["page_size"], cfg["sink_std"])
    names = ("q", "k_pages", "v_pages", "page_table", "cu_seqlens_q", "kv_lens", "sinks")
    dv = {n: to_dev(host[n], torch, device) for n in names}
    out = torch.empty_like(dv["q"])
    lse = torch.empty((dv["q"].shape[0], cfg["hq"]), dtype=torch.float32, device=device)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    q = q_lens.astype(np.int64)
    kv = kv_lens.astype(np.int64)
    pairs = int((q * (kv - q) + q * (q + 1) // 2).sum())
    flops = 4.0 * cfg["hq"] * cfg["d"] * pairs
    nbytes = int((kv * cfg["hkv"] * cfg["d"] * 2 * 2).sum() + q.sum() * cfg["hq"] * cfg["d"] * 2 * 2)

    def run():
        sa.sink_attn_prefill_paged(dv["q"], dv["k_pages"], dv["v_pages"], dv["page_table"],
                                   dv["cu_seqlens_q"], dv["kv_lens"], dv["sinks"], int(q.max()),
                                   cfg["sm_scale"], causal=True, out=out, lse=lse, stream=stream)

    for _ in range(3):
        run()
    times = []
    for _ in range(max(5, min(30, args.steps))):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run()
        e1.record(stream)
        times.append((e0, e1))
    torch.cuda.synchronize(device)
    each = sorted(a.elapsed_time(b) for a, b in times)
    ms = sum(each) / len(each)
    t_tc = flops / (pk["bf16"] * 1e12)
    t_hbm = nbytes / (pk["hbm"] * 1e9)
    bound = "tensor" if t_tc >= t_hbm else "hbm"
    return {"workload": "ragged_mixed: 32 paged seqs, half decode rows", "value": round(flops / (ms * 1e-3) / 1e12, 2),
            "unit": "TFLOP/s", "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1), "ms": round(ms, 4),
            "ms_median": round(each[len(each) // 2], 4), "flops": flops,
            "bytes": nbytes, "kernel": "sink_prefill_kernel", "bound": bound,
            "frac": round(max(t_tc, t_hbm) / (ms * 1e-3), 4), "tensor_frac": round(t_tc / (ms * 1e-3), 4),
            "hbm_frac": round(t_hbm / (ms * 1e-3), 4),
            "traffic": recorded_traffic("sink_prefill_kernel_mixed", PREFILL_SOURCES),
            "gpu_launches": len(times)}


def bench_tiny_prefill(args, sa, torch, device, pk):
    """The small parity case (1 x 128 tokens, causal, 4 query / 1 KV head): launch latency
    dominates, so it is reported as time per call; the roofline fraction is tiny by nature."""
    cfg = workloads.WORKLOADS["tiny_prefill"]
    host = workloads.make_prefill(cfg["seed"], [cfg["seqlen"]], cfg["hq"], cfg["hkv"], cfg["d"], cfg["sink_std"])
    q, k, v, sinks, cu = (to_dev(host[n], torch, device) for n in ("q", "k", "v", "sinks", "cu_seqlens"))
    out = torch.empty_like(q)
    lse = torch.empty((q.shape[0], q.shape[1]), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    def run():
        sa.sink_attn_prefill(q, k, v, sinks, cu, cfg["seqlen"], cfg["sm_scale"], causal=True, out=out, lse=lse,
                             stream=stream)

    for _ in range(10):
        run()
    reps = 200

    def timed(fn, n):
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(device)
        return e0.elapsed_time(e1) * 1e3

    us = timed(run, reps) / reps
    # the same calls captured once into a CUDA graph: device time without host enqueue gaps
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(device)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            for _ in range(20):
                sa.sink_attn_prefill(q, k, v, sinks, cu, cfg["seqlen"], cfg["sm_scale"], causal=True, out=out,
                                     lse=lse, stream=side)
    torch.cuda.synchronize(device)
    us_graph = timed(graph.replay, 10) / 200
    flops = prefill_flops(1, cfg["seqlen"], cfg["hq"], cfg["d"])
    tf = flops / (us_graph * 1e-6) / 1e12
    return {"workload": "1 x 128 tokens, 4/1 heads", "us_per_call": round(us, 2),
            "us_per_call_graph": round(us_graph, 2), "achieved": round(tf, 4), "unit": "TFLOP/s",
            "frac": round(tf / pk["bf16"], 6), "gpu_launches": reps + 10 + 200}


def bench_graph_decode(args, sa, torch, device, pk, nseq, kvl, seed_offset):
    """Decode at batch 1: one sequence of ``kvl`` cached tokens per step (64/8 heads, page 16)
    with the library's split count (1: one launch whose 16-CTA clusters merge on chip; a
    count above 1 adds the merge launch).  ``nseq`` steps cycle over ``nseq`` different
    sequences of one permuted page pool (32 x 4096 tokens = 256 MiB, 8 x 131072 = 2 GiB of KV,
    both larger than L2), run eagerly and as one captured CUDA graph of the same steps."""
    cfg = DECODE
    host = workloads.make_decode(cfg["seed"] + seed_offset, [kvl] * nseq, cfg["hq"], cfg["hkv"], cfg["d"],
                                 cfg["page_size"], cfg["sink_std"])
    dv = {n: to_dev(host[n], torch, device)
          for n in ("q", "k_pages", "v_pages", "page_table", "kv_lens", "sinks")}
    hq, d = cfg["hq"], cfg["d"]
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    splits = sa.sink_attn_decode_splits(1, cfg["hkv"], kvl, cfg["page_size"], sms)
    part_o = torch.empty((1, splits, hq, d), dtype=torch.float32, device=device)
    part_l = torch.empty((1, splits, hq), dtype=torch.float32, device=device)
    out = torch.empty((nseq, hq, d), dtype=torch.bfloat16, device=device)
    lse = torch.empty((nseq, hq), dtype=torch.float32, device=device)
    stream = torch.cuda.Stream(device)

    def steps():
        for i in range(nseq):
            sl = slice(i, i + 1)
            if splits > 1:
                sa.sink_attn_decode(dv["q"][sl], dv["k_pages"], dv["v_pages"], dv["page_table"][sl],
                                    dv["kv_lens"][sl], dv["sinks"], cfg["sm_scale"], num_splits=splits,
                                    out=part_o, lse=part_l, stream=stream)
                sa.sink_attn_merge(part_o, part_l, out=out[sl], lse=lse[sl], stream=stream)
            else:
                sa.sink_attn_decode(dv["q"][sl], dv["k_pages"], dv["v_pages"], dv["page_table"][sl],
                                    dv["kv_lens"][sl], dv["sinks"], cfg["sm_scale"], num_splits=1,
                                    out=out[sl], lse=lse[sl], stream=stream)

    stream.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(stream):
        for _ in range(3):
            steps()
    torch.cuda.synchronize(device)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        steps()
    torch.cuda.synchronize(device)
    reps = max(3, min(30, args.steps // 10))

    def timed(fn):
        with torch.cuda.stream(stream):
            fn()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
        torch.cuda.synchronize(device)
        return e0.elapsed_time(e1) * 1e3 / (reps * nseq)

    eager_us = timed(steps)
    graph_us = timed(graph.replay)
    step_bytes = decode_bytes(1, kvl, hq, cfg["hkv"], d, host["page_table"].shape[1])
    per_step = 2 if splits > 1 else 1
    del dv
    torch.cuda.empty_cache()
    return {"workload": f"1 x {kvl} tokens per step, {nseq} sequences", "num_splits": splits,
            "launches_per_step": per_step, "eager_us_per_step": round(eager_us, 2),
            "graph_us_per_step": round(graph_us, 2), "graph_gbs": round(step_bytes / (graph_us * 1e-6) / 1e9, 1),
            "gpu_launches": per_step * nseq * (2 * reps + 2)}


def flush_l2(buf):
    """Evict L2 before a timed launch: write a buffer larger than L2, then read it back.
    The read pushes the written (dirty) lines out to DRAM before the timed region starts
    and leaves only clean lines, so the timed kernel does not pay for their write-back.
    The read sums a float32 view: summing the uint8 buffer itself would first widen it to
    int64 (a 2 GiB cast copy)."""
    import torch
    buf.zero_()
    buf.view(torch.float32).sum()


def _timed_flushed(torch, device, stream, fn, reps):
    """Mean CUDA-event time (ms) of fn over reps launches, L2 flushed before each."""
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=device)
    for _ in range(3):
        fn()
    evs = []
    for _ in range(reps):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize(device)
    return sum(a.elapsed_time(b) for a, b in evs) / reps


def bench_around_attention(args, sa, torch, device, pk):
    """The two HBM-bound steps next to attention, on the causal-prefill batch
    (4 x 8192 = 32768 tokens): QKV bias + YaRN rotation (64/8 heads) and the
    Top-K-then-softmax router (128 experts, top 4)."""
    stream = torch.cuda.current_stream(device)
    reps = max(5, min(30, args.steps // 10))
    t, hq, hkv, e, k = 32768, PREFILL["hq"], PREFILL["hkv"], 128, 4
    cu = to_dev(workloads.cu_seqlens_from([8192] * 4), torch, device)
    inp = workloads.make_qkv(41, t, hq, hkv)
    qkv, bias = to_dev(inp["qkv"], torch, device), to_dev(inp["bias"], torch, device)
    q = torch.empty((t, hq, 64), dtype=torch.bfloat16, device=device)
    kk = torch.empty((t, hkv, 64), dtype=torch.bfloat16, device=device)
    vv = torch.empty_like(kk)
    rope_ms = _timed_flushed(torch, device, stream, lambda: sa.qkv_bias_rope(
        qkv, bias, cu, hq, hkv, q_out=q, k_out=kk, v_out=vv, stream=stream), reps)
    rope_bytes = 2 * t * (hq + 2 * hkv) * 64 * 2 + (hq + 2 * hkv) * 64 * 2 + cu.numel() * 4
    logits = to_dev(workloads.make_router_logits(42, t, e, std=2.0), torch, device)
    idx = torch.empty((t, k), dtype=torch.int32, device=device)
    w = torch.empty((t, k), dtype=torch.bfloat16, device=device)
    counts = torch.empty((e,), dtype=torch.int32, device=device)
    router_ms = _timed_flushed(torch, device, stream, lambda: sa.moe_router_topk_softmax(
        logits, k, topk_idx=idx, topk_weight=w, expert_counts=counts, stream=stream), reps)
    router_bytes = t * e * 2 + t * k * (4 + 2) + e * 4
    # the whole router: projection of 2880-wide hidden states + bias, then Top-K softmax,
    # fused into one kernel and as the two-kernel path
    rd = workloads.make_linear(43, t, e, 2880, std=1.0, w_std=0.05, bias_std=0.5)
    hx, rw, rb = (to_dev(rd[key], torch, device) for key in ("x", "w", "bias"))
    rlog = torch.empty((t, e), dtype=torch.bfloat16, device=device)
    fused_ms = _timed_flushed(torch, device, stream, lambda: sa.moe_router(
        hx, rw, rb, k, topk_idx=idx, topk_weight=w, expert_counts=counts, stream=stream), reps)
    two_ms = _timed_flushed(torch, device, stream, lambda: (
        sa.linear_bias(hx, rw, rb, out=rlog, stream=stream),
        sa.moe_router_topk_softmax(rlog, k, topk_idx=idx, topk_weight=w, expert_counts=counts, stream=stream)),
        reps)

    def hbm(kernel, srcs, ms, nbytes):
        gbs = nbytes / (ms * 1e-3) / 1e9
        return {"kernel": kernel, "us": round(ms * 1e3, 2), "bytes": nbytes, "achieved": round(gbs, 1),
                "unit": "GB/s", "frac": round(gbs / pk["hbm"], 4), "traffic": recorded_traffic(kernel, srcs)}
    fused_gbs = t * 2880 * 2 / (fused_ms * 1e-3) / 1e9  # the hidden states read once
    return {"qkv_bias_rope": hbm("qkv_rope_kernel", ROPE_SOURCES, rope_ms, rope_bytes),
            "moe_router": hbm("router_topk_kernel", ("router.cu", "router_args.h", "ptx.cuh"), router_ms,
                              router_bytes),
            "moe_router_fused": {"kernel": "linear_bias_kernel", "us": round(fused_ms * 1e3, 2),
                                 "two_kernels_us": round(two_ms * 1e3, 2), "achieved": round(fused_gbs, 1),
                                 "unit": "GB/s", "frac": round(fused_gbs / pk["hbm"], 4),
                                 "traffic": recorded_traffic("linear_bias_kernel_router",
                                                             ("linear.cu", "linear_args.h", "ptx.cuh"))},
            "gpu_launches": 2 * (reps + 3) + 3 * (reps + 3)}


def bench_fused_qkv(args, sa, torch, device, pk):
    """q taken from the QKV projection output and rotated inside the prefill, against the
    separate rotation kernel, on the causal-prefill batch (4 x 8192 tokens, 64/8 heads):
    unfused = qkv_bias_rope (writes q, k, v) + sink_attn_prefill; fused = qkv_bias_rope_kv
    (writes k, v and the (cos, sin) table) + sink_attn_prefill_qkv.  L2 flushed before
    each pair."""
    stream = torch.cuda.current_stream(device)
    t, hq, hkv = 32768, PREFILL["hq"], PREFILL["hkv"]
    cu = to_dev(workloads.cu_seqlens_from([8192] * 4), torch, device)
    inp = workloads.make_qkv(41, t, hq, hkv)
    qkv, bias = to_dev(inp["qkv"], torch, device), to_dev(inp["bias"], torch, device)
    sinks = to_dev(workloads.sinks_f32(0, hq, PREFILL["sink_std"]), torch, device)
    q = torch.empty((t, hq, 64), dtype=torch.bfloat16, device=device)
    k = torch.empty((t, hkv, 64), dtype=torch.bfloat16, device=device)
    v = torch.empty_like(k)
    table = torch.empty((t, 32, 2), dtype=torch.float32, device=device)
    out = torch.empty_like(q)
    lse = torch.empty((t, hq), dtype=torch.float32, device=device)
    reps = max(5, min(20, args.steps))

    def unfused():
        sa.qkv_bias_rope(qkv, bias, cu, hq, hkv, q_out=q, k_out=k, v_out=v, stream=stream)
        sa.sink_attn_prefill(q, k, v, sinks, cu, 8192, PREFILL["sm_scale"], out=out, lse=lse, stream=stream)

    def fused():
        sa.qkv_bias_rope_kv(qkv, bias, cu, hq, hkv, k_out=k, v_out=v, rope_table=table, stream=stream)
        sa.sink_attn_prefill_qkv(qkv, bias, table, k, v, sinks, cu, 8192, PREFILL["sm_scale"], hq, out=out,
                                 lse=lse, stream=stream)

    un_ms = _timed_flushed(torch, device, stream, unfused, reps)
    fu_ms = _timed_flushed(torch, device, stream, fused, reps)
    return {"workload": "4 x 8192 tokens", "unfused_us": round(un_ms * 1e3, 1), "fused_us": round(fu_ms * 1e3, 1),
            "fused_over_unfused": round(fu_ms / un_ms, 4), "gpu_launches": 4 * (reps + 3)}


def bench_linear(args, sa, torch, device, pk):
    """Bias-seeded tcgen05 linear layer at the attention output projection of the
    causal-prefill batch: 32768 tokens x (64 heads x 64) = 4096 inputs -> 2880 features
    (GPT-OSS hidden size, page "GPT-OSS on day 0", section "Performance tweaks").
    cuBLAS (torch's bf16 linear with bias) is timed beside it for context only."""
    stream = torch.cuda.current_stream(device)
    m, n, k = 32768, 2880, 4096
    d = workloads.make_linear(61, m, n, k)
    x, w, b = (to_dev(d[key], torch, device) for key in ("x", "w", "bias"))
    out = torch.empty((m, n), dtype=torch.bfloat16, device=device)
    reps = max(5, min(30, args.steps // 10))
    ms = _timed_flushed(torch, device, stream, lambda: sa.linear_bias(x, w, b, out=out, stream=stream), reps)
    ref_ms = _timed_flushed(torch, device, stream, lambda: torch.nn.functional.linear(x, w, b), reps)
    flops = 2.0 * m * n * k
    tf = flops / (ms * 1e-3) / 1e12
    return {"kernel": "linear_bias_kernel", "ms": round(ms, 4), "achieved": round(tf, 2), "unit": "TFLOP/s",
            "frac": round(tf / pk["bf16"], 4),
            "traffic": recorded_traffic("linear_bias_kernel", ("linear.cu", "linear_args.h", "ptx.cuh")),
            "cublas_tflops": round(flops / (ref_ms * 1e-3) / 1e12, 2), "gpu_launches": reps + 3}


def bench_prefill(args, sa, torch, device, pk):
    cfg = PREFILL
    lens = [cfg["seqlen"]] * cfg["batch"]
    host = workloads.make_prefill(cfg["seed"], lens, cfg["hq"], cfg["hkv"], cfg["d"], cfg["sink_std"])
    q, k, v = (to_dev(host[n], torch, device) for n in ("q", "k", "v"))
    sinks = to_dev(host["sinks"], torch, device)
    cu = to_dev(host["cu_seqlens"], torch, device)
    out = torch.empty_like(q)
    lse = torch.empty((q.shape[0], q.shape[1]), dtype=torch.float32, device=device)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    flops = prefill_flops(cfg["batch"], cfg["seqlen"], cfg["hq"], cfg["d"])

    def run():
        sa.sink_attn_prefill(q, k, v, sinks, cu, cfg["seqlen"], cfg["sm_scale"], causal=True,
                             out=out, lse=lse, stream=stream)

    for _ in range(max(3, args.warmup // 10)):
        run()
    steps = max(5, min(50, args.steps))
    times = []
    for _ in range(steps):
        flush_l2(flush)  # evict the previous launch's K/V from L2
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run()
        e1.record(stream)
        times.append((e0, e1))
    torch.cuda.synchronize(device)
    ms = sorted(a.elapsed_time(b) for a, b in times)
    avg = sum(ms) / len(ms)
    tflops = flops / (avg * 1e-3) / 1e12
    return {"workload": "causal_prefill: 4 x 8192 tokens, 64/8 heads", "value": round(tflops, 2),
            "unit": "TFLOP/s", "ms": round(avg, 4), "ms_median": round(ms[len(ms) // 2], 4), "flops": flops,
            "bound": "tensor",
            "kernel": "sink_prefill_kernel", "achieved": round(tflops, 2), "peak": pk["bf16"],
            "frac": round(tflops / pk["bf16"], 4), "peak_source": pk["source"] + " bf16 burst",
            "traffic": recorded_traffic("sink_prefill_kernel", PREFILL_SOURCES), "l2": "flushed before each launch",
            "gpu_launches": steps}


# ----------------------------------------------------------------------------- CPU baseline
def host_description():
    """Core count and CPU model of this host (for the CPU-baseline records)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None and os.path.exists("/proc/cpuinfo"):
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    import platform
    return {"nproc": os.cpu_count() or 1, "cpu_model": model or platform.processor() or platform.machine(),
            "machine": platform.machine()}


def oracle_decode_groups(host, cfg, groups, workers, max_tokens=None):
    """The oracle over (sequence, KV head) groups of a decode workload, on ``workers``
    threads (one BLAS thread each); returns (seconds, algorithmic bytes).  ``max_tokens``
    limits each group to its sequence's first tokens (a shorter sample of the same work)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    g = cfg["hq"] // cfg["hkv"]
    nb = len(host["kv_lens"])

    def one(u):
        b, kvh = divmod(u % (nb * cfg["hkv"]), cfg["hkv"])
        kv = int(host["kv_lens"][b])
        if max_tokens is not None:
            kv = min(kv, int(max_tokens))
        kb = oracle.widen_bf16(oracle.gather_pages(host["k_pages"][:, kvh:kvh + 1], host["page_table"][b], kv)[:, 0])
        vb = oracle.widen_bf16(oracle.gather_pages(host["v_pages"][:, kvh:kvh + 1], host["page_table"][b], kv)[:, 0])
        qf = oracle.widen_bf16(host["q"][b, kvh * g:(kvh + 1) * g])
        for hh in range(g):
            oracle.attention_with_sink(qf[hh][None], kb, vb, float(host["sinks"][kvh * g + hh]), cfg["sm_scale"])
        return kv * cfg["d"] * 2 * 2 + g * cfg["d"] * 2 * 2 + g * 4

    t0 = time.perf_counter()
    if workers <= 1:
        nbytes = sum(one(u) for u in groups)
    else:
        with ThreadPoolExecutor(max_workers=workers) as ex:
            nbytes = sum(ex.map(one, groups))
    return time.perf_counter() - t0, nbytes


def cpu_baseline(host, budget_s=12.0):
    """The oracle on the headline workload (8 x 131072-token decode), every host core, on
    a bounded sample of (sequence, KV head) groups."""
    cfg = LONG
    hd = host_description()
    workers = hd["nproc"]
    groups_total = len(host["kv_lens"]) * cfg["hkv"]
    t1, _ = oracle_decode_groups(host, cfg, range(workers), workers)       # warm-up, one group per thread
    rounds = max(1, int(budget_s / max(t1, 1e-3)))
    secs, nbytes = oracle_decode_groups(host, cfg, range(rounds * workers), workers)
    n = rounds * workers
    return {"value": round(nbytes / secs / 1e9, 4), "unit": "GB/s", "cores": workers, "kind": "oracle",
            "sample": f"{n} (sequence, KV head) groups of the 8 x 131072 decode ({n / groups_total:.2f} passes), "
                      f"{secs:.1f} s, fp64 numpy, {workers} threads x 1 BLAS thread",
            "nproc": hd["nproc"], "cpu_model": hd["cpu_model"], "machine": hd["machine"],
            "threads": workers, "blas_threads_per_thread": 1}


def cpu_baselines_per_row(budget_s=3.0):
    """The oracle timed beside every other measured row, on bounded samples of the same
    workloads (single thread, fp64): prefill rows, QKV bias + YaRN tokens, router rows,
    linear-layer rows.  Values in the unit of the row's own measurement."""
    import oracle
    from oracle import moe, rope
    res = {}
    # prefill: rows of sequence 0 of the causal-prefill workload at spread positions
    cfg = PREFILL
    data = workloads.make_prefill(cfg["seed"], [cfg["seqlen"]], cfg["hq"], cfg["hkv"], cfg["d"], cfg["sink_std"])
    g = cfg["hq"] // cfg["hkv"]
    kf = oracle.widen_bf16(data["k"][:, 0])
    vf = oracle.widen_bf16(data["v"][:, 0])
    rng = np.random.default_rng(9)
    flops, t0, n = 0.0, time.perf_counter(), 0
    while time.perf_counter() - t0 < budget_s:
        i = int(rng.integers(0, cfg["seqlen"]))
        h = int(rng.integers(0, g))
        oracle.attention_with_sink(oracle.widen_bf16(data["q"][i:i + 1, h]), kf[:i + 1], vf[:i + 1],
                                   float(data["sinks"][h]), cfg["sm_scale"])
        flops += 4.0 * cfg["d"] * (i + 1)
        n += 1
    secs = time.perf_counter() - t0
    res["prefill"] = {"value": round(flops / secs / 1e12, 6), "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                      "sample": f"{n} causal query rows of one 8192-token sequence, {secs:.1f} s"}
    # QKV bias + YaRN: 256 tokens
    inp = workloads.make_qkv(41, 256, cfg["hq"], cfg["hkv"])
    inv = rope.yarn_inv_freq(64, 150000.0, 32.0, 4096, 32.0, 1.0)
    cu = workloads.cu_seqlens_from([256])
    t0 = time.perf_counter()
    reps = 0
    while time.perf_counter() - t0 < budget_s / 3 or reps == 0:
        rope.qkv_bias_rope(inp["qkv"], inp["bias"], cu, None, cfg["hq"], cfg["hkv"], 64, inv, rope.yarn_mscale(32.0))
        reps += 1
    secs = time.perf_counter() - t0
    nbytes = reps * 2 * 256 * (cfg["hq"] + 2 * cfg["hkv"]) * 64 * 2
    res["qkv_bias_rope"] = {"value": round(nbytes / secs / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                            "sample": f"{reps} x 256 tokens, {secs:.1f} s"}
    # router: 256 rows of 128 logits, top 4
    lg = workloads.make_router_logits(42, 256, 128, std=2.0)
    t0 = time.perf_counter()
    reps = 0
    while time.perf_counter() - t0 < budget_s / 3 or reps == 0:
        moe.router_topk_softmax(lg, 4)
        reps += 1
    secs = time.perf_counter() - t0
    res["moe_router"] = {"value": round(reps * 256 * (128 * 2 + 4 * 6) / secs / 1e9, 6), "unit": "GB/s",
                         "cores": 1, "kind": "oracle", "sample": f"{reps} x 256 rows, {secs:.1f} s"}
    # linear: 64 rows of the output projection
    d = workloads.make_linear(61, 64, 2880, 4096)
    t0 = time.perf_counter()
    reps = 0
    while time.perf_counter() - t0 < budget_s / 3 or reps == 0:
        moe.linear_bias(d["x"], d["w"], d["bias"])
        reps += 1
    secs = time.perf_counter() - t0
    res["linear_bias"] = {"value": round(reps * 2.0 * 64 * 2880 * 4096 / secs / 1e12, 6), "unit": "TFLOP/s",
                          "cores": 1, "kind": "oracle", "sample": f"{reps} x 64 rows of [., 4096] x [2880, 4096]^T, {secs:.1f} s"}
    return res


def run_reference(args, budget_s=90.0):
    """The oracle as the reference arm: each step is one (sequence, KV head) group per host
    core of the headline workload (8 x 131072-token decode), all cores busy.  The first
    warm-up step times a full step; when the requested warm-up + timed steps would take
    longer than ``budget_s``, every group is cut to its sequence's first tokens so that the
    run stays within about that long (the line says so in its sample)."""
    cfg = LONG
    host = workloads.make_decode(cfg["seed"], [cfg["kv_len"]] * cfg["batch"], cfg["hq"], cfg["hkv"],
                                 cfg["d"], cfg["page_size"], cfg["sink_std"])
    hd = host_description()
    workers = hd["nproc"]
    t_full, _ = oracle_decode_groups(host, cfg, range(workers), workers)
    max_tokens = None
    if (args.warmup + args.steps) * t_full > budget_s:
        frac = budget_s / ((args.warmup + args.steps) * t_full)
        ps = cfg["page_size"]
        max_tokens = max(ps, int(cfg["kv_len"] * frac) // ps * ps)
    for w in range(1, args.warmup):
        oracle_decode_groups(host, cfg, range(w * workers, (w + 1) * workers), workers, max_tokens)
    tot_s = 0.0
    tot_b = 0
    for k in range(args.steps):
        secs, nb = oracle_decode_groups(host, cfg, range(k * workers, (k + 1) * workers), workers, max_tokens)
        tot_s += secs
        tot_b += nb
    value = tot_b / tot_s / 1e9
    span = (f"the first {max_tokens} of each sequence's {cfg['kv_len']} tokens" if max_tokens
            else f"all {cfg['kv_len']} tokens")
    sample = (f"{workers} (sequence, KV head) groups of the 8 x 131072 decode per step ({span}), fp64 numpy, "
              f"{workers} threads x 1 BLAS thread")
    return {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(tot_s / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": LONG_WORKLOAD},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": workers, "kind": "oracle",
                         "sample": sample, "nproc": hd["nproc"], "cpu_model": hd["cpu_model"]},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- ncu cases
def run_profile_case(case):
    """Small launches of one kernel for ncu captures: 2 warm-up launches, then 3.

    decode:  32 sequences x 4096 tokens (256 MiB of KV, larger than L2), 64/8 heads, 4 splits.
    decode_long: 2 sequences x 131072 tokens (512 MiB of KV), 64/8 heads, 32 splits.
    decode_one: one sequence of 4096 tokens per launch (16-CTA clusters merged on chip),
             launches cycling over 32 sequences of a 256 MiB pool.
    prefill: 1 x 8192 tokens causal, 64/8 heads.
    prefill_persistent: 8192 + 8191 tokens causal (the persistent schedule), 64/8 heads.
    mixed:   the ragged mixed batch (32 sequences, paged, GQA-packed decode rows).
    linear:  [32768, 4096] x [2880, 4096]^T + bias (the bench's output projection, ~470 MB).
    rope:    32768 tokens, 64/8 heads, bias + YaRN.
    router:  32768 tokens x 128 experts, top 4, counts.
    router_fused: the router projection [32768, 2880] x [128, 2880]^T + bias with the Top-K epilogue.
    """
    import torch
    import attention_softmax_sinks_gb300 as sa
    from attention_softmax_sinks_gb300 import _build
    _build.build()
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    if case == "decode":
        cfg = DECODE
        host = workloads.make_decode(cfg["seed"], [cfg["kv_len"]] * 32, cfg["hq"], cfg["hkv"], cfg["d"],
                                     cfg["page_size"], cfg["sink_std"])
        dev = {n: to_dev(host[n], torch, device)
               for n in ("q", "k_pages", "v_pages", "page_table", "kv_lens", "sinks")}
        for _ in range(5):
            po, pl = sa.sink_attn_decode(dev["q"], dev["k_pages"], dev["v_pages"], dev["page_table"],
                                         dev["kv_lens"], dev["sinks"], cfg["sm_scale"], num_splits=4)
            sa.sink_attn_merge(po, pl)
    elif case == "decode_long":
        cfg = workloads.WORKLOADS["long_decode"]
        host = workloads.make_decode(cfg["seed"], [cfg["kv_len"]] * 2, cfg["hq"], cfg["hkv"], cfg["d"],
                                     cfg["page_size"], cfg["sink_std"])
        dev = {n: to_dev(host[n], torch, device)
               for n in ("q", "k_pages", "v_pages", "page_table", "kv_lens", "sinks")}
        for _ in range(5):
            po, pl = sa.sink_attn_decode(dev["q"], dev["k_pages"], dev["v_pages"], dev["page_table"],
                                         dev["kv_lens"], dev["sinks"], cfg["sm_scale"], num_splits=cfg["num_splits"])
            sa.sink_attn_merge(po, pl)
    elif case == "decode_one":
        cfg = DECODE
        host = workloads.make_decode(cfg["seed"] + 7, [cfg["kv_len"]] * 32, cfg["hq"], cfg["hkv"], cfg["d"],
                                     cfg["page_size"], cfg["sink_std"])
        dev = {n: to_dev(host[n], torch, device)
               for n in ("q", "k_pages", "v_pages", "page_table", "kv_lens", "sinks")}
        for i in range(5):
            sl = slice(i, i + 1)
            sa.sink_attn_decode(dev["q"][sl], dev["k_pages"], dev["v_pages"], dev["page_table"][sl],
                                dev["kv_lens"][sl], dev["sinks"], cfg["sm_scale"], num_splits=1)
    elif case == "prefill_persistent":
        cfg = PREFILL
        lens = [cfg["seqlen"], cfg["seqlen"] - 1]  # not uniform: the persistent schedule
        host = workloads.make_prefill(cfg["seed"], lens, cfg["hq"], cfg["hkv"], cfg["d"], cfg["sink_std"])
        q, k, v, sinks, cu = (to_dev(host[n], torch, device) for n in ("q", "k", "v", "sinks", "cu_seqlens"))
        for _ in range(5):
            sa.sink_attn_prefill(q, k, v, sinks, cu, cfg["seqlen"], cfg["sm_scale"], causal=True)
    elif case == "mixed":
        cfg = workloads.WORKLOADS["ragged_mixed"]
        q_lens, kv_lens = workloads.ragged_mixed_lengths(cfg["seed"] + 2, cfg["num_seqs"], cfg["max_kv"])
        host = workloads.make_mixed(cfg["seed"], q_lens, kv_lens, cfg["hq"], cfg["hkv"], cfg["d"],
                                    cfg["page_size"], cfg["sink_std"])
        dv = {n: to_dev(host[n], torch, device)
              for n in ("q", "k_pages", "v_pages", "page_table", "cu_seqlens_q", "kv_lens", "sinks")}
        for _ in range(5):
            sa.sink_attn_prefill_paged(dv["q"], dv["k_pages"], dv["v_pages"], dv["page_table"], dv["cu_seqlens_q"],
                                       dv["kv_lens"], dv["sinks"], int(q_lens.max()), cfg["sm_scale"], causal=True)
    elif case == "router_fused":
        d = workloads.make_linear(43, 32768, 128, 2880, std=1.0, w_std=0.05, bias_std=0.5)
        x, w, b = (to_dev(d[key], torch, device) for key in ("x", "w", "bias"))
        for _ in range(5):
            sa.moe_router(x, w, b, 4, return_counts=True)
    elif case == "linear":
        d = workloads.make_linear(61, 32768, 2880, 4096)
        x, w, b = (to_dev(d[key], torch, device) for key in ("x", "w", "bias"))
        out = torch.empty((32768, 2880), dtype=torch.bfloat16, device=device)
        for _ in range(5):
            sa.linear_bias(x, w, b, out=out)
    elif case == "rope":
        cu = to_dev(workloads.cu_seqlens_from([8192] * 4), torch, device)
        inp = workloads.make_qkv(41, 32768, 64, 8)
        qkv, bias = to_dev(inp["qkv"], torch, device), to_dev(inp["bias"], torch, device)
        for _ in range(5):
            sa.qkv_bias_rope(qkv, bias, cu, 64, 8)
    elif case == "router":
        logits = to_dev(workloads.make_router_logits(42, 32768, 128, std=2.0), torch, device)
        for _ in range(5):
            sa.moe_router_topk_softmax(logits, 4, return_counts=True)
    else:
        cfg = PREFILL
        host = workloads.make_prefill(cfg["seed"], [cfg["seqlen"]], cfg["hq"], cfg["hkv"], cfg["d"],
                                      cfg["sink_std"])
        q, k, v, sinks, cu = (to_dev(host[n], torch, device) for n in ("q", "k", "v", "sinks", "cu_seqlens"))
        for _ in range(5):
            sa.sink_attn_prefill(q, k, v, sinks, cu, cfg["seqlen"], cfg["sm_scale"], causal=True)
    torch.cuda.synchronize(device)
    print(json.dumps({"profile_case": case, "device_status": sa.sink_attn_device_status(True)}))


# ----------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-prefill", action="store_true", help="skip the prefill measurement")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing")
    ap.add_argument("--profile", choices=["decode", "decode_long", "decode_one", "prefill", "prefill_persistent", "mixed", "linear",
                                          "rope", "router", "router_fused"], default=None,
                    help="run a small case of one kernel for an ncu capture, then exit")
    args = ap.parse_args()
    if args.profile:
        run_profile_case(args.profile)
        return
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    import torch
    local = int(os.environ.get("LOCAL_RANK", "0"))
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=device)
    line, host = run_ours(args, rank, world, device)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(host)
            per_row = cpu_baselines_per_row()
            # the oracle beside the other rows: value in the row's unit, one thread
            if "prefill" in line:
                line["prefill"]["cpu_baseline"] = {k: per_row["prefill"][k] for k in ("value", "cores", "sample")}
            for key, row in (("qkv_bias_rope", "qkv_bias_rope"), ("moe_router", "moe_router"),
                             ("linear_bias", "linear")):
                if "around" in line and row in line["around"]:
                    line["around"][row]["cpu_baseline"] = per_row[key]["value"]
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
