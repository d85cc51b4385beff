#!/usr/bin/env python
"""Benchmark of the GB300 verify attention (MLA, paged KV cache, draft tree).

One step = one verify call (split-KV partial kernel + LSE combine) over the
decode-batch workload (B=8 requests, 4096-token prefix each, T=8 chain
drafts, H=64 heads, page_size=1 scattered slots in a 65536-slot cache, 1% of
keys x8), inputs resident in HBM.  Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the fp64 CPU oracle as reference arm

Timing: every step writes a 512 MB buffer (larger than the 126 MB L2) before
the call, then CUDA events on the call's stream bracket the call; an event
the library records between its two kernels splits partial and combine.
Under torchrun every rank runs an independent replica (the operation has no
cross-request exchange), and the slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 512 << 20


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default="decode_batch")
    ap.add_argument("--e2e-steps", type=int, default=300)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    return ap.parse_args(argv)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            return {k: float(d[k]) for k in FALLBACK_PEAKS if k in d}, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash():
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "paged_mla_speculative_gb300", "csrc")
    for name in ("common.cuh", "tc_ptx.cuh", "partial_tc.cu"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic(workload):
    """DRAM bytes per launch of the partial kernel from a committed ncu
    summary, if it was taken on the current kernel source and workload."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get("partial_tc_kernel", {})
        if e.get("source_sha1") == kernel_source_hash() and e.get("workload") == workload:
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def compaction_timing(mb, plan, inp, w, flush, stream, steps):
    """µs and GB/s of compacting the step's requests into fresh 64-row pages
    (L2 flushed before each call); bytes = rows read + rows written."""
    import torch
    if inp.page_size != 1:
        return None
    pages_needed = sum((int(n) + 63) // 64 for n in inp.kv_lens.tolist())
    dst = torch.empty((pages_needed * 64, 576), dtype=torch.bfloat16, device="cuda")
    free = torch.arange(pages_needed, dtype=torch.int32, device="cuda")
    table = torch.empty(pages_needed, dtype=torch.int32, device="cuda")
    pin = torch.empty(w.batch + 1, dtype=torch.int32, device="cuda")

    def call():
        mb.compact_kv(plan, inp.kv_cache, inp.kv_indices, inp.kv_indptr, inp.kv_lens, free, dst,
                      table, pin, stream=stream)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    assert plan.get_error() == 0 and torch.equal(table, free)
    ea = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    eb = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        ea[i].record(stream)
        call()
        eb[i].record(stream)
    torch.cuda.synchronize()
    us = statistics.fmean(a.elapsed_time(b) for a, b in zip(ea, eb)) * 1e3
    rows = int(inp.kv_lens.sum())
    nbytes = rows * 1152 * 2 + rows * 4 + pages_needed * 8 + (w.batch + 1) * 8
    peaks, _ = load_peaks()
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"us_per_call": us, "pages": pages_needed, "algorithmic_bytes": nbytes, "gbs": gbs,
            "frac_of_hbm": gbs / hbm, "bound": "hbm", "launches": 2}


def small_r_timing(mb, W, name, flush, stream, steps):
    """µs per call, KV GB/s and the fraction of the HBM roof for one of the
    small-R workloads (L2 flushed before every call, events on the stream)."""
    import torch
    w = W.WORKLOADS[name]
    inp = W.make_inputs(w, device="cuda")
    work = W.algorithmic_work(inp.prefix, w.num_drafts, w.num_heads)
    plan = mb.Plan(w.batch, w.num_drafts, w.num_heads, w.page_size, w.num_slots,
                   max(inp.kv_lens.tolist()))
    out, lse = plan.new_outputs(w.batch)

    def call():
        mb.mla_verify_attn(plan, inp.q, inp.kv_cache, inp.kv_indices, inp.kv_indptr,
                           inp.kv_lens, inp.draft_parent, inp.scale, out, lse, stream=stream)

    for _ in range(3):
        flush.zero_()
        call()
    torch.cuda.synchronize()
    ea = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    eb = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        ea[i].record(stream)
        call()
        eb[i].record(stream)
    torch.cuda.synchronize()
    assert plan.get_error() == 0
    us = statistics.fmean(a.elapsed_time(b) for a, b in zip(ea, eb)) * 1e3
    peaks, _ = load_peaks()
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    kv_gbs = work["kv_bytes"] / (us * 1e-6) / 1e9
    tc = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    t_hbm, t_tc = work["bytes"] / (hbm * 1e9), work["flops"] / (tc * 1e12)
    t_roof = max(t_hbm, t_tc) * 1e6
    res = {"us_per_call": us, "kv_gbs": kv_gbs, "kv_frac_of_hbm": kv_gbs / hbm,
           "roofline_time_us": t_roof, "frac_of_roofline": t_roof / us,
           "bound": "hbm" if t_hbm > t_tc else "tensor",
           "nsplit": plan.nsplit(w.batch), "rows_per_request": w.num_drafts * w.num_heads}
    plan.close()
    return res


def kernels_of(kernel, ns, pack_stay=0):
    """The library kernels one call launches, for the JSON line (pack_stay >
    0: the pack that overlaps the attention kernel)."""
    from paged_mla_speculative_gb300 import binding as mb
    pack = "pack_kv_overlap_kernel" if pack_stay > 0 else "pack_kv_kernel"
    names = {mb.KERNEL_TC: [pack, "partial_tc_kernel"],
             mb.KERNEL_MMA: ["partial_mma_kernel"]}[kernel]
    return " + ".join(names + (["combine_kernel"] if ns > 1 else []))


def index_builder_timing(mb, plan, inp, w, flush, stream, steps):
    """Mean µs of mla_verify_build_indices for this step's requests (L2
    flushed before each build), its algorithmic bytes and GB/s."""
    import torch
    B = w.batch
    lens = inp.kv_lens.to(torch.int64)
    ptr = inp.kv_indptr.to(torch.int64)
    stride = plan.max_kv_len
    gen = torch.Generator().manual_seed(w.seed + 29)
    pool_of = torch.randperm(B + 5, generator=gen)[:B]
    table = torch.full((B + 5, stride), -1, dtype=torch.int32, device="cuda")
    if inp.page_size == 1:
        for b in range(B):
            table[pool_of[b], :int(lens[b])] = inp.kv_indices[int(ptr[b]):int(ptr[b]) + int(lens[b])]
    else:
        for b in range(B):
            pages = inp.kv_indices[int(ptr[b]):int(ptr[b + 1])].to(torch.int64)
            slots = (pages[:, None] * 64 + torch.arange(64, device="cuda")[None, :]).reshape(-1)
            table[pool_of[b], :int(lens[b])] = slots[:int(lens[b])].to(torch.int32)
    pools = pool_of.to(torch.int32).cuda()
    prefix = (inp.kv_lens - w.num_drafts).to(torch.int32).cuda()
    idx = torch.empty(int(ptr[-1]) + 64, dtype=torch.int32, device="cuda")
    iptr = torch.empty(B + 1, dtype=torch.int32, device="cuda")
    ilens = torch.empty(B, dtype=torch.int32, device="cuda")
    for _ in range(3):
        mb.build_indices(plan, table, pools, prefix, idx, iptr, ilens, stream=stream)
    torch.cuda.synchronize()
    assert torch.equal(iptr, inp.kv_indptr) and torch.equal(ilens, inp.kv_lens)
    assert torch.equal(idx[:int(ptr[-1])], inp.kv_indices), "built indices differ from the workload's"
    ea = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    eb = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        ea[i].record(stream)
        mb.build_indices(plan, table, pools, prefix, idx, iptr, ilens, stream=stream)
        eb[i].record(stream)
    torch.cuda.synchronize()
    us = statistics.fmean(a.elapsed_time(b) for a, b in zip(ea, eb)) * 1e3
    # Device time without host gaps: 20 builds captured in one graph, replayed.
    g = torch.cuda.CUDAGraph()
    gs = torch.cuda.Stream()
    gs.wait_stream(stream)
    with torch.cuda.graph(g, stream=gs):
        for _ in range(20):
            mb.build_indices(plan, table, pools, prefix, idx, iptr, ilens, stream=gs)
    ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g.replay()
    torch.cuda.synchronize()
    ga.record(stream)
    for _ in range(10):
        g.replay()
    gb.record(stream)
    torch.cuda.synchronize()
    us_warm = ga.elapsed_time(gb) * 1e3 / 200
    entries = int(ptr[-1])
    # per entry: one table slot read (a page's first slot for page_size 64) and
    # one index written; per request: pool row, prefix, kv_len; plus indptr
    nbytes = entries * (4 + 4) + B * (4 + 4 + 4) + (B + 1) * 4
    return {"us_per_step": us, "us_per_step_graph_warm_l2": us_warm, "entries": entries,
            "algorithmic_bytes": nbytes, "gbs": nbytes / (us * 1e-6) / 1e9,
            "launches": 1 if B <= 1024 else 2,
            "note": "us_per_step: L2 flushed before each build, launched from Python like the "
                    "attention; us_per_step_graph_warm_l2: device time of builds replayed from "
                    "a CUDA graph. At this size the build is bound by latency, not bandwidth"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.proc = None
        self.uuid = uuid

    def __enter__(self):
        try:
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "100"]
            if self.uuid:
                cmd += ["-i", self.uuid]
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            parts = [x.strip() for x in l.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(args):
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(ws, value):
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def config_of(w, extra=None):
    prefix = w.prefix if w.prefix[0] != "uniform" else f"U[{w.prefix[1]},{w.prefix[2]}]"
    c = {"workload": w.name, "batch": w.batch,
         "context": prefix[0] if isinstance(prefix, tuple) and len(set(prefix)) == 1 else prefix,
         "drafts": w.num_drafts, "tree": w.tree, "heads": w.num_heads, "page_size": w.page_size,
         "cache_slots": w.num_slots, "spiky_keys": f"{w.spike_frac:.0%} x{w.spike_mult:g}",
         "input_dtype": "bf16", "out_dtype": "fp32", "parallelism": "replicas",
         "l2": "flushed: 512 MB write before every call"}
    if extra:
        c.update(extra)
    return c


def _bits(t):
    """bf16 tensor -> numpy uint16 bit patterns (the oracle's input form)."""
    import torch
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


def oracle_seconds_per_call(inp, budget_s):
    """CPU oracle on whole requests, round robin, until the budget is spent."""
    import numpy as np
    import oracle
    qb, cb = _bits(inp.q), _bits(inp.kv_cache)
    idx = inp.kv_indices.cpu().numpy()
    ptr = inp.kv_indptr.cpu().numpy()
    lens = inp.kv_lens.cpu().numpy()
    par = inp.draft_parent.cpu().numpy()
    B = len(lens)
    done, t0 = 0, time.perf_counter()
    while True:
        b = done % B
        sub_ptr = np.array([0, ptr[b + 1] - ptr[b]], dtype=np.int64)
        oracle.mla_verify(qb[b:b + 1], cb, idx[ptr[b]:ptr[b + 1]], sub_ptr, lens[b:b + 1],
                          par[b:b + 1], inp.scale, inp.page_size)
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return el / done * B, done


def run_reference(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import numpy as np
    import oracle
    from paged_mla_speculative_gb300 import workloads as W
    w = W.WORKLOADS[args.workload]
    inp = W.make_inputs(w, device="cpu")
    qb, cb = _bits(inp.q), _bits(inp.kv_cache)
    idx, ptr = inp.kv_indices.numpy(), inp.kv_indptr.numpy()
    lens, par = inp.kv_lens.numpy(), inp.draft_parent.numpy()
    B, T, H = w.batch, w.num_drafts, w.num_heads
    rows_per_call = B * T * H

    def step(i, nrows):
        b, t = (i // T) % B, i % T
        rows = [(b, t, h) for h in range(nrows)]
        oracle.mla_verify_rows(rows, qb, cb, idx, ptr, lens, par, inp.scale, inp.page_size)

    # Size the per-step sample so warm-up + steps end within ~150 s.
    t0 = time.perf_counter()
    step(0, 1)
    t_row = max(time.perf_counter() - t0, 1e-4)
    budget = 150.0 / max(1, args.steps + args.warmup)
    nrows = max(1, min(H, int(budget / t_row)))
    for i in range(args.warmup):
        step(i, nrows)
    times, t_start = [], time.perf_counter()
    steps_run = 0
    for i in range(args.steps):
        s0 = time.perf_counter()
        step(i, nrows)
        times.append(time.perf_counter() - s0)
        steps_run += 1
        if time.perf_counter() - t_start > 180.0:
            break
    per_row = sum(times) / (steps_run * nrows)
    us_per_call = per_row * rows_per_call * 1e6
    cores = len(os.sched_getaffinity(0))
    line = {
        "impl": "reference", "metric": "verify_attn_us_per_call", "value": us_per_call,
        "unit": "us/call", "n_gpus": ws, "steps": args.steps, "steps_run": steps_run,
        "warmup": args.warmup, "ms_per_step": sum(times) / steps_run * 1e3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded), generated on the host",
        "config": config_of(w),
        "cpu_baseline": {"value": us_per_call, "unit": "us/call", "cores": cores, "kind": "oracle",
                         "sample": f"{nrows} query rows of one (request, draft) per step, "
                                   f"gather included, scaled to {rows_per_call} rows per call"},
        "e2e": {"value": us_per_call, "unit": "us/call", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_gb300(args):
    import torch
    ws, rank, local = dist_setup(args)
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device (the verify attention has no CPU path)")
    torch.cuda.set_device(local)
    from paged_mla_speculative_gb300 import binding as mb
    from paged_mla_speculative_gb300 import build as mbuild
    from paged_mla_speculative_gb300 import workloads as W
    if rank == 0:
        mbuild.build()
    barrier(ws)

    w = W.WORKLOADS[args.workload]
    inp = W.make_inputs(w, device="cuda")
    work = W.algorithmic_work(inp.prefix, w.num_drafts, w.num_heads)
    max_len = max(inp.kv_lens.tolist())
    plan = mb.Plan(w.batch, w.num_drafts, w.num_heads, w.page_size, w.num_slots, max_len)
    ns = plan.nsplit(w.batch)
    out, lse = plan.new_outputs(w.batch)
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    def call():
        mb.mla_verify_attn(plan, inp.q, inp.kv_cache, inp.kv_indices, inp.kv_indptr,
                           inp.kv_lens, inp.draft_parent, inp.scale, out, lse, stream=stream)

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        call()
    torch.cuda.synchronize()
    assert plan.get_error() == 0, "device error word set during warm-up"

    K = args.steps
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        pass

    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(uuid) as clk:
        t0 = time.perf_counter()
        for i in range(K):
            flush.zero_()
            ev_a[i].record(stream)
            call()
            ev_b[i].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    barrier(ws)
    call_ms = [a.elapsed_time(b) for a, b in zip(ev_a, ev_b)]

    # Per-kernel split: a second, shorter pass with events between the
    # kernels.  The library then runs the kernels back to back (no launch
    # overlap), so each difference times one kernel alone; the partial
    # kernel's time here is the roofline's denominator.
    kp = min(K, 300)
    pa = [torch.cuda.Event(enable_timing=True) for _ in range(kp)]
    pk = [torch.cuda.Event(enable_timing=True) for _ in range(kp)]
    pm = [torch.cuda.Event(enable_timing=True) for _ in range(kp)]
    pb = [torch.cuda.Event(enable_timing=True) for _ in range(kp)]
    for e in pk + pm:
        e.record(stream)
    torch.cuda.synchronize()
    for i in range(kp):
        flush.zero_()
        plan.set_profile_events(pk[i], pm[i])
        pa[i].record(stream)
        call()
        pb[i].record(stream)
    torch.cuda.synchronize()
    plan.set_profile_events(None, None)
    pack_ms = [a.elapsed_time(k) for a, k in zip(pa, pk)]
    part_ms = [k.elapsed_time(m) for k, m in zip(pk, pm)]
    comb_ms = [m.elapsed_time(b) for m, b in zip(pm, pb)]
    prof_call_ms = [a.elapsed_time(b) for a, b in zip(pa, pb)]

    mean_call = max_over_ranks(ws, statistics.fmean(call_ms))
    mean_pack = max_over_ranks(ws, statistics.fmean(pack_ms))
    mean_part = max_over_ranks(ws, statistics.fmean(part_ms))
    mean_comb = max_over_ranks(ws, statistics.fmean(comb_ms))
    us_per_call = mean_call * 1e3 / ws          # whole job: ws replicas in parallel
    q = statistics.quantiles(call_ms, n=10)

    # Per-step index builder on the same step: the request-to-token table
    # holds each request's slots (pool rows permuted); time the build alone.
    ib = index_builder_timing(mb, plan, inp, w, flush, stream, min(K, 300))

    # KV compaction of this step's requests into fresh 64-row pages.
    compaction = compaction_timing(mb, plan, inp, w, flush, stream, min(K, 200))

    # The small-R regime (a tensor-parallel head slice, one-token decode):
    # HBM is the roof there; same call protocol, fewer calls.
    small_r = {name: small_r_timing(mb, W, name, flush, stream, min(K, 200))
               for name in ("decode_tp8", "decode_t1")}

    # CUDA-graph replay of the same call (capture-safe path), device timed.
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(stream)
    with torch.cuda.stream(s):
        call_s = lambda: mb.mla_verify_attn(plan, inp.q, inp.kv_cache, inp.kv_indices,  # noqa: E731
                                            inp.kv_indptr, inp.kv_lens, inp.draft_parent,
                                            inp.scale, out, lse, stream=s)
        call_s()
    s.synchronize()
    with torch.cuda.graph(g, stream=s):
        call_s()
    gk = min(K, 500)
    ga = [torch.cuda.Event(enable_timing=True) for _ in range(gk)]
    gb = [torch.cuda.Event(enable_timing=True) for _ in range(gk)]
    for i in range(gk):
        flush.zero_()
        ga[i].record(stream)
        g.replay()
        gb[i].record(stream)
    torch.cuda.synchronize()
    graph_us = statistics.fmean(a.elapsed_time(b) for a, b in zip(ga, gb)) * 1e3

    # End to end through the host-buffer entry point: H2D of the step's
    # inputs from pinned memory, the call, D2H of out/lse, stream sync.
    hq = inp.q.cpu().pin_memory()
    hidx = inp.kv_indices.cpu().pin_memory()
    hptr = inp.kv_indptr.cpu().pin_memory()
    hlen = inp.kv_lens.cpu().pin_memory()
    hpar = inp.draft_parent.cpu().pin_memory()
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    hlse = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    for _ in range(3):
        mb.mla_verify_attn_host(plan, hq, inp.kv_cache, hidx, hptr, hlen, hpar, inp.scale,
                                hout, hlse, stream=stream)
    e2e_steps = min(args.e2e_steps, K)
    barrier(ws)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        mb.mla_verify_attn_host(plan, hq, inp.kv_cache, hidx, hptr, hlen, hpar, inp.scale,
                                hout, hlse, stream=stream)
    e2e_s = max_over_ranks(ws, time.perf_counter() - t0)
    e2e_us = e2e_s / e2e_steps / ws * 1e6
    h2d = sum(t.numel() * t.element_size() for t in (hq, hidx, hptr, hlen, hpar))
    d2h = hout.numel() * hout.element_size() + hlse.numel() * 4
    assert torch.equal(hout, out.cpu()), "host entry point disagrees with device entry point"
    assert plan.get_error() == 0

    peaks, peak_src = load_peaks()
    flops = work["flops"]
    achieved = flops / (mean_part * 1e-3) / 1e12
    peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    kv_gbs = work["kv_bytes"] / (mean_call * 1e-3) / 1e9
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    t_roof_us = max(work["bytes"] / (hbm * 1e9), flops / (peak * 1e12)) * 1e6
    clocks = clk.summary()
    pack_wide, pack_stay = plan.pack_schedule(w.batch)
    launches = K * (len(kernels_of(plan.kernel(), ns, pack_stay).split(" + ")))

    line = {
        "metric": "verify_attn_us_per_call", "value": us_per_call, "unit": "us/call",
        "n_gpus": ws, "steps": K, "warmup": args.warmup, "ms_per_step": mean_call,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16", "data": "synthetic (seeded), bf16 inputs resident in HBM",
        "config": config_of(w, {"nsplit": ns, "kernels": kernels_of(plan.kernel(), ns, pack_stay),
                                "pack_schedule": {"wide_positions": pack_wide, "overlap_ctas": pack_stay}}),
        "us_per_call_p10_p50_p90": [q[0] * 1e3, statistics.median(call_ms) * 1e3, q[-1] * 1e3],
        "pack_us": mean_pack * 1e3, "partial_us": mean_part * 1e3, "combine_us": mean_comb * 1e3,
        "serialised_us_per_call": statistics.fmean(prof_call_ms) * 1e3,
        "graph_replay_us_per_call": graph_us,
        "kv_gbs": kv_gbs, "kv_frac_of_hbm": kv_gbs / hbm,
        "roofline_time_us": t_roof_us, "frac_of_roofline": t_roof_us / (mean_call * 1e3),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": profiled_traffic(w.name),
                     "kernel": "partial_tc_kernel",
                     "peak_source": f"{peak_src} bf16 burst (fp16 has the same tensor rate)"},
        "index_builder": ib,
        "small_r": small_r,
        "compaction": compaction,
        "clocks": clocks, "gpu_launches": launches,
        "e2e": {"value": e2e_us, "unit": "us/call", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "timed_wall_s": wall,
    }
    if ws == 1 and rank == 0 and not args.no_cpu_baseline:
        sec, nreq = oracle_seconds_per_call(inp, args.cpu_seconds)
        line["cpu_baseline"] = {"value": sec * 1e6, "unit": "us/call",
                                "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
                                "sample": f"{nreq} whole requests of the same inputs (fp64 NumPy), "
                                          f"scaled to {w.batch} requests per call"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    plan.close()
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_gb300(args)


if __name__ == "__main__":
    sys.exit(main())
