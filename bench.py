#!/usr/bin/env python
"""Benchmark of the GB300 verify attention (MLA, paged KV cache, draft tree).

The metric is µs per call and KV-read GB/s against context.  One step is one
verify call (key pack + split-KV partial kernel + LSE combine), replayed from
a CUDA graph, over one point of the context sweep: B=1 request, T=8 chain
drafts, H=64 heads, page_size=1 slots scattered in a 131072-slot cache, 1% of
the keys x8, prefix P in {1024, 4096, 16384, 65536, 93184}.  The K timed
steps run at the largest point (P=93184), which is the line's `value`; every
sweep point and every other workload (decode batch, tree, the two ragged
batches, tiny, the small-R shapes) is timed the same way, with fewer calls,
and reported under `workloads`.  Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the fp64 CPU oracle as reference arm

Timing: every step writes a 512 MB buffer (larger than the 126 MB L2) before
the replay, then CUDA events on the replay stream bracket it.  A second pass
of eager calls with events the library records between its kernels splits
pack, partial and combine.  Under torchrun every rank runs an independent
replica (requests have no cross-request exchange) and the slowest rank's
time is reported.
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
METRIC = "MLA verify attn \u00b5s/call and KV-read GB/s (% of GB300 HBM roofline) vs context"
CURVE_NAME = "context_sweep"
SWEEP = ["sweep_p1024", "sweep_p4096", "sweep_p16384", "sweep_p65536", "sweep_p93184"]
HEADLINE = "sweep_p93184"      # the largest sweep point: the line's value
OTHERS = ["tiny", "decode_batch", "tree", "ragged_ps1", "ragged_ps64", "decode_tp8", "decode_t1"]


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default=CURVE_NAME,
                    help=f"{CURVE_NAME} (default: the sweep plus every other workload) or one workload")
    ap.add_argument("--other-steps", type=int, default=200,
                    help="timed calls per workload besides the headline point")
    ap.add_argument("--e2e-steps", type=int, default=300)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--calls-only", choices=["attn", "index", "compact"], default=None,
                    help="no timing: issue --steps calls of one workload (a target for a profiler)")
    ap.add_argument("--kernel", choices=["auto", "pair", "tc", "mma"], default="auto")
    ap.add_argument("--pack-schedule", choices=["auto", "whole", "idle_sms", "none"], default="auto")
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


PARTIAL_SOURCES = {"partial_tc_kernel": "partial_tc.cu", "partial_pair_kernel": "partial_pair.cu",
                   "partial_mma_kernel": "partial_mma.cu"}


def kernel_source_hash(kernel="partial_pair_kernel"):
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "paged_mla_speculative_gb300", "csrc")
    for name in ("common.cuh", "tc_ptx.cuh", PARTIAL_SOURCES[kernel]):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic(workload, kernel="partial_pair_kernel"):
    """DRAM bytes per launch of the attention kernel from a committed ncu
    summary, if it was taken on the current kernel source and workload."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(kernel, {})
        if e.get("source_sha1") == kernel_source_hash(kernel) and e.get("workload") == workload:
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


PACK_NAMES = {1: "whole", 2: "idle_sms", 4: "none"}
PACK_KERNELS = {"whole": "pack_kv_kernel", "idle_sms": "pack_kv_overlap_kernel"}
PARTIAL_NAMES = {1: "partial_mma_kernel", 2: "partial_tc_kernel", 3: "partial_pair_kernel"}


def kernels_of(kernel, ns, schedule="whole"):
    """The library kernels one call launches, for the JSON line (schedule:
    the key-pack schedule, "none" when the attention CTAs gather their own
    keys)."""
    from paged_mla_speculative_gb300 import binding as mb
    tc = ["partial_tc_kernel"] if schedule == "none" else [PACK_KERNELS[schedule], "partial_tc_kernel"]
    pair = [PACK_KERNELS.get(schedule, "pack_kv_kernel"), "partial_pair_kernel"]
    names = {mb.KERNEL_TC: tc, mb.KERNEL_MMA: ["partial_mma_kernel"], mb.KERNEL_PAIR: pair}[kernel]
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


def workload_config(w):
    prefix = w.prefix if w.prefix[0] != "uniform" else f"U[{w.prefix[1]},{w.prefix[2]}]"
    return {"workload": w.name, "batch": w.batch,
            "context": prefix[0] if isinstance(prefix, tuple) and len(set(prefix)) == 1 else prefix,
            "drafts": w.num_drafts, "tree": w.tree, "heads": w.num_heads, "page_size": w.page_size,
            "cache_slots": w.num_slots, "spiky_keys": f"{w.spike_frac:.0%} x{w.spike_mult:g}"}


def config_of(name):
    """The line's `config`: identical in both arms for the same workload."""
    from paged_mla_speculative_gb300 import workloads as W
    common = {"input_dtype": "bf16", "out_dtype": "fp32", "parallelism": "replicas",
              "l2": "flushed: 512 MB write before every call"}
    if name == CURVE_NAME:
        w = W.WORKLOADS[HEADLINE]
        c = workload_config(w)
        c.update({"workload": CURVE_NAME, "headline_point": HEADLINE,
                  "context": [W.WORKLOADS[n].prefix[0] for n in SWEEP]})
    else:
        c = workload_config(W.WORKLOADS[name])
    c.update(common)
    return c


def _bits(t):
    """bf16 tensor -> numpy uint16 bit patterns (the oracle's input form)."""
    import torch
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


def oracle_call(inp):
    """The fp64 oracle over one whole call's inputs (all requests)."""
    import oracle
    idx, ptr = inp["idx"], inp["ptr"]
    return oracle.mla_verify(inp["q"], inp["cache"], idx, ptr, inp["lens"], inp["par"], inp["scale"],
                             inp["ps"])


def oracle_inputs(inp):
    return {"q": _bits(inp.q), "cache": _bits(inp.kv_cache), "idx": inp.kv_indices.cpu().numpy(),
            "ptr": inp.kv_indptr.cpu().numpy(), "lens": inp.kv_lens.cpu().numpy(),
            "par": inp.draft_parent.cpu().numpy(), "scale": inp.scale, "ps": inp.page_size}


def oracle_seconds_per_call(inp, budget_s):
    """CPU oracle on whole calls of the same inputs until the budget is spent
    (at least one call).  Returns (seconds per call, calls run)."""
    oi = oracle_inputs(inp)
    done, t0 = 0, time.perf_counter()
    while True:
        oracle_call(oi)
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return el / done, done


def run_reference(args):
    """The reference arm: the fp64 oracle on this machine's host cores, timed
    per whole call on the workload the GPU arm's `value` is quoted on."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from paged_mla_speculative_gb300 import workloads as W
    name = HEADLINE if args.workload == CURVE_NAME else args.workload
    w = W.WORKLOADS[name]
    oi = oracle_inputs(W.make_inputs(w, device="cpu"))
    budget = 150.0                       # wall seconds for warm-up + steps
    t_start = time.perf_counter()
    for _ in range(args.warmup):
        oracle_call(oi)
        if time.perf_counter() - t_start > budget / 3:
            break
    times = []
    for _ in range(args.steps):
        s0 = time.perf_counter()
        oracle_call(oi)
        times.append(time.perf_counter() - s0)
        if time.perf_counter() - t_start > budget:
            break
    us_per_call = statistics.fmean(times) * 1e6
    cores = len(os.sched_getaffinity(0))
    line = {
        "impl": "reference", "metric": METRIC, "value": us_per_call,
        "unit": "us/call", "n_gpus": ws, "steps": args.steps, "steps_run": len(times),
        "warmup": args.warmup, "ms_per_step": us_per_call / 1e3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded), generated on the host",
        "config": config_of(args.workload),
        "cpu_baseline": {"value": us_per_call, "unit": "us/call", "cores": cores, "kind": "oracle",
                         "sample": f"whole calls of {name} (fp64 NumPy, gather + masked softmax + "
                                   f"weighted sum), {len(times)} timed"},
        "e2e": {"value": us_per_call, "unit": "us/call", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


KERNEL_IDS = {"auto": 0, "mma": 1, "tc": 2, "pair": 3}   # MLA_VERIFY_KERNEL_*


def measure_workload(mb, W, name, flush, steps, clocks=None, kernel="auto", nsplit=0, pack=None):
    """µs per call of one workload: `steps` CUDA-graph replays (the capture-
    safe production path), each after an L2 flush, bracketed by events on the
    replay stream; then eager calls, and eager calls with the library's
    events between its kernels (pack / partial / combine split)."""
    import torch
    w = W.WORKLOADS[name]
    inp = W.make_inputs(w, device="cuda")
    work = W.algorithmic_work(inp.prefix, w.num_drafts, w.num_heads)
    plan = mb.Plan(w.batch, w.num_drafts, w.num_heads, w.page_size, w.num_slots,
                   max(inp.kv_lens.tolist()))
    plan.set_kernel(KERNEL_IDS[kernel])
    if nsplit:
        plan.set_nsplit(nsplit)
    if pack is not None:
        plan.set_pack_schedule(pack)
    ns = plan.nsplit(w.batch)
    out, lse = plan.new_outputs(w.batch)
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())

    def call():
        mb.mla_verify_attn(plan, inp.q, inp.kv_cache, inp.kv_indices, inp.kv_indptr,
                           inp.kv_lens, inp.draft_parent, inp.scale, out, lse, stream=st)

    with torch.cuda.stream(st):
        for _ in range(3):
            flush.zero_()
            call()
    st.synchronize()
    err = plan.get_error()
    assert err == 0, f"{name}: device error word {err:#x} set during warm-up"
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        call()

    def timed(n, fn, events=False):
        ea = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        eb = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        pk = [torch.cuda.Event(enable_timing=True) for _ in range(n)] if events else None
        pm = [torch.cuda.Event(enable_timing=True) for _ in range(n)] if events else None
        if events:
            for e in pk + pm:
                e.record(st)
            st.synchronize()
        with torch.cuda.stream(st):
            for i in range(n):
                flush.zero_()
                if events:
                    plan.set_profile_events(pk[i], pm[i])
                ea[i].record(st)
                fn()
                eb[i].record(st)
        st.synchronize()
        if events:
            plan.set_profile_events(None, None)
            return ([a.elapsed_time(k) for a, k in zip(ea, pk)],
                    [k.elapsed_time(m) for k, m in zip(pk, pm)],
                    [m.elapsed_time(b) for m, b in zip(pm, eb)],
                    [a.elapsed_time(b) for a, b in zip(ea, eb)])
        return [a.elapsed_time(b) for a, b in zip(ea, eb)]

    t0 = time.perf_counter()
    if clocks is not None:
        with clocks:
            graph_ms = timed(steps, g.replay)
    else:
        graph_ms = timed(steps, g.replay)
    wall = time.perf_counter() - t0
    k2 = min(steps, 100)
    eager_ms = timed(k2, call)
    pack_ms, part_ms, comb_ms, ser_ms = timed(k2, call, events=True)
    err = plan.get_error()
    assert err == 0, f"{name}: device error word {err:#x} set while timing"
    peaks, peak_src = load_peaks()
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    tc = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    us = statistics.fmean(graph_ms) * 1e3
    q = statistics.quantiles(graph_ms, n=10) if len(graph_ms) >= 10 else [min(graph_ms), max(graph_ms)]
    t_hbm, t_tc = work["bytes"] / (hbm * 1e9), work["flops"] / (tc * 1e12)
    t_roof = max(t_hbm, t_tc) * 1e6
    part_us = statistics.fmean(part_ms) * 1e3
    sched = PACK_NAMES[plan.pack_mode(w.batch)]
    kv_gbs = work["kv_bytes"] / (us * 1e-6) / 1e9
    res = {
        "us_per_call": us, "us_p10_p50_p90": [q[0] * 1e3, statistics.median(graph_ms) * 1e3, q[-1] * 1e3],
        "eager_us_per_call": statistics.fmean(eager_ms) * 1e3,
        "kv_gbs": kv_gbs, "kv_frac_of_hbm": kv_gbs / hbm,
        "roofline_time_us": t_roof, "frac_of_roofline": t_roof / us,
        "bound": "hbm" if t_hbm > t_tc else "tensor",
        "pack_us": statistics.fmean(pack_ms) * 1e3, "partial_us": part_us,
        "combine_us": statistics.fmean(comb_ms) * 1e3,
        "serialised_us_per_call": statistics.fmean(ser_ms) * 1e3,
        "partial_tflops": work["flops"] / (part_us * 1e-6) / 1e12,
        "partial_frac_of_tensor_peak": work["flops"] / (part_us * 1e-6) / 1e12 / tc,
        "keys": work["keys"], "kv_bytes": work["kv_bytes"], "flops": work["flops"],
        "nsplit": ns, "pack_schedule": sched, "kernels": kernels_of(plan.call_kernel(w.batch), ns, sched),
        "partial_kernel": PARTIAL_NAMES[plan.call_kernel(w.batch)],
        "calls_timed": len(graph_ms),
    }
    state = {"inp": inp, "plan": plan, "out": out, "lse": lse, "work": work, "wall": wall,
             "peak_src": peak_src, "tc_peak": tc, "stream": st}
    return res, state


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

    head = HEADLINE if args.workload == CURVE_NAME else args.workload
    others = ([n for n in SWEEP + OTHERS if n != head] if args.workload == CURVE_NAME else [])
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        pass
    K = args.steps
    for _ in range(max(args.warmup, 3)):
        flush.zero_()
    barrier(ws)
    torch.cuda.synchronize()
    clk = ClockSampler(uuid)
    res, st = measure_workload(mb, W, head, flush, K, clocks=clk, kernel=args.kernel)
    barrier(ws)
    plan, inp, out, work = st["plan"], st["inp"], st["out"], st["work"]
    w = W.WORKLOADS[head]
    mean_call_ms = max_over_ranks(ws, res["us_per_call"] / 1e3)
    mean_part_ms = max_over_ranks(ws, res["partial_us"] / 1e3)
    us_per_call = mean_call_ms * 1e3 / ws          # whole job: ws replicas in parallel

    # End to end through the host-buffer entry point: H2D of the step's
    # inputs from pinned memory, the call, D2H of out/lse, stream sync.
    hq = inp.q.cpu().pin_memory()
    hidx = inp.kv_indices.cpu().pin_memory()
    hptr = inp.kv_indptr.cpu().pin_memory()
    hlen = inp.kv_lens.cpu().pin_memory()
    hpar = inp.draft_parent.cpu().pin_memory()
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    hlse = torch.empty(st["lse"].shape, dtype=torch.float32).pin_memory()
    stream = st["stream"]
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
    launches = K * len(res["kernels"].split(" + "))

    extra = {}
    if head == "decode_batch" or args.workload == CURVE_NAME:
        # NEXT rows measured on the decode-batch step: the per-step index
        # builder and KV compaction of its requests.
        db_inp = inp if head == "decode_batch" else W.make_inputs(W.WORKLOADS["decode_batch"], device="cuda")
        dbw = W.WORKLOADS["decode_batch"]
        db_plan = plan if head == "decode_batch" else mb.Plan(
            dbw.batch, dbw.num_drafts, dbw.num_heads, dbw.page_size, dbw.num_slots,
            max(db_inp.kv_lens.tolist()))
        cur = torch.cuda.current_stream()     # the flush and the timed call share a stream
        extra["index_builder"] = index_builder_timing(mb, db_plan, db_inp, dbw, flush, cur, min(K, 300))
        extra["compaction"] = compaction_timing(mb, db_plan, db_inp, dbw, flush, cur, min(K, 200))
        if db_plan is not plan:
            db_plan.close()
        del db_inp

    tc_peak = st["tc_peak"]
    achieved = work["flops"] / (mean_part_ms * 1e-3) / 1e12
    # When the planner gave up SMs to run the pack beside the attention
    # kernel (fewer splits), the same kernel on the whole grid -- the split
    # count that fills every SM, the pack first -- for its own fraction of
    # the peak.  The headline value stays the planner's call.
    full_grid = None
    if res["pack_schedule"] == "idle_sms" and res["partial_kernel"] == "partial_pair_kernel":
        wl = W.WORKLOADS[head]
        units = wl.batch * -(-wl.num_drafts * wl.num_heads // 128)
        ns_full = (torch.cuda.get_device_properties(0).multi_processor_count // 2) // units
        if ns_full > res["nsplit"]:
            rf, sf = measure_workload(mb, W, head, flush, min(args.other_steps, K), kernel=args.kernel,
                                      nsplit=ns_full, pack=mb.PACK_WHOLE)
            sf["plan"].close()
            del sf
            a_full = work["flops"] / (rf["partial_us"] * 1e-6) / 1e12
            full_grid = {"nsplit": rf["nsplit"], "pack_schedule": rf["pack_schedule"],
                         "us_per_call": rf["us_per_call"], "partial_us": rf["partial_us"],
                         "achieved": a_full, "peak": tc_peak, "unit": "TFLOP/s", "frac": a_full / tc_peak}
    line = {
        "metric": METRIC, "value": us_per_call, "unit": "us/call",
        "n_gpus": ws, "steps": K, "warmup": args.warmup, "ms_per_step": mean_call_ms,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16", "data": "synthetic (seeded), bf16 inputs resident in HBM",
        "config": config_of(args.workload),
        "headline": {"workload": head, **{k: res[k] for k in (
            "kv_gbs", "kv_frac_of_hbm", "roofline_time_us", "frac_of_roofline", "bound", "nsplit",
            "pack_schedule", "kernels", "us_p10_p50_p90", "eager_us_per_call", "pack_us",
            "partial_us", "combine_us")}},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s",
                     "frac": achieved / tc_peak, "traffic": profiled_traffic(head, res["partial_kernel"]),
                     "kernel": res["partial_kernel"], "workload": head,
                     "peak_source": f"{st['peak_src']} bf16 burst (fp16 has the same tensor rate)"},
        "roofline_full_grid": full_grid,
        "clocks": clk.summary(), "gpu_launches": launches,
        "e2e": {"value": e2e_us, "unit": "us/call", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "timed_wall_s": st["wall"],
    }
    line.update(extra)
    cpu_inp = inp if (ws == 1 and rank == 0 and not args.no_cpu_baseline) else None
    plan.close()
    del st, out
    torch.cuda.empty_cache()

    # The rest of the curve and every other workload, same protocol.
    if others:
        curve = {head: {**res}}
        for n in others:
            r, s2 = measure_workload(mb, W, n, flush, min(args.other_steps, K), kernel=args.kernel)
            s2["plan"].close()
            del s2
            torch.cuda.empty_cache()
            curve[n] = r
        line["workloads"] = {n: curve[n] for n in SWEEP + OTHERS if n in curve}
        line["curve"] = [{"context": W.WORKLOADS[n].prefix[0], "us_per_call": curve[n]["us_per_call"],
                          "kv_gbs": curve[n]["kv_gbs"], "frac_of_roofline": curve[n]["frac_of_roofline"],
                          "partial_frac_of_tensor_peak": curve[n]["partial_frac_of_tensor_peak"]}
                         for n in SWEEP]
    if cpu_inp is not None:
        sec, ncalls = oracle_seconds_per_call(cpu_inp, args.cpu_seconds)
        line["cpu_baseline"] = {"value": sec * 1e6, "unit": "us/call",
                                "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
                                "sample": f"{ncalls} whole calls of {head} (fp64 NumPy, same inputs)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_calls_only(args):
    """Issue --steps calls of one workload and check the device word: no
    timing, no extra passes (a short, fixed launch sequence to profile)."""
    import torch
    from paged_mla_speculative_gb300 import binding as mb
    from paged_mla_speculative_gb300 import build as mbuild
    from paged_mla_speculative_gb300 import workloads as W
    mbuild.build()
    name = HEADLINE if args.workload == CURVE_NAME else args.workload
    w = W.WORKLOADS[name]
    inp = W.make_inputs(w, device="cuda")
    plan = mb.Plan(w.batch, w.num_drafts, w.num_heads, w.page_size, w.num_slots, max(inp.kv_lens.tolist()))
    plan.set_kernel(KERNEL_IDS[args.kernel])
    plan.set_pack_schedule({"auto": mb.PACK_AUTO, "whole": mb.PACK_WHOLE, "idle_sms": mb.PACK_IDLE_SMS,
                            "none": mb.PACK_NONE}[args.pack_schedule])
    stream = torch.cuda.current_stream()
    for _ in range(args.steps):
        if args.calls_only == "attn":
            mb.mla_verify_attn(plan, inp.q, inp.kv_cache, inp.kv_indices, inp.kv_indptr, inp.kv_lens,
                               inp.draft_parent, inp.scale)
        elif args.calls_only == "index":
            index_builder_timing(mb, plan, inp, w, torch.empty(1 << 20, dtype=torch.uint8, device="cuda"),
                                 stream, 1)
        else:
            compaction_timing(mb, plan, inp, w, torch.empty(1 << 20, dtype=torch.uint8, device="cuda"),
                              stream, 1)
    torch.cuda.synchronize()
    assert plan.get_error() == 0
    print(json.dumps({"calls_only": args.calls_only, "workload": name, "calls": args.steps,
                      "nsplit": plan.nsplit(w.batch), "pack_schedule": PACK_NAMES[plan.pack_mode(w.batch)]}))
    plan.close()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.calls_only:
        return run_calls_only(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_gb300(args)


if __name__ == "__main__":
    sys.exit(main())
