"""The whole call records into a CUDA graph and replays with new data.

Static buffers are captured once; between replays the metadata (kv_lens,
indices, parents), q and the cache change, so a replay that baked any device
value into the graph would give the wrong answer.  Every replay must equal
an eager call on the same buffers bit for bit, and match the oracle.  Each
key-pack schedule (pack overlapping the attention kernel on idle SMs, whole
pack first, attention CTAs gathering directly -- automatic with one row tile,
forced with several), page size 64, bf16 output, the CTA-pair and mma.sync
families and full-size workloads are captured.
"""
import dataclasses

import pytest
import torch

from paged_mla_speculative_gb300 import binding as mb
from paged_mla_speculative_gb300 import workloads as W
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_mla_speculative_gb300 import build
    build.build()


def _inputs(seed, prefix, tree, T, H, ps):
    w = W.Workload(name="cap", batch=3, num_drafts=T, num_heads=H, prefix=prefix, tree=tree,
                   num_slots=8192, page_size=ps, spike_frac=0.01, seed=seed)
    return W.make_inputs(w)


# name: (T, H, page_size, out dtype, kernel, nsplit, forced pack schedule, expected mode)
CASES = {
    "idle_sms": (8, 16, 1, torch.float32, mb.KERNEL_TC, 4, mb.PACK_IDLE_SMS, mb.PACK_IDLE_SMS),
    "idle_sms_ps64_bf16": (8, 16, 64, torch.bfloat16, mb.KERNEL_TC, 4, mb.PACK_IDLE_SMS, mb.PACK_IDLE_SMS),
    "idle_sms_one_split": (8, 16, 1, torch.float32, mb.KERNEL_TC, 1, mb.PACK_IDLE_SMS, mb.PACK_IDLE_SMS),
    "whole": (8, 64, 1, torch.float32, mb.KERNEL_TC, 6, mb.PACK_WHOLE, mb.PACK_WHOLE),
    "whole_ps64_bf16": (8, 64, 64, torch.bfloat16, mb.KERNEL_TC, 6, mb.PACK_WHOLE, mb.PACK_WHOLE),
    "forced_no_pack": (8, 64, 1, torch.float32, mb.KERNEL_TC, 3, mb.PACK_NONE, mb.PACK_NONE),
    "auto": (8, 32, 1, torch.float32, mb.KERNEL_TC, 0, mb.PACK_AUTO, None),
    "direct": (4, 16, 1, torch.float32, mb.KERNEL_TC, 4, mb.PACK_AUTO, mb.PACK_NONE),
    "direct_ps64_bf16": (4, 16, 64, torch.bfloat16, mb.KERNEL_TC, 3, mb.PACK_AUTO, mb.PACK_NONE),
    "direct_one_split": (4, 16, 1, torch.float32, mb.KERNEL_TC, 1, mb.PACK_AUTO, mb.PACK_NONE),
    "mma": (8, 16, 1, torch.float32, mb.KERNEL_MMA, 3, mb.PACK_AUTO, mb.PACK_NONE),
    "pair_idle_sms": (8, 16, 1, torch.float32, mb.KERNEL_PAIR, 4, mb.PACK_IDLE_SMS, mb.PACK_IDLE_SMS),
    "pair_whole_ps64_bf16": (8, 64, 64, torch.bfloat16, mb.KERNEL_PAIR, 6, mb.PACK_WHOLE, mb.PACK_WHOLE),
    "pair_auto": (8, 32, 1, torch.float32, mb.KERNEL_AUTO, 0, mb.PACK_AUTO, None),
}


@pytest.mark.parametrize("case", list(CASES))
def test_graph_replay_with_changing_metadata(case):
    T, H, ps, odt, kernel, nsplit, forced, expect = CASES[case]
    cases = [_inputs(1, (1000, 300, 20), "chain", T, H, ps),
             _inputs(2, (64, 1500, 999), "random", T, H, ps),
             _inputs(3, (0, 7, 1800), "star", T, H, ps)]
    max_idx = max(c.kv_indices.numel() for c in cases)
    dev = torch.device("cuda")
    q = torch.empty_like(cases[0].q, device=dev)
    cache = torch.empty_like(cases[0].kv_cache, device=dev)
    idx = torch.zeros(max_idx, dtype=torch.int32, device=dev)
    indptr = torch.empty(4, dtype=torch.int32, device=dev)
    lens = torch.empty(3, dtype=torch.int32, device=dev)
    par = torch.empty((3, T), dtype=torch.int32, device=dev)

    def load(c):
        q.copy_(c.q)
        cache.copy_(c.kv_cache)
        idx[:c.kv_indices.numel()].copy_(c.kv_indices)
        indptr.copy_(c.kv_indptr)
        lens.copy_(c.kv_lens)
        par.copy_(c.draft_parent)

    plan = mb.Plan(3, T, H, ps, 8192, 2000, odt)
    plan.set_kernel(kernel)
    plan.set_nsplit(nsplit)
    plan.set_pack_schedule(forced)
    if expect is not None:
        assert plan.pack_mode(3) == expect, (case, plan.pack_mode(3))
    out, lse = plan.new_outputs(3)
    s = torch.cuda.Stream()
    load(cases[0])
    torch.cuda.synchronize()
    with torch.cuda.stream(s):   # warm-up outside capture
        mb.mla_verify_attn(plan, q, cache, idx, indptr, lens, par, cases[0].scale, out, lse, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        mb.mla_verify_attn(plan, q, cache, idx, indptr, lens, par, cases[0].scale, out, lse, stream=s)
    for c in cases + cases[::-1]:
        load(c)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        go, gl = out.clone(), lse.clone()
        eo, el = mb.mla_verify_attn(plan, q, cache, idx, indptr, lens, par, c.scale)
        torch.cuda.synchronize()
        assert torch.equal(go, eo) and torch.equal(gl, el)
        ref_o, ref_l = G.oracle_full(c)
        if odt == torch.float32:
            G.assert_parity(go.cpu().numpy(), gl.cpu().numpy(), ref_o, ref_l, case)
        else:
            G.assert_bf16_parity(go.cpu(), gl.cpu().numpy(), ref_o, ref_l, case)
    assert plan.get_error() == 0
    plan.close()


@pytest.mark.parametrize("name", ["decode_batch", "sweep_p65536", "decode_tp8", "decode_t1"])
def test_full_size_graph_replay(name):
    """A full-size workload captured in its benchmark configuration: two
    replays with different q, each bit-identical to an eager call."""
    w = W.WORKLOADS[name]
    inp = W.make_inputs(w, device="cuda")
    with G.make_plan(inp) as plan:
        out, lse = plan.new_outputs(w.batch)
        q = inp.q.clone()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())

        def call(st):
            mb.mla_verify_attn(plan, q, inp.kv_cache, inp.kv_indices, inp.kv_indptr, inp.kv_lens,
                               inp.draft_parent, inp.scale, out, lse, stream=st)

        with torch.cuda.stream(s):
            call(s)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            call(s)
        gen = torch.Generator(device="cuda").manual_seed(5)
        for i in range(2):
            if i:
                q.copy_(torch.randn(q.shape, generator=gen, device="cuda").to(torch.bfloat16))
            g.replay()
            torch.cuda.synchronize()
            go, gl = out.clone(), lse.clone()
            call(torch.cuda.current_stream())
            torch.cuda.synchronize()
            assert torch.equal(go, out) and torch.equal(gl, lse), name
        assert plan.get_error() == 0
        assert torch.isfinite(out).all()
