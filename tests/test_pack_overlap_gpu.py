"""The key pack overlapping the attention kernel, and the whole-pack schedule.

When the attention grid leaves SMs idle, the pack keeps running on them while
the attention kernel streams each 128-key block as soon as its ready flags
carry the call's tag; otherwise the whole pack runs first.  Both schedules
must give the oracle's answer, and the flags must not let a call read a
block packed by an earlier call (repeated calls and graph replays with new
data in the same buffers).
"""
import numpy as np
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


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _attention_ctas(plan, batch, rows):
    if plan.call_kernel(batch) == mb.KERNEL_PAIR:
        return plan.nsplit(batch) * ((rows + 127) // 128) * batch * 2
    return plan.nsplit(batch) * ((rows + 63) // 64) * batch


def _positions(plan, batch, blocks):
    """Block positions per split: one per 128-key block, or two per pair
    block when the splits take pairs of blocks."""
    ns = plan.nsplit(batch)
    if plan.call_kernel(batch) == mb.KERNEL_PAIR:
        return 2 * (-(-(-(-blocks // 2)) // ns))
    return -(-blocks // ns)


@pytest.mark.parametrize("kernel", [pytest.param(mb.KERNEL_TC, id="tc"), pytest.param(mb.KERNEL_PAIR, id="pair")])
def test_decode_batch_shape_schedule(kernel):
    """8 requests x 512 rows x 4104 keys.  The pack either runs whole first
    (stay 0, every position wide) or keeps the SMs the attention grid leaves
    idle and packs only the leading positions first.  The single-SM family
    leaves enough SMs idle for the second; the pair family's split steps
    take two blocks each, and the planner runs the whole pack first."""
    plan = mb.Plan(8, 8, 64, 1, 65536, 4104)
    plan.set_kernel(kernel)
    assert plan.call_kernel(8) == kernel
    wide, stay = plan.pack_schedule(8)
    idle = _sms() - _attention_ctas(plan, 8, 512)
    positions = _positions(plan, 8, 33)
    if stay == 0:
        assert wide == positions
    else:
        assert stay == idle and idle >= 16
        assert 1 <= wide and 2 * wide <= positions
    if kernel == mb.KERNEL_TC and idle >= 16:
        assert stay == idle
    plan.set_kernel(mb.KERNEL_MMA)
    assert plan.pack_schedule(8) == (0, 0)
    plan.close()


@pytest.mark.parametrize("kernel", [pytest.param(mb.KERNEL_TC, id="tc"), pytest.param(mb.KERNEL_PAIR, id="pair")])
def test_overlapping_pack_repeated_calls(kernel):
    w = W.Workload(name="ov", batch=4, num_drafts=8, num_heads=64, prefix=(1500, 900, 2000, 33),
                   tree="random", num_slots=8192, spike_frac=0.01, seed=610)
    inp = W.make_inputs(w)
    g = G.to_cuda(inp)
    with G.make_plan(g, kernel=kernel) as plan:
        plan.set_pack_schedule(mb.PACK_IDLE_SMS)
        wide, stay = plan.pack_schedule(4)
        assert stay > 0, (wide, stay)
        first = None
        for _ in range(4):
            out, lse = G.run(plan, g)
            assert plan.get_error() == 0
            if first is None:
                first = (out.clone(), lse.clone())
            else:
                assert torch.equal(out, first[0]) and torch.equal(lse, first[1])
    ref_o, ref_l = G.oracle_full(inp)
    G.assert_parity(first[0].cpu().numpy(), first[1].cpu().numpy(), ref_o, ref_l)


@pytest.mark.parametrize("kernel", [pytest.param(mb.KERNEL_TC, id="tc"), pytest.param(mb.KERNEL_PAIR, id="pair")])
def test_overlapping_pack_new_data_each_call(kernel):
    """Same buffers, different keys and lengths every call: a block packed by
    the previous call must never be read as this call's."""
    cases = [W.make_inputs(W.Workload(name="ovd", batch=3, num_drafts=4, num_heads=32,
                                      prefix=pre, tree="random", num_slots=8192,
                                      spike_frac=0.01, seed=620 + i))
             for i, pre in enumerate([(1800, 700, 1200), (300, 1900, 64), (1000, 1000, 1000)])]
    dev = torch.device("cuda")
    q = torch.empty_like(cases[0].q, device=dev)
    cache = torch.empty_like(cases[0].kv_cache, device=dev)
    idx = torch.zeros(max(c.kv_indices.numel() for c in cases), dtype=torch.int32, device=dev)
    indptr = torch.empty(4, dtype=torch.int32, device=dev)
    lens = torch.empty(3, dtype=torch.int32, device=dev)
    par = torch.empty((3, 4), dtype=torch.int32, device=dev)
    plan = mb.Plan(3, 4, 32, 1, 8192, 1904)
    plan.set_kernel(kernel)
    plan.set_nsplit(2)
    plan.set_pack_schedule(mb.PACK_IDLE_SMS)
    assert plan.pack_schedule(3)[1] > 0
    for c in cases + cases[::-1]:
        q.copy_(c.q)
        cache.copy_(c.kv_cache)
        idx[:c.kv_indices.numel()].copy_(c.kv_indices)
        indptr.copy_(c.kv_indptr)
        lens.copy_(c.kv_lens)
        par.copy_(c.draft_parent)
        out, lse = mb.mla_verify_attn(plan, q, cache, idx, indptr, lens, par, c.scale)
        torch.cuda.synchronize()
        ref_o, ref_l = G.oracle_full(c)
        G.assert_parity(out.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l)
    assert plan.get_error() == 0
    plan.close()


@pytest.mark.parametrize("kernel", [pytest.param(mb.KERNEL_TC, id="tc"), pytest.param(mb.KERNEL_PAIR, id="pair")])
def test_hand_off_tags_past_2_32(kernel):
    """The pack's ready flags carry 64-bit tags.  A first call packs long
    requests (its flags hold tag 1); the epoch is then moved to 2^32 - 3
    (MLA_VERIFY_FAULT_EPOCH_NEAR_WRAP), short calls take the tags across
    2^32, and long calls with new data follow.  With 32-bit tags the epoch
    would wrap and a later call would reuse tag 1, finding the first call's
    flags on blocks it has not packed yet."""
    def make(pre, seed):
        return W.make_inputs(W.Workload(name="tag", batch=3, num_drafts=4, num_heads=32, prefix=pre,
                                        tree="random", num_slots=8192, spike_frac=0.01, seed=seed))
    long_a, long_b = make((1800, 1900, 1500), 640), make((1700, 1890, 1600), 641)
    short = make((64, 100, 33), 642)
    dev = torch.device("cuda")
    q = torch.empty_like(long_a.q, device=dev)
    cache = torch.empty_like(long_a.kv_cache, device=dev)
    idx = torch.zeros(max(c.kv_indices.numel() for c in (long_a, long_b, short)), dtype=torch.int32, device=dev)
    indptr = torch.empty(4, dtype=torch.int32, device=dev)
    lens = torch.empty(3, dtype=torch.int32, device=dev)
    par = torch.empty((3, 4), dtype=torch.int32, device=dev)
    with mb.Plan(3, 4, 32, 1, 8192, 1904) as plan:
        plan.set_kernel(kernel)
        plan.set_nsplit(2)
        plan.set_pack_schedule(mb.PACK_IDLE_SMS)
        for i, c in enumerate([long_a, short, short, long_b, long_a, long_b]):
            if i == 1:
                plan.inject_fault(mb.FAULT_EPOCH_NEAR_WRAP)
            q.copy_(c.q)
            cache.copy_(c.kv_cache)
            idx[:c.kv_indices.numel()].copy_(c.kv_indices)
            indptr.copy_(c.kv_indptr)
            lens.copy_(c.kv_lens)
            par.copy_(c.draft_parent)
            out, lse = mb.mla_verify_attn(plan, q, cache, idx, indptr, lens, par, c.scale)
            torch.cuda.synchronize()
            ref_o, ref_l = G.oracle_full(c)
            G.assert_parity(out.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l)
        assert plan.get_error() == 0


@pytest.mark.parametrize("kernel", [pytest.param(mb.KERNEL_TC, id="tc"), pytest.param(mb.KERNEL_PAIR, id="pair")])
def test_two_plans_on_two_streams_at_once(kernel):
    """Two plans, each with its own pack hand-off, issue calls on two streams
    with no synchronisation between them, so their pack and attention kernels
    share the GPU.  A call's attention kernel becomes launchable only once
    every CTA of its own pack kernel has started (each triggers the dependent
    launch at its entry), so its flag waits never depend on CTAs that cannot
    get an SM.  Every output must be the oracle's."""
    cases = [W.make_inputs(W.Workload(name=f"two{i}", batch=2, num_drafts=8, num_heads=32, prefix=pre,
                                      tree="random", num_slots=16384, spike_frac=0.01, seed=660 + i))
             for i, pre in enumerate([(3000, 2100), (2600, 3100)])]
    gpu = [G.to_cuda(c) for c in cases]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    plans = []
    for c in cases:
        pl = mb.Plan(2, 8, 32, 1, 16384, max(int(x) for x in c.kv_lens))
        pl.set_kernel(kernel)
        pl.set_nsplit(3)
        pl.set_pack_schedule(mb.PACK_IDLE_SMS)
        plans.append(pl)
    torch.cuda.synchronize()
    results = []
    for rep in range(4):
        for i in (0, 1):
            g = gpu[i]
            with torch.cuda.stream(streams[i]):
                out, lse = mb.mla_verify_attn(plans[i], g.q, g.kv_cache, g.kv_indices, g.kv_indptr, g.kv_lens,
                                              g.draft_parent, g.scale, stream=streams[i])
            results.append((i, out, lse))
    torch.cuda.synchronize()
    refs = [G.oracle_full(c) for c in cases]
    for i, out, lse in results:
        G.assert_parity(out.cpu().numpy(), lse.cpu().numpy(), refs[i][0], refs[i][1])
    for pl in plans:
        assert pl.get_error() == 0
        pl.close()


def test_whole_pack_when_no_sm_is_idle():
    """As many attention CTAs as SMs: the whole pack runs first."""
    tiles = 8                                   # 512 rows
    batch = max(1, _sms() // tiles)
    w = W.Workload(name="whole", batch=batch, num_drafts=8, num_heads=64, prefix=(120,) * batch,
                   tree="chain", num_slots=8192, spike_frac=0.01, seed=630)
    inp = W.make_inputs(w)
    g = G.to_cuda(inp)
    with G.make_plan(g, nsplit=1) as plan:
        wide, stay = plan.pack_schedule(batch)
        if _sms() - _attention_ctas(plan, batch, 512) < 16:
            assert stay == 0 and wide == _positions(plan, batch, 1)
        out, lse = G.run(plan, g)
        assert plan.get_error() == 0
    ref_o, ref_l = G.oracle_full(inp)
    G.assert_parity(out.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l)


def test_profiling_events_use_the_whole_pack():
    """With profiling events between the kernels the same overlapping-shape
    call runs the kernels back to back; results are bit-identical."""
    w = W.Workload(name="ev", batch=4, num_drafts=8, num_heads=64, prefix=(1500, 900, 2000, 33),
                   tree="random", num_slots=8192, spike_frac=0.01, seed=610)
    g = G.to_cuda(W.make_inputs(w))
    with G.make_plan(g) as plan:
        o1, l1 = G.run(plan, g)
        o1, l1 = o1.clone(), l1.clone()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        plan.set_profile_events(e0, e1)
        o2, l2 = G.run(plan, g)
        assert plan.get_error() == 0
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("page_size,out_dtype", [(64, torch.float32), (1, torch.bfloat16),
                                                 (64, torch.bfloat16)])
@pytest.mark.parametrize("kernel", [pytest.param(mb.KERNEL_TC, id="tc"), pytest.param(mb.KERNEL_PAIR, id="pair")])
def test_overlapping_pack_pages_and_bf16(page_size, out_dtype, kernel):
    """The overlapping schedule with a 64-row page table and with bf16 output
    (bf16 must equal the fp32 result rounded)."""
    w = W.Workload(name="ovp", batch=4, num_drafts=8, num_heads=64, prefix=(1500, 900, 2000, 33),
                   tree="random", num_slots=16384, page_size=page_size, spike_frac=0.01, seed=640)
    inp = W.make_inputs(w)
    g = G.to_cuda(inp)
    with G.make_plan(g, out_dtype=out_dtype, kernel=kernel) as plan:
        plan.set_pack_schedule(mb.PACK_IDLE_SMS)
        assert plan.pack_schedule(4)[1] > 0
        out, lse = G.run(plan, g)
        assert plan.get_error() == 0
    with G.make_plan(g, kernel=kernel) as plan32:
        plan32.set_pack_schedule(mb.PACK_IDLE_SMS)
        o32, l32 = G.run(plan32, g)
    if out_dtype == torch.bfloat16:
        assert torch.equal(out, o32.to(torch.bfloat16)) and torch.equal(lse, l32)
    ref_o, ref_l = G.oracle_full(inp)
    G.assert_parity(o32.cpu().numpy(), l32.cpu().numpy(), ref_o, ref_l)


def test_schedules_alternate_on_one_plan():
    """Calls on one plan switch between the whole pack (a full attention grid)
    and the overlapping pack (few requests); every call must still read only
    blocks packed in that call."""
    tiles = 8                                   # 512 rows
    big = max(1, _sms() // tiles)
    wbig = W.Workload(name="alt_big", batch=big, num_drafts=8, num_heads=64,
                      prefix=tuple(100 + 37 * i for i in range(big)), tree="random",
                      num_slots=16384, spike_frac=0.01, seed=650)
    wsmall = W.Workload(name="alt_small", batch=3, num_drafts=8, num_heads=64,
                        prefix=(1400, 700, 1800), tree="random", num_slots=16384,
                        spike_frac=0.01, seed=651)
    ibig, ismall = W.make_inputs(wbig), W.make_inputs(wsmall)
    gbig, gsmall = G.to_cuda(ibig), G.to_cuda(ismall)
    plan = mb.Plan(big, 8, 64, 1, 16384, 1808)
    plan.set_nsplit(1)
    sched = {big: plan.pack_schedule(big), 3: plan.pack_schedule(3)}
    if _sms() - big * tiles < 16:
        assert sched[big][1] == 0
    refs = {}
    for i in range(6):
        g, inp = (gbig, ibig) if i % 2 == 0 else (gsmall, ismall)
        out, lse = mb.mla_verify_attn(plan, g.q, g.kv_cache, g.kv_indices, g.kv_indptr, g.kv_lens,
                                      g.draft_parent, g.scale)
        torch.cuda.synchronize()
        key = inp.workload.name
        if key not in refs:
            refs[key] = G.oracle_full(inp)
            G.assert_parity(out.cpu().numpy(), lse.cpu().numpy(), *refs[key])
            refs[key + "_out"] = (out.clone(), lse.clone())
        else:
            assert torch.equal(out, refs[key + "_out"][0]) and torch.equal(lse, refs[key + "_out"][1])
    assert plan.get_error() == 0
    plan.close()


@pytest.mark.parametrize("nsplit", [1, 3])
def test_one_row_tile_gathers_directly(nsplit):
    """T*H <= 64: no pack; every attention CTA gathers its own key blocks.
    Ragged lengths (a request shorter than one block, one ending mid-block),
    repeated calls bit-identical, parity with the oracle."""
    w = W.Workload(name="direct", batch=3, num_drafts=4, num_heads=16, prefix=(900, 129, 0),
                   tree="random", num_slots=4096, spike_frac=0.01, seed=700)
    inp = W.make_inputs(w)
    g = G.to_cuda(inp)
    with G.make_plan(g, nsplit=nsplit) as plan:
        assert plan.pack_schedule(3) == (0, 0)
        o1, l1 = G.run(plan, g)
        o1, l1 = o1.clone(), l1.clone()
        o2, l2 = G.run(plan, g)
        assert plan.get_error() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    ref_o, ref_l = G.oracle_full(inp)
    G.assert_parity(o1.cpu().numpy(), l1.cpu().numpy(), ref_o, ref_l)
