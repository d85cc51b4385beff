"""Error behaviour: host-visible problems return a status; problems only
visible in device data set the sticky device word and never fault.

Every bad index here is caught by the kernels' own range checks before any
memory access (the key is masked or the request is written as NaN)."""
import ctypes
import dataclasses

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


def _case(seed=1, **kw):
    base = dict(name="e", batch=2, num_drafts=4, num_heads=16, prefix=(200, 100),
                tree="random", num_slots=2048, seed=seed)
    base.update(kw)
    return G.to_cuda(W.make_inputs(W.Workload(**base)))


def _raw(plan, inp, batch=None, **over):
    lib = mb.load_library()
    out, lse = plan.new_outputs(inp.q.shape[0])
    a = dict(q=inp.q.data_ptr(), kv=inp.kv_cache.data_ptr(), idx=inp.kv_indices.data_ptr(),
             indptr=inp.kv_indptr.data_ptr(), lens=inp.kv_lens.data_ptr(),
             par=inp.draft_parent.data_ptr(), scale=inp.scale, out=out.data_ptr(),
             lse=lse.data_ptr())
    a.update(over)
    return lib.mla_verify_attn(plan.handle, batch or inp.q.shape[0], a["q"], a["kv"], a["idx"],
                               a["indptr"], a["lens"], a["par"], ctypes.c_float(a["scale"]),
                               a["out"], a["lse"], None)


def test_host_argument_errors():
    inp = _case()
    with G.make_plan(inp) as plan:
        assert _raw(plan, inp) == 0
        assert _raw(plan, inp, q=None) == -1
        assert _raw(plan, inp, lse=None) == -1
        assert _raw(plan, inp, q=inp.q.data_ptr() + 2) == -2
        assert _raw(plan, inp, batch=3) == -4
        assert _raw(plan, inp, scale=float("nan")) == -5
        assert _raw(plan, inp, scale=float("inf")) == -5
        assert plan.set_nsplit(0) is None
        with pytest.raises(mb.MlaVerifyError):
            plan.set_nsplit(33)
        torch.cuda.synchronize()
        assert plan.get_error() == 0


def test_slot_out_of_range_is_masked_and_reported():
    """A prefix key whose slot lies outside the cache is masked: the result
    equals the oracle on the request with that key removed."""
    inp = _case(seed=2)
    bad = inp.kv_indices.clone()
    bad[5] = 2048                       # request 0, prefix key 5: one past the cache
    bad[204 + 46] = -7                  # request 1, prefix key 46: negative
    import dataclasses
    binp = dataclasses.replace(inp, kv_indices=bad)
    with G.make_plan(binp) as plan:
        out, lse = G.run(plan, binp)
        assert plan.get_error() & mb.DEV_BAD_SLOT
        assert plan.get_error() == 0    # cleared by the previous read
    keep = torch.ones(inp.kv_indices.numel(), dtype=torch.bool)
    keep[5] = False
    keep[204 + 46] = False
    cpu = W.make_inputs(inp.workload)
    ref_inp = dataclasses.replace(
        cpu, kv_indices=cpu.kv_indices[keep],
        kv_lens=cpu.kv_lens - 1,
        kv_indptr=torch.tensor([0, 203, 203 + 103], dtype=torch.int32))
    ref_o, ref_l = G.oracle_full(ref_inp)
    G.assert_parity(out.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l)


def test_bad_parent_is_reported_and_treated_as_root():
    inp = _case(seed=3, tree="chain")
    par = inp.draft_parent.clone()
    par[0, 2] = 2          # self-parent: not an earlier draft
    import dataclasses
    binp = dataclasses.replace(inp, draft_parent=par)
    star_par = par.clone()
    star_par[0, 2] = -1
    sinp = dataclasses.replace(inp, draft_parent=star_par)
    with G.make_plan(binp) as plan:
        o1, l1 = G.run(plan, binp)
        assert plan.get_error() & mb.DEV_BAD_PARENT
        o2, l2 = G.run(plan, sinp)
        assert plan.get_error() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("nsplit", [1, 3])
def test_bad_length_gives_nan_request_and_flag(nsplit):
    inp = _case(seed=4)
    lens = inp.kv_lens.clone()
    lens[1] = 2            # fewer rows than drafts
    import dataclasses
    binp = dataclasses.replace(inp, kv_lens=lens)
    with G.make_plan(inp, nsplit=nsplit) as plan:
        out, lse = G.run(plan, binp)
        assert plan.get_error() & (mb.DEV_BAD_LEN | mb.DEV_BAD_INDPTR)
        good_o, good_l = G.run(plan, inp)
    assert torch.isnan(out[1]).all() and torch.isnan(lse[1]).all()
    assert torch.equal(out[0], good_o[0]) and torch.equal(lse[0], good_l[0])


def test_indptr_mismatch_is_reported():
    inp = _case(seed=5)
    ip = inp.kv_indptr.clone()
    ip[1] -= 1
    import dataclasses
    binp = dataclasses.replace(inp, kv_indptr=ip)
    with G.make_plan(inp) as plan:
        out, lse = G.run(plan, binp)
        assert plan.get_error() & mb.DEV_BAD_INDPTR
    assert torch.isnan(out).all()


@pytest.mark.parametrize("memory", ["pinned", "mixed", "pageable"])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_host_entry_point_matches_device_entry_point(memory, out_dtype):
    """The host-buffer entry moves its inputs and results with one copy
    kernel per direction when every host buffer is page-locked (mapped into
    the device's address space), else with one DMA copy per array; both give
    the device entry's bits, repeated calls included."""
    inp = _case(seed=6)
    pin = {"pinned": lambda t: t.pin_memory(), "pageable": lambda t: t,
           "mixed": None}[memory]

    def host(t, i):
        t = t.cpu()
        if memory == "mixed":
            return t.pin_memory() if i % 2 == 0 else t
        return pin(t)

    with G.make_plan(inp, out_dtype=out_dtype) as plan:
        o_dev, l_dev = G.run(plan, inp)
        B = inp.q.shape[0]
        out = host(torch.empty((B, 4, 16, 512), dtype=out_dtype), 0)
        lse = host(torch.empty((B, 4, 16), dtype=torch.float32), 1)
        args = [host(t, i) for i, t in enumerate((inp.q, inp.kv_indices, inp.kv_indptr, inp.kv_lens,
                                                  inp.draft_parent))]
        for _ in range(3):
            out.zero_()
            lse.zero_()
            mb.mla_verify_attn_host(plan, args[0], inp.kv_cache, args[1], args[2], args[3], args[4],
                                    inp.scale, out, lse)
            assert torch.equal(out, o_dev.cpu()) and torch.equal(lse, l_dev.cpu())
        assert plan.get_error() == 0


@pytest.mark.parametrize("memory", ["pinned", "pageable"])
def test_host_entry_on_smaller_batches(memory):
    """The host-buffer entry on a plan sized for 5 requests, called with 2,
    then 5, then 1 requests, each with its own inputs: the staged copies,
    the index count taken from kv_indptr[batch] and the results (stored
    straight into mapped host buffers when the call ends in the combine)
    follow each call's batch.  Each result against the oracle."""
    shapes = [(700, 90), (300, 1200, 0, 64, 900), (1500,)]
    cases = [W.make_inputs(W.Workload(name=f"hb{i}", batch=len(pre), num_drafts=4, num_heads=16, prefix=pre,
                                      tree="random", num_slots=4096, spike_frac=0.01, seed=1950 + i))
             for i, pre in enumerate(shapes)]
    pin = (lambda t: t.pin_memory()) if memory == "pinned" else (lambda t: t)
    max_kv = max(int(c.kv_lens.max()) for c in cases)
    with mb.Plan(5, 4, 16, 1, 4096, max_kv) as plan:
        for c in cases:
            B = c.q.shape[0]
            cache = c.kv_cache.cuda()
            out = pin(torch.full((B, 4, 16, 512), float("nan")))
            lse = pin(torch.full((B, 4, 16), float("nan")))
            mb.mla_verify_attn_host(plan, pin(c.q), cache, pin(c.kv_indices), pin(c.kv_indptr), pin(c.kv_lens),
                                    pin(c.draft_parent), c.scale, out, lse)
            ref_o, ref_l = G.oracle_full(c)
            G.assert_parity(out.numpy(), lse.numpy(), ref_o, ref_l)
        assert plan.get_error() == 0


@pytest.mark.parametrize("kernel", [pytest.param(mb.KERNEL_PAIR, id="pair"), pytest.param(mb.KERNEL_TC, id="tc")])
@pytest.mark.parametrize("nsplit", [1, 2])
def test_bounded_wait_runs_out_and_reports_timeout(nsplit, kernel):
    """Fault injected on the host: the attention kernel waits for ready flags
    that nothing sets.  Every wait gives up after its cycle limit (about a
    second): the rows are NaN, the status word reports the timeout, and the
    context stays usable -- the next call is correct."""
    inp = _case(seed=7, prefix=(300, 77), num_heads=32)
    with G.make_plan(inp, nsplit=nsplit, kernel=kernel) as plan:
        assert plan.call_kernel(inp.workload.batch) == kernel
        plan.inject_fault(mb.FAULT_SKIP_PACK)
        out, lse = G.run(plan, inp)
        assert plan.get_error() & mb.DEV_TIMEOUT
        assert torch.isnan(out).all() and torch.isnan(lse).all()
        o2, l2 = G.run(plan, inp)
        assert plan.get_error() == 0
    ref_o, ref_l = G.oracle_full(W.make_inputs(inp.workload))
    G.assert_parity(o2.cpu().numpy(), l2.cpu().numpy(), ref_o, ref_l)


def test_unknown_fault_is_rejected():
    inp = _case(seed=8)
    with G.make_plan(inp) as plan:
        with pytest.raises(mb.MlaVerifyError):
            plan.inject_fault(99)


@pytest.mark.parametrize("where", ["key", "query"])
@pytest.mark.parametrize("mode", ["pair", "packed", "direct", "mma"])
def test_value_outside_fp16_range_sets_the_range_bit(where, mode):
    """A bf16 value of 1e5 has no fp16 counterpart: the kernel that widens it
    reports MLA_VERIFY_DEV_RANGE; an unaffected call leaves the bit clear."""
    H = 16 if mode == "direct" else 32          # one 64-row tile -> direct gather
    inp = _case(seed=40, num_heads=H, tree="chain")
    kernel = {"mma": mb.KERNEL_MMA, "pair": mb.KERNEL_PAIR}.get(mode, mb.KERNEL_TC)
    with G.make_plan(inp, kernel=kernel) as plan:
        G.run(plan, inp)
        assert plan.get_error() == 0
        if where == "key":
            slot = int(inp.kv_indices[5])
            cache = inp.kv_cache.clone()
            cache[slot, 17] = 1.0e5
            bad = dataclasses.replace(inp, kv_cache=cache)
        else:
            q = inp.q.clone()
            q[1, 2, 3, 100] = -1.0e5
            bad = dataclasses.replace(inp, q=q)
        G.run(plan, bad)
        assert plan.get_error() & mb.DEV_RANGE
        G.run(plan, inp)
        assert plan.get_error() == 0


def test_get_error_waits_for_the_call_without_a_device_sync():
    """get_error returns the bits of the last call once it is done, while work
    on another stream is left running (no device-wide synchronisation)."""
    inp = _case(seed=41)
    bad_idx = inp.kv_indices.clone()
    bad_idx[3] = 10 ** 6
    bad = dataclasses.replace(inp, kv_indices=bad_idx)
    other = torch.cuda.Stream()
    with G.make_plan(inp) as plan:
        torch.cuda.synchronize()
        # a one-CTA kernel that spins for a bounded ~0.5 s on another stream
        with torch.cuda.stream(other):
            torch.cuda._sleep(1_000_000_000)
        ev = torch.cuda.Event()
        ev.record(other)
        mb.mla_verify_attn(plan, bad.q, bad.kv_cache, bad.kv_indices, bad.kv_indptr, bad.kv_lens,
                           bad.draft_parent, bad.scale)
        assert plan.get_error() & mb.DEV_BAD_SLOT
        assert not ev.query(), "get_error waited for another stream's work"
        other.synchronize()
