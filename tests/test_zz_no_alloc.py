"""The allocation-free entry point agrees with the plan-based one.

mla_verify_attn_static serves callers that cannot allocate device memory
(a memory pool that owns the whole device, a serving loop that must not
allocate after start-up, a layer that is only handed pointers).  It keeps its
split partials in a fixed device array instead of a plan's workspace.  This
test calls it twice in a row through the C ABI and compares each result with
mla_verify_attn on the same inputs, same kernel family and same split count,
and with the fp64 oracle, within the parity tolerances used everywhere else
(out max abs 1e-2, mean abs 1e-3; lse max abs 1e-3), for page sizes 1 and 64.  It lives in a file collected last so that a run
stopping at the first failure has already run every other test.
"""
import ctypes

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


def _static_call(inp, nsplit, out, lse, status):
    w = inp.workload
    lib = mb.load_library()
    return lib.mla_verify_attn_static(
        w.batch, w.num_drafts, w.num_heads, inp.page_size, inp.kv_cache.shape[0],
        int(inp.kv_lens.max()), nsplit, inp.q.data_ptr(), inp.kv_cache.data_ptr(),
        inp.kv_indices.data_ptr(), inp.kv_indptr.data_ptr(), inp.kv_lens.data_ptr(),
        inp.draft_parent.data_ptr(), ctypes.c_float(inp.scale), out.data_ptr(), lse.data_ptr(),
        status.data_ptr() if status is not None else None,
        torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("ps", [1, 64])
@pytest.mark.parametrize("nsplit", [3, 1])
def test_static_entry_matches_plan_entry_twice(nsplit, ps):
    raw = [
        W.make_inputs(W.Workload(name="na", batch=3, num_drafts=8, num_heads=16,
                                 prefix=(900, 65, 300), tree="random", num_slots=4096,
                                 page_size=ps, spike_frac=0.01, seed=901)),
        W.make_inputs(W.Workload(name="nb", batch=3, num_drafts=8, num_heads=16,
                                 prefix=(10, 1200, 0), tree="chain", num_slots=4096,
                                 page_size=ps, spike_frac=0.01, seed=902)),
    ]
    inputs = [G.to_cuda(r) for r in raw]
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    for inp, cpu in zip(inputs, raw):          # two calls in a row, different data
        out = torch.full((3, 8, 16, 512), float("nan"), device="cuda")
        lse = torch.full((3, 8, 16), float("nan"), device="cuda")
        st = _static_call(inp, nsplit, out, lse, status)
        assert st == 0, mb.strerror(st)
        with G.make_plan(inp, nsplit=nsplit, kernel=mb.KERNEL_MMA,
                         max_kv_len=int(inp.kv_lens.max())) as plan:
            ref_o, ref_l = G.run(plan, inp)
        torch.cuda.synchronize()
        assert int(status[0]) == 0
        G.assert_parity(out.cpu().numpy(), lse.cpu().numpy(), ref_o.cpu().numpy().astype(np.float64),
                        ref_l.cpu().numpy().astype(np.float64), "static vs plan entry")
        or_o, or_l = G.oracle_full(cpu)
        G.assert_parity(out.cpu().numpy(), lse.cpu().numpy(), or_o, or_l, "static vs oracle")


def test_static_entry_rejects_oversized_calls_and_reports_device_errors():
    inp = G.to_cuda(W.make_inputs(W.Workload(name="nc", batch=2, num_drafts=4, num_heads=16,
                                             prefix=(100, 40), tree="chain", num_slots=1024,
                                             seed=903)))
    out = torch.empty((2, 4, 16, 512), device="cuda")
    lse = torch.empty((2, 4, 16), device="cuda")
    # batch x nsplit x T*H x 2052 bytes must fit the fixed array.
    too_many_rows = W.Workload(name="nd", batch=1, num_drafts=32, num_heads=128, prefix=(64,),
                               tree="chain", num_slots=1024, seed=904)
    big = G.to_cuda(W.make_inputs(too_many_rows))
    bout = torch.empty((1, 32, 128, 512), device="cuda")
    blse = torch.empty((1, 32, 128), device="cuda")
    assert _static_call(big, 32, bout, blse, None) == -10
    # A slot outside the cache is masked and reported through device_status.
    bad = inp.kv_indices.clone()
    bad[3] = 1024
    import dataclasses
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _static_call(dataclasses.replace(inp, kv_indices=bad), 2, out, lse, status) == 0
    torch.cuda.synchronize()
    assert int(status[0]) & mb.DEV_BAD_SLOT
    assert torch.isfinite(out).all()
