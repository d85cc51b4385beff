"""GPU parity of KV compaction into 64-row pages, through the C ABI.

Byte work: the destination cache (written rows and untouched ones), the page
table, the page offsets and the device status bits must equal the oracle's
(oracle/compact_ref.py) exactly.  End to end, the verify attention over the
compacted cache with the new page_size 64 table returns the same bits as
over the source cache with the page_size 1 table.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle.compact_ref as cr
from paged_mla_speculative_gb300 import binding as mb
from paged_mla_speculative_gb300 import workloads as W
from tests import gpu_util as G
from tests.conftest import bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_mla_speculative_gb300 import build
    build.build()


def _case(seed, prefix=(300, 60, 129, 1000), T=4):
    w = W.Workload(name="cg", batch=len(prefix), num_drafts=T, num_heads=16, prefix=prefix,
                   tree="random", num_slots=4096, spike_frac=0.01, seed=seed)
    return w, W.make_inputs(w)


def _compare(plan, src, idx, ptr, lens, free, dst_pages, max_kv_len, expect_flags=None):
    """Run the GPU compaction and the oracle on the same inputs; compare all."""
    dst0 = torch.full((dst_pages * 64, 576), 0x7FC0, dtype=torch.int16).view(torch.bfloat16)
    dst_gpu = dst0.cuda()
    plan.get_error()
    table, pin = mb.compact_kv(plan, src.cuda(), idx.cuda(), ptr.cuda(), lens.cuda(),
                               torch.as_tensor(free, dtype=torch.int32).cuda(), dst_gpu)
    torch.cuda.synchronize()
    flags = plan.get_error()
    want_dst, want_table, want_pin, want_flags = cr.compact_kv(
        bits(src), idx.tolist(), ptr.tolist(), lens.tolist(), list(free), bits(dst0), max_kv_len)
    assert pin.cpu().tolist() == want_pin
    assert table[:want_pin[-1]].cpu().tolist() == want_table
    assert np.array_equal(bits(dst_gpu.cpu()), want_dst)
    assert flags == want_flags
    if expect_flags is not None:
        assert flags == expect_flags
    return dst_gpu, table, pin


@pytest.mark.parametrize("seed", [0, 1])
def test_compaction_matches_the_oracle(seed):
    w, inp = _case(seed)
    free = np.random.default_rng(seed).permutation(64)
    with G.make_plan(G.to_cuda(inp)) as plan:
        _compare(plan, inp.kv_cache, inp.kv_indices, inp.kv_indptr, inp.kv_lens, free, 64,
                 int(inp.kv_lens.max()), expect_flags=0)


def test_capacity_bad_slots_bad_pages_bad_lengths():
    w, inp = _case(5)
    mx = int(inp.kv_lens.max())
    with G.make_plan(G.to_cuda(inp)) as plan:
        idx = inp.kv_indices.clone()
        idx[7] = 4096          # outside the 4096-slot source cache: zero row, BAD_SLOT
        idx[400] = -3
        free = np.arange(10)   # requests need 5, 1, 3, 17 pages: the last is cut
        _compare(plan, inp.kv_cache, idx, inp.kv_indptr, inp.kv_lens, free, 64, mx,
                 expect_flags=cr.BAD_SLOT | cr.CAPACITY)
        free2 = np.array([1, 2, 99, 4, 5] + list(range(6, 40)))   # page 99 outside a 64-page cache
        _compare(plan, inp.kv_cache, inp.kv_indices, inp.kv_indptr, inp.kv_lens, free2, 64, mx,
                 expect_flags=cr.BAD_SLOT)
        lens = inp.kv_lens.clone()
        lens[1] = 65           # indptr range holds 64 slots: no pages, BAD_INDPTR
        _compare(plan, inp.kv_cache, inp.kv_indices, inp.kv_indptr, lens, np.arange(64), 64, mx,
                 expect_flags=cr.BAD_INDPTR)


def test_attention_on_the_compacted_cache_is_bitwise_the_same():
    w, inp = _case(9, prefix=(2000, 130, 700), T=8)
    g = G.to_cuda(inp)
    free = np.random.default_rng(9).permutation(80)
    with G.make_plan(g, nsplit=3) as plan:
        o1, l1 = G.run(plan, g)
        dst = torch.zeros((80 * 64, 576), dtype=torch.bfloat16, device="cuda")
        table, pin = mb.compact_kv(plan, g.kv_cache, g.kv_indices, g.kv_indptr, g.kv_lens,
                                   torch.as_tensor(free, dtype=torch.int32).cuda(), dst)
        torch.cuda.synchronize()
        assert plan.get_error() == 0
    paged = dataclasses.replace(g, kv_cache=dst, kv_indices=table[:int(pin[-1])].contiguous(),
                                kv_indptr=pin, page_size=64)
    with G.make_plan(paged, nsplit=3) as plan64:
        o2, l2 = G.run(plan64, paged)
        assert plan64.get_error() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_host_argument_errors():
    w, inp = _case(11)
    g = G.to_cuda(inp)
    with G.make_plan(g) as plan:
        lib = mb.load_library()
        dst = torch.zeros((64 * 64, 576), dtype=torch.bfloat16, device="cuda")
        free = torch.arange(64, dtype=torch.int32, device="cuda")
        tab = torch.empty(64, dtype=torch.int32, device="cuda")
        pin = torch.empty(len(w.prefix) + 1, dtype=torch.int32, device="cuda")

        def call(**k):
            return lib.mla_verify_compact_kv(
                plan.handle, k.get("batch", w.batch), g.kv_cache.data_ptr(), 4096,
                g.kv_indices.data_ptr(), g.kv_indptr.data_ptr(), g.kv_lens.data_ptr(),
                free.data_ptr(), 64, k.get("dst", dst.data_ptr()), k.get("dst_slots", 64 * 64),
                tab.data_ptr(), pin.data_ptr(), None)
        assert call() == 0
        assert call(dst=None) == -1
        assert call(dst=dst.data_ptr() + 8) == -2
        assert call(batch=w.batch + 1) == -4
        assert call(dst_slots=64 * 64 - 1) == -9
        torch.cuda.synchronize()
