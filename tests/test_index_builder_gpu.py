"""GPU parity of the per-step index builder, through the C ABI.

Integer work: kv_lens, kv_indptr, kv_indices and the device status bits must
equal the oracle's (oracle/index_builder_ref.py) exactly, for page sizes 1
and 64, invalid pool rows and prefixes, capacity cuts, misaligned pages, and
batches larger than one scan chunk.  End to end, indices built on the GPU
make mla_verify_attn return the same bits as the workload's own indices,
also when the builder and the attention are captured into one CUDA graph.
"""
import numpy as np
import pytest
import torch

import oracle.index_builder_ref as ib
from paged_mla_speculative_gb300 import binding as mb
from paged_mla_speculative_gb300 import workloads as W
from tests import gpu_util as G
from tests.test_index_builder_pins import workload_table

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_mla_speculative_gb300 import build
    build.build()


def _check(plan, table, pools, prefix, T, ps, max_kv_len, capacity):
    t = torch.as_tensor(np.asarray(table), dtype=torch.int32).cuda().contiguous()
    pl = torch.as_tensor(np.asarray(pools), dtype=torch.int32).cuda()
    pf = torch.as_tensor(np.asarray(prefix), dtype=torch.int32).cuda()
    buf = torch.full((capacity + 64,), -7, dtype=torch.int32, device="cuda")
    ptr = torch.full((len(pools) + 1,), -7, dtype=torch.int32, device="cuda")
    lens = torch.full((len(pools),), -7, dtype=torch.int32, device="cuda")
    plan.get_error()
    st = mb.load_library().mla_verify_build_indices(
        plan.handle, len(pools), t.data_ptr(), int(t.stride(0)), int(t.shape[0]), pl.data_ptr(),
        pf.data_ptr(), buf.data_ptr(), capacity, ptr.data_ptr(), lens.data_ptr(), None)
    assert st == 0, mb.strerror(st)
    torch.cuda.synchronize()
    flags = plan.get_error()
    want_lens, want_ptr, want_idx, want_flags = ib.build_indices(
        np.asarray(table), pools, prefix, T, ps, max_kv_len, capacity)
    assert lens.cpu().tolist() == want_lens
    assert ptr.cpu().tolist() == want_ptr
    n = want_ptr[-1]
    assert buf[:n].cpu().tolist() == want_idx
    assert (buf[n:] == -7).all(), "wrote past the last entry"
    assert flags == want_flags


def _plan(batch, T, ps, max_kv_len, num_slots=1 << 20):
    return mb.Plan(batch, T, 1, ps, num_slots, max_kv_len)


@pytest.mark.parametrize("ps", [1, 64])
@pytest.mark.parametrize("seed", [0, 1])
def test_random_steps_match_the_oracle(ps, seed):
    rng = np.random.default_rng(100 + seed)
    T, max_kv_len, pool_size, B = 4, 700, 40, 37
    if ps == 1:
        table = rng.integers(0, 1 << 20, size=(pool_size, max_kv_len + 3))
    else:   # whole pages, a few rows with a misaligned page start
        pages = rng.integers(0, (1 << 20) // 64, size=(pool_size, (max_kv_len + 63) // 64 + 1))
        table = (pages[:, :, None] * 64 + np.arange(64)[None, None, :]).reshape(pool_size, -1)
        table = table[:, :max_kv_len + 3].copy()
        table[3, 64] += 5
        table[7, 0] = -1
    pools = rng.integers(-1, pool_size + 1, size=B)
    prefix = rng.integers(-2, max_kv_len - T + 3, size=B)
    with _plan(B, T, ps, max_kv_len) as plan:
        for capacity in (10 ** 6, 3000 if ps == 1 else 40, 0):
            _check(plan, table, pools, prefix, T, ps, max_kv_len, capacity)


def test_batch_larger_than_one_scan_chunk():
    rng = np.random.default_rng(7)
    T, max_kv_len, pool_size, B = 2, 40, 3000, 2500
    table = rng.integers(0, 1 << 20, size=(pool_size, max_kv_len))
    pools = rng.permutation(pool_size)[:B]
    prefix = rng.integers(0, max_kv_len - T + 1, size=B)
    with _plan(B, T, 1, max_kv_len) as plan:
        total = int((prefix + T).sum())
        for capacity in (total, total - 1, total // 2, 10 ** 6):
            _check(plan, table, pools, prefix, T, 1, max_kv_len, capacity)


def test_host_argument_errors():
    with _plan(4, 2, 1, 100) as plan:
        t = torch.zeros((3, 100), dtype=torch.int32, device="cuda")
        i4 = torch.zeros(4, dtype=torch.int32, device="cuda")
        buf = torch.zeros(64, dtype=torch.int32, device="cuda")
        lib = mb.load_library()
        call = lambda **k: lib.mla_verify_build_indices(  # noqa: E731
            plan.handle, k.get("batch", 4), k.get("table", t.data_ptr()), k.get("stride", 100), 3,
            i4.data_ptr(), i4.data_ptr(), buf.data_ptr(), k.get("cap", 64), buf.data_ptr(),
            i4.data_ptr(), None)
        assert call() == 0
        assert call(table=None) == -1
        assert call(table=t.data_ptr() + 4) == -2
        assert call(batch=5) == -4
        assert call(stride=99) == -9
        assert call(cap=-1) == -9
        assert call(cap=1 << 31) == -9
        torch.cuda.synchronize()


@pytest.mark.parametrize("ps", [1, 64])
def test_built_indices_drive_the_attention_bit_for_bit(ps):
    w = W.Workload(name="ibe", batch=4, num_drafts=8, num_heads=16, prefix=(500, 64, 1300, 7),
                   tree="random", num_slots=16384, page_size=ps, spike_frac=0.01, seed=47)
    raw = W.make_inputs(w)
    inp = G.to_cuda(raw)
    table, pools, prefix = workload_table(raw)
    with G.make_plan(inp, nsplit=3) as plan:
        ref_o, ref_l = G.run(plan, inp)
        idx, ptr, lens = mb.build_indices(
            plan, torch.as_tensor(table, dtype=torch.int32).cuda(),
            torch.as_tensor(pools, dtype=torch.int32).cuda(),
            torch.as_tensor(prefix, dtype=torch.int32).cuda())
        import dataclasses
        built = dataclasses.replace(inp, kv_indices=idx, kv_indptr=ptr, kv_lens=lens)
        o, l = G.run(plan, built)
        assert plan.get_error() == 0
    assert torch.equal(ptr.cpu(), raw.kv_indptr) and torch.equal(lens.cpu(), raw.kv_lens)
    assert torch.equal(o, ref_o) and torch.equal(l, ref_l)


def test_builder_and_attention_in_one_graph():
    w = W.Workload(name="ibg", batch=3, num_drafts=4, num_heads=16, prefix=(300, 900, 40),
                   tree="chain", num_slots=8192, seed=53)
    raw = W.make_inputs(w)
    inp = G.to_cuda(raw)
    table, pools, prefix = workload_table(raw)
    table = np.pad(table, ((0, 0), (0, 1000 - table.shape[1])), constant_values=-1)  # stride >= max_kv_len
    t = torch.as_tensor(table, dtype=torch.int32).cuda()
    pl = torch.as_tensor(pools, dtype=torch.int32).cuda()
    pf = torch.as_tensor(prefix, dtype=torch.int32).cuda()
    with G.make_plan(inp, max_kv_len=1000) as plan:
        idx = torch.empty(w.batch * 1000, dtype=torch.int32, device="cuda")
        ptr = torch.empty(w.batch + 1, dtype=torch.int32, device="cuda")
        lens = torch.empty(w.batch, dtype=torch.int32, device="cuda")
        out, lse = plan.new_outputs(w.batch)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())

        def step():
            mb.build_indices(plan, t, pl, pf, idx, ptr, lens, stream=s)
            mb.mla_verify_attn(plan, inp.q, inp.kv_cache, idx, ptr, lens, inp.draft_parent,
                               inp.scale, out, lse, stream=s)

        with torch.cuda.stream(s):
            step()
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step()
        # New step data in the same buffers: every prefix halved.
        pf.copy_(torch.as_tensor(np.asarray(prefix) // 2, dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        got_o, got_l = out.clone(), lse.clone()
        with torch.cuda.stream(s):
            step()
        s.synchronize()
        assert plan.get_error() == 0
    assert torch.equal(got_o, out) and torch.equal(got_l, lse)
    assert lens.cpu().tolist() == [int(x) // 2 + 4 for x in np.asarray(prefix)]
