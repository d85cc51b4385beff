"""Parity of the CTA-pair kernel (128 query rows per cluster of two CTAs,
256-key pair blocks, O^T split by value dim across the pair) against the
fp64 oracle, element by element.

The cases reach every structural edge of the pair kernel: a key range with an
odd number of 128-key blocks (the last pair block holds one block, so the odd
CTA has no keys there), splits that start on either parity, a partial 128-row
tile (rows past R), several pair tiles per request, page size 64, bf16 output,
tree masks and empty splits.
"""
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


def _check(w, nsplit=0, out_dtype=torch.float32, pack=mb.PACK_AUTO, expect_pack=None):
    raw = W.make_inputs(w)
    inp = G.to_cuda(raw)
    with G.make_plan(inp, nsplit=nsplit, out_dtype=out_dtype, kernel=mb.KERNEL_PAIR) as plan:
        plan.set_pack_schedule(pack)
        assert plan.call_kernel(w.batch) == mb.KERNEL_PAIR
        if expect_pack is not None:
            assert plan.pack_mode(w.batch) == expect_pack
        out, lse = G.run(plan, inp)
        assert plan.get_error() == 0
    ref_o, ref_l = G.oracle_full(raw)
    if out_dtype == torch.float32:
        return G.assert_parity(out.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l)
    return G.assert_bf16_parity(out.cpu(), lse.cpu().numpy(), ref_o, ref_l, "pair bf16")


def _w(**kw):
    base = dict(name="pair", batch=1, num_drafts=8, num_heads=16, prefix=(1100,), tree="chain",
                num_slots=8192, spike_frac=0.01, seed=900)
    base.update(kw)
    return W.Workload(**base)


@pytest.mark.parametrize("nsplit", [1, 2, 3, 5])
def test_one_pair_tile_odd_blocks(nsplit):
    # 1108 keys = 9 blocks of 128: pair blocks (0,1) .. (6,7), (8,-).
    _check(_w(seed=901 + nsplit), nsplit=nsplit)


@pytest.mark.parametrize("prefix", [(0,), (120,), (128,), (248,), (2000,)])
def test_key_counts(prefix):
    # 8 keys (one block, the odd CTA idle), 128, 136, 256 and 2008 keys.
    _check(_w(prefix=prefix, seed=920 + prefix[0] % 97))


def test_partial_row_tile():
    # R = 3 * 32 = 96 rows: rows 96..127 of the pair tile are past R.
    _check(_w(num_drafts=3, num_heads=32, tree="random", seed=931))


@pytest.mark.parametrize("nsplit", [0, 4])
def test_several_pair_tiles_batch(nsplit):
    w = _w(batch=3, num_drafts=8, num_heads=64, prefix=(3000, 700, 129), tree="random", seed=940)
    _check(w, nsplit=nsplit)


def test_page_size_64_bf16_out():
    w = _w(batch=2, num_heads=32, prefix=(1500, 77), page_size=64, tree="star", seed=950)
    _check(w, out_dtype=torch.bfloat16)


@pytest.mark.parametrize("pack", [mb.PACK_WHOLE, mb.PACK_IDLE_SMS])
def test_pack_schedules(pack):
    w = _w(batch=2, num_heads=32, prefix=(4000, 2500), seed=960)
    _check(w, nsplit=3, pack=pack, expect_pack=pack)


def test_empty_splits():
    # 32 splits over 3 pair blocks: most splits have no keys (weight 0).
    _check(_w(prefix=(600,), seed=970), nsplit=32)


def test_tree_sixteen_drafts_spiky():
    w = _w(batch=2, num_drafts=16, num_heads=16, prefix=(5000, 3000), tree="random",
           spike_frac=0.01, seed=980)
    _check(w)


@pytest.mark.parametrize("pack", [mb.PACK_WHOLE, mb.PACK_IDLE_SMS])
def test_odd_block_ends_many_replays(pack):
    """Splits whose last pair block holds one block (the odd CTA has nothing
    to load there): hundreds of graph replays, each after an L2 flush, leave
    the status word clear.  A version in which the even CTA's MMAs could run
    units ahead of the odd CTA's copy warps failed here about once in eight
    timing runs (a slot barrier two phases ahead of its waiter)."""
    w = _w(batch=4, num_drafts=8, num_heads=32, prefix=(4096, 1100, 3000, 16384 + 8), num_slots=32768,
           seed=990)
    raw = W.make_inputs(w)
    inp = G.to_cuda(raw)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    with G.make_plan(inp, kernel=mb.KERNEL_PAIR, nsplit=3) as plan:
        plan.set_pack_schedule(pack)
        out, lse = plan.new_outputs(w.batch)
        st = torch.cuda.Stream()
        st.wait_stream(torch.cuda.current_stream())

        def call():
            mb.mla_verify_attn(plan, inp.q, inp.kv_cache, inp.kv_indices, inp.kv_indptr, inp.kv_lens,
                               inp.draft_parent, inp.scale, out, lse, stream=st)

        with torch.cuda.stream(st):
            call()
        st.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            call()
        ref = None
        for k in range(300):
            with torch.cuda.stream(st):
                flush.zero_()
                g.replay()
            if k % 50 == 49:
                st.synchronize()
                assert plan.get_error() == 0, k
                if ref is None:
                    ref = (out.clone(), lse.clone())
                else:
                    assert torch.equal(out, ref[0]) and torch.equal(lse, ref[1])
    ref_o, ref_l = G.oracle_full(raw)
    G.assert_parity(ref[0].cpu().numpy(), ref[1].cpu().numpy(), ref_o, ref_l)
