"""Context-parallel split on one GPU, through the C ABI.

Every shard of a call runs in sequence on the same device
(mla_verify_attn_partial), the partials are stacked shard-major as an
all-gather leaves them, and mla_verify_combine_parts merges them.  Each
shard's partial is compared element by element with the oracle restricted to
that shard's keys, and the merged result with the unsharded oracle (out max
abs 1e-2, mean abs 1e-3; lse max abs 1e-3).  Multi-GPU runs differ only in
the gather, which tests/test_context_parallel_pins.py covers on gloo ranks.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_mla_speculative_gb300 import binding as mb
from paged_mla_speculative_gb300 import workloads as W
from tests import gpu_util as G
from tests.conftest import oracle_args

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_mla_speculative_gb300 import build
    build.build()


def _check_partial(po, pl, ref_o, ref_l, what):
    po = po.cpu().numpy().astype(np.float64)
    pl = pl.cpu().numpy().astype(np.float64)
    empty = np.isneginf(ref_l)
    assert (np.isneginf(pl) == empty).all(), f"{what}: -inf rows differ"
    assert (po[empty] == 0).all(), f"{what}: rows with no key must be 0"
    if (~empty).any():
        G.assert_parity(po[~empty], pl[~empty], ref_o[~empty], ref_l[~empty], what)


def run_shards(inp, S, kernel=mb.KERNEL_AUTO, out_dtype=torch.float32, check_parts=True):
    g = G.to_cuda(inp)
    args = oracle_args(inp)
    lens = inp.kv_lens.tolist()
    with G.make_plan(g, out_dtype=out_dtype, kernel=kernel) as plan:
        parts_o, parts_l = [], []
        for s in range(S):
            po, pl = mb.mla_verify_attn_partial(plan, g.q, g.kv_cache, g.kv_indices, g.kv_indptr,
                                                g.kv_lens, g.draft_parent, g.scale, s, S)
            torch.cuda.synchronize()
            if check_parts:
                rng = [oracle.shard_key_range(n, s, S) for n in lens]
                ro, rl = oracle.mla_verify_key_range(*args, [r[0] for r in rng], [r[1] for r in rng])
                _check_partial(po, pl, ro, rl, f"shard {s}/{S}")
            parts_o.append(po)
            parts_l.append(pl)
        out, lse = mb.mla_verify_combine_parts(plan, torch.stack(parts_o), torch.stack(parts_l))
        torch.cuda.synchronize()
        assert plan.get_error() == 0
    return out, lse


@pytest.mark.parametrize("kernel", [pytest.param(mb.KERNEL_PAIR, id="pair"), pytest.param(mb.KERNEL_TC, id="tc"),
                                    pytest.param(mb.KERNEL_MMA, id="mma")])
@pytest.mark.parametrize("S", [1, 2, 3, 7])
def test_shards_merge_to_the_oracle(kernel, S):
    w = W.Workload(name="cp", batch=3, num_drafts=8, num_heads=16, prefix=(900, 130, 0),
                   tree="random", num_slots=4096, spike_frac=0.01, seed=1200 + S)
    inp = W.make_inputs(w)
    out, lse = run_shards(inp, S, kernel)
    ref_o, ref_l = oracle.mla_verify(*oracle_args(inp))
    G.assert_parity(out.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, f"merged {S} shards")


@pytest.mark.parametrize("ps", [1, 64])
def test_shards_page_size_and_bf16_out(ps):
    w = W.Workload(name="cp64", batch=2, num_drafts=4, num_heads=32, prefix=(1500, 333),
                   tree="chain", num_slots=8192, page_size=ps, spike_frac=0.01, seed=1300 + ps)
    inp = W.make_inputs(w)
    o32, l32 = run_shards(inp, 2)
    o16, l16 = run_shards(inp, 2, out_dtype=torch.bfloat16, check_parts=False)
    assert torch.equal(o32.to(torch.bfloat16), o16) and torch.equal(l32, l16)
    ref_o, ref_l = oracle.mla_verify(*oracle_args(inp))
    G.assert_parity(o32.cpu().numpy(), l32.cpu().numpy(), ref_o, ref_l, f"ps{ps}")


def test_long_request_two_shards_full_size():
    """sweep_p16384 (R=512, 16392 keys) split over two shards."""
    inp = W.make_inputs(W.WORKLOADS["sweep_p16384"])
    out, lse = run_shards(inp, 2, check_parts=False)
    ref_o, ref_l = oracle.mla_verify(*oracle_args(inp))
    G.assert_parity(out.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, "sweep_p16384 / 2 shards")


def test_partial_and_combine_capture_into_one_graph():
    w = W.Workload(name="cpg", batch=2, num_drafts=8, num_heads=16, prefix=(700, 90),
                   tree="random", num_slots=4096, spike_frac=0.01, seed=1400)
    inp = G.to_cuda(W.make_inputs(w))
    S = 3
    with G.make_plan(inp, max_kv_len=1000) as plan:
        parts_o = torch.empty((S, 2, 8, 16, 512), device="cuda")
        parts_l = torch.empty((S, 2, 8, 16), device="cuda")
        out, lse = plan.new_outputs(2)
        st = torch.cuda.Stream()

        def call():
            for s in range(S):
                mb.mla_verify_attn_partial(plan, inp.q, inp.kv_cache, inp.kv_indices, inp.kv_indptr,
                                           inp.kv_lens, inp.draft_parent, inp.scale, s, S,
                                           parts_o[s], parts_l[s], stream=st)
            mb.mla_verify_combine_parts(plan, parts_o, parts_l, out, lse, stream=st)

        st.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(st):
            call()
        st.synchronize()
        eo, el = out.clone(), lse.clone()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            call()
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eo) and torch.equal(lse, el)
        assert plan.get_error() == 0


def test_bad_shard_arguments_are_rejected():
    w = W.Workload(name="cpb", batch=1, num_drafts=4, num_heads=16, prefix=(100,), tree="chain",
                   num_slots=1024, seed=1500)
    inp = G.to_cuda(W.make_inputs(w))
    with G.make_plan(inp) as plan:
        for shard, num in ((2, 2), (-1, 2), (0, 0), (0, 33)):
            with pytest.raises(mb.MlaVerifyError) as e:
                mb.mla_verify_attn_partial(plan, inp.q, inp.kv_cache, inp.kv_indices, inp.kv_indptr,
                                           inp.kv_lens, inp.draft_parent, inp.scale, shard, num)
            assert e.value.status == -9
        po = torch.empty((3, 1, 4, 16, 512), device="cuda")
        pl = torch.empty((3, 1, 4, 16), device="cuda")
        big = torch.empty((33, 1, 4, 16, 512), device="cuda")
        bigl = torch.empty((33, 1, 4, 16), device="cuda")
        with pytest.raises(mb.MlaVerifyError):
            mb.mla_verify_combine_parts(plan, big, bigl)
        mb.mla_verify_combine_parts(plan, po.zero_(), pl.fill_(0.0))
        torch.cuda.synchronize()


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
@pytest.mark.parametrize("S", [1, 2, 3, 4, 5, 8, 9, 16, 17, 25, 32])
def test_combine_parts_every_count_against_the_merge(S, out_dtype):
    """The combine on synthetic partials, for part counts across every launch
    shape of the combine kernel (1-2, 3-4, 5-8 and 9-16 parts in one round
    trip; 17-32 in two), against the oracle's fp64 LSE merge (the reduce step
    of "The Decisive A/B ...", section "The Context").  About a quarter of
    the (part, row) entries have no visible key: lse -inf and rows of NaN,
    which must carry weight 0 and never be read into the result.  One row
    has every part empty (lse -inf, out 0) and one row has a NaN lse in one
    part (the row becomes NaN)."""
    B, T, H = 2, 4, 16
    g = torch.Generator().manual_seed(1700 + S)
    po = torch.randn((S, B, T, H, 512), generator=g) * 4.0
    pl = torch.randn((S, B, T, H), generator=g) * 3.0 + 5.0
    empty = torch.rand((S, B, T, H), generator=g) < 0.25
    empty[:, 0, 0, 0] = True                      # a row with no visible key in any part
    pl[empty] = float("-inf")
    clean = po.clone()
    clean[empty] = 0.0
    po[empty] = float("nan")                      # never to be read
    nan_part = S // 2
    empty[nan_part, 1, 1, 1] = False
    pl[nan_part, 1, 1, 1] = float("nan")
    ref_o, ref_l = oracle.lse_merge(clean.numpy(), pl.numpy())

    w = W.Workload(name="cpm", batch=B, num_drafts=T, num_heads=H, prefix=(64, 64), tree="chain",
                   num_slots=1024, seed=1700)
    inp = G.to_cuda(W.make_inputs(w))
    with G.make_plan(inp, out_dtype=out_dtype) as plan:
        out, lse = mb.mla_verify_combine_parts(plan, po.cuda(), pl.cuda())
        torch.cuda.synchronize()
        assert plan.get_error() == 0
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.cpu().numpy().astype(np.float64)
    assert np.isnan(l[1, 1, 1]) and np.isnan(o[1, 1, 1]).all(), "a NaN part makes its row NaN"
    keep = np.ones((B, T, H), dtype=bool)
    keep[1, 1, 1] = False
    assert np.isneginf(l[0, 0, 0]) and (o[0, 0, 0] == 0).all(), "a row with no visible key"
    assert np.isfinite(o[keep]).all() and (np.isneginf(l[keep]) == np.isneginf(ref_l[keep])).all()
    fin = keep & np.isfinite(ref_l)
    assert np.abs(l[fin] - ref_l[fin]).max() <= 1e-4
    # fp32: the merge's own rounding; bf16: one rounding of the result on top.
    bound = 1e-4 if out_dtype == torch.float32 else 2.0 ** -8 * np.abs(ref_o[keep]).max() + 1e-4
    assert np.abs(o[keep] - ref_o[keep]).max() <= bound
