"""GPU parity of the verify attention against the fp64 oracle, through the C ABI.

Small cases (several 64-row tiles, several key blocks, ragged tails) and every
full-size workload, in the launch configuration the benchmark times, are
compared element by element.
Tolerances: out max abs 1e-2 and mean abs 1e-3, lse max abs 1e-3.
"""
import json
import os

import numpy as np
import pytest
import torch

from paged_mla_speculative_gb300 import binding as mb
from paged_mla_speculative_gb300 import workloads as W
from tests import gpu_util as G
from tests.conftest import bits

pytestmark = pytest.mark.gpu


def small(**kw):
    base = dict(name="s", batch=2, num_drafts=4, num_heads=16, prefix=(300, 77),
                tree="random", num_slots=4096, spike_frac=0.01, seed=100)
    base.update(kw)
    return W.Workload(**base)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_mla_speculative_gb300 import build
    build.build()


def check_full(inp, **plan_kw):
    g = G.to_cuda(inp)
    with G.make_plan(g, **plan_kw) as plan:
        out, lse = G.run(plan, g)
        assert plan.get_error() == 0
    ref_o, ref_l = G.oracle_full(inp)
    return G.assert_parity(out.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l)


KERNELS = [pytest.param(mb.KERNEL_PAIR, id="pair"), pytest.param(mb.KERNEL_TC, id="tc"),
           pytest.param(mb.KERNEL_MMA, id="mma")]


@pytest.mark.parametrize("kernel", KERNELS)
def test_tiny_workload_elementwise(kernel):
    check_full(W.make_inputs(W.WORKLOADS["tiny"]), kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("nsplit", [1, 3])
def test_kernel_families_small_ragged(kernel, nsplit):
    w = small(batch=3, prefix=(700, 129, 0), num_drafts=8, num_heads=16, seed=150)
    check_full(W.make_inputs(w), kernel=kernel, nsplit=nsplit)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("ps", [1, 64])
def test_thirty_two_drafts_deep_random_tree(kernel, ps):
    """The largest draft count (32: every bit of the ancestor words) on a
    random tree up to 12 deep, 8 heads (R = 256: two pair tiles, four
    single-SM tiles), ragged prefixes with an empty one, both page sizes."""
    w = small(batch=3, num_drafts=32, num_heads=8, prefix=(650, 37, 0), tree="random", max_depth=12,
              page_size=ps, seed=1800 + ps)
    check_full(W.make_inputs(w), kernel=kernel)


@pytest.mark.parametrize("kernel,ps", [
    pytest.param(mb.KERNEL_AUTO, 1, id="auto-ps1"), pytest.param(mb.KERNEL_AUTO, 64, id="auto-ps64"),
    pytest.param(mb.KERNEL_PAIR, 1, id="pair-ps1"), pytest.param(mb.KERNEL_TC, 1, id="tc-ps1"),
    pytest.param(mb.KERNEL_MMA, 1, id="mma-ps1")])
def test_one_plan_serves_smaller_batches(kernel, ps):
    """A plan sized for 6 requests serves calls of 6, 2, 5 and 1 requests in
    a row, each with its own inputs: the split count, the pack's layout and
    its epoch tags (counted over each call's grid) follow each call's batch."""
    T, H, slots = 8, 16, 8192
    shapes = [(900, 40, 0, 1300, 257, 64), (1500, 3), (100, 700, 1200, 9, 0), (2000,)]
    inputs = [W.make_inputs(W.Workload(name=f"mb{i}", batch=len(pre), num_drafts=T, num_heads=H, prefix=pre,
                                       tree="random", num_slots=slots, page_size=ps, spike_frac=0.01,
                                       seed=1900 + 10 * i + ps))
              for i, pre in enumerate(shapes)]
    max_kv = max(int(x.kv_lens.max()) for x in inputs)
    with mb.Plan(6, T, H, ps, slots, max_kv) as plan:
        plan.set_kernel(kernel)
        for inp in inputs:
            out, lse = G.run(plan, G.to_cuda(inp))
            assert plan.get_error() == 0
            ref_o, ref_l = G.oracle_full(inp)
            G.assert_parity(out.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("scale", [0.5, 1e-3], ids=["peaked", "flat"])
def test_softmax_scale_extremes(kernel, scale):
    """A large scale (0.5: a few keys carry nearly all the weight, so the
    running max moves often) and a tiny one (1e-3: near-uniform weights over
    every key, so the sums run long), against the oracle at the same scale."""
    w = small(batch=2, num_drafts=8, num_heads=16, prefix=(3000, 700), tree="random", scale=scale,
              seed=1830 if scale > 0.1 else 1831)
    check_full(W.make_inputs(w), kernel=kernel, nsplit=3)


@pytest.mark.parametrize("nsplit", [1, 2, 4])
@pytest.mark.parametrize("ps", [1, 64])
def test_fifteen_rows_direct_gather(nsplit, ps):
    """T·H = 15 (3 drafts x 5 heads): one partial 64-row tile, whose CTAs
    gather their own key rows (no pack); rows 15..63 of the tile are idle."""
    w = small(batch=2, num_drafts=3, num_heads=5, prefix=(520, 200), page_size=ps, seed=1820 + nsplit)
    check_full(W.make_inputs(w), nsplit=nsplit)


@pytest.mark.parametrize("kernel", KERNELS)
def test_kernel_families_spiky_long(kernel):
    """Spiky keys (1% x8) over a few thousand keys: the precision case."""
    w = small(batch=2, prefix=(3000, 2500), num_drafts=8, num_heads=64, tree="chain",
              num_slots=8192, spike_frac=0.01, seed=160)
    check_full(W.make_inputs(w), kernel=kernel)


@pytest.mark.parametrize("T,H", [(1, 64), (2, 16), (4, 16), (8, 64), (16, 64), (3, 5), (32, 2)])
def test_shapes_T_H(T, H):
    w = small(num_drafts=T, num_heads=H, prefix=(130, 64), seed=200 + T * 7 + H)
    check_full(W.make_inputs(w))


@pytest.mark.parametrize("prefix", [(0, 1), (63, 64), (65, 127), (128, 0), (1000, 5)])
@pytest.mark.parametrize("ps", [1, 64])
def test_prefix_edges_and_page_sizes(prefix, ps):
    w = small(prefix=prefix, page_size=ps, tree="chain", seed=300 + sum(prefix) + ps)
    check_full(W.make_inputs(w))


@pytest.mark.parametrize("nsplit", [1, 2, 3, 5, 32])
def test_split_counts(nsplit):
    # 32 splits over ~7 key blocks leaves most splits empty: weight 0.
    w = small(prefix=(400, 33), seed=400 + nsplit)
    check_full(W.make_inputs(w), nsplit=nsplit)


@pytest.mark.parametrize("nsplit", [2, 7])
def test_split_merge_repeats_bit_for_bit(nsplit):
    """Split partials and their LSE combine are deterministic: calls in a row
    on one plan give the same bits, also after a call with a rejected request
    (whose NaN rows must not leak into the next call), and match the oracle."""
    import dataclasses
    raw = W.make_inputs(small(batch=3, prefix=(900, 300, 1500), seed=111))
    inp = G.to_cuda(raw)
    lens = inp.kv_lens.clone()
    lens[1] = 2                      # fewer rows than drafts: request 1 rejected
    bad = dataclasses.replace(inp, kv_lens=lens)
    with G.make_plan(inp, nsplit=nsplit) as plan:
        o0, l0 = G.run(plan, inp)
        for i in range(4):
            if i == 2:
                G.run(plan, bad)
                assert plan.get_error() & mb.DEV_BAD_LEN
            o, l = G.run(plan, inp)
            assert torch.equal(o, o0) and torch.equal(l, l0)
        assert plan.get_error() == 0
    ref_o, ref_l = G.oracle_full(raw)
    G.assert_parity(o0.float().cpu().numpy(), l0.cpu().numpy(), ref_o, ref_l)


@pytest.mark.parametrize("tree", ["chain", "star", "random"])
def test_tree_shapes(tree):
    w = small(num_drafts=16, num_heads=8, tree=tree, prefix=(200, 90), seed=500)
    check_full(W.make_inputs(w))


def test_ragged_small_batch():
    w = small(batch=5, prefix=(1, 700, 64, 0, 333), num_drafts=8, num_heads=16, seed=600)
    check_full(W.make_inputs(w))


def test_bf16_output_is_the_rounded_fp32_output():
    inp = G.to_cuda(W.make_inputs(small(seed=700)))
    for ns in (1, 3):
        with G.make_plan(inp, nsplit=ns) as p32, G.make_plan(inp, torch.bfloat16, nsplit=ns) as p16:
            o32, l32 = G.run(p32, inp)
            o16, l16 = G.run(p16, inp)
        assert torch.equal(o32.to(torch.bfloat16), o16)
        assert torch.equal(l32, l16)


def test_slot_permutation_gives_identical_bits():
    a = W.make_inputs(small(seed=800, num_slots=2048))
    perm = torch.randperm(2048, generator=torch.Generator().manual_seed(9))
    b_cache = torch.full_like(a.kv_cache, float("nan"))
    b_cache[perm] = a.kv_cache
    import dataclasses
    b = dataclasses.replace(a, kv_cache=b_cache, kv_indices=perm[a.kv_indices.long()].to(torch.int32))
    ga, gb = G.to_cuda(a), G.to_cuda(b)
    with G.make_plan(ga) as plan:
        oa, la = G.run(plan, ga)
        ob, lb = G.run(plan, gb)
    assert torch.equal(oa, ob) and torch.equal(la, lb)


def test_page_size_64_matches_page_size_1_bits():
    """Same logical rows through a page table and through a slot table."""
    a = W.make_inputs(small(seed=900, page_size=64, num_slots=4096))
    n = a.kv_lens.tolist()
    slots = []
    for bb in range(2):
        pages = a.kv_indices[a.kv_indptr[bb]:a.kv_indptr[bb + 1]].long()
        j = torch.arange(n[bb])
        slots.append(pages[j // 64] * 64 + j % 64)
    import dataclasses
    b = dataclasses.replace(
        a, page_size=1, kv_indices=torch.cat(slots).to(torch.int32),
        kv_indptr=torch.tensor([0, n[0], n[0] + n[1]], dtype=torch.int32))
    ga, gb = G.to_cuda(a), G.to_cuda(b)
    with G.make_plan(ga) as pa, G.make_plan(gb) as pb:
        oa, la = G.run(pa, ga)
        ob, lb = G.run(pb, gb)
    assert torch.equal(oa, ob) and torch.equal(la, lb)


# ------------------------------------------------------------ full size
FULL = ["decode_batch", "tree", "sweep_p1024", "sweep_p4096", "sweep_p16384", "sweep_p65536",
        "sweep_p93184", "ragged_ps1", "ragged_ps64", "decode_tp8", "decode_t1"]


def _log_errors(name, errs):
    """Append a workload's errors to $MLA_VERIFY_PARITY_LOG (JSON lines), if set."""
    path = os.environ.get("MLA_VERIFY_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"workload": name, "out_max_abs": errs[0], "out_mean_abs": errs[1],
                                "lse_max_abs": errs[2]}) + "\n")


@pytest.mark.parametrize("name", FULL)
def test_full_size_every_element(name):
    """Every output element of a full-size workload, in the launch
    configuration the benchmark times, against the fp64 oracle."""
    w = W.WORKLOADS[name]
    inp = W.make_inputs(w, device="cuda")
    with G.make_plan(inp) as plan:   # the automatic configuration the benchmark times
        out, lse = G.run(plan, inp)
        assert plan.get_error() == 0
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    del out, lse
    ref_o, ref_l = G.oracle_full(inp)
    errs = G.assert_parity(o, l, ref_o, ref_l, name)
    _log_errors(name, errs)
