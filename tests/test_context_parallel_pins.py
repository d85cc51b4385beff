"""Pins of the context-parallel oracle functions (CPU only), and the exchange
step run by two gloo ranks.

``shard_key_range`` is checked against hand-worked ranges and for covering
every key exactly once; ``mla_verify_key_range`` against the pure-Python
brute force restricted to the same keys; ``lse_merge`` against a closed form;
and merging every shard's partial against the unsharded oracle.  The gloo
test runs ``context_parallel.run_sharded`` on two CPU ranks with oracle
partials, so the rank-to-shard mapping, the shard-major gather and the merge
are those a multi-GPU run uses.
"""
import math
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from oracle.brute import brute_verify
from paged_mla_speculative_gb300 import workloads as W
from tests.conftest import bits, oracle_args

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("n,S,expect", [
    (300, 1, [(0, 300)]),
    (300, 2, [(0, 128), (128, 300)]),                      # 3 blocks: 1 + 2
    (300, 4, [(0, 0), (0, 128), (128, 256), (256, 300)]),  # 3 blocks over 4 shards
    (256, 2, [(0, 128), (128, 256)]),
    (5, 3, [(0, 0), (0, 0), (0, 5)]),
    (1000, 3, [(0, 256), (256, 640), (640, 1000)]),        # 8 blocks: 2, 3, 3
])
def test_shard_ranges_by_hand(n, S, expect):
    assert [oracle.shard_key_range(n, s, S) for s in range(S)] == expect


def test_shards_cover_every_key_once():
    for n in (1, 2, 127, 128, 129, 1000, 4104, 93192):
        for S in (1, 2, 3, 5, 8, 32):
            cover = np.zeros(n, dtype=int)
            last = 0
            for s in range(S):
                lo, hi = oracle.shard_key_range(n, s, S)
                assert lo == last or lo == hi == last or lo >= last
                assert lo % 128 == 0 or lo == n
                cover[lo:hi] += 1
                last = max(last, hi)
            assert (cover == 1).all(), (n, S)


def _tiny(seed, prefix=(9, 5), tree="random", ps=1):
    w = W.Workload(name="cp", batch=2, num_drafts=3, num_heads=2, prefix=prefix, tree=tree,
                   num_slots=64, page_size=ps, spike_frac=0.2, seed=seed)
    return W.make_inputs(w)


@pytest.mark.parametrize("ranges", [
    [(0, 4), (2, 8)],       # prefix only / straddling the drafts
    [(9, 12), (0, 8)],      # the drafts only: rows whose ancestors lie outside see nothing
    [(3, 3), (5, 8)],       # an empty range
])
def test_key_range_partial_equals_brute_force(ranges):
    inp = _tiny(21)
    lo = [r[0] for r in ranges]
    hi = [r[1] for r in ranges]
    out, lse = oracle.mla_verify_key_range(*oracle_args(inp), lo, hi)
    bo, bl = brute_verify(bits(inp.q).astype(int).tolist(), bits(inp.kv_cache).astype(int).tolist(),
                          inp.kv_indices.tolist(), inp.kv_indptr.tolist(), inp.kv_lens.tolist(),
                          inp.draft_parent.tolist(), inp.scale, inp.page_size, key_ranges=ranges)
    bl = np.array(bl)
    np.testing.assert_array_equal(np.isinf(lse), np.isinf(bl))
    fin = np.isfinite(bl)
    np.testing.assert_allclose(lse[fin], bl[fin], rtol=0, atol=1e-12)
    np.testing.assert_allclose(out, np.array(bo), rtol=0, atol=1e-12)
    assert (out[np.isinf(lse)] == 0).all()


def test_lse_merge_closed_form():
    a = np.full((1, 512), 2.0)
    b = np.full((1, 512), -6.0)
    z = np.full((1, 512), 123.0)           # weight 0: never used
    parts_out = np.stack([a, b, z])
    parts_lse = np.array([[math.log(1.0)], [math.log(3.0)], [-np.inf]])
    out, lse = oracle.lse_merge(parts_out, parts_lse)
    np.testing.assert_allclose(out, (1.0 * a + 3.0 * b) / 4.0, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, [math.log(4.0)], rtol=0, atol=1e-15)
    out, lse = oracle.lse_merge(np.stack([z, z]), np.full((2, 1), -np.inf))
    assert (out == 0).all() and np.isneginf(lse).all()


@pytest.mark.parametrize("S", [1, 2, 3, 5])
@pytest.mark.parametrize("ps", [1, 64])
def test_merged_shards_equal_unsharded(S, ps):
    w = W.Workload(name="cp2", batch=3, num_drafts=4, num_heads=3, prefix=(700, 129, 0),
                   tree="random", num_slots=4096, page_size=ps, spike_frac=0.01, seed=31 + S)
    inp = W.make_inputs(w)
    args = oracle_args(inp)
    ref_o, ref_l = oracle.mla_verify(*args)
    lens = inp.kv_lens.tolist()
    po, pl = [], []
    for s in range(S):
        rng = [oracle.shard_key_range(n, s, S) for n in lens]
        o, l = oracle.mla_verify_key_range(*args, [r[0] for r in rng], [r[1] for r in rng])
        po.append(o)
        pl.append(l)
    out, lse = oracle.lse_merge(np.stack(po), np.stack(pl))
    np.testing.assert_allclose(out, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, rtol=0, atol=1e-12)


# ------------------------------------------------------------- two gloo ranks
def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _cp_rank(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    from paged_mla_speculative_gb300 import context_parallel as CP
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = W.Workload(name="cpg", batch=2, num_drafts=4, num_heads=2, prefix=(600, 140),
                       tree="random", num_slots=2048, spike_frac=0.01, seed=77)
        inp = W.make_inputs(w)
        args = oracle_args(inp)
        lens = inp.kv_lens.tolist()
        seen = {}

        def partial(shard, num_shards):
            seen["shard"] = (shard, num_shards)
            rng = [oracle.shard_key_range(n, shard, num_shards) for n in lens]
            o, l = oracle.mla_verify_key_range(*args, [r[0] for r in rng], [r[1] for r in rng])
            return torch.from_numpy(o), torch.from_numpy(l)

        def combine(parts_out, parts_lse):
            seen["parts"] = tuple(parts_out.shape)
            o, l = oracle.lse_merge(parts_out.numpy(), parts_lse.numpy())
            return torch.from_numpy(o), torch.from_numpy(l)

        out, lse = CP.run_sharded(partial, combine)
        ref_o, ref_l = oracle.mla_verify(*args)
        results[rank] = (seen["shard"], seen["parts"],
                         float(np.abs(out.numpy() - ref_o).max()),
                         float(np.abs(lse.numpy() - ref_l).max()))
    finally:
        dist.destroy_process_group()


def test_context_parallel_exchange_with_two_gloo_ranks():
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_cp_rank, args=(2, port, results), nprocs=2, join=True)
        res = dict(results)
    assert res[0][0] == (0, 2) and res[1][0] == (1, 2)
    for r in (0, 1):
        assert res[r][1] == (2, 2, 4, 2, 512)
        assert res[r][2] <= 1e-12 and res[r][3] <= 1e-12
