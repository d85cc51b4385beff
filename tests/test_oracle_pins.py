"""Pins of the fp64 oracle against things other than itself (CPU only).

Each test fixes the oracle to brute force, a closed form, or an invariant of
the definition, so that a dropped term, a wrong sign or index, or a
transposed operand in the oracle fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle.brute import brute_verify
from paged_mla_speculative_gb300 import workloads as W
from tests.conftest import bits, oracle_args

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def small(name="t", **kw):
    base = dict(name=name, batch=2, num_drafts=3, num_heads=2, prefix=(4, 7),
                tree="random", num_slots=64, seed=11)
    base.update(kw)
    return W.Workload(**base)


# ---------------------------------------------------------------- brute force
@pytest.mark.parametrize("ps,tree,prefix,seed", [
    (1, "random", (4, 7), 11),
    (1, "chain", (0, 3), 12),
    (4, "random", (5, 2), 13),
    (1, "star", (6, 1), 14),
])
def test_oracle_equals_brute_force(ps, tree, prefix, seed):
    w = small(page_size=ps, tree=tree, prefix=prefix, seed=seed, spike_frac=0.2)
    inp = W.make_inputs(w)
    out, lse = oracle.mla_verify(*oracle_args(inp))
    qb = bits(inp.q).astype(int).tolist()
    cb = bits(inp.kv_cache).astype(int).tolist()
    bo, bl = brute_verify(qb, cb, inp.kv_indices.tolist(), inp.kv_indptr.tolist(),
                          inp.kv_lens.tolist(), inp.draft_parent.tolist(),
                          inp.scale, ps)
    np.testing.assert_allclose(out, np.array(bo), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(bl), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- closed form
def _golden_inputs(g):
    B, T, H, P = g["batch"], g["num_drafts"], g["num_heads"], g["prefix_len"]
    n = P + T
    q = torch.zeros((B, T, H, W.D_QK), dtype=torch.bfloat16)
    q[:, :, 0, 0] = g["q_head0"]["dim0"]
    q[:, :, 0, 512] = g["q_head0"]["dim512"]
    cache = torch.full((g["num_slots"], W.D_QK), float("nan"), dtype=torch.bfloat16)
    for j, slot in enumerate(g["slots_of_keys"]):
        row = torch.zeros(W.D_QK)
        row[0] = g["key_dim0"][j]
        row[1] = j + 1
        row[2] = (-1) ** j
        row[512] = g["key_dim512"]
        cache[slot] = row.to(torch.bfloat16)
    idx = np.array(g["slots_of_keys"], dtype=np.int32)
    return (bits(q), bits(cache), idx, np.array([0, n], np.int32),
            np.array([n], np.int32), np.array([g["draft_parent"]], np.int32),
            g["scale"], g["page_size"])


def test_oracle_closed_form_golden():
    with open(os.path.join(GOLDEN, "closed_form_tree.json")) as f:
        g = json.load(f)
    out, lse = oracle.mla_verify(*_golden_inputs(g))
    hd = g["hand_derived"]
    for t, vis in enumerate(hd["visible_keys_per_draft"]):
        for h, scores in ((0, hd["head0_scores"]), (1, hd["head1_scores"])):
            e = [math.exp(scores[j]) for j in vis]
            z = sum(e)
            want = np.zeros(512)
            for ej, j in zip(e, vis):
                want[0] += ej / z * g["key_dim0"][j]
                want[1] += ej / z * (j + 1)
                want[2] += ej / z * (-1) ** j
            np.testing.assert_allclose(out[0, t, h], want, rtol=0, atol=1e-13)
            assert abs(lse[0, t, h] - math.log(z)) < 1e-13
    # head 1 (q = 0): uniform weights, lse = log(#visible)
    for t, vis in enumerate(hd["visible_keys_per_draft"]):
        assert abs(lse[0, t, 1] - math.log(len(vis))) < 1e-13
        assert abs(out[0, t, 1, 1] - np.mean([j + 1 for j in vis])) < 1e-13


# ---------------------------------------------------------- special cases
def test_one_visible_key_returns_its_value_exactly():
    # P = 0, chain: draft 0 sees only its own key.
    w = small(prefix=(0, 0), tree="chain", spike_frac=0.0)
    inp = W.make_inputs(w)
    out, lse = oracle.mla_verify(*oracle_args(inp))
    keys = oracle.gather_request_keys(bits(inp.kv_cache), inp.kv_indices.numpy(),
                                      inp.kv_indptr.numpy(), 0, 3, 1)
    q0 = oracle.bf16_bits_to_f64(bits(inp.q))[0, 0]
    assert np.array_equal(out[0, 0], np.broadcast_to(keys[0, :512], (2, 512)))
    np.testing.assert_allclose(lse[0, 0], inp.scale * q0 @ keys[0], rtol=0, atol=1e-12)


def test_identical_keys_give_that_value():
    w = small(spike_frac=0.0)
    inp = W.make_inputs(w)
    row = inp.kv_cache[inp.kv_indices[0].item()].clone()
    live = inp.kv_indices.long()
    inp.kv_cache[live] = row
    out, lse = oracle.mla_verify(*oracle_args(inp))
    v = oracle.bf16_bits_to_f64(bits(row))
    np.testing.assert_allclose(out, np.broadcast_to(v[:512], out.shape), rtol=0, atol=1e-12)
    qf = oracle.bf16_bits_to_f64(bits(inp.q))
    anc = [oracle.ancestor_sets(p) for p in inp.draft_parent.tolist()]
    for b in range(2):
        for t in range(3):
            nvis = inp.prefix[b] + len(anc[b][t])
            s = inp.scale * qf[b, t] @ v
            np.testing.assert_allclose(lse[b, t], s + math.log(nvis), rtol=0, atol=1e-12)


def test_equal_scores_give_mean_of_visible_values():
    w = small(spike_frac=0.0, tree="random", seed=21)
    inp = W.make_inputs(w)
    inp.q.zero_()
    out, lse = oracle.mla_verify(*oracle_args(inp))
    anc = [oracle.ancestor_sets(p) for p in inp.draft_parent.tolist()]
    for b in range(2):
        P = inp.prefix[b]
        keys = oracle.gather_request_keys(bits(inp.kv_cache), inp.kv_indices.numpy(),
                                          inp.kv_indptr.numpy(), b, P + 3, 1)
        for t in range(3):
            vis = list(range(P)) + [P + i for i in sorted(anc[b][t])]
            mean = keys[vis, :512].mean(axis=0)
            np.testing.assert_allclose(out[b, t], np.broadcast_to(mean, (2, 512)), atol=1e-12)
            np.testing.assert_allclose(lse[b, t], math.log(len(vis)), atol=1e-13)


# ---------------------------------------------------------------- invariants
def test_slot_placement_and_page_size_do_not_matter():
    w1 = small(page_size=1, seed=31, spike_frac=0.2, num_slots=256)
    a = W.make_inputs(w1)
    o1, l1 = oracle.mla_verify(*oracle_args(a))
    # Same logical rows, moved into 64-row pages of a different cache.
    P = a.prefix
    n = [p + 3 for p in P]
    cache = torch.full((512, W.D_QK), float("nan"), dtype=torch.bfloat16)
    pages = [[5, 2], [7, 0]]
    idx, rows = [], []
    for b in range(2):
        keys_slots = a.kv_indices[a.kv_indptr[b]:a.kv_indptr[b + 1]].long()
        for j in range(n[b]):
            cache[pages[b][j // 64] * 64 + j % 64] = a.kv_cache[keys_slots[j]]
        idx += pages[b][: -(-n[b] // 64)]
    indptr = np.array([0, 1, 2], np.int32)
    o2, l2 = oracle.mla_verify(bits(a.q), bits(cache), np.array(idx, np.int32), indptr,
                               a.kv_lens.numpy(), a.draft_parent.numpy(), a.scale, 64)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # A second random slot permutation of the same rows.
    perm = torch.randperm(256, generator=torch.Generator().manual_seed(5))
    cache3 = torch.full_like(a.kv_cache, float("nan"))
    cache3[perm] = a.kv_cache
    idx3 = perm[a.kv_indices.long()].to(torch.int32).numpy()
    o3, l3 = oracle.mla_verify(bits(a.q), bits(cache3), idx3, a.kv_indptr.numpy(),
                               a.kv_lens.numpy(), a.draft_parent.numpy(), a.scale, 1)
    assert np.array_equal(o1, o3) and np.array_equal(l1, l3)


def _single_draft_request(inp, b, keys_logical):
    """A T=1 request whose keys are the listed logical keys of request b;
    the last one plays the draft (parent -1)."""
    sl = inp.kv_indices[inp.kv_indptr[b]:inp.kv_indptr[b + 1]].numpy()
    idx = sl[np.array(keys_logical)]
    n = len(keys_logical)
    return idx.astype(np.int32), np.array([0, n], np.int32), np.array([n], np.int32)


@pytest.mark.parametrize("tree", ["chain", "star"])
def test_chain_is_causal_and_star_is_prefix_plus_self(tree):
    w = small(tree=tree, seed=41, spike_frac=0.2, num_drafts=4, prefix=(5, 9))
    inp = W.make_inputs(w)
    out, lse = oracle.mla_verify(*oracle_args(inp))
    qb = bits(inp.q)
    for b in range(2):
        P = inp.prefix[b]
        for t in range(4):
            if tree == "chain":       # key j visible iff j <= P + t
                keys = list(range(P + t + 1))
            else:                     # prefix plus the draft's own key
                keys = list(range(P)) + [P + t]
            idx, indptr, lens = _single_draft_request(inp, b, keys)
            o, l = oracle.mla_verify(qb[b:b + 1, t:t + 1], bits(inp.kv_cache), idx, indptr,
                                     lens, np.array([[-1]], np.int32), inp.scale, 1)
            np.testing.assert_allclose(out[b, t], o[0, 0], rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[b, t], l[0, 0], rtol=0, atol=1e-12)


def test_scale_invariance():
    w = small(seed=51, spike_frac=0.2)
    inp = W.make_inputs(w)
    o1, l1 = oracle.mla_verify(*oracle_args(inp))
    args = list(oracle_args(inp))
    args[0] = bits((inp.q.float() * 4).to(torch.bfloat16))   # exact: power of two
    args[6] = inp.scale / 4
    o2, l2 = oracle.mla_verify(*args)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


@pytest.mark.parametrize("nsplit", [1, 2, 3, 7])
def test_split_and_combine_equals_unsplit(nsplit):
    w = small(seed=61, spike_frac=0.2, prefix=(20, 3), num_drafts=4)
    inp = W.make_inputs(w)
    o1, l1 = oracle.mla_verify(*oracle_args(inp))
    o2, l2 = oracle.mla_verify_split_combine(*oracle_args(inp), nsplit=nsplit)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


def test_rows_subset_matches_whole_batch():
    w = small(seed=71, spike_frac=0.2)
    inp = W.make_inputs(w)
    o, l = oracle.mla_verify(*oracle_args(inp))
    rows = [(0, 2, 1), (1, 0, 0), (1, 2, 1)]
    o2, l2 = oracle.mla_verify_rows(rows, *oracle_args(inp))
    for i, (b, t, h) in enumerate(rows):
        np.testing.assert_allclose(o2[i], o[b, t, h], rtol=0, atol=1e-12)
        assert abs(l2[i] - l[b, t, h]) < 1e-12


def test_nan_sentinels_never_reach_output():
    inp = W.make_inputs(W.WORKLOADS["tiny"])
    assert torch.isnan(inp.kv_cache.float()).any()    # unused slots are NaN
    out, lse = oracle.mla_verify(*oracle_args(inp))
    assert np.isfinite(out).all() and np.isfinite(lse).all()


def test_bf16_widening_is_exact():
    x = torch.randn(1000).to(torch.bfloat16)
    assert np.array_equal(oracle.bf16_bits_to_f64(bits(x)), x.double().numpy())


# ---------------------------------------------------------- input generator
def test_random_tree_respects_depth_and_order():
    w = small(num_drafts=16, tree="random", batch=8, prefix=(1,) * 8, max_depth=6,
              num_slots=256, seed=3)
    par = W.draft_parents(w, torch.Generator().manual_seed(3))
    for p in par:
        depth = []
        for i, pi in enumerate(p):
            assert -1 <= pi < i
            depth.append(1 if pi < 0 else depth[pi] + 1)
        assert max(depth) <= 6


def test_generator_slots_disjoint_and_spikes_exact():
    w = small(num_slots=64, spike_frac=0.25, seed=81)
    inp = W.make_inputs(w)
    idx = inp.kv_indices.tolist()
    assert len(set(idx)) == len(idx)
    used = torch.zeros(64, dtype=torch.bool)
    used[inp.kv_indices.long()] = True
    assert torch.isnan(inp.kv_cache[~used].float()).all()
    assert torch.isfinite(inp.kv_cache[used].float()).all()
