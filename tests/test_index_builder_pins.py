"""Pins of the index-builder oracle (CPU only).

The builder turns the serving stack's request-to-token table into the slot
or page table the verify attention reads (the "marshaling" step, once per
step on the GPU).  Pinned here against: hand-derived cases in
tests/golden/index_builder_cases.json, the output invariants, and round trips
through the seeded workloads' own index arrays and the attention oracle's
gather; planted mistakes must fail them.
"""
import json
import os

import numpy as np
import pytest

import oracle.index_builder_ref as ib
import oracle.mla_verify_ref as ref
from paged_mla_speculative_gb300 import workloads as W
from tests.conftest import bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "index_builder_cases.json")


def table_from_runs(rows, pool_size, stride):
    t = np.full((pool_size, stride), -1, dtype=np.int64)
    for r, runs in enumerate(rows):
        for pos, slot, n in runs:
            t[r, pos:pos + n] = np.arange(slot, slot + n)
    return t


def golden_cases():
    with open(GOLDEN) as f:
        g = json.load(f)
    for case in g["cases"]:
        for run in case["runs"]:
            yield case, run


@pytest.mark.parametrize("case,run", list(golden_cases()),
                         ids=lambda x: x.get("name", str(x.get("capacity", ""))))
def test_hand_derived_cases(case, run):
    table = table_from_runs(case["rows"], case["pool_size"], case["stride"])
    lens, indptr, idx, flags = ib.build_indices(table, case["req_pool_indices"], case["prefix_lens"],
                                                case["T"], case["page_size"], case["max_kv_len"],
                                                run["capacity"])
    assert lens == run["kv_lens"]
    assert indptr == run["kv_indptr"]
    assert idx == run["kv_indices"]
    assert flags == run["flags"]


def workload_table(inp):
    """A request-to-token table holding each request's logical slots, pool
    rows in a shuffled order, plus the step's pool indices and prefixes."""
    w = inp.workload
    idx, ptr, lens = inp.kv_indices.numpy(), inp.kv_indptr.numpy(), inp.kv_lens.numpy()
    stride = int(lens.max()) + 7
    pool_size = w.batch + 3
    perm = np.random.default_rng(w.seed + 17).permutation(pool_size)[:w.batch]
    table = np.full((pool_size, stride), -1, dtype=np.int64)
    for b in range(w.batch):
        n = int(lens[b])
        if inp.page_size == 1:
            slots = idx[ptr[b]:ptr[b] + n]
        else:
            pages = idx[ptr[b]:ptr[b + 1]]
            slots = (pages[:, None] * 64 + np.arange(64)[None, :]).reshape(-1)[:n]
        table[perm[b], :n] = slots
    return table, perm, lens - w.num_drafts


@pytest.mark.parametrize("ps", [1, 64])
def test_round_trip_of_a_workload_index_table(ps):
    w = W.Workload(name="ib", batch=5, num_drafts=4, num_heads=2, prefix=(0, 63, 64, 300, 129),
                   tree="random", num_slots=8192, page_size=ps, seed=41)
    inp = W.make_inputs(w)
    table, pools, prefix = workload_table(inp)
    lens, indptr, idx, flags = ib.build_indices(table, pools, prefix, w.num_drafts, ps,
                                                int(inp.kv_lens.max()), 10 ** 9)
    assert flags == 0
    assert lens == inp.kv_lens.tolist()
    assert indptr == inp.kv_indptr.tolist()
    assert idx == inp.kv_indices.tolist()


def test_page_and_slot_tables_gather_the_same_rows():
    """Built from one page-aligned table, the page_size 64 and page_size 1
    index arrays make the attention oracle gather identical key rows."""
    w = W.Workload(name="ib2", batch=3, num_drafts=8, num_heads=2, prefix=(120, 7, 250),
                   tree="chain", num_slots=4096, page_size=64, seed=43)
    inp = W.make_inputs(w)
    table, pools, prefix = workload_table(inp)
    cache = bits(inp.kv_cache)
    mx = int(inp.kv_lens.max())
    l1, p1, i1, f1 = ib.build_indices(table, pools, prefix, 8, 1, mx, 10 ** 9)
    l64, p64, i64, f64 = ib.build_indices(table, pools, prefix, 8, 64, mx, 10 ** 9)
    assert f1 == 0 and f64 == 0 and l1 == l64
    for b in range(w.batch):
        a = ref.gather_request_keys(cache, np.array(i1), np.array(p1), b, l1[b], 1)
        c = ref.gather_request_keys(cache, np.array(i64), np.array(p64), b, l64[b], 64)
        assert np.array_equal(a, c)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_output_invariants_on_random_steps(seed):
    rng = np.random.default_rng(seed)
    pool_size, stride, T = 12, 300, 3
    table = rng.integers(0, 10 ** 6, size=(pool_size, stride))
    B = 9
    pools = rng.integers(-2, pool_size + 2, size=B)
    prefix = rng.integers(-3, stride, size=B)
    for ps in (1, 64):
        for cap in (0, 50, 400, 10 ** 6):
            lens, indptr, idx, flags = ib.build_indices(table, pools, prefix, T, ps, stride, cap)
            assert indptr[0] == 0 and all(a <= b for a, b in zip(indptr, indptr[1:]))
            assert indptr[-1] == len(idx) <= cap
            for b in range(B):
                n = lens[b]
                want = 0 if n == 0 else (n if ps == 1 else -(-n // 64))
                assert indptr[b + 1] - indptr[b] == want
                assert n == 0 or T <= n <= stride


def _mutated(monkeypatch, fn):
    monkeypatch.setattr(ib, "build_indices", fn)


def _pins_fail():
    try:
        for case, run in golden_cases():
            test_hand_derived_cases(case, run)
        test_round_trip_of_a_workload_index_table(64)
    except AssertionError:
        return True
    return False


_orig = ib.build_indices


def _floor_pages(table, pools, prefix, T, ps, mx, cap):
    lens, indptr, idx, flags = _orig(table, pools, prefix, T, ps, mx, cap)
    if ps == 64:   # a plausible slip: floor instead of ceil for the page count
        counts = [n // 64 for n in lens]
        indptr = [0]
        for c in counts:
            indptr.append(indptr[-1] + c)
    return lens, indptr, idx, flags


def _no_drafts(table, pools, prefix, T, ps, mx, cap):
    return _orig(table, pools, prefix, 0, ps, mx, cap)   # forgets the draft rows


def _inclusive_indptr(table, pools, prefix, T, ps, mx, cap):
    lens, indptr, idx, flags = _orig(table, pools, prefix, T, ps, mx, cap)
    return lens, indptr[1:] + [indptr[-1]], idx, flags


@pytest.mark.parametrize("fn", [_floor_pages, _no_drafts, _inclusive_indptr],
                         ids=["floor page count", "draft rows left out", "inclusive prefix sum"])
def test_planted_mistakes_are_caught(fn, monkeypatch):
    monkeypatch.setattr(ib, "build_indices", fn)
    assert _pins_fail()
