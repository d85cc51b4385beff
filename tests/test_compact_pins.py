"""Pins of the KV-compaction oracle (CPU only).

Compaction copies each request's scattered page_size 1 rows into fresh
64-row pages from a free list and returns the page_size 64 table of the
same requests.  Pinned here against a hand-derived case, and by round trips:
the attention oracle gathers bit-identical key rows (hence identical
results) from the compacted cache with the new page table as from the
source cache with the old slot table; planted mistakes must fail.
"""
import numpy as np
import pytest

import oracle.compact_ref as cr
import oracle.mla_verify_ref as ref
from paged_mla_speculative_gb300 import workloads as W
from tests.conftest import bits, oracle_args


def test_hand_derived_case():
    # Source cache: 200 slots, row s holds the value s in both of its columns.
    src = np.repeat(np.arange(200, dtype=np.int64)[:, None], 2, axis=1)
    dst = np.full((10 * 64, 2), -1, dtype=np.int64)
    # Request 0: 70 rows at slots 100..169 in reverse order; request 1: 5 rows
    # at slots 7, 3, 250 (outside the cache), 0, 199.
    idx = list(range(169, 99, -1)) + [7, 3, 250, 0, 199]
    ptr = [0, 70, 75]
    lens = [70, 5]
    out, table, pin, flags = cr.compact_kv(src, idx, ptr, lens, [3, 9, 4, 0], dst, 100)
    assert table == [3, 9, 4] and pin == [0, 2, 3]
    assert flags == cr.BAD_SLOT          # slot 250 is outside the 200-slot cache
    # request 0: rows 0..63 on page 3, rows 64..69 on page 9
    assert np.array_equal(out[3 * 64:4 * 64, 0], np.arange(169, 105, -1))
    assert np.array_equal(out[9 * 64:9 * 64 + 6, 0], np.arange(105, 99, -1))
    assert (out[9 * 64 + 6:10 * 64] == -1).all()          # rest of the last page untouched
    # request 1 on page 4: 7, 3, zeros for the bad slot, 0, 199
    assert out[4 * 64:4 * 64 + 5, 0].tolist() == [7, 3, 0, 0, 199]
    # untouched pages
    assert (out[:3 * 64] == -1).all() and (out[5 * 64:9 * 64] == -1).all()
    # capacity: with 2 free pages only request 0 keeps its pages
    out2, table2, pin2, flags2 = cr.compact_kv(src, idx, ptr, lens, [3, 9], dst, 100)
    assert table2 == [3, 9] and pin2 == [0, 2, 2] and flags2 == cr.CAPACITY
    # a length beyond max_kv_len: that request gets no pages
    _, t3, p3, f3 = cr.compact_kv(src, idx, ptr, lens, [3, 9, 4], dst, 69)
    assert p3 == [0, 0, 1] and t3 == [3] and f3 == cr.BAD_LEN | cr.BAD_SLOT


def compacted_workload(seed, page_shuffle=True):
    w = W.Workload(name="cp", batch=3, num_drafts=4, num_heads=2, prefix=(300, 60, 129),
                   tree="random", num_slots=2048, spike_frac=0.01, seed=seed)
    inp = W.make_inputs(w)
    src = bits(inp.kv_cache)
    n_pages = 40
    rng = np.random.default_rng(seed)
    free = rng.permutation(n_pages) if page_shuffle else np.arange(n_pages)
    dst = np.full((n_pages * 64, src.shape[1]), 0x7FC0, dtype=src.dtype)
    out, table, pin, flags = cr.compact_kv(src, inp.kv_indices.tolist(), inp.kv_indptr.tolist(),
                                           inp.kv_lens.tolist(), free.tolist(), dst,
                                           int(inp.kv_lens.max()))
    return inp, src, out, table, pin, flags


@pytest.mark.parametrize("seed", [1, 2])
def test_compacted_pages_gather_the_same_rows(seed):
    inp, src, out, table, pin, flags = compacted_workload(seed)
    assert flags == 0
    for b in range(3):
        n = int(inp.kv_lens[b])
        a = ref.gather_request_keys(src, inp.kv_indices.numpy(), inp.kv_indptr.numpy(), b, n, 1)
        c = ref.gather_request_keys(out, np.array(table), np.array(pin), b, n, 64)
        assert np.array_equal(a, c)


def test_attention_on_compacted_cache_is_identical():
    inp, src, out, table, pin, flags = compacted_workload(3)
    q, kv, idx, ptr, lens, par, scale, ps = oracle_args(inp)
    o1, l1 = ref.mla_verify(q, kv, idx, ptr, lens, par, scale, 1)
    o2, l2 = ref.mla_verify(q, out, np.array(table), np.array(pin), lens, par, scale, 64)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


_orig = cr.compact_kv


def _floor_pages(src, idx, ptr, lens, free, dst, mx):
    # a plausible slip: one page too few when n is not a multiple of 64
    return _orig(src, idx, ptr, [(n // 64) * 64 for n in lens], free, dst, mx)


def _row_offset(src, idx, ptr, lens, free, dst, mx):
    out, t, p, f = _orig(src, idx, ptr, lens, free, dst, mx)
    return np.roll(out, 1, axis=0), t, p, f


def _reuse_first_page(src, idx, ptr, lens, free, dst, mx):
    return _orig(src, idx, ptr, lens, [free[0]] * len(free), dst, mx)


@pytest.mark.parametrize("fn", [_floor_pages, _row_offset, _reuse_first_page],
                         ids=["page count floored", "rows off by one", "one page reused"])
def test_planted_mistakes_are_caught(fn, monkeypatch):
    monkeypatch.setattr(cr, "compact_kv", fn)
    caught = False
    try:
        test_hand_derived_case()
        for seed in (1, 2):
            test_compacted_pages_gather_the_same_rows(seed)
    except AssertionError:
        caught = True
    assert caught
