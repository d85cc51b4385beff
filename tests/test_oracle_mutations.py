"""Planted mistakes in the oracle must be caught by its pins (CPU only).

Each case replaces one piece of the oracle with a plausibly wrong version
(dropped scale, wrong value dims, a draft not seeing itself, the prefix-only
mask, a base-2 LSE, a shifted page gather, a parent walk that skips links)
and checks that the brute-force comparison or the closed-form fixture then
fails.  The mistakes are planted in the oracle only, never in the GPU path.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import oracle.mla_verify_ref as ref
from oracle.brute import brute_verify
from paged_mla_speculative_gb300 import workloads as W
from tests.conftest import bits, oracle_args
from tests.test_oracle_pins import _golden_inputs, GOLDEN


def _pins_detect():
    """True if any pin fails with the (possibly mutated) oracle."""
    try:
        for ps, tree, prefix, seed in [(1, "random", (4, 7), 11), (1, "chain", (0, 3), 12),
                                       (4, "random", (5, 2), 13), (1, "star", (6, 1), 14)]:
            w = W.Workload(name="m", batch=2, num_drafts=3, num_heads=2, prefix=prefix, tree=tree,
                           num_slots=64, page_size=ps, spike_frac=0.2, seed=seed)
            inp = W.make_inputs(w)
            out, lse = ref.mla_verify(*oracle_args(inp))
            bo, bl = brute_verify(bits(inp.q).astype(int).tolist(), bits(inp.kv_cache).astype(int).tolist(),
                                  inp.kv_indices.tolist(), inp.kv_indptr.tolist(), inp.kv_lens.tolist(),
                                  inp.draft_parent.tolist(), inp.scale, ps)
            np.testing.assert_allclose(out, np.array(bo), rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse, np.array(bl), rtol=0, atol=1e-12)
        with open(os.path.join(GOLDEN, "closed_form_tree.json")) as f:
            g = json.load(f)
        out, lse = ref.mla_verify(*_golden_inputs(g))
        hd = g["hand_derived"]
        for t, vis in enumerate(hd["visible_keys_per_draft"]):
            z = sum(math.exp(hd["head0_scores"][j]) for j in vis)
            assert abs(lse[0, t, 0] - math.log(z)) < 1e-13
    except AssertionError:
        return True
    return False


def test_unmutated_oracle_passes_its_pins():
    assert not _pins_detect()


def _attend_no_scale(qrows, keys, vis, scale):
    return _orig_attend(qrows, keys, vis, 1.0)


def _attend_wrong_value_dims(qrows, keys, vis, scale):
    shifted = np.concatenate([keys[:, 64:], keys[:, :64]], axis=1)   # values from dims 64..575
    out, lse = _orig_attend(qrows, keys, vis, scale)
    kv = keys[vis]
    s = scale * (qrows @ kv.T)
    e = np.exp(s - lse[:, None])
    return e @ shifted[vis][:, :512], lse


def _attend_log2(qrows, keys, vis, scale):
    out, lse = _orig_attend(qrows, keys, vis, scale)
    return out, lse / math.log(2.0)


def _ancestors_without_self(parent):
    return [s - {t} for t, s in enumerate(_orig_ancestors(parent))]


def _ancestors_prefix_only(parent):
    return [set() for _ in parent]


def _ancestors_parent_only(parent):
    return [{t} | ({int(parent[t])} if parent[t] >= 0 else set()) for t in range(len(parent))]


def _gather_shifted_page(kv_cache, kv_indices, kv_indptr, b, n, page_size):
    if page_size == 1:
        return _orig_gather(kv_cache, kv_indices, kv_indptr, b, n, page_size)
    rows = _orig_gather(kv_cache, kv_indices, kv_indptr, b, n, page_size)
    return np.roll(rows, 1, axis=0)


_orig_attend = ref._attend
_orig_ancestors = ref.ancestor_sets
_orig_gather = ref.gather_request_keys

MUTATIONS = {
    "dropped scale": ("_attend", _attend_no_scale),
    "values from the wrong dims": ("_attend", _attend_wrong_value_dims),
    "base-2 lse": ("_attend", _attend_log2),
    "draft does not see itself": ("ancestor_sets", _ancestors_without_self),
    "drafts see only the prefix": ("ancestor_sets", _ancestors_prefix_only),
    "only the direct parent is visible": ("ancestor_sets", _ancestors_parent_only),
    "page gather off by one row": ("gather_request_keys", _gather_shifted_page),
}


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(ref, attr, fn)
    assert _pins_detect(), f"pins missed: {name}"
