"""fp64 CPU oracle for speculative-verify MLA attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path imports,
links or runs this package: only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference arm of ``bench.py`` use it.  It shares no code
with the CUDA path (no kernels, headers, helpers, tables or pre/post
processing); both sides only consume the same seeded inputs.

What it computes (the plain definition, evaluated without blocking or
splitting of the key axis):

  for request b with n_b = kv_lens[b] cached rows, of which the last T are
  the draft tokens' own rows (prefix length P_b = n_b - T), for draft t and
  head h:
      k_j      = cache row of logical key j (gathered through the slot or
                 page table), as fp64
      visible  = j < P_b, or j - P_b is t or an ancestor of t in the draft
                 tree given by draft_parent
      s_j      = scale * <q[b,t,h,:576], k_j[:576]>
      lse      = log sum_{visible j} exp(s_j)            (natural log)
      out      = sum_{visible j} exp(s_j - lse) * k_j[:512]

Sources: the verify step (drafter tokens attending to the target model's MLA
KV, scattered page_size=1 reads) is described in "The Decisive A/B: When
Benchmarking Honesty Reveals the Real Bottleneck", section "The Context"; the
tree-shaped drafts in "The Moment of Truth: Benchmarking a Custom sm_120
Verify Kernel Against Triton", section "The Raw Numbers" (the kdtree verify
switch).  The pages state no formula; the definition above is the plain
reading of MLA decode attention with absorbed queries (one shared latent KV
head, values = the 512 latent dims of each key row) plus a causal-prefix and
tree mask.

``index_builder_ref.build_indices`` restates the per-step index builder (the
request-to-token table turned into the slot or page table the attention
reads); its pins are in tests/test_index_builder_pins.py.
``shard_key_range``, ``mla_verify_key_range`` and ``lse_merge`` restate the
context-parallel split: one shard's partial over its keys and the reduce of
the shards' partials (pins: tests/test_context_parallel_pins.py).  ``compact_ref.compact_kv``
restates KV compaction into 64-row pages (pins: tests/test_compact_pins.py).

Pins (tests/test_oracle_pins.py): pure-Python brute force on tiny inputs, a
hand-derived closed-form fixture (tests/golden/), one-visible-key, identical
keys/scores, slot-permutation and page-size invariance, chain == causal,
star == prefix+self, scale invariance, split-and-combine == unsplit, and
NaN-sentinel isolation.
"""
from .mla_verify_ref import (  # noqa: F401
    bf16_bits_to_f64,
    ancestor_sets,
    gather_request_keys,
    mla_verify,
    mla_verify_rows,
    mla_verify_split_combine,
    shard_key_range,
    mla_verify_key_range,
    lse_merge,
)
