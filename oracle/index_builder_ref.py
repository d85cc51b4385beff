"""Plain reference for the per-step index builder (the "marshaling" step).

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

The pages trace the custom verify kernel's short-context loss to host-side
marshaling: index arrays rebuilt in Python for every layer, and name two
remedies, building the combined indices once per step, or moving that work
into a kernel on the GPU ("The Moment of Truth: Benchmarking a Custom sm_120
Verify Kernel Against Triton", sections "Interpreting the Crossover: The
Marshaling Tax" and "Assumptions and Their Validity").  The pages give no
layout; the reading used here is the serving stack's request-to-token table:

  req_to_token[pool, j] = cache slot of token position j of the request
                          held in pool row `pool`;
  a verify step for request b (pool row req_pool_indices[b], prefix length
  prefix_lens[b]) reads positions 0 .. prefix_lens[b] + T - 1, the last T of
  them being the draft tokens' own rows.

What the builder returns for a batch (written out sequentially below, one
request at a time):

  kv_lens[b]    = prefix_lens[b] + T, or 0 when the request is invalid: pool
                  row outside [0, pool_size), negative prefix, or more than
                  max_kv_len rows (flag BAD_POOL);
  count[b]      = kv_lens[b] table entries (page_size 1) or ceil(kv_lens[b]/64)
                  page ids (page_size 64);
  kv_indptr     = exclusive prefix sum of count;
  capacity      : the longest leading run of requests whose entries fit in
                  `capacity` keeps its entries; every later request gets
                  kv_lens = 0 and no entries (flag CAPACITY);
  kv_indices    = page_size 1: req_to_token[pool, 0 .. n-1];
                  page_size 64: req_to_token[pool, 64 i] // 64 for page i --
                  a whole page holds 64 consecutive slots starting at a
                  multiple of 64, so its first slot names it; a first slot
                  that is negative or not a multiple of 64 gives page id -1
                  (flag BAD_SLOT).

The flags are the library's device status bits of the same names.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

import numpy as np

PAGE = 64

BAD_SLOT = 1
BAD_POOL = 64
CAPACITY = 128


def build_indices(req_to_token: np.ndarray, req_pool_indices: Sequence[int],
                  prefix_lens: Sequence[int], T: int, page_size: int, max_kv_len: int,
                  capacity: int) -> Tuple[List[int], List[int], List[int], int]:
    """Return (kv_lens, kv_indptr, kv_indices, flags) for one verify step."""
    table = np.asarray(req_to_token)
    pool_size = table.shape[0]
    B = len(req_pool_indices)
    flags = 0
    kv_lens: List[int] = []
    counts: List[int] = []
    for b in range(B):
        pool = int(req_pool_indices[b])
        n = int(prefix_lens[b]) + T
        valid = 0 <= pool < pool_size and int(prefix_lens[b]) >= 0 and n <= max_kv_len
        if not valid:
            flags |= BAD_POOL
            kv_lens.append(0)
            counts.append(0)
            continue
        kv_lens.append(n)
        counts.append(n if page_size == 1 else (n + PAGE - 1) // PAGE)

    # Longest leading run of requests whose entries fit.
    kept = B
    running = 0
    for b in range(B):
        if running + counts[b] > capacity:
            kept = b
            break
        running += counts[b]
    for b in range(kept, B):
        if counts[b] > 0:
            flags |= CAPACITY
        kv_lens[b] = 0
        counts[b] = 0

    kv_indptr = [0]
    for b in range(B):
        kv_indptr.append(kv_indptr[-1] + counts[b])

    kv_indices: List[int] = []
    for b in range(B):
        if counts[b] == 0:
            continue
        row = table[int(req_pool_indices[b])]
        if page_size == 1:
            kv_indices.extend(int(x) for x in row[:counts[b]])
        else:
            for i in range(counts[b]):
                first = int(row[PAGE * i])
                if first >= 0 and first % PAGE == 0:
                    kv_indices.append(first // PAGE)
                else:
                    flags |= BAD_SLOT
                    kv_indices.append(-1)
    return kv_lens, kv_indptr, kv_indices, flags
