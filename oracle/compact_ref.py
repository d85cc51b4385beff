"""Plain reference for KV compaction into 64-row pages.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

The pages name KV defragmentation as a next step after the custom verify
kernel ("The Moment of Truth: Benchmarking a Custom sm_120 Verify Kernel
Against Triton", section "The Broader Context: From Kernel to System"), the
problem being the page_size=1 layout that scatters every KV access ("The
Decisive A/B: When Benchmarking Honesty Reveals the Real Bottleneck", section
"The Context").  They give no procedure; the reading used here:

  for each request b of the call, in order, with n_b = kv_lens[b] rows whose
  slots are kv_indices[kv_indptr[b] .. kv_indptr[b] + n_b - 1] (page_size 1):
    pages_b     = the next ceil(n_b / 64) entries of `free_pages`;
    row j of b  is copied to slot pages_b[j // 64] * 64 + j % 64 of kv_dst;
  page_indptr   = exclusive prefix sum of the page counts, page_table = the
                  consumed prefix of free_pages -- together the page_size 64
                  table of the same requests (kv_lens unchanged);
  the remaining rows of a request's last page are left as they were.

Failures never stop the call, they set flags (the library's device status
bits of the same names):
  a request whose length is outside [0, max_kv_len] or whose indptr range
  does not hold n_b slots gets no pages (BAD_LEN / BAD_INDPTR);
  when the free list runs out, the longest leading run of requests whose
  pages fit keeps them and every later request gets none (CAPACITY);
  a source slot outside the source cache is copied as zeros, a destination
  page outside the destination cache is not written (BAD_SLOT).
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

import numpy as np

PAGE = 64

BAD_SLOT = 1
BAD_LEN = 2
BAD_INDPTR = 8
CAPACITY = 128


def compact_kv(kv_src: np.ndarray, kv_indices: Sequence[int], kv_indptr: Sequence[int],
               kv_lens: Sequence[int], free_pages: Sequence[int], kv_dst: np.ndarray,
               max_kv_len: int) -> Tuple[np.ndarray, List[int], List[int], int]:
    """Return (kv_dst after the copies, page_table, page_indptr, flags).

    kv_src / kv_dst are [slots, row] arrays of any dtype (rows are copied
    exactly); kv_dst is not modified in place.
    """
    src = np.asarray(kv_src)
    dst = np.array(kv_dst, copy=True)
    B = len(kv_lens)
    flags = 0
    counts: List[int] = []
    for b in range(B):
        n = int(kv_lens[b])
        if n < 0 or n > max_kv_len:
            flags |= BAD_LEN
            counts.append(0)
            continue
        if int(kv_indptr[b + 1]) - int(kv_indptr[b]) != n or int(kv_indptr[b]) < 0:
            flags |= BAD_INDPTR
            counts.append(0)
            continue
        counts.append((n + PAGE - 1) // PAGE)

    kept = B
    running = 0
    for b in range(B):
        if running + counts[b] > len(free_pages):
            kept = b
            break
        running += counts[b]
    for b in range(kept, B):
        if counts[b] > 0:
            flags |= CAPACITY
        counts[b] = 0

    page_indptr = [0]
    for b in range(B):
        page_indptr.append(page_indptr[-1] + counts[b])
    page_table = [int(x) for x in free_pages[:page_indptr[-1]]]

    src_slots, dst_pages = src.shape[0], dst.shape[0] // PAGE
    for b in range(B):
        if counts[b] == 0:
            continue
        n = int(kv_lens[b])
        for j in range(n):
            page = page_table[page_indptr[b] + j // PAGE]
            if page < 0 or page >= dst_pages:
                flags |= BAD_SLOT
                continue
            slot = int(kv_indices[int(kv_indptr[b]) + j])
            if 0 <= slot < src_slots:
                dst[page * PAGE + j % PAGE] = src[slot]
            else:
                flags |= BAD_SLOT
                dst[page * PAGE + j % PAGE] = 0
    return dst, page_table, page_indptr, flags
