"""Pure-Python brute force of the verify attention, for tiny inputs only.

TEST INFRASTRUCTURE ONLY.  It exists to pin ``oracle.mla_verify``: it walks
every (b, t, h, key, dim) with plain loops and ``math.fsum``, takes slots one
key at a time, decides visibility by asking, for each draft key, whether it
lies on the path from t to the root, and never subtracts a running max.  It
shares no helper with ``mla_verify_ref``.
"""
from __future__ import annotations

import math
import struct


def _bf16(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


def _on_root_path(parent, t: int, i: int) -> bool:
    cur = t
    for _ in range(len(parent) + 1):
        if cur == i:
            return True
        p = parent[cur]
        if p < 0 or p >= cur:
            return False
        cur = p
    return False


def brute_verify(q_bits, cache_bits, kv_indices, kv_indptr, kv_lens, parent,
                 scale, page_size, key_ranges=None):
    """q_bits: nested lists [B][T][H][576] of bf16 bit patterns (ints);
    cache_bits: list of rows of bf16 bit patterns.  Returns nested lists
    out[B][T][H][512], lse[B][T][H].  key_ranges: optional [(lo, hi)] per
    request; only keys lo <= j < hi count, and a row with no counted key
    gets lse -inf and a zero out."""
    B = len(q_bits)
    T = len(q_bits[0])
    H = len(q_bits[0][0])
    out, lse = [], []
    for b in range(B):
        n = kv_lens[b]
        P = n - T
        rows = []
        for j in range(n):
            if page_size == 1:
                slot = kv_indices[kv_indptr[b] + j]
            else:
                slot = kv_indices[kv_indptr[b] + j // page_size] * page_size + j % page_size
            rows.append([_bf16(x) for x in cache_bits[slot]])
        ob, lb = [], []
        for t in range(T):
            ot, lt = [], []
            for h in range(H):
                qv = [_bf16(x) for x in q_bits[b][t][h]]
                weights, vis_rows = [], []
                for j in range(n):
                    if key_ranges is not None and not key_ranges[b][0] <= j < key_ranges[b][1]:
                        continue
                    if j >= P and not _on_root_path(parent[b], t, j - P):
                        continue
                    s = scale * math.fsum(qv[d] * rows[j][d] for d in range(576))
                    weights.append(math.exp(s))
                    vis_rows.append(rows[j])
                z = math.fsum(weights)
                if not weights:
                    ot.append([0.0] * 512)
                    lt.append(-math.inf)
                    continue
                ot.append([math.fsum(w * r[d] for w, r in zip(weights, vis_rows)) / z
                           for d in range(512)])
                lt.append(math.log(z))
            ob.append(ot)
            lb.append(lt)
        out.append(ob)
        lse.append(lb)
    return out, lse
