"""fp64 NumPy oracle: gather, masked softmax, weighted sum.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

Inputs are NumPy arrays.  bf16 tensors are passed as their raw 16-bit
patterns (``uint16``/``int16``) or as any float dtype that holds the bf16
values exactly; ``bf16_bits_to_f64`` widens them exactly.
"""
from __future__ import annotations

from typing import Iterable, List, Optional, Sequence, Set, Tuple

import numpy as np

D_QK = 576
D_V = 512


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 values to fp64.

    A bf16 number is the upper half of an IEEE binary32 pattern, so shifting
    its 16 bits left by 16 gives the binary32 of the same value, which fp64
    holds exactly.  Float inputs are taken to hold bf16 values already.
    """
    a = np.asarray(a)
    if a.dtype in (np.uint16, np.int16):
        bits = a.astype(np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def ancestor_sets(parent: Sequence[int]) -> List[Set[int]]:
    """anc[t] = {t} plus every draft reached by following parent links.

    parent[i] is -1 (the draft hangs off the prefix) or an earlier draft.
    Walking the links is the plain reading of a tree given by a parent array;
    a link that does not point to an earlier draft ends the walk (the library
    reports such a link as an input error).
    """
    T = len(parent)
    out = []
    for t in range(T):
        s, cur = {t}, t
        while True:
            p = int(parent[cur])
            if p < 0 or p >= cur:
                break
            s.add(p)
            cur = p
        out.append(s)
    return out


def gather_request_keys(kv_cache: np.ndarray, kv_indices: np.ndarray,
                        kv_indptr: np.ndarray, b: int, n: int,
                        page_size: int) -> np.ndarray:
    """Rows of request b's n logical keys, in logical order, as fp64 [n, 576].

    page_size 1: logical key j lives in slot kv_indices[indptr[b] + j].
    page_size p: it lives in row j % p of page kv_indices[indptr[b] + j // p],
    i.e. slot page * p + j % p.  (Scattered page_size=1 reads are the case
    named in "The Decisive A/B ...", section "The Context".)
    """
    base = int(kv_indptr[b])
    j = np.arange(n, dtype=np.int64)
    if page_size == 1:
        slots = np.asarray(kv_indices[base:base + n], dtype=np.int64)
    else:
        pages = np.asarray(kv_indices, dtype=np.int64)[base + j // page_size]
        slots = pages * page_size + j % page_size
    return bf16_bits_to_f64(kv_cache[slots])


def _visible(P: int, n: int, anc_t: Set[int]) -> np.ndarray:
    vis = np.zeros(n, dtype=bool)
    vis[:P] = True
    for i in anc_t:
        vis[P + i] = True
    return vis


def _attend(qrows: np.ndarray, keys: np.ndarray, vis: np.ndarray,
            scale: float) -> Tuple[np.ndarray, np.ndarray]:
    """Masked softmax attention of query rows over the visible keys (fp64).

    qrows [m, 576], keys [n, 576], vis [n] -> out [m, 512], lse [m].
    The max is subtracted before exp only to avoid overflow; it cancels
    exactly in the definition.
    """
    kv = keys[vis]
    s = scale * (qrows @ kv.T)                      # [m, n_vis]
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    z = e.sum(axis=1, keepdims=True)
    lse = (m + np.log(z))[:, 0]
    out = (e / z) @ kv[:, :D_V]
    return out, lse


def mla_verify(q, kv_cache, kv_indices, kv_indptr, kv_lens, draft_parent,
               scale: float, page_size: int = 1):
    """Whole-batch oracle.  q [B,T,H,576] -> out [B,T,H,512], lse [B,T,H]."""
    qf = bf16_bits_to_f64(q)
    B, T, H, _ = qf.shape
    out = np.empty((B, T, H, D_V))
    lse = np.empty((B, T, H))
    for b in range(B):
        n = int(kv_lens[b])
        P = n - T
        keys = gather_request_keys(kv_cache, kv_indices, kv_indptr, b, n, page_size)
        anc = ancestor_sets(np.asarray(draft_parent)[b])
        for t in range(T):
            o, l = _attend(qf[b, t], keys, _visible(P, n, anc[t]), scale)
            out[b, t], lse[b, t] = o, l
    return out, lse


def mla_verify_rows(rows: Iterable[Tuple[int, int, int]], q, kv_cache,
                    kv_indices, kv_indptr, kv_lens, draft_parent, scale: float,
                    page_size: int = 1):
    """Oracle evaluated only at the given (b, t, h) query rows.

    Used for sampled checks on workloads too large to evaluate whole.
    Returns out [len(rows), 512], lse [len(rows)].
    """
    rows = list(rows)
    T = np.asarray(q).shape[1]
    out = np.empty((len(rows), D_V))
    lse = np.empty(len(rows))
    by_req = {}
    for i, (b, t, h) in enumerate(rows):
        by_req.setdefault(int(b), []).append((i, int(t), int(h)))
    for b, items in by_req.items():
        n = int(kv_lens[b])
        P = n - T
        keys = gather_request_keys(kv_cache, kv_indices, kv_indptr, b, n, page_size)
        anc = ancestor_sets(np.asarray(draft_parent)[b])
        for i, t, h in items:
            qr = bf16_bits_to_f64(np.asarray(q)[b, t, h])[None, :]
            o, l = _attend(qr, keys, _visible(P, n, anc[t]), scale)
            out[i], lse[i] = o[0], l[0]
    return out, lse


def mla_verify_split_combine(q, kv_cache, kv_indices, kv_indptr, kv_lens,
                             draft_parent, scale: float, page_size: int,
                             nsplit: int):
    """The oracle evaluated on nsplit key ranges, then merged by their LSEs.

    This is the partial + reduce structure of "The Decisive A/B ...",
    section "The Context" (KV split across workers, partials merged by a
    reduce step), written in fp64: each range r yields o_r (its own softmax
    over the visible keys in range, normalised) and lse_r; then
        lse = log sum_r exp(lse_r),  out = sum_r exp(lse_r - lse) * o_r.
    A range with no visible key has lse_r = -inf and weight 0.
    """
    qf = bf16_bits_to_f64(q)
    B, T, H, _ = qf.shape
    out = np.zeros((B, T, H, D_V))
    lse = np.empty((B, T, H))
    for b in range(B):
        n = int(kv_lens[b])
        P = n - T
        keys = gather_request_keys(kv_cache, kv_indices, kv_indptr, b, n, page_size)
        anc = ancestor_sets(np.asarray(draft_parent)[b])
        edges = np.linspace(0, n, nsplit + 1).round().astype(int)
        for t in range(T):
            vis = _visible(P, n, anc[t])
            parts = []
            for r in range(nsplit):
                lo, hi = edges[r], edges[r + 1]
                vr = np.zeros(n, dtype=bool)
                vr[lo:hi] = vis[lo:hi]
                if not vr.any():
                    parts.append((np.zeros((H, D_V)), np.full(H, -np.inf)))
                    continue
                parts.append(_attend(qf[b, t], keys, vr, scale))
            L = np.stack([p[1] for p in parts])          # [nsplit, H]
            mx = L.max(axis=0)
            tot = mx + np.log(np.exp(L - mx).sum(axis=0))
            w = np.exp(L - tot)                            # exp(-inf) = 0
            out[b, t] = sum(w[r][:, None] * parts[r][0] for r in range(nsplit))
            lse[b, t] = tot
    return out, lse


def shard_key_range(n: int, shard: int, num_shards: int, block: int = 128) -> Tuple[int, int]:
    """Logical keys [lo, hi) that shard `shard` of `num_shards` covers in a
    request of n keys (the context-parallel split of the partial + reduce
    design, "The Decisive A/B ...", section "The Context").

    The request's ceil(n / 128) blocks of 128 consecutive keys are dealt out
    evenly: shard s takes blocks floor(s * nb / S) .. floor((s+1) * nb / S) - 1,
    so a shard boundary never cuts a block; the range is clipped to n.
    """
    nb = -(-int(n) // block)
    b0 = (shard * nb) // num_shards
    b1 = ((shard + 1) * nb) // num_shards
    return min(int(n), b0 * block), min(int(n), b1 * block)


def mla_verify_key_range(q, kv_cache, kv_indices, kv_indptr, kv_lens,
                         draft_parent, scale: float, page_size: int,
                         lo: Sequence[int], hi: Sequence[int]):
    """The definition restricted to the logical keys [lo[b], hi[b]) of each
    request: a key counts iff it is in range and visible as usual.

    Returns out [B,T,H,512] (normalised over the counted keys) and lse
    [B,T,H] (their log-sum-exp).  A row with no counted key has lse = -inf
    and out = 0, the weight-0 partial of the reduce step.
    """
    qf = bf16_bits_to_f64(q)
    B, T, H, _ = qf.shape
    out = np.zeros((B, T, H, D_V))
    lse = np.full((B, T, H), -np.inf)
    for b in range(B):
        n = int(kv_lens[b])
        P = n - T
        keys = gather_request_keys(kv_cache, kv_indices, kv_indptr, b, n, page_size)
        anc = ancestor_sets(np.asarray(draft_parent)[b])
        inr = np.zeros(n, dtype=bool)
        inr[int(lo[b]):int(hi[b])] = True
        for t in range(T):
            vis = _visible(P, n, anc[t]) & inr
            if vis.any():
                out[b, t], lse[b, t] = _attend(qf[b, t], keys, vis, scale)
    return out, lse


def lse_merge(parts_out, parts_lse):
    """The reduce step over S partials, in fp64: parts_out [S, ..., 512],
    parts_lse [S, ...] ->
        lse = log sum_s exp(lse_s),  out = sum_s exp(lse_s - lse) * out_s.
    Partials with lse_s = -inf have weight 0; when every partial of a row has
    -inf the row is lse = -inf, out = 0.
    """
    po = np.asarray(parts_out, dtype=np.float64)
    pl = np.asarray(parts_lse, dtype=np.float64)
    mx = pl.max(axis=0)
    base = np.where(np.isfinite(mx), mx, 0.0)
    w = np.exp(pl - base)                            # exp(-inf) = 0
    tot = w.sum(axis=0)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(tot > 0, base + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)
        wn = np.where(tot > 0, w / np.where(tot > 0, tot, 1.0), 0.0)
    out = (wn[..., None] * po).sum(axis=0)
    return out, lse
