"""Seeded synthetic inputs for speculative-verify MLA attention.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  It is the one module that both the CUDA path and the
fp64 oracle consume (the oracle never imports it: tests and the bench call it
and hand the resulting tensors to each side).

Shapes follow the verify step described in "The Decisive A/B: When
Benchmarking Honesty Reveals the Real Bottleneck" (section "The Context"): the
drafter's T speculative tokens, each with H absorbed query heads of
576 = 512 latent + 64 rope dims, attend to the target model's cached latent KV
rows, which sit in a page_size=1 slot table (scattered rows) or a paged table.

Recipe (one seed per workload):
  * structure (prefix lengths, draft-tree parents, spiky-key choice, slot or
    page permutation) comes from a CPU ``torch.Generator`` seeded with
    ``seed``, so it is identical whichever device holds the values;
  * values (q and the KV rows) are drawn ~N(0,1) in fp32 from a generator on
    the target device seeded with ``seed + VALUE_SEED_OFFSET`` and rounded to
    bf16 (round-to-nearest-even, torch's cast);
  * a fraction of each request's key rows (``floor(frac * n)`` rows, without
    replacement) is multiplied by 8 after rounding, which is exact in bf16;
  * slots (page_size=1) or pages (page_size=64) are drawn without replacement
    across the whole batch, so requests never share a slot; a request's
    logical key order is the order of its slots in the permutation;
  * every cache slot that no request owns holds bf16 NaN, so a mis-gather
    shows up in the output.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import torch

D_QK = 576          # absorbed query / latent-KV row width (512 latent + 64 rope)
D_V = 512           # value width: the latent part of each cached row
VALUE_SEED_OFFSET = 1_000_003
BF16_NAN_BITS = 0x7FC0


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic verify workload.

    ``prefix`` is either a tuple of per-request prefix lengths P_b, or
    ``("uniform", lo, hi)`` for lengths drawn uniformly in [lo, hi].
    ``tree`` is "chain" (draft i's parent is i-1), "star" (every parent is
    the prefix) or "random" (parent uniform over the prefix and the earlier
    drafts whose depth is below ``max_depth``).
    """
    name: str
    batch: int
    num_drafts: int
    num_heads: int
    prefix: tuple
    tree: str
    num_slots: int
    page_size: int = 1
    spike_frac: float = 0.0
    spike_mult: float = 8.0
    max_depth: int = 6
    scale: float = 1.0 / math.sqrt(192.0)
    seed: int = 0

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _sweep(p: int) -> Workload:
    return Workload(name=f"sweep_p{p}", batch=1, num_drafts=8, num_heads=64,
                    prefix=(p,), tree="chain", num_slots=131072,
                    spike_frac=0.01, seed=3)


# The workloads of the verify benchmark.  "tiny" is the small case the oracle
# finishes in well under a second; the rest are the full-size shapes.
WORKLOADS = {
    "tiny": Workload(name="tiny", batch=1, num_drafts=4, num_heads=16,
                     prefix=(256,), tree="chain", num_slots=1024,
                     spike_frac=0.01, seed=0),
    "decode_batch": Workload(name="decode_batch", batch=8, num_drafts=8,
                             num_heads=64, prefix=(4096,) * 8, tree="chain",
                             num_slots=65536, spike_frac=0.01, seed=1),
    "tree": Workload(name="tree", batch=4, num_drafts=16, num_heads=64,
                     prefix=(16384,) * 4, tree="random", num_slots=131072,
                     seed=2),
    **{f"sweep_p{p}": _sweep(p) for p in (1024, 4096, 16384, 65536, 93184)},
    "ragged_ps1": Workload(name="ragged_ps1", batch=32, num_drafts=16,
                           num_heads=64, prefix=("uniform", 512, 131072),
                           tree="random", num_slots=4194304, page_size=1,
                           seed=4),
    "ragged_ps64": Workload(name="ragged_ps64", batch=32, num_drafts=16,
                            num_heads=64, prefix=("uniform", 512, 131072),
                            tree="random", num_slots=4194304, page_size=64,
                            seed=4),
    # The small-R regime, where one key row serves few query rows and HBM is
    # the roof: a tensor-parallel slice of the heads (16 of them) verifying 4
    # drafts, and plain one-token decode over all 128 heads.
    "decode_tp8": Workload(name="decode_tp8", batch=16, num_drafts=4,
                           num_heads=16, prefix=(4096,) * 16, tree="chain",
                           num_slots=131072, spike_frac=0.01, seed=5),
    "decode_t1": Workload(name="decode_t1", batch=32, num_drafts=1,
                          num_heads=128, prefix=(2048,) * 32, tree="chain",
                          num_slots=131072, spike_frac=0.01, seed=6),
}


def prefix_lengths(w: Workload, g: torch.Generator) -> List[int]:
    if len(w.prefix) == 3 and w.prefix[0] == "uniform":
        lo, hi = int(w.prefix[1]), int(w.prefix[2])
        return [int(x) for x in torch.randint(lo, hi + 1, (w.batch,), generator=g)]
    assert len(w.prefix) == w.batch, "one prefix length per request"
    return [int(p) for p in w.prefix]


def draft_parents(w: Workload, g: torch.Generator) -> List[List[int]]:
    """Parent of draft i: -1 (the prefix) or an earlier draft j < i."""
    out = []
    for _ in range(w.batch):
        if w.tree == "chain":
            par = [i - 1 for i in range(w.num_drafts)]
        elif w.tree == "star":
            par = [-1] * w.num_drafts
        elif w.tree == "random":
            par, depth = [], []
            for i in range(w.num_drafts):
                cand = [-1] + [j for j in range(i) if depth[j] < w.max_depth]
                pick = cand[int(torch.randint(len(cand), (1,), generator=g))]
                par.append(pick)
                depth.append(1 if pick < 0 else depth[pick] + 1)
        else:
            raise ValueError(f"unknown tree kind {w.tree!r}")
        out.append(par)
    return out


@dataclasses.dataclass
class VerifyInputs:
    q: torch.Tensor            # [B, T, H, 576] bf16
    kv_cache: torch.Tensor     # [S, 576] bf16, unused slots NaN
    kv_indices: torch.Tensor   # int32: slot ids (page_size 1) or page ids (64)
    kv_indptr: torch.Tensor    # int32 [B+1]
    kv_lens: torch.Tensor      # int32 [B]   = P_b + T
    draft_parent: torch.Tensor  # int32 [B, T]
    scale: float
    page_size: int
    workload: Workload
    prefix: List[int]
    parents: List[List[int]]

    @property
    def num_keys(self) -> int:
        return int(sum(self.prefix)) + self.workload.batch * self.workload.num_drafts


def make_inputs(w: Workload, device="cpu", *, prefix: Optional[Sequence[int]] = None,
                parents: Optional[Sequence[Sequence[int]]] = None,
                chunk_rows: int = 1 << 18) -> VerifyInputs:
    """Draw the inputs of workload ``w`` on ``device``.

    ``prefix`` / ``parents`` override the drawn structure (edge-case tests).
    """
    device = torch.device(device)
    gs = torch.Generator(device="cpu").manual_seed(w.seed)
    gv = torch.Generator(device=device).manual_seed(w.seed + VALUE_SEED_OFFSET)
    B, T, H, ps = w.batch, w.num_drafts, w.num_heads, w.page_size
    P = list(prefix) if prefix is not None else prefix_lengths(w, gs)
    par = [list(p) for p in parents] if parents is not None else draft_parents(w, gs)
    n = [p + T for p in P]
    total = sum(n)

    q = torch.randn((B, T, H, D_QK), generator=gv, device=device,
                    dtype=torch.float32).to(torch.bfloat16)

    # Slot assignment: disjoint across requests.
    if ps == 1:
        if total > w.num_slots:
            raise ValueError(f"{total} keys do not fit {w.num_slots} slots")
        perm = torch.randperm(w.num_slots, generator=gs)[:total]
        slot_of, indices, off = [], [], 0
        for nb in n:
            s = perm[off:off + nb]
            slot_of.append(s)
            indices.append(s)
            off += nb
        counts = n
    else:
        pages_needed = [-(-nb // ps) for nb in n]
        if sum(pages_needed) * ps > w.num_slots:
            raise ValueError("pages do not fit the cache")
        perm = torch.randperm(w.num_slots // ps, generator=gs)[:sum(pages_needed)]
        slot_of, indices, off = [], [], 0
        for nb, npg in zip(n, pages_needed):
            pg = perm[off:off + npg]
            j = torch.arange(nb)
            slot_of.append(pg[j // ps] * ps + j % ps)
            indices.append(pg)
            off += npg
        counts = pages_needed

    spikes = []
    for nb in n:
        k = int(math.floor(w.spike_frac * nb))
        spikes.append(torch.randperm(nb, generator=gs)[:k] if k else None)

    cache = torch.empty((w.num_slots, D_QK), dtype=torch.bfloat16, device=device)
    cache.view(torch.int16).fill_(BF16_NAN_BITS)
    for b in range(B):
        slots_b = slot_of[b].to(device)
        for r0 in range(0, n[b], chunk_rows):
            r1 = min(n[b], r0 + chunk_rows)
            rows = torch.randn((r1 - r0, D_QK), generator=gv, device=device,
                               dtype=torch.float32).to(torch.bfloat16)
            if spikes[b] is not None:
                sel = spikes[b][(spikes[b] >= r0) & (spikes[b] < r1)] - r0
                if sel.numel():
                    sel = sel.to(device)
                    rows[sel] = rows[sel] * w.spike_mult
            cache[slots_b[r0:r1]] = rows

    indptr = [0]
    for c in counts:
        indptr.append(indptr[-1] + c)
    kv_indices = torch.cat([x.to(torch.int32) for x in indices]).to(device)
    return VerifyInputs(
        q=q, kv_cache=cache, kv_indices=kv_indices,
        kv_indptr=torch.tensor(indptr, dtype=torch.int32, device=device),
        kv_lens=torch.tensor(n, dtype=torch.int32, device=device),
        draft_parent=torch.tensor(par, dtype=torch.int32, device=device).reshape(B, T),
        scale=float(w.scale), page_size=ps, workload=w, prefix=P, parents=par)


def algorithmic_work(prefix: Sequence[int], T: int, H: int, out_bytes: int = 4):
    """Bytes and flops one verify call must move/do, by definition.

    bytes: every key row once (1152 B), q once, out/lse once, one int32
    index per key.  flops: 2*(576+512) per query row and key.
    """
    keys = sum(prefix) + len(prefix) * T
    R = T * H
    kv = keys * D_QK * 2
    byt = kv + len(prefix) * R * (D_QK * 2 + D_V * out_bytes + 4) + keys * 4
    flops = 2 * (D_QK + D_V) * R * keys
    return {"kv_bytes": kv, "bytes": byt, "flops": flops, "keys": keys}
