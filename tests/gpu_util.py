"""Helpers shared by the GPU parity tests (not a test module)."""
import numpy as np
import torch

import oracle
from paged_mla_speculative_gb300 import binding as mb
from paged_mla_speculative_gb300 import workloads as W
from tests.conftest import bits

# Tolerances of the verify attention against the fp64 oracle.
OUT_MAX_ABS = 1e-2
OUT_MEAN_ABS = 1e-3
LSE_MAX_ABS = 1e-3


def to_cuda(inp: W.VerifyInputs) -> W.VerifyInputs:
    import dataclasses
    return dataclasses.replace(
        inp, q=inp.q.cuda(), kv_cache=inp.kv_cache.cuda(), kv_indices=inp.kv_indices.cuda(),
        kv_indptr=inp.kv_indptr.cuda(), kv_lens=inp.kv_lens.cuda(),
        draft_parent=inp.draft_parent.cuda())


def make_plan(inp: W.VerifyInputs, out_dtype=torch.float32, nsplit=0, max_kv_len=None,
              max_batch=None, kernel=mb.KERNEL_AUTO):
    w = inp.workload
    mk = max_kv_len or max(int(x) for x in inp.kv_lens.tolist())
    plan = mb.Plan(max_batch or w.batch, w.num_drafts, w.num_heads, inp.page_size,
                   inp.kv_cache.shape[0], mk, out_dtype)
    plan.set_kernel(kernel)
    if nsplit:
        plan.set_nsplit(nsplit)
    return plan


def run(plan, inp, stream=None):
    out, lse = mb.mla_verify_attn(plan, inp.q, inp.kv_cache, inp.kv_indices, inp.kv_indptr,
                                  inp.kv_lens, inp.draft_parent, inp.scale, stream=stream)
    torch.cuda.synchronize()
    return out, lse


def oracle_full(inp):
    return oracle.mla_verify(bits(inp.q), bits(inp.kv_cache), inp.kv_indices.cpu().numpy(),
                             inp.kv_indptr.cpu().numpy(), inp.kv_lens.cpu().numpy(),
                             inp.draft_parent.cpu().numpy(), inp.scale, inp.page_size)


def oracle_rows(inp, rows, cache_bits=None):
    cb = cache_bits if cache_bits is not None else bits(inp.kv_cache)
    return oracle.mla_verify_rows(rows, bits(inp.q), cb, inp.kv_indices.cpu().numpy(),
                                  inp.kv_indptr.cpu().numpy(), inp.kv_lens.cpu().numpy(),
                                  inp.draft_parent.cpu().numpy(), inp.scale, inp.page_size)


def assert_parity(out, lse, ref_out, ref_lse, what=""):
    o = np.asarray(out, dtype=np.float64)
    l = np.asarray(lse, dtype=np.float64)
    assert np.isfinite(o).all() and np.isfinite(l).all(), f"{what}: non-finite output"
    eo = np.abs(o - ref_out)
    el = np.abs(l - ref_lse)
    assert eo.max() <= OUT_MAX_ABS, f"{what}: out max abs err {eo.max():.3g}"
    assert eo.mean() <= OUT_MEAN_ABS, f"{what}: out mean abs err {eo.mean():.3g}"
    assert el.max() <= LSE_MAX_ABS, f"{what}: lse max abs err {el.max():.3g}"
    return float(eo.max()), float(eo.mean()), float(el.max())


def sample_rows(inp, per_request=3, seed=0):
    """(b, t, h) rows: for every request the last draft, the first draft and a
    random one, each with a random head."""
    g = np.random.default_rng(seed)
    w = inp.workload
    rows = []
    for b in range(w.batch):
        ts = [w.num_drafts - 1, 0] + list(g.integers(0, w.num_drafts, max(0, per_request - 2)))
        for t in ts[:per_request]:
            rows.append((b, int(t), int(g.integers(0, w.num_heads))))
    return rows


def assert_bf16_parity(out_bf16, lse, ref_out, ref_lse, what=""):
    """bf16 output: each element within the fp32 tolerance plus one bf16 ulp
    of the reference (the rounding of the output itself); lse as for fp32."""
    o = out_bf16.float().numpy().astype(np.float64)
    l = np.asarray(lse, dtype=np.float64)
    assert np.isfinite(o).all() and np.isfinite(l).all(), f"{what}: non-finite output"
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref_out), 2.0 ** -126))) - 7)
    bad = np.abs(o - ref_out) > OUT_MAX_ABS + ulp
    assert not bad.any(), f"{what}: {int(bad.sum())} bf16 elements beyond tolerance + 1 ulp"
    el = np.abs(l - ref_lse)
    assert el.max() <= LSE_MAX_ABS, f"{what}: lse max abs err {el.max():.3g}"
