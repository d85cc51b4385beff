"""The whole call records into a CUDA graph and replays with new data.

The metadata (kv_lens, indices, parents) and q change between replays, so a
replay that baked any device value into the graph would give the wrong
answer; every replay must equal an eager call on the same buffers bit for
bit, and match the oracle.
"""
import numpy as np
import pytest
import torch

from paged_mla_speculative_gb300 import binding as mb
from paged_mla_speculative_gb300 import workloads as W
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_mla_speculative_gb300 import build
    build.build()


def _inputs(seed, prefix, tree):
    w = W.Workload(name="cap", batch=3, num_drafts=8, num_heads=16, prefix=prefix, tree=tree,
                   num_slots=8192, spike_frac=0.01, seed=seed)
    return W.make_inputs(w)


@pytest.mark.parametrize("nsplit", [1, 4])
def test_graph_replay_with_changing_metadata(nsplit):
    cases = [_inputs(1, (1000, 300, 20), "chain"), _inputs(2, (64, 1500, 999), "random"),
             _inputs(3, (0, 7, 1800), "star")]
    max_idx = max(c.kv_indices.numel() for c in cases)
    dev = torch.device("cuda")
    # Static buffers, sized for the largest case.
    q = torch.empty_like(cases[0].q, device=dev)
    cache = torch.empty_like(cases[0].kv_cache, device=dev)
    idx = torch.zeros(max_idx, dtype=torch.int32, device=dev)
    indptr = torch.empty(4, dtype=torch.int32, device=dev)
    lens = torch.empty(3, dtype=torch.int32, device=dev)
    par = torch.empty((3, 8), dtype=torch.int32, device=dev)

    def load(c):
        q.copy_(c.q)
        cache.copy_(c.kv_cache)
        idx[:c.kv_indices.numel()].copy_(c.kv_indices)
        indptr.copy_(c.kv_indptr)
        lens.copy_(c.kv_lens)
        par.copy_(c.draft_parent)

    plan = mb.Plan(3, 8, 16, 1, 8192, 2000)
    plan.set_nsplit(nsplit)
    out, lse = plan.new_outputs(3)
    s = torch.cuda.Stream()
    load(cases[0])
    torch.cuda.synchronize()
    with torch.cuda.stream(s):   # warm-up outside capture
        mb.mla_verify_attn(plan, q, cache, idx, indptr, lens, par, cases[0].scale, out, lse, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        mb.mla_verify_attn(plan, q, cache, idx, indptr, lens, par, cases[0].scale, out, lse, stream=s)
    for c in cases + cases[::-1]:
        load(c)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        go, gl = out.clone(), lse.clone()
        eo, el = mb.mla_verify_attn(plan, q, cache, idx, indptr, lens, par, c.scale)
        torch.cuda.synchronize()
        assert torch.equal(go, eo) and torch.equal(gl, el)
        ref_o, ref_l = G.oracle_full(c)
        G.assert_parity(go.cpu().numpy(), gl.cpu().numpy(), ref_o, ref_l)
    assert plan.get_error() == 0
    plan.close()
