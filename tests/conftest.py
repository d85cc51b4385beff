import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running")


def bits(t):
    """bf16 torch tensor -> numpy uint16 bit patterns (what the oracle takes)."""
    import torch
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


def oracle_args(inp):
    """Positional oracle arguments from a workloads.VerifyInputs."""
    return (bits(inp.q), bits(inp.kv_cache), inp.kv_indices.cpu().numpy(),
            inp.kv_indptr.cpu().numpy(), inp.kv_lens.cpu().numpy(),
            inp.draft_parent.cpu().numpy(), inp.scale, inp.page_size)
