"""GB300-native speculative-decoding verify attention for MLA over a paged KV cache.

The product is the C-ABI library ``libmla_verify.so`` (``include/mla_verify.h``);
this package holds its CUDA sources (``csrc/``), the in-tree build
(``build.py``), a thin ctypes binding (``binding.py``) and the seeded
synthetic-input generator (``workloads.py``).
"""
from .binding import (  # noqa: F401
    KERNEL_AUTO,
    KERNEL_MMA,
    KERNEL_TC,
    OUT_BF16,
    OUT_F32,
    MlaVerifyError,
    Plan,
    load_library,
    mla_verify_attn,
    mla_verify_attn_host,
    strerror,
)
