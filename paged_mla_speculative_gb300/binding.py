"""ctypes binding of libmla_verify.so (argument marshalling only).

Every step of the verify attention runs in the library's CUDA kernels; this
module checks tensor dtypes, shapes, devices and contiguity, passes raw
pointers and the current CUDA stream, and turns status codes into
exceptions.  There is no fallback: if the library is missing or fails to
load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libmla_verify.so")

OUT_F32 = 0
OUT_BF16 = 1
KERNEL_AUTO = 0
KERNEL_MMA = 1
KERNEL_TC = 2
KERNEL_PAIR = 3
PACK_AUTO = 0
PACK_WHOLE = 1
PACK_IDLE_SMS = 2
PACK_NONE = 4
FAULT_NONE = 0
FAULT_SKIP_PACK = 1
FAULT_EPOCH_NEAR_WRAP = 2
MAX_NSPLIT = 32

DEV_BAD_SLOT = 1
DEV_BAD_LEN = 2
DEV_BAD_PARENT = 4
DEV_BAD_INDPTR = 8
DEV_TIMEOUT = 16
DEV_INTERNAL = 32
DEV_BAD_POOL = 64
DEV_CAPACITY = 128
DEV_RANGE = 256

STATUS = {0: "OK", -1: "ERR_NULL", -2: "ERR_ALIGN", -3: "ERR_SHAPE", -4: "ERR_BATCH",
          -5: "ERR_SCALE", -6: "ERR_CUDA", -7: "ERR_DEVICE", -8: "ERR_OOM", -9: "ERR_ARG",
          -10: "ERR_SCRATCH"}
STATIC_SCRATCH_BYTES = 32 << 20

# name -> (restype, argtypes): every entry point the header declares.
_P = ctypes.c_void_p
_I = ctypes.c_int
SIGNATURES = {
    "mla_verify_plan_create": (_I, [ctypes.POINTER(_P), _I, _I, _I, _I, ctypes.c_int64, _I, _I, _I]),
    "mla_verify_plan_destroy": (None, [_P]),
    "mla_verify_plan_set_nsplit": (_I, [_P, _I]),
    "mla_verify_plan_get_nsplit": (_I, [_P, _I]),
    "mla_verify_plan_inject_fault": (_I, [_P, _I]),
    "mla_verify_plan_get_pack_schedule": (_I, [_P, _I, ctypes.POINTER(ctypes.c_int),
                                              ctypes.POINTER(ctypes.c_int)]),
    "mla_verify_plan_set_pack_schedule": (_I, [_P, _I]),
    "mla_verify_plan_get_pack_mode": (_I, [_P, _I]),
    "mla_verify_plan_set_kernel": (_I, [_P, _I]),
    "mla_verify_plan_get_kernel": (_I, [_P]),
    "mla_verify_plan_get_call_kernel": (_I, [_P, _I]),
    "mla_verify_plan_workspace_bytes": (ctypes.c_size_t, [_P]),
    "mla_verify_plan_set_profile_events": (_I, [_P, _P, _P]),
    "mla_verify_attn": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P]),
    "mla_verify_attn_host": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P]),
    "mla_verify_attn_partial": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, ctypes.c_float, _I, _I, _P, _P,
                                     _P]),
    "mla_verify_combine_parts": (_I, [_P, _I, _I, _P, _P, _P, _P, _P]),
    "mla_verify_get_error": (_I, [_P, ctypes.POINTER(_I), _I]),
    "mla_verify_attn_static": (_I, [_I, _I, _I, _I, ctypes.c_int64, _I, _I, _P, _P, _P, _P, _P, _P,
                                    ctypes.c_float, _P, _P, _P, _P]),
    "mla_verify_build_indices": (_I, [_P, _I, _P, ctypes.c_int64, _I, _P, _P, _P, ctypes.c_int64,
                                      _P, _P, _P]),
    "mla_verify_compact_kv": (_I, [_P, _I, _P, ctypes.c_int64, _P, _P, _P, _P, ctypes.c_int64, _P,
                                   ctypes.c_int64, _P, _P, _P]),
    "mla_verify_strerror": (ctypes.c_char_p, [_I]),
    "mla_verify_version": (_I, []),
}

_lib = None


class MlaVerifyError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({strerror(status)})")


def load_library(path: Optional[str] = None):
    """Load (once) and return the ctypes handle; raises if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"{p} is missing: build it with `python -m paged_mla_speculative_gb300.build` "
            "(the verify attention has no non-CUDA implementation)")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def strerror(status: int) -> str:
    return load_library().mla_verify_strerror(int(status)).decode()


def _check(status: int, what: str):
    if status != 0:
        raise MlaVerifyError(status, what)


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: torch.Tensor) -> int:
    return int(t.data_ptr())


class Plan:
    """Owns one mla_verify_plan (its workspace and error word)."""

    def __init__(self, max_batch: int, num_drafts: int, num_heads: int, page_size: int,
                 num_slots: int, max_kv_len: int, out_dtype=torch.float32,
                 device: Optional[int] = None):
        lib = load_library()
        if device is None:
            device = torch.cuda.current_device()
        od = {torch.float32: OUT_F32, torch.bfloat16: OUT_BF16}[out_dtype]
        h = ctypes.c_void_p()
        _check(lib.mla_verify_plan_create(ctypes.byref(h), max_batch, num_drafts, num_heads,
                                          page_size, num_slots, max_kv_len, od, device),
               "mla_verify_plan_create")
        self._h = h
        self.max_batch, self.T, self.H = max_batch, num_drafts, num_heads
        self.page_size, self.num_slots, self.max_kv_len = page_size, num_slots, max_kv_len
        self.out_dtype, self.device = out_dtype, device

    @property
    def handle(self):
        if self._h is None:
            raise RuntimeError("plan already destroyed")
        return self._h

    def close(self):
        if getattr(self, "_h", None) is not None:
            load_library().mla_verify_plan_destroy(self._h)
            self._h = None

    __del__ = close

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def set_nsplit(self, nsplit: int):
        _check(load_library().mla_verify_plan_set_nsplit(self.handle, nsplit), "set_nsplit")

    def nsplit(self, batch: int) -> int:
        v = load_library().mla_verify_plan_get_nsplit(self.handle, batch)
        if v < 0:
            raise MlaVerifyError(v, "get_nsplit")
        return v

    def pack_schedule(self, batch: int):
        """(wide, stay) of the key pack for `batch` requests: stay > 0 when the
        pack overlaps the attention kernel (see the C header)."""
        wide, stay = ctypes.c_int(), ctypes.c_int()
        rc = load_library().mla_verify_plan_get_pack_schedule(self.handle, batch, ctypes.byref(wide),
                                                              ctypes.byref(stay))
        if rc != 0:
            raise MlaVerifyError(rc, "get_pack_schedule")
        return wide.value, stay.value

    def set_pack_schedule(self, schedule: int):
        """Force a key-pack schedule (PACK_WHOLE / PACK_IDLE_SMS / PACK_NONE)
        or PACK_AUTO."""
        _check(load_library().mla_verify_plan_set_pack_schedule(self.handle, schedule),
               "set_pack_schedule")

    def pack_mode(self, batch: int) -> int:
        """The pack schedule a call with `batch` requests uses (PACK_NONE: no pack)."""
        v = load_library().mla_verify_plan_get_pack_mode(self.handle, batch)
        if v < 0:
            raise MlaVerifyError(v, "get_pack_mode")
        return v

    def inject_fault(self, fault: int):
        """Testing hook: inject a host-side fault into the next call (see the
        C header, FAULT_SKIP_PACK)."""
        _check(load_library().mla_verify_plan_inject_fault(self.handle, fault), "inject_fault")

    def set_kernel(self, kernel: int):
        _check(load_library().mla_verify_plan_set_kernel(self.handle, kernel), "set_kernel")

    def kernel(self) -> int:
        """The kernel family selected (KERNEL_MMA, KERNEL_TC or KERNEL_PAIR)."""
        v = load_library().mla_verify_plan_get_kernel(self.handle)
        if v < 0:
            raise MlaVerifyError(v, "get_kernel")
        return v

    def call_kernel(self, batch: int) -> int:
        """The partial kernel a call with `batch` requests launches
        (KERNEL_MMA, KERNEL_TC or KERNEL_PAIR)."""
        v = load_library().mla_verify_plan_get_call_kernel(self.handle, batch)
        if v < 0:
            raise MlaVerifyError(v, "get_call_kernel")
        return v

    def set_profile_events(self, after_pack=None, after_partial=None):
        """Record torch.cuda.Events (timing enabled) after the pack kernel and
        after the partial kernel of every later call; None stops either."""
        ptrs = []
        for ev in (after_pack, after_partial):
            if ev is None:
                ptrs.append(None)
                continue
            if int(ev.cuda_event) == 0:   # torch creates the event on first record
                ev.record()
                ev.synchronize()
            ptrs.append(int(ev.cuda_event))
        _check(load_library().mla_verify_plan_set_profile_events(self.handle, *ptrs),
               "set_profile_events")
        self._profile_events = (after_pack, after_partial)

    def workspace_bytes(self) -> int:
        return int(load_library().mla_verify_plan_workspace_bytes(self.handle))

    def get_error(self, clear: bool = True) -> int:
        v = ctypes.c_int(0)
        _check(load_library().mla_verify_get_error(self.handle, ctypes.byref(v), int(clear)),
               "get_error")
        return v.value

    def new_outputs(self, batch: int):
        dev = torch.device("cuda", self.device)
        out = torch.empty((batch, self.T, self.H, 512), dtype=self.out_dtype, device=dev)
        lse = torch.empty((batch, self.T, self.H), dtype=torch.float32, device=dev)
        return out, lse


def _expect(t: torch.Tensor, name: str, dtype, device=None, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def mla_verify_attn(plan: Plan, q, kv_cache, kv_indices, kv_indptr, kv_lens, draft_parent,
                    scale: float, out=None, lse=None, stream=None):
    """Verify attention on the plan's device; returns (out, lse).

    q [B,T,H,576] bf16, kv_cache [S,576] bf16, kv_indices/kv_indptr/kv_lens/
    draft_parent int32, out [B,T,H,512] (plan's dtype), lse [B,T,H] fp32.
    Enqueued on ``stream`` (default: the current torch stream); no sync.
    """
    B = q.shape[0]
    dev = torch.device("cuda", plan.device)
    _expect(q, "q", torch.bfloat16, dev, (B, plan.T, plan.H, 576))
    _expect(kv_cache, "kv_cache", torch.bfloat16, dev)
    if kv_cache.dim() != 2 or kv_cache.shape[1] != 576 or kv_cache.shape[0] != plan.num_slots:
        raise ValueError(f"kv_cache must be [{plan.num_slots}, 576]")
    _expect(kv_indices, "kv_indices", torch.int32, dev)
    _expect(kv_indptr, "kv_indptr", torch.int32, dev, (B + 1,))
    _expect(kv_lens, "kv_lens", torch.int32, dev, (B,))
    _expect(draft_parent, "draft_parent", torch.int32, dev, (B, plan.T))
    if out is None or lse is None:
        o2, l2 = plan.new_outputs(B)
        out = o2 if out is None else out
        lse = l2 if lse is None else lse
    _expect(out, "out", plan.out_dtype, dev, (B, plan.T, plan.H, 512))
    _expect(lse, "lse", torch.float32, dev, (B, plan.T, plan.H))
    st = load_library().mla_verify_attn(
        plan.handle, B, _ptr(q), _ptr(kv_cache), _ptr(kv_indices), _ptr(kv_indptr),
        _ptr(kv_lens), _ptr(draft_parent), float(scale), _ptr(out), _ptr(lse),
        _stream_ptr(stream))
    _check(st, "mla_verify_attn")
    return out, lse


def mla_verify_attn_partial(plan: Plan, q, kv_cache, kv_indices, kv_indptr, kv_lens,
                            draft_parent, scale: float, shard: int, num_shards: int,
                            part_out=None, part_lse=None, stream=None):
    """One context-parallel shard of the verify attention; returns (part_out
    fp32 [B,T,H,512], part_lse fp32 [B,T,H]) over the keys of shard `shard`
    of `num_shards` (see the C header).  Enqueued on ``stream``; no sync."""
    B = q.shape[0]
    dev = torch.device("cuda", plan.device)
    _expect(q, "q", torch.bfloat16, dev, (B, plan.T, plan.H, 576))
    _expect(kv_cache, "kv_cache", torch.bfloat16, dev)
    _expect(kv_indices, "kv_indices", torch.int32, dev)
    _expect(kv_indptr, "kv_indptr", torch.int32, dev, (B + 1,))
    _expect(kv_lens, "kv_lens", torch.int32, dev, (B,))
    _expect(draft_parent, "draft_parent", torch.int32, dev, (B, plan.T))
    if part_out is None:
        part_out = torch.empty((B, plan.T, plan.H, 512), dtype=torch.float32, device=dev)
    if part_lse is None:
        part_lse = torch.empty((B, plan.T, plan.H), dtype=torch.float32, device=dev)
    _expect(part_out, "part_out", torch.float32, dev, (B, plan.T, plan.H, 512))
    _expect(part_lse, "part_lse", torch.float32, dev, (B, plan.T, plan.H))
    st = load_library().mla_verify_attn_partial(
        plan.handle, B, _ptr(q), _ptr(kv_cache), _ptr(kv_indices), _ptr(kv_indptr),
        _ptr(kv_lens), _ptr(draft_parent), float(scale), int(shard), int(num_shards),
        _ptr(part_out), _ptr(part_lse), _stream_ptr(stream))
    _check(st, "mla_verify_attn_partial")
    return part_out, part_lse


def mla_verify_combine_parts(plan: Plan, parts_out, parts_lse, out=None, lse=None, stream=None):
    """Merge shard partials laid out shard-major (parts_out fp32 [S,B,T,H,512],
    parts_lse fp32 [S,B,T,H]) into (out, lse) in the plan's output dtype."""
    S, B = parts_out.shape[0], parts_out.shape[1]
    dev = torch.device("cuda", plan.device)
    _expect(parts_out, "parts_out", torch.float32, dev, (S, B, plan.T, plan.H, 512))
    _expect(parts_lse, "parts_lse", torch.float32, dev, (S, B, plan.T, plan.H))
    if out is None or lse is None:
        o2, l2 = plan.new_outputs(B)
        out = o2 if out is None else out
        lse = l2 if lse is None else lse
    _expect(out, "out", plan.out_dtype, dev, (B, plan.T, plan.H, 512))
    _expect(lse, "lse", torch.float32, dev, (B, plan.T, plan.H))
    st = load_library().mla_verify_combine_parts(plan.handle, B, S, _ptr(parts_out), _ptr(parts_lse),
                                                 _ptr(out), _ptr(lse), _stream_ptr(stream))
    _check(st, "mla_verify_combine_parts")
    return out, lse


def build_indices(plan: Plan, req_to_token, req_pool_indices, prefix_lens, kv_indices=None,
                  kv_indptr=None, kv_lens=None, stream=None):
    """Per-step index builder on the plan's device; returns (kv_indices,
    kv_indptr, kv_lens) ready for mla_verify_attn.

    req_to_token int32 [pool_size, stride >= max_kv_len] (cache slot of each
    token position per pool row), req_pool_indices / prefix_lens int32 [B].
    kv_indices defaults to a buffer of B * (entries of max_kv_len) int32; its
    length is the capacity.  Enqueued on ``stream``; no sync.
    """
    B = req_pool_indices.shape[0]
    dev = torch.device("cuda", plan.device)
    _expect(req_to_token, "req_to_token", torch.int32, dev)
    if req_to_token.dim() != 2 or req_to_token.stride(1) != 1:
        raise ValueError("req_to_token must be a 2-D int32 tensor with unit column stride")
    _expect(req_pool_indices, "req_pool_indices", torch.int32, dev, (B,))
    _expect(prefix_lens, "prefix_lens", torch.int32, dev, (B,))
    per_req = plan.max_kv_len if plan.page_size == 1 else -(-plan.max_kv_len // 64)
    if kv_indices is None:
        kv_indices = torch.empty(B * per_req, dtype=torch.int32, device=dev)
    if kv_indptr is None:
        kv_indptr = torch.empty(B + 1, dtype=torch.int32, device=dev)
    if kv_lens is None:
        kv_lens = torch.empty(B, dtype=torch.int32, device=dev)
    _expect(kv_indices, "kv_indices", torch.int32, dev)
    _expect(kv_indptr, "kv_indptr", torch.int32, dev, (B + 1,))
    _expect(kv_lens, "kv_lens", torch.int32, dev, (B,))
    st = load_library().mla_verify_build_indices(
        plan.handle, B, _ptr(req_to_token), int(req_to_token.stride(0)), int(req_to_token.shape[0]),
        _ptr(req_pool_indices), _ptr(prefix_lens), _ptr(kv_indices), int(kv_indices.numel()),
        _ptr(kv_indptr), _ptr(kv_lens), _stream_ptr(stream))
    _check(st, "mla_verify_build_indices")
    return kv_indices, kv_indptr, kv_lens


def compact_kv(plan: Plan, kv_src, kv_indices, kv_indptr, kv_lens, free_pages, kv_dst,
               page_table=None, page_indptr=None, stream=None):
    """KV compaction into 64-row pages on the plan's device; returns
    (page_table, page_indptr), the page_size 64 table of the same requests.

    kv_src [S, 576] / kv_dst [S2, 576] bf16 (S2 a multiple of 64),
    kv_indices / kv_indptr / kv_lens int32 (page_size 1 table), free_pages
    int32 destination page ids used in order.  Enqueued on ``stream``; no sync.
    """
    B = kv_lens.shape[0]
    dev = torch.device("cuda", plan.device)
    for t, name in ((kv_src, "kv_src"), (kv_dst, "kv_dst")):
        _expect(t, name, torch.bfloat16, dev)
        if t.dim() != 2 or t.shape[1] != 576:
            raise ValueError(f"{name} must be [slots, 576]")
    _expect(kv_indices, "kv_indices", torch.int32, dev)
    _expect(kv_indptr, "kv_indptr", torch.int32, dev, (B + 1,))
    _expect(kv_lens, "kv_lens", torch.int32, dev, (B,))
    _expect(free_pages, "free_pages", torch.int32, dev)
    if page_table is None:
        page_table = torch.empty(max(free_pages.numel(), 4), dtype=torch.int32, device=dev)
    if page_indptr is None:
        page_indptr = torch.empty(B + 1, dtype=torch.int32, device=dev)
    _expect(page_table, "page_table", torch.int32, dev)
    _expect(page_indptr, "page_indptr", torch.int32, dev, (B + 1,))
    st = load_library().mla_verify_compact_kv(
        plan.handle, B, _ptr(kv_src), int(kv_src.shape[0]), _ptr(kv_indices), _ptr(kv_indptr),
        _ptr(kv_lens), _ptr(free_pages), int(free_pages.numel()), _ptr(kv_dst),
        int(kv_dst.shape[0]), _ptr(page_table), _ptr(page_indptr), _stream_ptr(stream))
    _check(st, "mla_verify_compact_kv")
    return page_table, page_indptr


def mla_verify_attn_host(plan: Plan, q, kv_cache, kv_indices, kv_indptr, kv_lens,
                         draft_parent, scale: float, out, lse, stream=None):
    """Host-buffer variant: q/indices/indptr/lens/parent/out/lse are CPU
    tensors (pinned for speed), kv_cache is on the device.  Copies in, runs,
    copies back and synchronises ``stream``."""
    B = q.shape[0]
    cpu = torch.device("cpu")
    dev = torch.device("cuda", plan.device)
    _expect(q, "q", torch.bfloat16, cpu, (B, plan.T, plan.H, 576))
    _expect(kv_cache, "kv_cache", torch.bfloat16, dev)
    _expect(kv_indices, "kv_indices", torch.int32, cpu)
    _expect(kv_indptr, "kv_indptr", torch.int32, cpu, (B + 1,))
    _expect(kv_lens, "kv_lens", torch.int32, cpu, (B,))
    _expect(draft_parent, "draft_parent", torch.int32, cpu, (B, plan.T))
    _expect(out, "out", plan.out_dtype, cpu, (B, plan.T, plan.H, 512))
    _expect(lse, "lse", torch.float32, cpu, (B, plan.T, plan.H))
    if kv_indices.numel() < int(kv_indptr[B]):
        raise ValueError("kv_indices shorter than kv_indptr[B]")
    st = load_library().mla_verify_attn_host(
        plan.handle, B, _ptr(q), _ptr(kv_cache), _ptr(kv_indices), _ptr(kv_indptr),
        _ptr(kv_lens), _ptr(draft_parent), float(scale), _ptr(out), _ptr(lse),
        _stream_ptr(stream))
    _check(st, "mla_verify_attn_host")
    return out, lse
