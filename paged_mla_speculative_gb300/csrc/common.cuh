// Shared device-side definitions of the verify-attention kernels.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mlav {

constexpr int D_QK = 576;                 // latent 512 + rope 64
constexpr int D_V = 512;                  // value = latent part of each row
constexpr int ROW_BYTES = D_QK * 2;       // 1152 bytes per bf16/fp16 row
constexpr int ROW_CHUNKS = ROW_BYTES / 16;  // 72 sixteen-byte chunks per row
constexpr int PAGE = 64;                  // the paged layout's rows per page
constexpr int MAX_T = 32;                 // drafts per request (one mask bit each)
constexpr int MAX_NSPLIT = 32;

// Device error bits (mirrors MLA_VERIFY_DEV_* in the public header).
enum : int {
  ERR_SLOT = 1,
  ERR_LEN = 2,
  ERR_PARENT = 4,
  ERR_INDPTR = 8,
  ERR_TIMEOUT = 16,
  ERR_INTERNAL = 32,
  ERR_POOL = 64,       // index builder: pool row, prefix or length out of range
  ERR_CAPACITY = 128,  // index builder: kv_indices capacity exceeded
  ERR_RANGE = 256,     // an input value widened to fp16 is outside its range
};

// Arguments of one verify call, shared by every kernel of the call.
struct Params {
  const uint16_t* q;            // bf16 [B, R, 576], R = T*H
  const uint16_t* kv;           // bf16 [num_slots, 576]
  const int32_t* kv_indices;
  const int32_t* kv_indptr;     // [B+1]
  const int32_t* kv_lens;       // [B]
  const int32_t* draft_parent;  // [B, T]
  float scale_log2;             // scale * log2(e): scores kept in base 2
  int batch, T, H, R;
  int page_size;                // 1 or 64
  int64_t num_slots;
  int max_kv_len;
  int nsplit;
  float* ws_o;                  // [B][nsplit][R][512] normalised split outputs
  float* ws_lse;                // [B][nsplit][R] natural-log split LSEs
  void* out;                    // fp32 or bf16 [B, R, 512]
  float* lse;                   // [B, R]
  int out_bf16;
  int* err;                     // sticky device error word
  const uint8_t* packed;        // packed fp16 key blocks (TC kernel), see pack_kv.cu
  int packed_max_blocks;        // 128-key blocks reserved per request in `packed`
  int pack_flags;               // 1: the pack publishes per-unit ready flags
                                // (overlapping pack); 0: wait for its grid
  int direct_all;               // 1: no pack; every attention CTA gathers its
                                // own key blocks from the cache
  // Context-parallel shard of this call: every request's 128-key blocks are
  // dealt out evenly over num_shards and the call covers shard `shard` only
  // (0 and 1 for a whole call).
  int shard, num_shards;
  // 1: splits divide a request's 128-key blocks in pairs (the CTA-pair
  // kernel works on 256-key pair blocks); 0: block by block.
  int split_pairs;
  // Workspace row of split s of request b, query row r:
  // b * ws_stride_b + s * ws_stride_s + r (rows of 512 floats / one lse).
  long long ws_stride_b, ws_stride_s;
  // Hand-off between the pack and the attention kernel of one call, 32-bit
  // words: [0..1] epoch (64-bit: calls completed), [2] ticket (attention
  // CTAs done this call), then 64-bit flags from word PACK_SYNC_HEADER on:
  // flag 32 * (b * packed_max_blocks + kb) + g = epoch + 1 once keys
  // 4g .. 4g+3 of block kb of request b are packed in this call.  64-bit
  // tags never repeat in practice: with 32-bit ones, a flag left by a call
  // 2^32 calls earlier (a block position nothing packed since) would pass
  // for this call's after the wrap.
  unsigned* pack_sync;
};

constexpr int PACK_SYNC_HEADER = 4;   // 32-bit words before the flags (16 bytes)
constexpr int PACK_SYNC_TICKET = 2;   // word of the ticket

__device__ __forceinline__ unsigned long long pack_epoch(const unsigned* pack_sync) {
  return *reinterpret_cast<const volatile unsigned long long*>(pack_sync);
}
__device__ __forceinline__ unsigned long long* pack_flags(unsigned* pack_sync) {
  return reinterpret_cast<unsigned long long*>(pack_sync + PACK_SYNC_HEADER);
}

// Per-request facts every CTA of the request derives the same way.
struct Request {
  int n;        // kv_len: prefix + drafts
  int P;        // prefix length
  int ip0;      // first index position
  int lo, hi;   // logical keys [lo, hi) this call covers (its shard)
  bool ok;      // length and indptr consistent
};

constexpr int SHARD_KEYS = 128;   // shard boundaries fall on multiples of this

__device__ __forceinline__ Request load_request(const Params& p, int b) {
  Request r;
  r.n = p.kv_lens[b];
  r.P = r.n - p.T;
  r.ip0 = p.kv_indptr[b];
  const int ip1 = p.kv_indptr[b + 1];
  const int ipn = p.kv_indptr[p.batch];
  const long long need = p.page_size == 1 ? (long long)r.n : ((long long)r.n + PAGE - 1) / PAGE;
  const bool len_ok = r.n >= p.T && r.n <= p.max_kv_len;
  const bool ptr_ok = r.ip0 >= 0 && ip1 >= r.ip0 && ip1 <= ipn && (long long)(ip1 - r.ip0) == need;
  r.ok = len_ok && ptr_ok;
  // Shard s of S takes the request's 128-key blocks floor(s*nb/S) ..
  // floor((s+1)*nb/S) - 1, clipped to n.
  const long long nb = (static_cast<long long>(r.n) + SHARD_KEYS - 1) / SHARD_KEYS;
  const long long b0 = nb * p.shard / p.num_shards, b1 = nb * (p.shard + 1) / p.num_shards;
  r.lo = static_cast<int>(min(static_cast<long long>(r.n), b0 * SHARD_KEYS));
  r.hi = static_cast<int>(min(static_cast<long long>(r.n), b1 * SHARD_KEYS));
  if (!r.ok) r.lo = r.hi = 0;
  return r;
}

// Units [u0, u1) that part `part` of `parts` takes of `n` units: n / parts
// each, the remainder to the first parts.  The last part of a request's keys
// holds its draft keys (the tree-masked block, the slowest one) and, with
// pair blocks, possibly a lone block: it gets the smaller share.  (An even
// division by floor(n * part / parts) gives the last part the larger one;
// measured on the 93k sweep point the last split then ended ~5 us after the
// other long splits and set the kernel's end.)
__device__ __forceinline__ void split_units(long long n, int part, int parts, long long& u0, long long& u1) {
  const long long q = n / parts, r = n % parts;
  u0 = part * q + min(static_cast<long long>(part), r);
  u1 = u0 + q + (part < r ? 1 : 0);
}

// Blocks [kb0, kb1) of `bn` keys that split `split` of `nsplit` takes of the
// request's range [lo, hi).
__device__ __forceinline__ void split_blocks(const Request& rq, int bn, int split, int nsplit, int& kb0,
                                             int& kb1) {
  const int a = rq.lo / bn, z = (rq.hi + bn - 1) / bn;
  long long u0, u1;
  split_units(z > a ? z - a : 0, split, nsplit, u0, u1);
  kb0 = a + static_cast<int>(u0);
  kb1 = a + static_cast<int>(u1);
}

// The 128-key blocks [kb0, kb1) that split `split` takes of the request's
// range: its blocks, or its pairs of blocks when the attention kernel works
// on pair blocks (a range with an odd block count ends on a lone block).
// The pack and the attention kernel both use it, so the pack order follows
// the order the attention kernel reads blocks in.
__device__ __forceinline__ void split_range(const Params& p, const Request& rq, int split, int& kb0,
                                            int& kb1) {
  if (!p.split_pairs) {
    split_blocks(rq, 128, split, p.nsplit, kb0, kb1);
    return;
  }
  const int a = rq.lo / 128, z = (rq.hi + 127) / 128;
  long long u0, u1;
  split_units(z > a ? (z - a + 1) / 2 : 0, split, p.nsplit, u0, u1);
  kb0 = a + 2 * static_cast<int>(u0);
  kb1 = min(z, a + 2 * static_cast<int>(u1));
}

// First workspace row of split s of request b.
__device__ __forceinline__ size_t ws_base(const Params& p, int b, int s) {
  return static_cast<size_t>(b * p.ws_stride_b + s * p.ws_stride_s);
}

// Bit i of the result is set iff draft i is t itself or an ancestor of t.
// A parent that is not an earlier draft ends the walk and is reported.
__device__ __forceinline__ uint32_t ancestor_mask(const int32_t* parent, int t, int* err) {
  uint32_t m = 1u << t;
  int cur = t;
  for (int it = 0; it < MAX_T; ++it) {
    const int par = parent[cur];
    if (par < 0) {
      if (par != -1) atomicOr(err, ERR_PARENT);
      break;
    }
    if (par >= cur) {
      atomicOr(err, ERR_PARENT);
      break;
    }
    m |= 1u << par;
    cur = par;
  }
  return m;
}

// Slot of logical key j, or -1 when the table points outside the cache.
__device__ __forceinline__ long long key_slot(const Params& p, int ip0, int j) {
  if (p.page_size == 1) {
    const long long s = p.kv_indices[ip0 + j];
    return (s >= 0 && s < p.num_slots) ? s : -1;
  }
  const long long pg = p.kv_indices[ip0 + j / PAGE];
  return (pg >= 0 && pg < p.num_slots / PAGE) ? pg * PAGE + (j % PAGE) : -1;
}

// bf16 pair -> fp16 pair (round to nearest).  Exact for |x| in [2^-14,
// 65504]; a magnitude of 65536 or more becomes inf, which `bad` records (it
// is also set by a NaN input) so the caller can report ERR_RANGE.
__device__ __forceinline__ uint32_t widen_bf16x2(uint32_t w, bool& bad) {
  const float lo = __uint_as_float(w << 16);
  const float hi = __uint_as_float(w & 0xffff0000u);
  __half2 h = __floats2half2_rn(lo, hi);
  const uint32_t r = *reinterpret_cast<uint32_t*>(&h);
  bad |= ((r & 0x7c00u) == 0x7c00u) | ((r & 0x7c000000u) == 0x7c000000u);
  return r;
}
__device__ __forceinline__ uint4 widen_bf16x8(uint4 v, bool& bad) {
  return make_uint4(widen_bf16x2(v.x, bad), widen_bf16x2(v.y, bad), widen_bf16x2(v.z, bad),
                    widen_bf16x2(v.w, bad));
}
// One atomic per warp for a per-thread range flag (all lanes must call).
__device__ __forceinline__ void report_range(bool bad, int* err) {
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(err, ERR_RANGE);
}

__device__ __forceinline__ uint32_t smem_u32(const void* ptr) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

}  // namespace mlav
