// KV pack: gathers each request's scattered cache rows once per call into a
// dense, MMA-ready staging buffer, widening bf16 to fp16 on the way.
//
// The pages name KV defragmentation as the step after the custom verify
// kernel ("The Moment of Truth: Benchmarking a Custom sm_120 Verify Kernel
// Against Triton", section "The Broader Context": page_size=1 scatters every
// KV access).  Here the defragmentation is per call: every query-row tile of
// a request reads the same key blocks, so gathering them once (a bandwidth-
// bound pass over the request's rows) replaces eight or sixteen scattered
// gathers of the same rows inside the attention kernel, and the attention
// kernel then streams each block with plain bulk copies.
//
// Layout: block kb of request b occupies 147456 contiguous bytes at
// packed + (b * max_blocks + kb) * 147456: nine 16 KB chunk tiles (dims
// 64c .. 64c+63), each [128 keys][128 bytes] with the 16-byte granules of
// key j permuted by XOR with (j & 7) -- the 128-byte-swizzled operand tile
// tcgen05 reads.  Keys past the end of the request, or whose slot lies
// outside the cache (reported), are zero.
//
// Two kernels, same layout:
//  * pack_kv_kernel: one 256-thread CTA per quarter block (every thread has
//    its nine 16-byte loads in flight at once), the whole grid ahead of the
//    attention kernel, whose copy warp waits for it with griddepcontrol.wait.
//  * pack_kv_overlap_kernel: when the attention grid leaves SMs idle
//    (decode batches: 128 attention CTAs on 152 SMs), a persistent grid of
//    1024-thread CTAs, one per SM, in two phases: the CTAs beyond the idle
//    count pack the first block positions of every split and exit -- their
//    SMs take the attention CTAs (programmatic dependent launch) -- while
//    the others pack the rest on the idle SMs as the attention kernel runs.
//    Each warp packs 4-key units and publishes every unit with a release
//    store of this call's tag (epoch + 1) into pack_sync, 32 flags per
//    block, which the attention kernel's copy warp waits for block by block.
//    Units run in split-position order (the i-th block of every (request,
//    split) before any (i+1)-th), so every attention CTA finds its next
//    block packed while it works on the last.
#include <cuda_fp16.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace mlav {
namespace {

constexpr int BN = 128;
constexpr int NTHREADS = 256;           // pack_kv_kernel
constexpr int OV_THREADS = 1024;        // pack_kv_overlap_kernel
constexpr int BLOCK_BYTES = 9 * BN * 128;

// The key rows are read exactly once per call: load them past L1 and mark
// them first to leave L2, so the packed blocks the attention kernel reads
// next stay there.
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint4 load_row_granule(const uint4* src, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(src), "l"(pol));
  return v;
}

constexpr int QUARTER = BN / 4;   // keys per CTA of pack_kv_kernel

// One CTA packs a quarter block (32 keys x 72 granules): every thread has
// its nine 16-byte loads in flight at once, and several CTAs per SM keep
// enough bytes in flight to cover DRAM latency.
__global__ void __launch_bounds__(NTHREADS) pack_kv_kernel(const Params p, uint8_t* packed,
                                                           int max_blocks) {
  __shared__ int s_slot[QUARTER];
  // The attention kernel may be scheduled as soon as every pack CTA runs:
  // only its copy warp reads the packed blocks, after griddepcontrol.wait.
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const int kb = blockIdx.x >> 2, quarter = blockIdx.x & 3, b = blockIdx.y, tid = threadIdx.x;
  const Request rq = load_request(p, b);
  if (!rq.ok) return;                      // the attention kernel reports the request
  if (kb < rq.lo / BN || kb >= (rq.hi + BN - 1) / BN) return;   // outside the call's keys
  const int key0 = quarter * QUARTER;      // first key of this quarter within the block
  if (tid < QUARTER) {
    const int j = kb * BN + key0 + tid;
    long long s = -1;
    if (j >= rq.lo && j < rq.hi) {
      s = key_slot(p, rq.ip0, j);
      if (s < 0) atomicOr(p.err, ERR_SLOT);
    }
    s_slot[tid] = static_cast<int>(s);
  }
  __syncthreads();
  uint8_t* dst = packed + (static_cast<size_t>(b) * max_blocks + kb) * BLOCK_BYTES;
  constexpr int PER_THREAD = QUARTER * ROW_CHUNKS / NTHREADS;   // 9
  static_assert(QUARTER * ROW_CHUNKS == PER_THREAD * NTHREADS, "even split");
  const uint64_t pol = evict_first_policy();
  uint4 v[PER_THREAD];
  int off[PER_THREAD];
#pragma unroll
  for (int u = 0; u < PER_THREAD; ++u) {
    const int e = tid + u * NTHREADS;
    const int jl = e / ROW_CHUNKS, q = e - jl * ROW_CHUNKS;
    const int j = key0 + jl;                // key within the block
    const int slot = s_slot[jl];
    off[u] = (q >> 3) * (BN * 128) + j * 128 + (((q & 7) ^ (j & 7)) << 4);
    v[u] = slot >= 0 ? load_row_granule(reinterpret_cast<const uint4*>(p.kv + static_cast<long long>(slot) * D_QK) + q, pol)
                     : make_uint4(0, 0, 0, 0);
  }
  bool bad = false;
#pragma unroll
  for (int u = 0; u < PER_THREAD; ++u) *reinterpret_cast<uint4*>(dst + off[u]) = widen_bf16x8(v[u], bad);
  report_range(bad, p.err);
}

constexpr int UNIT_KEYS = 4;                        // keys per warp unit
constexpr int UNITS_PER_BLOCK = BN / UNIT_KEYS;     // 32: one ready flag each
constexpr int PER_LANE = ROW_CHUNKS / 8;               // 9 granules per lane (8 lanes per key)
static_assert(UNIT_KEYS * 8 == 32 && PER_LANE * 8 == ROW_CHUNKS, "8 lanes per key");
static_assert(UNITS_PER_BLOCK == 32, "one flag per lane of the reader's warp");

// Packed blocks whose descriptions every pack CTA tabulates in shared memory
// (16 bytes each); larger calls describe each block as they reach it.
constexpr int TABLE_BLOCKS = 12288;

// Block q of the pack order: split q % nsplit, request (q / nsplit) %
// batch, position q / nsplit / batch within the split.  Returns (packed
// block b * max_blocks + kb, first index position of the request, first key
// kb * 128, end of the call's keys), or x = -1 when there is nothing to pack
// (past the split, or the request is invalid -- the attention kernel reports
// it).  A shard's keys start on a block boundary, so every key of a block
// from its first key up to the end is in the call's range.
__device__ __noinline__ int4 block_info(const Params& p, int q, int max_blocks) {
  const int split = q % p.nsplit;
  const int r = q / p.nsplit;
  const int b = r % p.batch, pos = r / p.batch;
  const Request rq = load_request(p, b);
  if (!rq.ok) return make_int4(-1, 0, 0, 0);
  int kb0, kb1;   // the attention kernel's division of the call's keys
  split_range(p, rq, split, kb0, kb1);
  const int kb = kb0 + pos;
  if (kb >= kb1) return make_int4(-1, 0, 0, 0);
  return make_int4(b * max_blocks + kb, rq.ip0, kb * BN, rq.hi);
}

// Unit u: 4-key group u % 32 of block u / 32 of the pack order.  blk: the
// packed block, or -1 (nothing to pack).  slot: lanes 0..3 hold the cache
// slot of key `lane` of the unit (-1: none / outside).
struct Unit {
  int blk, slot;
};

__device__ __forceinline__ Unit locate(const Params& p, const int4* s_tab, int max_blocks, int u,
                                       int lane) {
  Unit t;
  const int grp = u & (UNITS_PER_BLOCK - 1);
  const int4 e = s_tab ? s_tab[u / UNITS_PER_BLOCK] : block_info(p, u / UNITS_PER_BLOCK, max_blocks);
  t.blk = e.x;
  t.slot = -1;
  const int j = e.z + grp * UNIT_KEYS + lane;
  if (e.x >= 0 && lane < UNIT_KEYS && j < e.w) {
    const long long s = key_slot(p, e.y, j);
    if (s < 0) atomicOr(p.err, ERR_SLOT);
    t.slot = static_cast<int>(s);
  }
  return t;
}

// Lane l moves granules l % 8, l % 8 + 8, .. of key l / 8 of the unit:
// granule l % 8 of each of the nine 64-dim chunks.
__device__ __forceinline__ void load_unit(const Params& p, const Unit& t, int lane, uint4 (&v)[PER_LANE]) {
  const int sk = __shfl_sync(0xffffffffu, t.slot, lane >> 3);
  const uint4* src = reinterpret_cast<const uint4*>(p.kv + static_cast<long long>(sk) * D_QK) + (lane & 7);
#pragma unroll
  for (int i = 0; i < PER_LANE; ++i) v[i] = make_uint4(0, 0, 0, 0);
  if (sk >= 0) {   // streamed once
    const uint64_t pol = evict_first_policy();
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) v[i] = load_row_granule(src + 8 * i, pol);
  }
}

__device__ __forceinline__ void store_unit(uint8_t* packed, const Unit& t, int grp, int lane,
                                           const uint4 (&v)[PER_LANE], bool& bad) {
  const int j = grp * UNIT_KEYS + (lane >> 3);   // key within the block
  uint8_t* dst = packed + static_cast<size_t>(t.blk) * BLOCK_BYTES + j * 128 +
                 (((lane & 7) ^ (j & 7)) << 4);
#pragma unroll
  for (int i = 0; i < PER_LANE; ++i) *reinterpret_cast<uint4*>(dst + i * (BN * 128)) = widen_bf16x8(v[i], bad);
}

// Pack units first, first + stride, .. below `end`.  Per round a warp
// locates unit k+1, stores unit k, issues the row loads of unit k+1 and only
// then publishes unit k: the release waits for those loads, which the next
// round needs anyway, so the fence does not sit between two row loads.
__device__ __forceinline__ void pack_units(const Params& p, const int4* s_tab, uint8_t* packed,
                                           int max_blocks, int u, int end, int stride, int lane,
                                           unsigned tag) {
  if (u >= end) return;
  bool bad = false;
  Unit cur = locate(p, s_tab, max_blocks, u, lane);
  uint4 v[PER_LANE];
  if (cur.blk >= 0) load_unit(p, cur, lane, v);
#pragma unroll 1
  for (; u < end; u += stride) {
    const bool more = u + stride < end;
    const Unit nxt = locate(p, s_tab, max_blocks, more ? u + stride : u, lane);
    if (cur.blk >= 0) {
      store_unit(packed, cur, u & (UNITS_PER_BLOCK - 1), lane, v, bad);
      // The stores must reach the reader's bulk copies (async proxy).
      asm volatile("fence.proxy.async.global;\n" ::: "memory");
    }
    if (more && nxt.blk >= 0) load_unit(p, nxt, lane, v);
    if (cur.blk >= 0) {
      // Publish unit k: the release store orders the warp's stores (made
      // visible to lane 0 by the warp barrier) before the flag.
      __syncwarp();
      if (lane == 0) {
        unsigned* flag = p.pack_sync + PACK_SYNC_HEADER + UNITS_PER_BLOCK * static_cast<size_t>(cur.blk) +
                         (u & (UNITS_PER_BLOCK - 1));
        asm volatile("st.release.gpu.global.u32 [%0], %1;\n" ::"l"(flag), "r"(tag) : "memory");
      }
    }
    cur = nxt;
  }
  report_range(bad, p.err);
}

// Two phases in one launch.  CTAs from `stay` on pack the units of the
// first `wide_units` (the first positions of every split), spread CTA by
// CTA so that they all finish together, and exit: their SMs take attention
// CTAs.  CTAs 0 .. stay-1 start on the rest at once and pack it while the
// attention kernel runs.
__global__ void __maxnreg__(64) pack_kv_overlap_kernel(const Params p, uint8_t* packed, int max_blocks,
                                                       int per_split, int wide_units, int stay) {
  extern __shared__ int4 s_tab_buf[];
  // The attention kernel may be scheduled as soon as every pack CTA runs:
  // its copy warp waits for each block's flags before reading it.
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const int cta = static_cast<int>(blockIdx.x);
  if (cta >= stay && cta - stay >= wide_units) return;   // no unit in the wide phase: free the SM
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nq = p.nsplit * p.batch * per_split;   // blocks in the pack order
  const int4* s_tab = nullptr;
  if (nq <= TABLE_BLOCKS) {
    for (int q = threadIdx.x; q < nq; q += OV_THREADS) s_tab_buf[q] = block_info(p, q, max_blocks);
    __syncthreads();
    s_tab = s_tab_buf;
  }
  constexpr int WPC = OV_THREADS / 32;               // warps per CTA
  const int units = UNITS_PER_BLOCK * nq;            // < 2^31 (host check)
  const int wide_end = min(wide_units, units);
  const unsigned tag = *reinterpret_cast<volatile unsigned*>(p.pack_sync) + 1u;
  const int n = gridDim.x - stay;     // CTAs of the wide phase: warp w of CTA c takes units
  const bool wide = cta >= stay;      // w * n + c, w * n + c + 32 n, ..
  const int first = wide ? warp * n + (cta - stay) : wide_end + cta * WPC + warp;
  pack_units(p, s_tab, packed, max_blocks, first, wide ? wide_end : units, (wide ? n : stay) * WPC, lane, tag);
}

}  // namespace

size_t packed_block_bytes() { return BLOCK_BYTES; }

cudaError_t pack_kv_prepare() {
  // Room for the block table; the attention kernel's shared-memory
  // configuration (an SM whose carveout differs drains before the other
  // kernel's CTAs can start on it).
  cudaError_t e = cudaFuncSetAttribute(pack_kv_overlap_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(sizeof(int4)) * TABLE_BLOCKS);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(pack_kv_overlap_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                              cudaSharedmemCarveoutMaxShared);
}

cudaError_t launch_pack_kv(const Params& p, void* packed, int max_blocks, cudaStream_t stream) {
  const dim3 grid(4 * max_blocks, p.batch);
  pack_kv_kernel<<<grid, NTHREADS, 0, stream>>>(p, static_cast<uint8_t*>(packed), max_blocks);
  return cudaGetLastError();
}

cudaError_t launch_pack_kv_overlap(const Params& p, void* packed, int max_blocks, int num_ctas,
                                   int wide_positions, int stay, cudaStream_t stream) {
  // Positions per split: at most ceil(max_blocks / nsplit) blocks, or twice
  // ceil(pairs / nsplit) when splits take pairs of blocks.
  const int per_split = p.split_pairs ? 2 * (((max_blocks + 1) / 2 + p.nsplit - 1) / p.nsplit)
                                      : (max_blocks + p.nsplit - 1) / p.nsplit;
  const long long nq = 1LL * p.nsplit * p.batch * per_split;
  if (UNITS_PER_BLOCK * nq > 0x7fffffffLL || stay < 1 || stay >= num_ctas)
    return cudaErrorInvalidConfiguration;
  const int wide_units =
      static_cast<int>(1LL * UNITS_PER_BLOCK * p.nsplit * p.batch * std::min(wide_positions, per_split));
  const size_t smem = nq <= TABLE_BLOCKS ? sizeof(int4) * nq : 0;
  pack_kv_overlap_kernel<<<num_ctas, OV_THREADS, smem, stream>>>(p, static_cast<uint8_t*>(packed),
                                                                 max_blocks, per_split, wide_units, stay);
  return cudaGetLastError();
}

}  // namespace mlav
