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
//    one 768-thread CTA per SM, in two phases: the CTAs beyond the idle
//    count pack the first block positions of every split and exit -- their
//    SMs take the attention CTAs (programmatic dependent launch) -- while
//    the others pack the rest on the idle SMs as the attention kernel runs.
//    Each warp packs 4-key units through two shared-memory stages (16-byte
//    cp.async of the unit's rows, so one unit's loads stay in flight while
//    it widens and stores the other, without registers held per load) and
//    publishes every unit with a release store of this call's tag (epoch +
//    1) into pack_sync, 32 flags per block, which the attention kernel's
//    copy warp waits for block by block.  Units run in split-position order
//    (the i-th block of every (request, split) before any (i+1)-th), so
//    every attention CTA finds its next block packed while it works on the
//    last.
#include <cuda_fp16.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace mlav {
namespace {

constexpr int BN = 128;
constexpr int NTHREADS = 256;           // pack_kv_kernel
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
constexpr int PER_LANE = ROW_CHUNKS / 8;            // 9 granules per lane (8 lanes per key)
static_assert(UNIT_KEYS * 8 == 32 && PER_LANE * 8 == ROW_CHUNKS, "8 lanes per key");
static_assert(UNITS_PER_BLOCK == 32, "one flag per lane of the reader's warp");

// pack_kv_overlap_kernel: warps per CTA and units staged per warp.  24
// warps of two stages fill shared memory; measured on GB300 (the narrow phase
// alone, 93k scattered keys, 24 SMs): ~36 GB/s of rows read per SM, against
// ~32 with 16 warps of three stages, ~29 with 12 of four, ~23 with 8 of six,
// and ~23 with the units held in registers.  Every unit's publication waits
// for the warp's outstanding memory operations, so the parallel warps, not
// the depth, carry the throughput.
constexpr int OV_WARPS = 24;
constexpr int OV_DEPTH = 2;
constexpr int UNIT_BYTES = UNIT_KEYS * ROW_BYTES;   // 4608: a unit's rows as they are in the cache
constexpr int OV_SMEM = OV_WARPS * OV_DEPTH * UNIT_BYTES;

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

// A warp's units u0, u0 + stride, .. in groups of eight: lane l describes
// key l & 3 of unit l >> 2 of the group -- `blk` the packed block (-1:
// nothing to pack, or past `end`), `slot` the key's cache slot (-1: none,
// or outside the cache, which is reported).
__device__ __forceinline__ void locate8(const Params& p, int max_blocks, int u0, int end, int stride, int lane,
                                        int& blk, int& slot) {
  const int u = u0 + (lane >> 2) * stride;
  blk = -1;
  slot = -1;
  if (u >= end) return;
  const int4 e = block_info(p, u / UNITS_PER_BLOCK, max_blocks);
  blk = e.x;
  const int j = e.z + (u & (UNITS_PER_BLOCK - 1)) * UNIT_KEYS + (lane & 3);
  if (e.x >= 0 && j < e.w) {
    const long long s = key_slot(p, e.y, j);
    if (s < 0) atomicOr(p.err, ERR_SLOT);
    slot = static_cast<int>(s);
  }
}

// Start the copy of a unit's rows into a stage: lane l moves granules l % 8,
// l % 8 + 8, .. of row l / 8 (slot `sk`; zero-filled when sk < 0).  The
// rows are read once per call: marked first to leave L2.
__device__ __forceinline__ void stage_unit(const Params& p, uint32_t stage, int sk, int lane, uint64_t pol) {
  const uint16_t* src = p.kv + static_cast<long long>(sk < 0 ? 0 : sk) * D_QK + (lane & 7) * 8;
  const uint32_t dst = stage + ((lane >> 3) * ROW_CHUNKS + (lane & 7)) * 16;
  const int bytes = sk < 0 ? 0 : 16;
#pragma unroll
  for (int i = 0; i < PER_LANE; ++i)
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;\n"
                 ::"r"(dst + 128 * i), "l"(src + 64 * i), "r"(bytes), "l"(pol)
                 : "memory");
}

// Pack this warp's units u, u + stride, .. below `end` through its
// OV_DEPTH stages: unit k lands in stage k % OV_DEPTH while the next
// OV_DEPTH - 1 units are in flight; each lane widens and stores exactly the granules it
// copied (its own cp.async data, visible to it after the group wait), into
// chunk i of key j at the swizzled granule, then the warp publishes the unit.
__device__ __forceinline__ void pack_units(const Params& p, uint8_t* packed, int max_blocks, int u, int end,
                                           int stride, int lane, unsigned long long tag, uint32_t stages) {
  if (u >= end) return;
  bool bad = false;
  const uint64_t pol = evict_first_policy();
  int cur_blk, cur_slot, next_blk, next_slot;   // this group of eight units and the next
  locate8(p, max_blocks, u, end, stride, lane, cur_blk, cur_slot);
  locate8(p, max_blocks, u + 8 * stride, end, stride, lane, next_blk, next_slot);
  // Packed block of units k .. k + OV_DEPTH - 2 (already issued).
  int blk[OV_DEPTH - 1];
#pragma unroll
  for (int d = 0; d < OV_DEPTH - 1; ++d) {
    blk[d] = __shfl_sync(0xffffffffu, cur_blk, 4 * d);
    const int sk = __shfl_sync(0xffffffffu, cur_slot, 4 * d + (lane >> 3));
    if (blk[d] >= 0) stage_unit(p, stages + d * UNIT_BYTES, sk, lane, pol);
    asm volatile("cp.async.commit_group;\n" ::: "memory");
  }
#pragma unroll 1
  for (int k = 0; u < end; u += stride, ++k) {
    // Issue unit k + OV_DEPTH - 1 into the stage unit k - 1 has left.
    const int ka = k + OV_DEPTH - 1;
    if ((ka & 7) == 0) {
      cur_blk = next_blk;
      cur_slot = next_slot;
      locate8(p, max_blocks, u + (OV_DEPTH - 1 + 8) * stride, end, stride, lane, next_blk, next_slot);
    }
    const int ba = __shfl_sync(0xffffffffu, cur_blk, 4 * (ka & 7));
    const int sa = __shfl_sync(0xffffffffu, cur_slot, 4 * (ka & 7) + (lane >> 3));
    if (ba >= 0) stage_unit(p, stages + (ka % OV_DEPTH) * UNIT_BYTES, sa, lane, pol);
    asm volatile("cp.async.commit_group;\n" ::: "memory");
    const int cblk = blk[0];
#pragma unroll
    for (int d = 0; d < OV_DEPTH - 2; ++d) blk[d] = blk[d + 1];
    blk[OV_DEPTH - 2] = ba;
    asm volatile("cp.async.wait_group %0;\n" ::"n"(OV_DEPTH - 1) : "memory");
    if (cblk < 0) continue;
    const int j = (u & (UNITS_PER_BLOCK - 1)) * UNIT_KEYS + (lane >> 3);   // key within the block
    uint8_t* dst = packed + static_cast<size_t>(cblk) * BLOCK_BYTES + j * 128 + (((lane & 7) ^ (j & 7)) << 4);
    const uint32_t src = stages + (k % OV_DEPTH) * UNIT_BYTES + ((lane >> 3) * ROW_CHUNKS + (lane & 7)) * 16;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
      uint4 v;
      asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                   : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                   : "r"(src + 128 * i));
      *reinterpret_cast<uint4*>(dst + i * (BN * 128)) = widen_bf16x8(v, bad);
    }
    // The stores must reach the reader's bulk copies (async proxy); the
    // release store orders the warp's stores (made visible to lane 0 by the
    // warp barrier) before the flag.
    asm volatile("fence.proxy.async.global;\n" ::: "memory");
    __syncwarp();
    if (lane == 0) {
      unsigned long long* flag = pack_flags(p.pack_sync) + UNITS_PER_BLOCK * static_cast<size_t>(cblk) +
                       (u & (UNITS_PER_BLOCK - 1));
      asm volatile("st.release.gpu.global.u64 [%0], %1;\n" ::"l"(flag), "l"(tag) : "memory");
    }
  }
  asm volatile("cp.async.wait_all;\n" ::: "memory");
  report_range(bad, p.err);
}

// Two phases in one launch.  CTAs from `stay` on pack the units of the
// first `wide_units` (the first positions of every split), spread CTA by
// CTA so that they all finish together, and exit: their SMs take attention
// CTAs.  CTAs 0 .. stay-1 start on the rest at once and pack it while the
// attention kernel runs.
__global__ void __launch_bounds__(OV_WARPS * 32, 1)
    pack_kv_overlap_kernel(const Params p, uint8_t* packed, int max_blocks, int per_split, int wide_units,
                           int stay) {
  extern __shared__ __align__(128) uint8_t ov_stages[];
  // The attention kernel may be scheduled as soon as every pack CTA runs:
  // its copy warp waits for each block's flags before reading it.
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const int cta = static_cast<int>(blockIdx.x);
  if (cta >= stay && cta - stay >= wide_units) return;   // no unit in the wide phase: free the SM
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nq = p.nsplit * p.batch * per_split;     // blocks in the pack order
  const int units = UNITS_PER_BLOCK * nq;            // < 2^31 (host check)
  const int wide_end = min(wide_units, units);
  const unsigned long long tag = pack_epoch(p.pack_sync) + 1ull;
  const int n = gridDim.x - stay;     // CTAs of the wide phase: warp w of CTA c takes units
  const bool wide = cta >= stay;      // w * n + c, w * n + c + 16 n, ..
  const int first = wide ? warp * n + (cta - stay) : wide_end + cta * OV_WARPS + warp;
  pack_units(p, packed, max_blocks, first, wide ? wide_end : units, (wide ? n : stay) * OV_WARPS, lane, tag,
             smem_u32(ov_stages) + warp * OV_DEPTH * UNIT_BYTES);
}

}  // namespace

size_t packed_block_bytes() { return BLOCK_BYTES; }

cudaError_t pack_kv_prepare() {
  // Room for the warps' stages; the attention kernel's shared-memory
  // configuration (an SM whose carveout differs drains before the other
  // kernel's CTAs can start on it).
  cudaError_t e = cudaFuncSetAttribute(pack_kv_overlap_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       OV_SMEM);
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
  pack_kv_overlap_kernel<<<num_ctas, OV_WARPS * 32, OV_SMEM, stream>>>(p, static_cast<uint8_t*>(packed),
                                                                 max_blocks, per_split, wide_units, stay);
  return cudaGetLastError();
}

}  // namespace mlav
