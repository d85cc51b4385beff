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
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"

namespace mlav {
namespace {

constexpr int BN = 128;
constexpr int NTHREADS = 256;
constexpr int BLOCK_BYTES = 9 * BN * 128;

__device__ __forceinline__ uint32_t widen(uint32_t w) {
  const float lo = __uint_as_float(w << 16);
  const float hi = __uint_as_float(w & 0xffff0000u);
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

constexpr int QUARTER = BN / 4;   // keys per CTA

// One CTA packs a quarter block (32 keys x 72 granules): every thread has
// its nine 16-byte loads in flight at once, and four CTAs per block keep
// enough bytes in flight per SM to cover DRAM latency.
__global__ void __launch_bounds__(NTHREADS) pack_kv_kernel(const Params p, uint8_t* packed,
                                                           int max_blocks) {
  __shared__ int s_slot[QUARTER];
  // The attention kernel may be scheduled as soon as every pack CTA runs:
  // only its copy warp reads the packed blocks, after griddepcontrol.wait.
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const int kb = blockIdx.x >> 2, quarter = blockIdx.x & 3, b = blockIdx.y, tid = threadIdx.x;
  const Request rq = load_request(p, b);
  if (!rq.ok) return;                      // the attention kernel reports the request
  const int nblk = (rq.n + BN - 1) / BN;
  if (kb >= nblk) return;
  const int key0 = quarter * QUARTER;      // first key of this quarter within the block
  if (tid < QUARTER) {
    const int j = kb * BN + key0 + tid;
    long long s = -1;
    if (j < rq.n) {
      s = key_slot(p, rq.ip0, j);
      if (s < 0) atomicOr(p.err, ERR_SLOT);
    }
    s_slot[tid] = static_cast<int>(s);
  }
  __syncthreads();
  uint8_t* dst = packed + (static_cast<size_t>(b) * max_blocks + kb) * BLOCK_BYTES;
  constexpr int PER_THREAD = QUARTER * ROW_CHUNKS / NTHREADS;   // 9
  static_assert(QUARTER * ROW_CHUNKS == PER_THREAD * NTHREADS, "even split");
  uint4 v[PER_THREAD];
  int off[PER_THREAD];
#pragma unroll
  for (int u = 0; u < PER_THREAD; ++u) {
    const int e = tid + u * NTHREADS;
    const int jl = e / ROW_CHUNKS, q = e - jl * ROW_CHUNKS;
    const int j = key0 + jl;                // key within the block
    const int slot = s_slot[jl];
    off[u] = (q >> 3) * (BN * 128) + j * 128 + (((q & 7) ^ (j & 7)) << 4);
    v[u] = slot >= 0 ? __ldg(reinterpret_cast<const uint4*>(p.kv + static_cast<long long>(slot) * D_QK) + q)
                     : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int u = 0; u < PER_THREAD; ++u)
    *reinterpret_cast<uint4*>(dst + off[u]) =
        make_uint4(widen(v[u].x), widen(v[u].y), widen(v[u].z), widen(v[u].w));
}

}  // namespace

size_t packed_block_bytes() { return BLOCK_BYTES; }

cudaError_t launch_pack_kv(const Params& p, void* packed, int max_blocks, cudaStream_t stream) {
  const dim3 grid(4 * max_blocks, p.batch);
  pack_kv_kernel<<<grid, NTHREADS, 0, stream>>>(p, static_cast<uint8_t*>(packed), max_blocks);
  return cudaGetLastError();
}

}  // namespace mlav
