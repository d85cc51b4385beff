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

__global__ void __launch_bounds__(NTHREADS) pack_kv_kernel(const Params p, uint8_t* packed,
                                                           int max_blocks) {
  __shared__ int s_slot[BN];
  const int kb = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const Request rq = load_request(p, b);
  if (!rq.ok) return;                      // the attention kernel reports the request
  const int nblk = (rq.n + BN - 1) / BN;
  if (kb >= nblk) return;
  if (tid < BN) {
    const int j = kb * BN + tid;
    long long s = -1;
    if (j < rq.n) {
      s = key_slot(p, rq.ip0, j);
      if (s < 0) atomicOr(p.err, ERR_SLOT);
    }
    s_slot[tid] = static_cast<int>(s);
  }
  __syncthreads();
  uint8_t* dst = packed + (static_cast<size_t>(b) * max_blocks + kb) * BLOCK_BYTES;
  // 128 rows x 72 granules; consecutive threads take consecutive granules of
  // a row (coalesced 16-byte loads), eight loads in flight per thread.
#pragma unroll 1
  for (int e0 = tid; e0 < BN * ROW_CHUNKS; e0 += 8 * NTHREADS) {
    uint4 v[8];
    int off[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = e0 + u * NTHREADS;
      off[u] = -1;
      v[u] = make_uint4(0, 0, 0, 0);
      if (e < BN * ROW_CHUNKS) {
        const int j = e / ROW_CHUNKS, q = e - j * ROW_CHUNKS;
        const int slot = s_slot[j];
        off[u] = (q >> 3) * (BN * 128) + j * 128 + (((q & 7) ^ (j & 7)) << 4);
        if (slot >= 0)
          v[u] = __ldg(reinterpret_cast<const uint4*>(p.kv + static_cast<long long>(slot) * D_QK) + q);
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (off[u] < 0) continue;
      const uint4 w = make_uint4(widen(v[u].x), widen(v[u].y), widen(v[u].z), widen(v[u].w));
      *reinterpret_cast<uint4*>(dst + off[u]) = w;
    }
  }
}

}  // namespace

size_t packed_block_bytes() { return BLOCK_BYTES; }

cudaError_t launch_pack_kv(const Params& p, void* packed, int max_blocks, cudaStream_t stream) {
  const dim3 grid(max_blocks, p.batch);
  pack_kv_kernel<<<grid, NTHREADS, 0, stream>>>(p, static_cast<uint8_t*>(packed), max_blocks);
  return cudaGetLastError();
}

}  // namespace mlav
