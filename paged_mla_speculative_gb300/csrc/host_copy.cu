// Host <-> device transfers of the host-buffer entry point as one kernel per
// direction.
//
// The host entry copies five input arrays in and two results out on every
// call.  As seven DMA copies each one costs a copy-engine round trip on the
// stream.  When the caller's buffers are page-locked and mapped into the
// device's address space (pinned memory on a unified-address system: on
// GB300 the Grace host memory is reached over NVLink-C2C), one kernel moves
// all regions of a direction at once: every thread keeps several 16-byte
// loads in flight, so the small arrays cost no more than the large one.
#include <cstdint>

#include "kernels.h"

namespace mlav {
namespace {

constexpr int COPY_THREADS = 256;
constexpr int COPY_UNROLL = 4;

__device__ __forceinline__ bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// Region r of `c`: 16-byte words while both ends are aligned and whole,
// then (or otherwise) 4-byte words.  Byte counts are multiples of 4.
__global__ void __launch_bounds__(COPY_THREADS) copy_regions_kernel(const CopyRegions c) {
  const long long tid = static_cast<long long>(blockIdx.x) * COPY_THREADS + threadIdx.x;
  const long long nthreads = static_cast<long long>(gridDim.x) * COPY_THREADS;
  for (int r = 0; r < c.n; ++r) {
    const uint8_t* src = static_cast<const uint8_t*>(c.src[r]);
    uint8_t* dst = static_cast<uint8_t*>(c.dst[r]);
    const long long bytes = c.bytes[r];
    long long done = 0;
    if (aligned16(src) && aligned16(dst)) {
      const long long n16 = bytes / 16;
      const uint4* s4 = reinterpret_cast<const uint4*>(src);
      uint4* d4 = reinterpret_cast<uint4*>(dst);
      for (long long i = tid; i < n16; i += nthreads * COPY_UNROLL) {
        uint4 v[COPY_UNROLL];
#pragma unroll
        for (int u = 0; u < COPY_UNROLL; ++u) {
          const long long k = i + u * nthreads;
          if (k < n16) v[u] = s4[k];
        }
#pragma unroll
        for (int u = 0; u < COPY_UNROLL; ++u) {
          const long long k = i + u * nthreads;
          if (k < n16) d4[k] = v[u];
        }
      }
      done = n16 * 16;
    }
    const uint32_t* s1 = reinterpret_cast<const uint32_t*>(src + done);
    uint32_t* d1 = reinterpret_cast<uint32_t*>(dst + done);
    const long long n4 = (bytes - done) / 4;
    for (long long i = tid; i < n4; i += nthreads) d1[i] = s1[i];
  }
}

}  // namespace

cudaError_t launch_copy_regions(const CopyRegions& c, cudaStream_t stream) {
  if (c.n < 0 || c.n > CopyRegions::kMax) return cudaErrorInvalidValue;
  long long total = 0;
  for (int r = 0; r < c.n; ++r) {
    if (c.bytes[r] < 0 || (c.bytes[r] & 3)) return cudaErrorInvalidValue;
    total += c.bytes[r];
  }
  if (total == 0) return cudaSuccess;
  // Enough threads for ~4 words in flight each over the largest region,
  // capped at a few CTAs per SM.
  const long long words = (total + 15) / 16;
  const long long want = (words + COPY_THREADS * COPY_UNROLL - 1) / (COPY_THREADS * COPY_UNROLL);
  const int grid = static_cast<int>(want < 1 ? 1 : (want > 1024 ? 1024 : want));
  copy_regions_kernel<<<grid, COPY_THREADS, 0, stream>>>(c);
  return cudaGetLastError();
}

}  // namespace mlav
