// KV compaction: each request's scattered page_size=1 rows copied, in logical
// order, into fresh 64-row pages taken from a free list, and the page_size=64
// table of the same requests written out.  The pages name KV defragmentation
// as a next step after the custom verify kernel ("The Moment of Truth:
// Benchmarking a Custom sm_120 Verify Kernel Against Triton", section "The
// Broader Context: From Kernel to System"), the page_size=1 layout scattering
// every KV access ("The Decisive A/B: When Benchmarking Honesty Reveals the
// Real Bottleneck", section "The Context").
//
// Definition (per request b, in batch order):
//   n_b        = kv_lens[b]; the request gets no pages when n_b is outside
//                [0, max_kv_len] (ERR_LEN) or its indptr range does not hold
//                n_b slots inside [0, kv_indptr[batch]) (ERR_INDPTR);
//   pages      = the next ceil(n_b / 64) free pages; the longest leading run of
//                requests whose pages fit keeps them, later requests get none
//                (ERR_CAPACITY);
//   row j      -> slot page[j / 64] * 64 + j % 64 of the destination cache (a
//                source slot outside the source cache is copied as zeros, a
//                page outside the destination cache is not written: ERR_SLOT);
//   page_indptr = exclusive prefix sum of the kept page counts; page_table =
//                the consumed prefix of the free list.
#include "common.cuh"
#include "kernels.h"

namespace mlav {
namespace {

constexpr int SCAN_THREADS = 1024;
constexpr int COPY_THREADS = 256;
constexpr int ROWS_PER_THREAD = PAGE * ROW_CHUNKS / COPY_THREADS;   // 18 vectors of 16 B
static_assert(ROWS_PER_THREAD * COPY_THREADS == PAGE * ROW_CHUNKS, "even split of a page");

__global__ void __launch_bounds__(SCAN_THREADS) compact_scan_kernel(const CompactArgs a) {
  __shared__ long long s_warp[SCAN_THREADS / 32];
  __shared__ long long s_fit[SCAN_THREADS / 32];
  __shared__ long long s_carry, s_last_fit;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    s_carry = 0;
    s_last_fit = 0;
    a.page_indptr[0] = 0;
  }
  __syncthreads();
  for (int base = 0; base < a.batch; base += SCAN_THREADS) {
    const int b = base + tid;
    long long count = 0;
    if (b < a.batch) {
      const long long n = a.kv_lens[b];
      const long long p0 = a.kv_indptr[b], p1 = a.kv_indptr[b + 1];
      if (n < 0 || n > a.max_kv_len) {
        atomicOr(a.err, ERR_LEN);
      } else if (p0 < 0 || p1 - p0 != n || p1 > a.kv_indptr[a.batch]) {
        atomicOr(a.err, ERR_INDPTR);
      } else {
        count = (n + PAGE - 1) / PAGE;
      }
    }
    long long x = count;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
      long long t = s_warp[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, t, o);
        if (lane >= o) t += y;
      }
      s_warp[lane] = t;
    }
    __syncthreads();
    const long long full_end = s_carry + (warp > 0 ? s_warp[warp - 1] : 0) + x;
    const bool fits = full_end <= a.num_free_pages;
    long long fit_end = (b < a.batch && fits) ? full_end : 0;
#pragma unroll
    for (int o = 16; o; o >>= 1) fit_end = max(fit_end, __shfl_xor_sync(0xffffffffu, fit_end, o));
    if (lane == 0) s_fit[warp] = fit_end;
    __syncthreads();
    if (tid == 0) {
      long long m = s_last_fit;
      for (int w = 0; w < SCAN_THREADS / 32; ++w) m = max(m, s_fit[w]);
      s_last_fit = m;
    }
    __syncthreads();
    if (b < a.batch) {
      if (!fits && count > 0) atomicOr(a.err, ERR_CAPACITY);
      a.page_indptr[b + 1] = static_cast<int32_t>(fits ? full_end : s_last_fit);
    }
    __syncthreads();
    if (tid == SCAN_THREADS - 1) s_carry = full_end;
    __syncthreads();
  }
  // The consumed prefix of the free list is the page table.
  const long long total = s_last_fit;
  for (long long i = tid; i < total; i += SCAN_THREADS) a.page_table[i] = a.free_pages[i];
}

// grid (ceil(max_kv_len / 64), batch): CTA (i, b) writes page i of request b.
__global__ void __launch_bounds__(COPY_THREADS) compact_copy_kernel(const CompactArgs a) {
  const int b = blockIdx.y, i = blockIdx.x, tid = threadIdx.x;
  const int p0 = a.page_indptr[b], p1 = a.page_indptr[b + 1];
  if (i >= p1 - p0) return;                 // request cut, invalid, or shorter
  const long long page = a.free_pages[p0 + i];
  if (page < 0 || (page + 1) * PAGE > a.dst_slots) {
    if (tid == 0) atomicOr(a.err, ERR_SLOT);
    return;
  }
  const int n = a.kv_lens[b];
  const int row0 = i * PAGE;
  const int rows = min(PAGE, n - row0);
  const int32_t* idx = a.kv_indices + a.kv_indptr[b] + row0;
  const uint4* src = static_cast<const uint4*>(a.kv_src);
  uint4* dst = static_cast<uint4*>(a.kv_dst) + page * PAGE * ROW_CHUNKS;
  uint4 v[ROWS_PER_THREAD];
  bool bad = false;
#pragma unroll
  for (int u = 0; u < ROWS_PER_THREAD; ++u) {
    const int e = tid + u * COPY_THREADS;
    const int r = e / ROW_CHUNKS, c = e - r * ROW_CHUNKS;
    v[u] = make_uint4(0, 0, 0, 0);
    if (r < rows) {
      const long long s = idx[r];
      if (s >= 0 && s < a.src_slots) v[u] = __ldg(src + s * ROW_CHUNKS + c);
      else bad = true;
    }
  }
#pragma unroll
  for (int u = 0; u < ROWS_PER_THREAD; ++u) {
    const int e = tid + u * COPY_THREADS;
    if (e / ROW_CHUNKS < rows) dst[e] = v[u];
  }
  if (bad) atomicOr(a.err, ERR_SLOT);
}

}  // namespace

cudaError_t launch_compact_kv(const CompactArgs& a, cudaStream_t stream) {
  compact_scan_kernel<<<1, SCAN_THREADS, 0, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 grid((a.max_kv_len + PAGE - 1) / PAGE, a.batch);
  compact_copy_kernel<<<grid, COPY_THREADS, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mlav
