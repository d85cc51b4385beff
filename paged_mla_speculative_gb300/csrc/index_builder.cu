// Per-step index builder: the request-to-token table of the serving stack
// turned into the kv_lens / kv_indptr / kv_indices the verify attention
// reads, on the GPU and in the same stream (so a whole step, indices and
// attention, can be captured into one CUDA graph).
//
// The pages trace the custom verify kernel's short-context loss to index
// arrays rebuilt on the host for every layer, and name two remedies: build the
// combined indices once per step, or do that work in a kernel on the GPU
// ("The Moment of Truth: Benchmarking a Custom sm_120 Verify Kernel Against
// Triton", sections "Interpreting the Crossover: The Marshaling Tax" and
// "Assumptions and Their Validity").  This is that kernel.
//
// Definition (per request b of the step):
//   n_b      = prefix_lens[b] + T, or 0 when the pool row, the prefix or n_b
//              is out of range (ERR_POOL; the attention then rejects b);
//   count_b  = n_b slots (page_size 1) or ceil(n_b / 64) page ids;
//   indptr   = exclusive prefix sum of count; the longest leading run of
//              requests whose entries fit in `capacity` keeps them, every
//              later request gets n_b = 0 (ERR_CAPACITY);
//   entries  = req_to_token[pool_b, 0 .. n_b-1] (page_size 1), or
//              req_to_token[pool_b, 64 i] / 64 for page i (page_size 64; a
//              first slot that is negative or not a multiple of 64 gives -1
//              and ERR_SLOT).
#include "common.cuh"
#include "kernels.h"

namespace mlav {
namespace {

constexpr int SCAN_THREADS = 1024;
constexpr int COPY_THREADS = 256;

// One CTA: validation, counts, prefix sums (64-bit), capacity cut.
__global__ void __launch_bounds__(SCAN_THREADS) index_scan_kernel(const IndexArgs a) {
  __shared__ long long s_warp[SCAN_THREADS / 32];
  __shared__ long long s_fit[SCAN_THREADS / 32];
  __shared__ long long s_carry, s_last_fit;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    s_carry = 0;
    s_last_fit = 0;
    a.kv_indptr[0] = 0;
  }
  __syncthreads();
  for (int base = 0; base < a.batch; base += SCAN_THREADS) {
    const int b = base + tid;
    long long n = 0, count = 0;
    if (b < a.batch) {
      const long long pool = a.req_pool_indices[b];
      const long long prefix = a.prefix_lens[b];
      n = prefix + a.T;
      const bool valid = pool >= 0 && pool < a.pool_size && prefix >= 0 && n <= a.max_kv_len;
      if (!valid) {
        atomicOr(a.err, ERR_POOL);
        n = 0;
      }
      count = a.page_size == 1 ? n : (n + PAGE - 1) / PAGE;
    }
    // Inclusive scan of count over the block: warp shuffles, then warp totals.
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
      s_warp[lane] = t;   // inclusive warp-total prefix
    }
    __syncthreads();
    const long long full_end = s_carry + (warp > 0 ? s_warp[warp - 1] : 0) + x;
    const bool fits = full_end <= a.capacity;
    // Entries end at full_end, which never decreases with b: the requests that
    // fit are a leading run, and a cut request's indptr repeats the end of the
    // last request that fits (this chunk's largest fitting end, or an earlier one).
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
      a.kv_lens[b] = fits ? static_cast<int32_t>(n) : 0;
      a.kv_indptr[b + 1] = static_cast<int32_t>(fits ? full_end : s_last_fit);
    }
    __syncthreads();
    if (tid == SCAN_THREADS - 1) s_carry = full_end;
    __syncthreads();
  }
}

// grid (ceil(max entries per request / 256), batch): one entry per thread.
__global__ void __launch_bounds__(COPY_THREADS) index_copy_kernel(const IndexArgs a) {
  const int b = blockIdx.y;
  const int n = a.kv_lens[b];
  if (n == 0) return;
  const int count = a.page_size == 1 ? n : (n + PAGE - 1) / PAGE;
  const int j = blockIdx.x * COPY_THREADS + threadIdx.x;
  if (j >= count) return;
  const int32_t* row = a.req_to_token + static_cast<long long>(a.req_pool_indices[b]) * a.stride;
  int32_t* dst = a.kv_indices + a.kv_indptr[b];
  if (a.page_size == 1) {
    dst[j] = row[j];
  } else {
    const int32_t first = row[static_cast<long long>(j) * PAGE];
    const bool ok = first >= 0 && first % PAGE == 0;
    if (!ok) atomicOr(a.err, ERR_SLOT);
    dst[j] = ok ? first / PAGE : -1;
  }
}

// Batches up to FUSED_MAX_BATCH: one launch.  CTA (x, b) scans the entry
// counts of requests 0..b itself (<= 4 per thread), which gives request b's
// offset and the capacity cut, then copies entries
// [x * FUSED_CHUNK, (x+1) * FUSED_CHUNK) of request b; the CTAs with x == 0
// also write kv_lens[b] and kv_indptr[b+1] (and b == 0 kv_indptr[0]).  Same
// results as the scan + copy pair, without the dependent round trip between
// two launches.
constexpr int FUSED_THREADS = 256;
constexpr int FUSED_MAX_BATCH = 1024;
constexpr int FUSED_PER_THREAD = FUSED_MAX_BATCH / FUSED_THREADS;   // 4
constexpr int FUSED_CHUNK = FUSED_THREADS * 8;                      // entries per CTA

__global__ void __launch_bounds__(FUSED_THREADS) index_fused_kernel(const IndexArgs a) {
  __shared__ long long s_warp[FUSED_THREADS / 32];
  __shared__ long long s_fit[FUSED_THREADS / 32];
  __shared__ long long s_end[FUSED_THREADS / 32];
  __shared__ long long s_n[FUSED_THREADS / 32];
  const int b = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // Requests tid*4 .. tid*4+3 (only those <= b matter).
  long long cnt[FUSED_PER_THREAD], n_own = 0;
  long long local = 0;
#pragma unroll
  for (int k = 0; k < FUSED_PER_THREAD; ++k) {
    const int i = tid * FUSED_PER_THREAD + k;
    long long c = 0;
    if (i <= b) {
      const long long pool = a.req_pool_indices[i];
      const long long prefix = a.prefix_lens[i];
      long long n = prefix + a.T;
      const bool valid = pool >= 0 && pool < a.pool_size && prefix >= 0 && n <= a.max_kv_len;
      if (!valid) n = 0;
      if (i == b) {
        n_own = n;
        if (!valid && blockIdx.x == 0) atomicOr(a.err, ERR_POOL);
      }
      c = a.page_size == 1 ? n : (n + PAGE - 1) / PAGE;
    }
    cnt[k] = c;
    local += c;
  }
  // Exclusive prefix of the per-thread totals over the block.
  long long x = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  long long before = x - local;
  for (int w = 0; w < warp; ++w) before += s_warp[w];
  // Inclusive ends of this thread's requests; the largest end that fits.
  long long end = before, fit = 0, end_b = 0;
#pragma unroll
  for (int k = 0; k < FUSED_PER_THREAD; ++k) {
    const int i = tid * FUSED_PER_THREAD + k;
    end += cnt[k];
    if (i <= b && end <= a.capacity) fit = max(fit, end);
    if (i == b) end_b = end;
  }
  // Only the thread holding request b knows its end and length: broadcast
  // them (the other threads contribute 0) with the largest fitting end.
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    fit = max(fit, __shfl_xor_sync(0xffffffffu, fit, o));
    end_b = max(end_b, __shfl_xor_sync(0xffffffffu, end_b, o));
    n_own = max(n_own, __shfl_xor_sync(0xffffffffu, n_own, o));
  }
  if (lane == 0) {
    s_fit[warp] = fit;
    s_end[warp] = end_b;
    s_n[warp] = n_own;
  }
  __syncthreads();
  long long last_fit = 0, full_end = 0;
  for (int w = 0; w < FUSED_THREADS / 32; ++w) {
    last_fit = max(last_fit, s_fit[w]);
    full_end = max(full_end, s_end[w]);
    n_own = max(n_own, s_n[w]);
  }
  const long long count = a.page_size == 1 ? n_own : (n_own + PAGE - 1) / PAGE;
  const bool fits = full_end <= a.capacity;
  if (blockIdx.x == 0 && tid == 0) {
    if (!fits && count > 0) atomicOr(a.err, ERR_CAPACITY);
    a.kv_lens[b] = fits ? static_cast<int32_t>(n_own) : 0;
    a.kv_indptr[b + 1] = static_cast<int32_t>(fits ? full_end : last_fit);
    if (b == 0) a.kv_indptr[0] = 0;
  }
  if (!fits || count == 0) return;
  const long long start = full_end - count;
  const int32_t* row = a.req_to_token + static_cast<long long>(a.req_pool_indices[b]) * a.stride;
  for (long long j = static_cast<long long>(blockIdx.x) * FUSED_CHUNK + tid;
       j < min(count, static_cast<long long>(blockIdx.x + 1) * FUSED_CHUNK); j += FUSED_THREADS) {
    if (a.page_size == 1) {
      a.kv_indices[start + j] = row[j];
    } else {
      const int32_t first = row[j * PAGE];
      const bool ok = first >= 0 && first % PAGE == 0;
      if (!ok) atomicOr(a.err, ERR_SLOT);
      a.kv_indices[start + j] = ok ? first / PAGE : -1;
    }
  }
}

}  // namespace

cudaError_t launch_build_indices(const IndexArgs& a, int max_kv_len, cudaStream_t stream) {
  const int max_entries = a.page_size == 1 ? max_kv_len : (max_kv_len + PAGE - 1) / PAGE;
  if (a.batch <= FUSED_MAX_BATCH) {
    const dim3 grid((max_entries + FUSED_CHUNK - 1) / FUSED_CHUNK, a.batch);
    index_fused_kernel<<<grid, FUSED_THREADS, 0, stream>>>(a);
    return cudaGetLastError();
  }
  index_scan_kernel<<<1, SCAN_THREADS, 0, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 grid((max_entries + COPY_THREADS - 1) / COPY_THREADS, a.batch);
  index_copy_kernel<<<grid, COPY_THREADS, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mlav
