// Allocation-free entry point: the verify attention for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc at all: code running inside a memory
// pool that owns the whole device, a host process that must not allocate
// after start-up (latency-critical serving loops), or a layer that is only
// handed pointers by an outer framework.  For them mla_verify_attn_static
// runs the mma.sync family's split-KV partial kernel and the LSE combine
// with the split partials kept in a file-scope device array of fixed size,
// instead of in a plan's cudaMalloc'd workspace.
//
// The array is a module-scope __device__ object: every GPU that loads this
// library holds it until the process exits, and every call on a device
// shares it.  Its device address is looked up with cudaGetSymbolAddress once
// per device, on that device's first call (which should therefore come
// before any stream capture).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "kernels.h"
#include "mla_verify.h"

namespace {

constexpr int kMaxDevices = 64;

// Split partials (normalised O and LSE per split) and one fallback error word.
static __device__ __align__(256) unsigned char g_static_scratch[MLA_VERIFY_STATIC_SCRATCH_BYTES];

std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices];
bool g_ready[kMaxDevices];

// Once per device, with that device current: the scratch array's device
// address and the partial kernel's shared-memory attribute.
int setup_device(int dev, void** scratch) {
  if (dev < 0 || dev >= kMaxDevices) return MLA_VERIFY_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_ready[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || ptr == nullptr)
      return MLA_VERIFY_ERR_CUDA;
    if (mlav::partial_mma_prepare() != cudaSuccess) return MLA_VERIFY_ERR_CUDA;
    g_scratch_addr[dev] = ptr;
    g_ready[dev] = true;
  }
  *scratch = g_scratch_addr[dev];
  return MLA_VERIFY_OK;
}

// A CUDA call of this entry failed: the cached address may belong to a
// context that no longer exists (cudaDeviceReset), so the next call on the
// device repeats the set-up.
int forget_device(int dev) {
  cudaGetLastError();
  std::lock_guard<std::mutex> lock(g_setup_mu);
  g_ready[dev] = false;
  return MLA_VERIFY_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int mla_verify_attn_static(int batch, int num_drafts, int num_heads, int page_size,
                                      int64_t num_slots, int max_kv_len, int nsplit,
                                      const void* q, const void* kv_cache,
                                      const int32_t* kv_indices, const int32_t* kv_indptr,
                                      const int32_t* kv_lens, const int32_t* draft_parent,
                                      float scale, float* out, float* lse, int* device_status,
                                      void* stream) {
  if (!q || !kv_cache || !kv_indices || !kv_indptr || !kv_lens || !draft_parent || !out || !lse)
    return MLA_VERIFY_ERR_NULL;
  if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(kv_indices) || !aligned16(kv_indptr) ||
      !aligned16(kv_lens) || !aligned16(draft_parent) || !aligned16(out) || !aligned16(lse))
    return MLA_VERIFY_ERR_ALIGN;
  if (batch < 1) return MLA_VERIFY_ERR_BATCH;
  if (num_drafts < 1 || num_drafts > mlav::MAX_T || num_heads < 1 ||
      static_cast<long long>(num_drafts) * num_heads > 4096 ||
      (page_size != 1 && page_size != mlav::PAGE) || num_slots < 1 || num_slots > INT32_MAX ||
      (page_size == mlav::PAGE && num_slots % mlav::PAGE) || max_kv_len < num_drafts ||
      nsplit < 1 || nsplit > mlav::MAX_NSPLIT)
    return MLA_VERIFY_ERR_SHAPE;
  if (!std::isfinite(scale)) return MLA_VERIFY_ERR_SCALE;
  const int R = num_drafts * num_heads;
  // Split partials plus the fallback error word must fit the fixed array.
  const unsigned long long need = nsplit > 1
      ? 1ULL * batch * nsplit * R * (mlav::D_V + 1) * sizeof(float) + 256
      : 256;
  if (need > MLA_VERIFY_STATIC_SCRATCH_BYTES) return MLA_VERIFY_ERR_SCRATCH;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_VERIFY_ERR_CUDA;
  void* scratch = nullptr;
  const int st = setup_device(dev, &scratch);
  if (st != MLA_VERIFY_OK) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned char* base = static_cast<unsigned char*>(scratch);
  int* err = device_status;
  if (!err) {
    // The fallback word is shared by every call and keeps the last call's
    // bits: clear it first.
    err = reinterpret_cast<int*>(base + MLA_VERIFY_STATIC_SCRATCH_BYTES - 256);
    if (cudaMemsetAsync(err, 0, sizeof(int), s) != cudaSuccess) return forget_device(dev);
  }

  mlav::Params p{};
  p.q = static_cast<const uint16_t*>(q);
  p.kv = static_cast<const uint16_t*>(kv_cache);
  p.kv_indices = kv_indices;
  p.kv_indptr = kv_indptr;
  p.kv_lens = kv_lens;
  p.draft_parent = draft_parent;
  p.scale_log2 = scale * mlav::kLog2e;
  p.batch = batch;
  p.T = num_drafts;
  p.H = num_heads;
  p.R = R;
  p.page_size = page_size;
  p.num_slots = num_slots;
  p.max_kv_len = max_kv_len;
  p.nsplit = nsplit;
  p.shard = 0;
  p.num_shards = 1;
  p.ws_stride_b = 1LL * nsplit * R;
  p.ws_stride_s = R;
  // Every (request, split, row) partial is written before the combine reads
  // it, so the array needs no clearing between calls.
  p.ws_o = reinterpret_cast<float*>(base);
  p.ws_lse = reinterpret_cast<float*>(base) + static_cast<size_t>(batch) * nsplit * R * mlav::D_V;
  p.out = out;
  p.lse = lse;
  p.out_bf16 = 0;
  p.err = err;
  if (mlav::launch_partial_mma(p, s) != cudaSuccess) return forget_device(dev);
  if (nsplit > 1 && mlav::launch_combine(p, s, false) != cudaSuccess) return forget_device(dev);
  return MLA_VERIFY_OK;
}
