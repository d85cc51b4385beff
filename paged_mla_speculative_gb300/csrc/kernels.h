// Internal launch interface between the C ABI and the kernels.
#pragma once

#include <cuda.h>   // CUtensorMap (a plain struct; the library does not link the driver)
#include <cuda_runtime.h>

#include "common.cuh"

namespace mlav {

// Split-KV partial kernel on warp-level mma.sync.
int partial_mma_smem_bytes();
cudaError_t partial_mma_prepare();
cudaError_t launch_partial_mma(const Params& p, cudaStream_t stream);

// Split-KV partial kernel on tcgen05 tensor cores with TMEM accumulators.
cudaError_t partial_tc_prepare();
// `overlap`: launch with programmatic stream serialisation, so the kernel's
// CTAs may start while the previous kernel on the stream (the pack) runs;
// the kernel then reads each packed block after its ready flags carry the
// call's tag (Params::pack_flags = 1), or after griddepcontrol.wait, which
// waits for the whole pack grid (pack_flags = 0).
cudaError_t launch_partial_tc(const Params& p, cudaStream_t stream, bool overlap);

// Split-KV partial kernel on CTA pairs (cta_group::2), 128 query rows and
// 256 keys per step, over the packed blocks (Params::split_pairs = 1);
// `overlap` as for launch_partial_tc.  The packed buffer is read through two
// TMA tensor maps (make_pack_maps): rows of 128 bytes, boxes of 256 rows (a
// chunk pair) and of 128 rows (one chunk).
struct PackMaps {
  CUtensorMap pair;    // box 64 x 256 fp16
  CUtensorMap chunk;   // box 64 x 128 fp16
};
cudaError_t make_pack_maps(PackMaps* maps, void* packed, size_t packed_bytes);
cudaError_t partial_pair_prepare();
cudaError_t launch_partial_pair(const Params& p, const PackMaps& maps, cudaStream_t stream, bool overlap);

// Per-call gather of the key rows into packed fp16 operand tiles.
size_t packed_block_bytes();
// The whole pack ahead of the attention kernel (Params::pack_flags = 0).
cudaError_t launch_pack_kv(const Params& p, void* packed, int max_blocks, cudaStream_t stream);
// The two-phase pack that overlaps the attention kernel (pack_flags = 1):
// num_ctas persistent CTAs (one per SM); CTAs stay .. num_ctas-1 pack the
// first `wide_positions` blocks of every split and exit, CTAs 0 .. stay-1
// pack the rest.  pack_kv_prepare sets its shared-memory attributes.
cudaError_t pack_kv_prepare();
cudaError_t launch_pack_kv_overlap(const Params& p, void* packed, int max_blocks, int num_ctas,
                                   int wide_positions, int stay, cudaStream_t stream);

// LSE combine of the split partials into out/lse (`overlap`: may be
// scheduled early; it waits for the partial kernel with griddepcontrol.wait).
cudaError_t launch_combine(const Params& p, cudaStream_t stream, bool overlap);

// Up to kMax copies between device-addressable regions (device memory, or
// page-locked host memory mapped into the device's address space) in one
// kernel launch.  Byte counts are multiples of 4.
struct CopyRegions {
  static constexpr int kMax = 8;
  const void* src[kMax];
  void* dst[kMax];
  long long bytes[kMax];
  int n;
};
cudaError_t launch_copy_regions(const CopyRegions& c, cudaStream_t stream);

// Per-step index builder (index_builder.cu).
struct IndexArgs {
  const int32_t* req_to_token;      // [pool_size][stride] cache slot of each token position
  long long stride;                 // entries per table row (>= max_kv_len)
  int pool_size;
  const int32_t* req_pool_indices;  // [batch]
  const int32_t* prefix_lens;       // [batch]
  int batch, T, page_size, max_kv_len;
  long long capacity;               // entries kv_indices holds (<= INT32_MAX)
  int32_t* kv_indices;
  int32_t* kv_indptr;               // [batch + 1]
  int32_t* kv_lens;                 // [batch]
  int* err;
};
cudaError_t launch_build_indices(const IndexArgs& a, int max_kv_len, cudaStream_t stream);

// KV compaction into 64-row pages (compact.cu).
struct CompactArgs {
  const void* kv_src;               // bf16 [src_slots][576]
  long long src_slots;
  const int32_t* kv_indices;        // page_size 1 slot table of the requests
  const int32_t* kv_indptr;         // [batch + 1]
  const int32_t* kv_lens;           // [batch]
  const int32_t* free_pages;        // [num_free_pages] destination page ids, used in order
  long long num_free_pages;
  void* kv_dst;                     // bf16 [dst_slots][576], dst_slots a multiple of 64
  long long dst_slots;
  int32_t* page_table;              // [num_free_pages] out
  int32_t* page_indptr;             // [batch + 1] out
  int batch, max_kv_len;
  int* err;
};
cudaError_t launch_compact_kv(const CompactArgs& a, cudaStream_t stream);

}  // namespace mlav
