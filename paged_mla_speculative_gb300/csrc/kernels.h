// Internal launch interface between the C ABI and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace mlav {

// Split-KV partial kernel on warp-level mma.sync.
int partial_mma_smem_bytes();
cudaError_t partial_mma_prepare();
cudaError_t launch_partial_mma(const Params& p, cudaStream_t stream);

// Split-KV partial kernel on tcgen05 tensor cores with TMEM accumulators.
cudaError_t partial_tc_prepare();
cudaError_t launch_partial_tc(const Params& p, const CUtensorMap& kv_map, cudaStream_t stream);

// 2-D tensor map over the cache rows ([num_slots, 576] bf16, 1152-byte rows)
// with a 64-element x 1-row box and 128-byte swizzle, for tile::gather4.
cudaError_t encode_kv_map(CUtensorMap* map, const void* kv_cache, long long num_slots);

// LSE combine of the split partials into out/lse.
cudaError_t launch_combine(const Params& p, cudaStream_t stream);

}  // namespace mlav
