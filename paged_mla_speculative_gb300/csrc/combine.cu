// Fixed-split LSE combine: the "reduce" half of the partial + reduce design in
// "The Decisive A/B: When Benchmarking Honesty Reveals the Real Bottleneck"
// (section "The Context").
//
// For each query row, with split s holding a normalised output o_s and its
// log-sum-exp lse_s:
//     lse = log sum_s exp(lse_s),   out = sum_s exp(lse_s - lse) * o_s.
// A split with no visible key has lse_s = -inf and weight 0 (its o_s is not
// used).  A NaN lse_s (request rejected by the partial kernel) makes the row
// NaN.  One warp per row; each lane owns 16 of the 512 value dims.
#include "common.cuh"
#include "kernels.h"

#include <cuda_bf16.h>

namespace mlav {
namespace {

constexpr int WARPS = 4;   // rows per CTA: more CTAs over the SMs for the few rows of a call
constexpr int EARLY = 2;   // splits whose rows are loaded before the weights are known
constexpr int GROUP = 4;   // later splits whose rows are in flight together

__global__ void __launch_bounds__(WARPS * 32) combine_kernel(const Params p) {
  // The split partials come from the kernel just before this one on the
  // stream (a no-op when launched without overlap).
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  const int lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * WARPS + (threadIdx.x >> 5);
  if (row >= static_cast<long long>(p.batch) * p.R) return;
  const int b = static_cast<int>(row / p.R);
  const int r = static_cast<int>(row - static_cast<long long>(b) * p.R);
  const int ns = p.nsplit;

  const float L = lane < ns ? p.ws_lse[ws_base(p, b, lane) + r] : -INFINITY;
  float4 early[EARLY][4];
#pragma unroll
  for (int s = 0; s < EARLY; ++s) {
    if (s < ns) {
      const float4* src = reinterpret_cast<const float4*>(p.ws_o + (ws_base(p, b, s) + r) * D_V);
#pragma unroll
      for (int k = 0; k < 4; ++k) early[s][k] = __ldcs(src + lane + 32 * k);
    }
  }
  const bool any_nan = __any_sync(0xffffffffu, L != L);
  float mx = L;
#pragma unroll
  for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const float base = mx == -INFINITY ? 0.f : mx;
  float w = (L == -INFINITY) ? 0.f : ex2((L - base) * kLog2e);
  float tot = w;
#pragma unroll
  for (int o = 16; o; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  w = tot > 0.f ? w / tot : 0.f;

  float4 acc[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  // The first EARLY splits' rows were loaded together with the LSEs (one
  // round trip instead of two); a split of weight 0 adds nothing (its row
  // may be unwritten: it is never used).
#pragma unroll
  for (int s = 0; s < EARLY; ++s) {
    if (s >= ns) break;
    const float ws = __shfl_sync(0xffffffffu, w, s);
    if (ws == 0.f) continue;  // uniform across the warp
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      acc[k].x += ws * early[s][k].x;
      acc[k].y += ws * early[s][k].y;
      acc[k].z += ws * early[s][k].z;
      acc[k].w += ws * early[s][k].w;
    }
  }
  // The rest GROUP splits at a time: every load of a group is issued before
  // any is used, one memory round trip per group instead of one per split.
  for (int s0 = EARLY; s0 < ns; s0 += GROUP) {
    float wg[GROUP];
    float4 v[GROUP][4];
#pragma unroll
    for (int g = 0; g < GROUP; ++g) {
      const int s = s0 + g;   // uniform across the warp, < 32
      wg[g] = s < ns ? __shfl_sync(0xffffffffu, w, s) : 0.f;
      if (wg[g] != 0.f) {
        const float4* src = reinterpret_cast<const float4*>(p.ws_o + (ws_base(p, b, s) + r) * D_V);
#pragma unroll
        for (int k = 0; k < 4; ++k) v[g][k] = __ldcs(src + lane + 32 * k);
      }
    }
#pragma unroll
    for (int g = 0; g < GROUP; ++g) {
      if (wg[g] == 0.f) continue;  // uniform across the warp
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc[k].x += wg[g] * v[g][k].x;
        acc[k].y += wg[g] * v[g][k].y;
        acc[k].z += wg[g] * v[g][k].z;
        acc[k].w += wg[g] * v[g][k].w;
      }
    }
  }
  const float nan = __int_as_float(0x7fc00000);
  const float lse = any_nan ? nan : (tot > 0.f ? base + logf(tot) : -INFINITY);
  if (any_nan) {
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] = make_float4(nan, nan, nan, nan);
  }
  const size_t orow = (static_cast<size_t>(b) * p.R + r) * D_V;
  if (p.out_bf16) {
    uint2* dst = reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(p.out) + orow);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc[k].x, acc[k].y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc[k].z, acc[k].w);
      dst[lane + 32 * k] = make_uint2(*reinterpret_cast<uint32_t*>(&lo),
                                      *reinterpret_cast<uint32_t*>(&hi));
    }
  } else {
    float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + orow);
#pragma unroll
    for (int k = 0; k < 4; ++k) dst[lane + 32 * k] = acc[k];
  }
  if (lane == 0) p.lse[static_cast<size_t>(b) * p.R + r] = lse;
}

}  // namespace

cudaError_t launch_combine(const Params& p, cudaStream_t stream, bool overlap) {
  const long long rows = static_cast<long long>(p.batch) * p.R;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((rows + WARPS - 1) / WARPS));
  cfg.blockDim = dim3(WARPS * 32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, combine_kernel, p);
}

}  // namespace mlav
