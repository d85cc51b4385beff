// Fixed-split LSE combine: the "reduce" half of the partial + reduce design in
// "The Decisive A/B: When Benchmarking Honesty Reveals the Real Bottleneck"
// (section "The Context").
//
// For each query row, with split s holding a normalised output o_s and its
// log-sum-exp lse_s:
//     lse = log sum_s exp(lse_s),   out = sum_s exp(lse_s - lse) * o_s.
// A split with no visible key has lse_s = -inf and weight 0 (its o_s is not
// used).  A NaN lse_s (request rejected by the partial kernel) makes the row
// NaN.  Each thread owns F float4 of a row's 512 value dims (F = 1, 2 or 4 by
// the split count, so that a thread loads at most 16 float4): it issues its
// loads of the row's LSEs and of its float4 of every split before it uses
// any -- one memory round trip (two past 16 splits) -- and the few rows of a
// long-context call spread over many threads (one warp per row would leave
// most SMs idle).  The weights come from a butterfly over a warp's lanes
// (lane l: split l), the accumulation runs in split order.
#include "common.cuh"
#include "kernels.h"

#include <cuda_bf16.h>

namespace mlav {
namespace {

constexpr int CTA = 128;   // threads per CTA
static_assert(MAX_NSPLIT <= 32, "one split per lane for the weights");

// F float4 per thread, CH splits' float4 in flight together.
template <int F, int CH>
__global__ void __launch_bounds__(CTA) combine_kernel(const Params p) {
  constexpr int TPR = D_V / 4 / F;   // threads per row: whole warps
  constexpr int ROWS = CTA / TPR;    // rows per CTA
  static_assert(TPR % 32 == 0 && CTA % TPR == 0, "whole warps per row");
  // The split partials come from the kernel just before this one on the
  // stream (a no-op when launched without overlap).
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  const int t = threadIdx.x % TPR, lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * ROWS + threadIdx.x / TPR;
  if (row >= static_cast<long long>(p.batch) * p.R) return;   // uniform per warp
  const int b = static_cast<int>(row / p.R);
  const int r = static_cast<int>(row - static_cast<long long>(b) * p.R);
  const int ns = p.nsplit;
  // Thread t's float4 of split s: t, t + TPR, .. (each warp load covers 512
  // contiguous bytes).
  auto load = [&](int s, float4 (&x)[F]) {
    const float4* src = reinterpret_cast<const float4*>(p.ws_o + (ws_base(p, b, s) + r) * D_V) + t;
#pragma unroll
    for (int f = 0; f < F; ++f) x[f] = __ldcs(src + TPR * f);
  };

  // Lane l of each warp takes split l's LSE (every warp of the row derives
  // the same weights).
  const float L = lane < ns ? p.ws_lse[ws_base(p, b, lane) + r] : -INFINITY;
  float4 v[CH][F];
#pragma unroll
  for (int s = 0; s < CH; ++s)
    if (s < ns) load(s, v[s]);
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

  // A split of weight 0 adds nothing (its row may be unwritten: never used).
  float4 acc[F];
#pragma unroll
  for (int f = 0; f < F; ++f) acc[f] = make_float4(0.f, 0.f, 0.f, 0.f);
  auto add = [&](int s, const float4 (&x)[F]) {
    const float ws = __shfl_sync(0xffffffffu, w, s);
    if (ws == 0.f) return;   // uniform across the warp
#pragma unroll
    for (int f = 0; f < F; ++f) {
      acc[f].x += ws * x[f].x;
      acc[f].y += ws * x[f].y;
      acc[f].z += ws * x[f].z;
      acc[f].w += ws * x[f].w;
    }
  };
#pragma unroll
  for (int s = 0; s < CH; ++s)
    if (s < ns) add(s, v[s]);
  // Past CH splits (only with F = 1, CH = 16: the launch picks F so that
  // ns <= CH otherwise), the rest in a second round trip.
  if constexpr (CH < MAX_NSPLIT) {
    if (ns > CH) {
      constexpr int REST = MAX_NSPLIT - CH < CH ? MAX_NSPLIT - CH : CH;
#pragma unroll
      for (int s = 0; s < REST; ++s)
        if (CH + s < ns) load(CH + s, v[s]);
#pragma unroll
      for (int s = 0; s < REST; ++s)
        if (CH + s < ns) add(CH + s, v[s]);
    }
  }
  const float nan = __int_as_float(0x7fc00000);
  const float lse = any_nan ? nan : (tot > 0.f ? base + logf(tot) : -INFINITY);
  const size_t orow = (static_cast<size_t>(b) * p.R + r) * D_V;
#pragma unroll
  for (int f = 0; f < F; ++f) {
    const float4 a = any_nan ? make_float4(nan, nan, nan, nan) : acc[f];
    if (p.out_bf16) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(a.z, a.w);
      reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(p.out) + orow)[t + TPR * f] =
          make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
    } else {
      reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + orow)[t + TPR * f] = a;
    }
  }
  if (t == 0) p.lse[static_cast<size_t>(b) * p.R + r] = lse;
}

}  // namespace

cudaError_t launch_combine(const Params& p, cudaStream_t stream, bool overlap) {
  const long long rows = static_cast<long long>(p.batch) * p.R;
  const int ns = p.nsplit;
  if (ns < 1 || ns > MAX_NSPLIT) return cudaErrorInvalidValue;
  // Float4 per thread and splits per round trip: every split in one round
  // trip up to 16 splits (CH >= ns), the rest of up to 32 in a second.
  const int f = ns > 8 ? 1 : (ns > 4 ? 2 : 4);
  const int rows_per_cta = CTA / (D_V / 4 / f);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((rows + rows_per_cta - 1) / rows_per_cta));
  cfg.blockDim = dim3(CTA);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  if (f == 1) return cudaLaunchKernelEx(&cfg, combine_kernel<1, 16>, p);
  if (f == 2) return cudaLaunchKernelEx(&cfg, combine_kernel<2, 8>, p);
  if (ns > 2) return cudaLaunchKernelEx(&cfg, combine_kernel<4, 4>, p);
  return cudaLaunchKernelEx(&cfg, combine_kernel<4, 2>, p);
}

}  // namespace mlav
