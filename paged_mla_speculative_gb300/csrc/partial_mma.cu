// Split-KV partial kernel built on warp-level mma.sync (m16n8k16, fp16 in,
// fp32 accumulate), O kept in registers.
//
// One CTA = one request b, one tile of 64 query rows (r = t*H + h), one key
// split.  The split's keys stream through shared memory in blocks of 64
// gathered rows (16-byte cp.async vectors, double buffered), which is the
// KV-split "partial" half of the partial + reduce design in "The Decisive
// A/B: When Benchmarking Honesty Reveals the Real Bottleneck" (sections "The
// Context" and "What This Reveals About the Bottleneck": KV split for
// occupancy, 128-bit vector loads of scattered page_size=1 rows).
//
// Per key block (8 warps; warp w owns rows 16*(w%4)..+16):
//   1. convert the staged bf16 block to fp16 in place;
//   2. S = Q K^T, warp w computing keys 32*(w/4)..+32 of its rows over 576 dims;
//   3. mask (prefix visible; draft key i visible to draft t iff i is t or an
//      ancestor of t), exact block max shared between the two warps of a row
//      group, P = 2^(S - m) rounded to fp16 into shared memory;
//   4. O = alpha * O + P V, warp w accumulating value dims 256*(w/4)..+256.
// The split's normalised O and natural-log LSE go to the workspace (or
// straight to out/lse when there is one split).
#include "common.cuh"
#include "kernels.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace mlav {
namespace {

constexpr int BM = 64;          // query rows per CTA
constexpr int BN = 64;          // keys per block
constexpr int NTHREADS = 256;
constexpr int SMEM_Q = BM * ROW_BYTES;
constexpr int SMEM_KV = BN * ROW_BYTES;
constexpr int SMEM_P = BM * BN * 2;
constexpr int OFF_KV0 = SMEM_Q;
constexpr int OFF_KV1 = OFF_KV0 + SMEM_KV;
constexpr int OFF_P = OFF_KV1 + SMEM_KV;
constexpr int OFF_RED = OFF_P + SMEM_P;          // float [2][64]: block max / row sums
constexpr int OFF_SLOT = OFF_RED + 2 * 64 * 4;    // int32 [3][64]: slot of each key, -1 if none
constexpr int OFF_MASK = OFF_SLOT + 3 * 64 * 4;   // uint32 [32]: ancestor masks
constexpr int OFF_PAR = OFF_MASK + MAX_T * 4;     // int32 [32]: draft parents
constexpr int SMEM_TOTAL = OFF_PAR + MAX_T * 4;
static_assert(SMEM_TOTAL <= 232448, "shared memory budget");

// Byte offset of 16-byte chunk `c` of row `r` in a tile of 72-chunk rows.
// XOR-ing the chunk with (r & 7) spreads the 8 rows an ldmatrix reads over
// all banks (the 1152-byte row stride is a multiple of 128).
__device__ __forceinline__ uint32_t sw_row(int r, int c) {
  return static_cast<uint32_t>(r * ROW_BYTES + ((c ^ (r & 7)) << 4));
}
// Same for the 64-key P tile (8 chunks per row).
__device__ __forceinline__ uint32_t sw_p(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// bf16 -> fp16 for a tile of `rows` 1152-byte rows, in place; `bad` records
// a value outside the fp16 range.
__device__ __forceinline__ void widen_tile(uint8_t* tile, int rows, int tid, bool& bad) {
  const int chunks = rows * ROW_CHUNKS;
  for (int c = tid; c < chunks; c += NTHREADS) {
    uint4* ptr = reinterpret_cast<uint4*>(tile + c * 16);
    *ptr = widen_bf16x8(*ptr, bad);
  }
}

// Slot of key r of block kb, or -1 past the end of the request or when the
// table points outside the cache (reported).
__device__ __forceinline__ int block_slot(const Params& p, const Request& rq, int kb, int r) {
  const int j = kb * BN + r;
  if (j < rq.lo || j >= rq.hi) return -1;
  const long long s = key_slot(p, rq.ip0, j);
  if (s < 0) atomicOr(p.err, ERR_SLOT);
  return static_cast<int>(s);
}

// Gather the 64 rows of one key block into a stage with 16-byte cp.async
// vectors; rows without a slot are zero-filled.
__device__ __forceinline__ void load_kv_block(const Params& p, const int* slots, uint8_t* stage,
                                              int tid) {
  const uint32_t base = smem_u32(stage);
#pragma unroll 2
  for (int c = tid; c < BN * ROW_CHUNKS; c += NTHREADS) {
    const int r = c / ROW_CHUNKS;
    const int ch = c - r * ROW_CHUNKS;
    const int slot = slots[r];
    const uint16_t* src = slot >= 0 ? p.kv + static_cast<long long>(slot) * D_QK + ch * 8 : p.kv;
    cp_async16(base + sw_row(r, ch), src, slot >= 0 ? 16 : 0);
  }
}

__global__ void __launch_bounds__(NTHREADS, 1) partial_mma_kernel(const Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int split = blockIdx.x, rt = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rg = warp & 3;       // row group: rows rg*16 .. +16
  const int half = warp >> 2;    // key half (for S) and value half (for O)
  const int row0 = rt * BM;

  float* s_red = reinterpret_cast<float*>(smem + OFF_RED);
  int* s_slot = reinterpret_cast<int*>(smem + OFF_SLOT);
  uint32_t* s_mask = reinterpret_cast<uint32_t*>(smem + OFF_MASK);

  const Request rq = load_request(p, b);
  const size_t ws_row = ws_base(p, b, split);

  // Rows of this thread's accumulator fragments (local to the 64-row tile).
  const int lrA = rg * 16 + (lane >> 2);
  const int lrB = lrA + 8;

  if (!rq.ok) {
    if (split == 0 && rt == 0 && tid == 0) {
      const int n = rq.n;
      atomicOr(p.err, (n < p.T || n > p.max_kv_len) ? ERR_LEN : ERR_INDPTR);
    }
    // The whole request is reported as NaN.
    const float nan = __int_as_float(0x7fc00000);
    for (int i = tid; i < BM * D_V; i += NTHREADS) {
      const int lr = i / D_V, d = i - lr * D_V;
      const int gr = row0 + lr;
      if (gr >= p.R) continue;
      if (p.nsplit == 1) {
        const size_t o = (static_cast<size_t>(b) * p.R + gr) * D_V + d;
        if (p.out_bf16) reinterpret_cast<uint16_t*>(p.out)[o] = 0x7fc0;
        else reinterpret_cast<float*>(p.out)[o] = nan;
        if (d == 0) p.lse[static_cast<size_t>(b) * p.R + gr] = nan;
      } else {
        p.ws_o[(ws_row + gr) * D_V + d] = nan;
        if (d == 0) p.ws_lse[ws_row + gr] = nan;
      }
    }
    return;
  }

  int kb0, kb1;
  split_blocks(rq, BN, split, p.nsplit, kb0, kb1);

  // Parents in one parallel load; the chains are walked in shared memory
  // after the barrier (a walk through global memory costs one round trip a
  // step), and the main loop's barriers order the masks before their use.
  int* s_par = reinterpret_cast<int*>(smem + OFF_PAR);
  if (tid < p.T) s_par[tid] = p.draft_parent[b * p.T + tid];
  // Slots of the first two blocks; later blocks' slots are fetched one
  // iteration ahead so the gather never waits on an index load.
  if (tid < BN && kb1 > kb0) {
    s_slot[tid] = block_slot(p, rq, kb0, tid);
    if (kb0 + 1 < kb1) s_slot[BN + tid] = block_slot(p, rq, kb0 + 1, tid);
  }
  __syncthreads();

  // Q tile: rows beyond R are zero.
  if (kb1 > kb0) {
    const uint32_t qbase = smem_u32(smem);
    const uint16_t* qb = p.q + static_cast<size_t>(b) * p.R * D_QK;
#pragma unroll 1
    for (int c = tid; c < BM * ROW_CHUNKS; c += NTHREADS) {
      const int r = c / ROW_CHUNKS, ch = c - r * ROW_CHUNKS;
      const int gr = row0 + r;
      const bool in = gr < p.R;
      cp_async16(qbase + sw_row(r, ch), in ? qb + static_cast<size_t>(gr) * D_QK + ch * 8 : p.q,
                 in ? 16 : 0);
    }
    cp_async_commit();
    load_kv_block(p, s_slot, smem + OFF_KV0, tid);
    cp_async_commit();
  }
  if (tid < p.T) s_mask[tid] = ancestor_mask(s_par, tid, p.err);

  float o[32][4];
#pragma unroll
  for (int i = 0; i < 32; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;

  const int grA = row0 + lrA, grB = row0 + lrB;
  const int tA = grA < p.R ? grA / p.H : -1;
  const int tB = grB < p.R ? grB / p.H : -1;

  const uint32_t sq = smem_u32(smem);
  const uint32_t sp = smem_u32(smem + OFF_P);

#pragma unroll 1
  for (int kb = kb0; kb < kb1; ++kb) {
    const int it = kb - kb0;
    const int st = it & 1;
    const int ring = it % 3;
    uint8_t* stage = smem + (st ? OFF_KV1 : OFF_KV0);
    int pending = -1;
    if (tid < BN && kb + 2 < kb1) pending = block_slot(p, rq, kb + 2, tid);
    if (kb + 1 < kb1) {
      load_kv_block(p, s_slot + ((it + 1) % 3) * BN, smem + (st ? OFF_KV0 : OFF_KV1), tid);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    {
      bool bad = false;
      widen_tile(stage, BN, tid, bad);
      if (kb == kb0) widen_tile(smem, BM, tid, bad);
      report_range(bad, p.err);
    }
    __syncthreads();

    const uint32_t skv = smem_u32(stage);
    // ---- S = Q K^T over 576 dims: 16 rows x 32 keys per warp.
    float s[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
    {
      const int arow = rg * 16 + (lane & 15);
      const int acol = lane >> 4;
      const int krow0 = half * 32 + ((lane >> 4) << 3) + (lane & 7);
      const int kcol = (lane >> 3) & 1;
#pragma unroll 4
      for (int ks = 0; ks < D_QK / 16; ++ks) {
        uint32_t a[4];
        ldsm4(a, sq + sw_row(arow, ks * 2 + acol));
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
          uint32_t bb[4];
          ldsm4(bb, skv + sw_row(krow0 + pr * 16, ks * 2 + kcol));
          mma16816(s[pr * 2 + 0], a, bb[0], bb[1]);
          mma16816(s[pr * 2 + 1], a, bb[2], bb[3]);
        }
      }
    }

    // ---- mask, scale to base 2, block max.
    const int* ok = s_slot + ring * BN;
    float bmA = -INFINITY, bmB = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int kl = half * 32 + nt * 8 + 2 * (lane & 3) + (e & 1);
        const int j = kb * BN + kl;
        const int t = (e < 2) ? tA : tB;
        bool vis = ok[kl] >= 0 && t >= 0;
        if (vis && j >= rq.P) vis = (s_mask[t] >> (j - rq.P)) & 1u;
        const float v = vis ? s[nt][e] * p.scale_log2 : -INFINITY;
        s[nt][e] = v;
        if (e < 2) bmA = fmaxf(bmA, v);
        else bmB = fmaxf(bmB, v);
      }
    }
    bmA = fmaxf(bmA, __shfl_xor_sync(0xffffffffu, bmA, 1));
    bmA = fmaxf(bmA, __shfl_xor_sync(0xffffffffu, bmA, 2));
    bmB = fmaxf(bmB, __shfl_xor_sync(0xffffffffu, bmB, 1));
    bmB = fmaxf(bmB, __shfl_xor_sync(0xffffffffu, bmB, 2));
    if ((lane & 3) == 0) {
      s_red[half * 64 + lrA] = bmA;
      s_red[half * 64 + lrB] = bmB;
    }
    __syncthreads();
    bmA = fmaxf(bmA, s_red[(half ^ 1) * 64 + lrA]);
    bmB = fmaxf(bmB, s_red[(half ^ 1) * 64 + lrB]);
    const float nmA = fmaxf(mA, bmA), nmB = fmaxf(mB, bmB);
    const float uA = nmA == -INFINITY ? 0.f : nmA;
    const float uB = nmB == -INFINITY ? 0.f : nmB;
    const float alA = ex2(mA - uA), alB = ex2(mB - uB);
    mA = nmA;
    mB = nmB;

    // ---- P = 2^(S - m) as fp16 into shared memory; partial row sums.
    float psA = 0.f, psB = 0.f;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const float p0 = ex2(s[nt][0] - uA), p1 = ex2(s[nt][1] - uA);
      const float p2 = ex2(s[nt][2] - uB), p3 = ex2(s[nt][3] - uB);
      const __half2 hA = __floats2half2_rn(p0, p1);
      const __half2 hB = __floats2half2_rn(p2, p3);
      // Sum what the PV product will see.
      const float2 fA = __half22float2(hA), fB = __half22float2(hB);
      psA += fA.x + fA.y;
      psB += fB.x + fB.y;
      const int kl = half * 32 + nt * 8 + 2 * (lane & 3);
      const uint32_t offA = sw_p(lrA, kl >> 3) + (kl & 7) * 2;
      const uint32_t offB = sw_p(lrB, kl >> 3) + (kl & 7) * 2;
      asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sp + offA), "r"(*reinterpret_cast<const uint32_t*>(&hA)));
      asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sp + offB), "r"(*reinterpret_cast<const uint32_t*>(&hB)));
    }
    lA = lA * alA + psA;
    lB = lB * alB + psB;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      o[i][0] *= alA;
      o[i][1] *= alA;
      o[i][2] *= alB;
      o[i][3] *= alB;
    }
    __syncthreads();

    // ---- O += P V: 16 rows x 256 value dims per warp, 64 keys.
    {
      const int arow = rg * 16 + (lane & 15);
      const int acol = lane >> 4;
      const int mi = lane >> 3;
      const int vrow_off = ((mi & 1) << 3) + (lane & 7);
      const int vcol0 = half * 32 + (mi >> 1);
#pragma unroll
      for (int ks = 0; ks < BN / 16; ++ks) {
        uint32_t a[4];
        ldsm4(a, sp + sw_p(arow, ks * 2 + acol));
        const int vrow = ks * 16 + vrow_off;
#pragma unroll
        for (int np = 0; np < 16; ++np) {
          uint32_t bb[4];
          ldsm4_t(bb, skv + sw_row(vrow, vcol0 + np * 2));
          mma16816(o[np * 2 + 0], a, bb[0], bb[1]);
          mma16816(o[np * 2 + 1], a, bb[2], bb[3]);
        }
      }
    }
    if (tid < BN && kb + 2 < kb1) s_slot[((it + 2) % 3) * BN + tid] = pending;
    __syncthreads();
  }

  // ---- finish: combine the two key halves' row sums, normalise, store.
  lA += __shfl_xor_sync(0xffffffffu, lA, 1);
  lA += __shfl_xor_sync(0xffffffffu, lA, 2);
  lB += __shfl_xor_sync(0xffffffffu, lB, 1);
  lB += __shfl_xor_sync(0xffffffffu, lB, 2);
  if ((lane & 3) == 0) {
    s_red[half * 64 + lrA] = lA;
    s_red[half * 64 + lrB] = lB;
  }
  __syncthreads();
  lA += s_red[(half ^ 1) * 64 + lrA];
  lB += s_red[(half ^ 1) * 64 + lrB];
  const float invA = lA > 0.f ? 1.f / lA : 0.f;
  const float invB = lB > 0.f ? 1.f / lB : 0.f;
  const float lseA = lA > 0.f ? (mA + __log2f(lA)) * kLn2 : -INFINITY;
  const float lseB = lB > 0.f ? (mB + __log2f(lB)) * kLn2 : -INFINITY;

  const int dcol = half * 256 + 2 * (lane & 3);
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int gr = rr ? grB : grA;
    if (gr >= p.R) continue;
    const float inv = rr ? invB : invA;
    if (p.nsplit == 1) {
      const size_t orow = (static_cast<size_t>(b) * p.R + gr) * D_V;
      if (p.out_bf16) {
        uint32_t* dst = reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(p.out) + orow);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          __nv_bfloat162 v = __floats2bfloat162_rn(o[i][rr * 2] * inv, o[i][rr * 2 + 1] * inv);
          dst[(dcol + i * 8) >> 1] = *reinterpret_cast<uint32_t*>(&v);
        }
      } else {
        float* dst = reinterpret_cast<float*>(p.out) + orow;
#pragma unroll
        for (int i = 0; i < 32; ++i)
          *reinterpret_cast<float2*>(dst + dcol + i * 8) =
              make_float2(o[i][rr * 2] * inv, o[i][rr * 2 + 1] * inv);
      }
      if (half == 0 && (lane & 3) == 0) p.lse[static_cast<size_t>(b) * p.R + gr] = rr ? lseB : lseA;
    } else {
      float* dst = p.ws_o + (ws_row + gr) * D_V;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        *reinterpret_cast<float2*>(dst + dcol + i * 8) =
            make_float2(o[i][rr * 2] * inv, o[i][rr * 2 + 1] * inv);
      if (half == 0 && (lane & 3) == 0) p.ws_lse[ws_row + gr] = rr ? lseB : lseA;
    }
  }
}

}  // namespace

int partial_mma_smem_bytes() { return SMEM_TOTAL; }

cudaError_t partial_mma_prepare() {
  return cudaFuncSetAttribute(partial_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              SMEM_TOTAL);
}

cudaError_t launch_partial_mma(const Params& p, cudaStream_t stream) {
  const dim3 grid(p.nsplit, (p.R + BM - 1) / BM, p.batch);
  partial_mma_kernel<<<grid, NTHREADS, SMEM_TOTAL, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mlav
