// Split-KV partial kernel on the sm_103a tensor cores (tcgen05 + TMEM).
//
// One CTA = one request b, one tile of 64 query rows (r = t*H + h), one key
// split: the KV-split "partial" half of the partial + reduce design in "The
// Decisive A/B: When Benchmarking Honesty Reveals the Real Bottleneck"
// (sections "The Context" and "What This Reveals About the Bottleneck").
//
// The products are taken transposed so that every MMA has M = 128:
//     S^T[key, row] = K_block[128 x 576] . Q_tile[64 x 576]^T          (bf16)
//     O^T[dim, row] += V_block^T[512 x 128] . P^T[128 x 64]              (fp16)
// O^T lives in tensor memory for the whole split (4 tiles of 128 dims x 64
// rows = 256 columns) and S^T in another 64 columns.  With one thread per
// key, the softmax reduces each query row across the 128 TMEM lanes
// (redux.sync per warp, shared memory across the four warps).  The running
// row max is exact (P <= 1, and the key holding the max has P = 1 exactly):
// a lazily moved max would round the dominant key's weight to fp16 too, which
// measurably doubles the worst-case output error on spiky keys.  O^T columns
// are rescaled in TMEM only for the 32-row groups whose max moved.
//
// Per 128-key block:
//   A. gather the 128 scattered 1152-byte rows with 16-byte cp.async vectors
//      into nine 128-byte-swizzled 16 KB chunk tiles (the MMA operand layout);
//   B. one thread issues the 36 S^T MMAs (bf16 operands, fp32 in TMEM);
//   C. warps 0-3: softmax of S^T, P^T as fp16 into the (now unused) rope
//      chunk tile; warps 4-7: widen the value chunks 0-7 to fp16 in place
//      (P in bf16 would cost more than the 1e-2 output tolerance allows);
//   D. rescale the O^T columns of the 32-row groups whose max moved;
//   E. one thread issues the 32 O^T MMAs (fp16 operands).
// The next block's slots are read and its rows prefetched into L2 while the
// tensor core runs step B.
#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace mlav {
namespace {

constexpr int BM = 64;          // query rows per CTA: MMA N
constexpr int BN = 128;         // keys per block: MMA M of S^T
constexpr int NTHREADS = 256;
constexpr int Q_CHUNK = BM * 128;   // one 64-dim chunk of the Q tile
constexpr int KV_CHUNK = BN * 128;  // one 64-dim chunk of the key block
constexpr int OFF_Q = 0;
constexpr int OFF_KV = OFF_Q + 9 * Q_CHUNK;
constexpr int OFF_P = OFF_KV + 8 * KV_CHUNK;   // rope chunk tile, reused for P^T
constexpr int OFF_RED = OFF_KV + 9 * KV_CHUNK;  // float [4][64] per-warp column max / sums
constexpr int OFF_MREF = OFF_RED + 4 * 64 * 4;  // float [64] running row max (base 2)
constexpr int OFF_ALPHA = OFF_MREF + 64 * 4;    // float [64] rescale factor of this block
constexpr int OFF_L = OFF_ALPHA + 64 * 4;       // float [64] final row sums
constexpr int OFF_SLOT = OFF_L + 64 * 4;        // int [2][128] slots of this / next block
constexpr int OFF_MASK = OFF_SLOT + 2 * BN * 4; // uint32 [32] ancestor masks
constexpr int OFF_TOFR = OFF_MASK + MAX_T * 4;  // int [64] draft of each row, -1 past R
constexpr int OFF_MBAR = OFF_TOFR + 64 * 4;     // uint64 [2]: S^T done, O^T done
constexpr int OFF_MISC = OFF_MBAR + 16;         // uint32 tmem base, int rescale flags [2]
constexpr int SMEM_TOTAL = OFF_MISC + 16;
static_assert(SMEM_TOTAL <= 232448, "shared memory budget");
static_assert(OFF_KV % 1024 == 0 && OFF_P % 1024 == 0, "swizzled tiles need 1024-byte alignment");

constexpr int TMEM_COLS = 512;
constexpr uint32_t TM_S = 256;                  // S^T columns; O^T tile d at d * 64
constexpr long long WAIT_LIMIT = 1LL << 31;     // cycles before a wait gives up

constexpr uint32_t IDESC_S = tc::idesc_f16(128, BM, 1, 0, 0);   // bf16, both K-major
constexpr uint32_t IDESC_O = tc::idesc_f16(128, BM, 0, 1, 1);   // fp16, both MN-major

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
}
__device__ __forceinline__ void named_sync_softmax() {
  asm volatile("bar.sync 1, 128;\n" ::: "memory");
}

// Slot of key r of 128-key block kb, or -1 past the end of the request or
// when the table points outside the cache (reported).
__device__ __forceinline__ int block_slot(const Params& p, const Request& rq, int kb, int r) {
  const int j = kb * BN + r;
  if (j >= rq.n) return -1;
  const long long s = key_slot(p, rq.ip0, j);
  if (s < 0) atomicOr(p.err, ERR_SLOT);
  return static_cast<int>(s);
}

__device__ __forceinline__ uint32_t widen_word(uint32_t w) {
  const float lo = __uint_as_float(w << 16);
  const float hi = __uint_as_float(w & 0xffff0000u);
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void write_nan_rows(const Params& p, int b, int split, int row0, int tid) {
  const float nan = __int_as_float(0x7fc00000);
  const size_t ws_row = (static_cast<size_t>(b) * p.nsplit + split) * p.R;
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
}

__global__ void __launch_bounds__(NTHREADS, 1) partial_tc_kernel(const Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int split = blockIdx.x, rt = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3;       // TMEM lanes 32*quad .. +32 are this warp's
  const int row0 = rt * BM;

  float* s_red = reinterpret_cast<float*>(smem + OFF_RED);
  float* s_mref = reinterpret_cast<float*>(smem + OFF_MREF);
  float* s_alpha = reinterpret_cast<float*>(smem + OFF_ALPHA);
  float* s_l = reinterpret_cast<float*>(smem + OFF_L);
  int* s_slot = reinterpret_cast<int*>(smem + OFF_SLOT);
  uint32_t* s_mask = reinterpret_cast<uint32_t*>(smem + OFF_MASK);
  int* s_tofr = reinterpret_cast<int*>(smem + OFF_TOFR);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* s_flag = reinterpret_cast<int*>(smem + OFF_MISC + 4);
  const uint32_t mbar_s = smem_u32(smem + OFF_MBAR);
  const uint32_t mbar_o = mbar_s + 8;
  const uint32_t sbase = smem_u32(smem);

  const Request rq = load_request(p, b);
  if (!rq.ok) {
    if (split == 0 && rt == 0 && tid == 0)
      atomicOr(p.err, (rq.n < p.T || rq.n > p.max_kv_len) ? ERR_LEN : ERR_INDPTR);
    write_nan_rows(p, b, split, row0, tid);
    return;
  }
  if (sbase & 1023) {   // swizzled operand tiles need a 1024-byte aligned base
    if (tid == 0) atomicOr(p.err, ERR_INTERNAL);
    write_nan_rows(p, b, split, row0, tid);
    return;
  }

  const int nblk = (rq.n + BN - 1) / BN;
  const int kb0 = static_cast<int>((static_cast<long long>(split) * nblk) / p.nsplit);
  const int kb1 = static_cast<int>((static_cast<long long>(split + 1) * nblk) / p.nsplit);

  if (tid < p.T) s_mask[tid] = ancestor_mask(p.draft_parent + b * p.T, tid, p.err);
  if (tid < BM) {
    s_tofr[tid] = row0 + tid < p.R ? (row0 + tid) / p.H : -1;
    s_mref[tid] = -INFINITY;
  }
  if (tid < BN && kb1 > kb0) s_slot[tid] = block_slot(p, rq, kb0, tid);
  if (tid == 0) {
    tc::mbar_init(mbar_s, 1);
    tc::mbar_init(mbar_o, 1);
    tc::mbar_fence_init();
    s_flag[0] = 0;
    s_flag[1] = 0;
  }
  if (warp == 0) tc::tmem_alloc<TMEM_COLS>(smem_u32(s_tmem));
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;

  // Q tile: 64 rows x 9 swizzled chunks; rows beyond R are zero.
  if (kb1 > kb0) {
    const uint16_t* qb = p.q + static_cast<size_t>(b) * p.R * D_QK;
#pragma unroll 1
    for (int e = tid; e < BM * ROW_CHUNKS; e += NTHREADS) {
      const int r = e / ROW_CHUNKS, q = e - r * ROW_CHUNKS;
      const int gr = row0 + r;
      const bool in = gr < p.R;
      cp_async16(sbase + OFF_Q + (q >> 3) * Q_CHUNK + r * 128 + (((q & 7) ^ (r & 7)) << 4),
                 in ? qb + static_cast<size_t>(gr) * D_QK + q * 8 : p.q, in ? 16 : 0);
    }
  }

  const bool all_rows = row0 + BM <= p.R;
  const float scale2 = p.scale_log2;
  float lpart[BM];   // softmax threads: this key's share of every row sum
#pragma unroll
  for (int c = 0; c < BM; ++c) lpart[c] = 0.f;
  bool alive = true;

#pragma unroll 1
  for (int kb = kb0; kb < kb1; ++kb) {
    const int it = kb - kb0;
    const int cur = it & 1;
    const uint32_t par = static_cast<uint32_t>(it & 1);

    // ---- A. gather the key block (cp.async, 36 vectors per thread).
    {
      const int* slots = s_slot + cur * BN;
#pragma unroll 4
      for (int e = tid; e < BN * ROW_CHUNKS; e += NTHREADS) {
        const int j = e / ROW_CHUNKS, q = e - j * ROW_CHUNKS;
        const int slot = slots[j];
        cp_async16(sbase + OFF_KV + (q >> 3) * KV_CHUNK + j * 128 + (((q & 7) ^ (j & 7)) << 4),
                   slot >= 0 ? p.kv + static_cast<long long>(slot) * D_QK + q * 8 : p.kv,
                   slot >= 0 ? 16 : 0);
      }
      cp_async_wait_all();
      tc::fence_async_smem();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    // ---- B. S^T = K Q^T, issued by one thread.
    if (tid == 0) {
#pragma unroll 4
      for (int k = 0; k < D_QK / 16; ++k) {
        const uint64_t a = tc::desc_sw128(sbase + OFF_KV + (k >> 2) * KV_CHUNK + (k & 3) * 32, 16, 1024);
        const uint64_t bq = tc::desc_sw128(sbase + OFF_Q + (k >> 2) * Q_CHUNK + (k & 3) * 32, 16, 1024);
        tc::mma_ss(tmem + TM_S, a, bq, IDESC_S, k > 0);
      }
      tc::commit(mbar_s);
    }
    // Meanwhile: the next block's slots, and its rows into L2.
    int pending = -1;
    if (tid < BN && kb + 1 < kb1) {
      pending = block_slot(p, rq, kb + 1, tid);
      if (pending >= 0) {
        const char* row = reinterpret_cast<const char*>(p.kv + static_cast<long long>(pending) * D_QK);
#pragma unroll
        for (int l = 0; l < ROW_BYTES / 128; ++l)
          asm volatile("prefetch.global.L2 [%0];\n" ::"l"(row + l * 128));
      }
    }
    alive = tc::mbar_wait_bounded(mbar_s, par, WAIT_LIMIT);
    tc::fence_after_sync();
    if (__syncthreads_or(!alive)) break;

    // ---- C. softmax (warps 0-3) and fp16 widening of the values (warps 4-7).
    if (warp < 4) {
      const int j = tid;                  // key of this thread = TMEM lane
      const int jg = kb * BN + j;
      const bool key_ok = s_slot[cur * BN + j] >= 0;
      uint32_t sr_lo[32], sr_hi[32];
      {
        const uint32_t ta = tmem + (static_cast<uint32_t>(quad * 32) << 16) + TM_S;
        tc::tmem_ld32(ta, sr_lo);
        tc::tmem_ld32(ta + 32, sr_hi);
        tc::tmem_wait_ld();
      }
#define SR(c) ((c) < 32 ? sr_lo[(c)] : sr_hi[(c) - 32])
      float s[BM];
      if (!key_ok) {
#pragma unroll
        for (int c = 0; c < BM; ++c) s[c] = -INFINITY;
      } else if (jg < rq.P && all_rows) {
#pragma unroll
        for (int c = 0; c < BM; ++c) s[c] = __uint_as_float(SR(c)) * scale2;
      } else {
        const int di = jg - rq.P;   // draft index when >= 0
#pragma unroll
        for (int c = 0; c < BM; ++c) {
          const int t = s_tofr[c];
          bool vis = t >= 0;
          if (vis && di >= 0) vis = (s_mask[t] >> di) & 1u;
          s[c] = vis ? __uint_as_float(SR(c)) * scale2 : -INFINITY;
        }
      }
#undef SR
      // Column (query row) max over this warp's 32 keys, then over 4 warps.
#pragma unroll
      for (int c = 0; c < BM; ++c) {
        const float m = tc::warp_max(s[c]);
        if ((c & 31) == lane) s_red[warp * BM + c] = m;
      }
      named_sync_softmax();
      if (tid < BM) {
        const float bm = fmaxf(fmaxf(s_red[tid], s_red[BM + tid]),
                               fmaxf(s_red[2 * BM + tid], s_red[3 * BM + tid]));
        const float old = s_mref[tid];
        float alpha = 1.f;
        if (bm > old) {
          s_mref[tid] = bm;
          if (old != -INFINITY) {
            alpha = ex2(old - bm);
            s_flag[tid >> 5] = 1;
          }
        }
        s_alpha[tid] = alpha;
      }
      named_sync_softmax();
      // P^T row of this key (64 query rows) as fp16, 128-byte swizzled.
      uint32_t pk[BM / 2];
#pragma unroll
      for (int c = 0; c < BM; c += 2) {
        const float m0 = s_mref[c], m1 = s_mref[c + 1];
        const float p0 = s[c] == -INFINITY ? 0.f : ex2(s[c] - m0);
        const float p1 = s[c + 1] == -INFINITY ? 0.f : ex2(s[c + 1] - m1);
        lpart[c] = lpart[c] * s_alpha[c] + p0;
        lpart[c + 1] = lpart[c + 1] * s_alpha[c + 1] + p1;
        __half2 h = __floats2half2_rn(p0, p1);
        pk[c >> 1] = *reinterpret_cast<uint32_t*>(&h);
      }
      uint8_t* prow = smem + OFF_P + j * 128;
#pragma unroll
      for (int g = 0; g < 8; ++g)
        *reinterpret_cast<uint4*>(prow + ((g ^ (j & 7)) << 4)) =
            make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
    } else {
      const int t2 = tid - 128;
#pragma unroll 4
      for (int e = t2; e < 8 * KV_CHUNK / 16; e += 128) {
        uint4* ptr = reinterpret_cast<uint4*>(smem + OFF_KV + e * 16);
        uint4 v = *ptr;
        v.x = widen_word(v.x);
        v.y = widen_word(v.y);
        v.z = widen_word(v.z);
        v.w = widen_word(v.w);
        *ptr = v;
      }
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    // ---- D. rescale the O^T columns of the row groups whose max moved.
    const bool rescale0 = s_flag[0] != 0, rescale1 = s_flag[1] != 0;
    if (rescale0 || rescale1) {
      const int d0 = (warp >> 2) * 2;   // warps 0-3: tiles 0,1; warps 4-7: tiles 2,3
#pragma unroll 1
      for (int d = d0; d < d0 + 2; ++d) {
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          if (!(h ? rescale1 : rescale0)) continue;
          const uint32_t ta = tmem + (static_cast<uint32_t>(quad * 32) << 16) + d * BM + h * 32;
          uint32_t v[32];
          tc::tmem_ld32(ta, v);
          tc::tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c)
            v[c] = __float_as_uint(__uint_as_float(v[c]) * s_alpha[h * 32 + c]);
          tc::tmem_st32(ta, v);
        }
      }
      tc::tmem_wait_st();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0) {
      s_flag[0] = 0;
      s_flag[1] = 0;
    }

    // ---- E. O^T += V^T P^T, issued by one thread.
    if (tid == 0) {
#pragma unroll 1
      for (int d = 0; d < 4; ++d) {
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          const uint64_t a = tc::desc_sw128(sbase + OFF_KV + 2 * d * KV_CHUNK + k * 2048, KV_CHUNK, 1024);
          const uint64_t bp = tc::desc_sw128(sbase + OFF_P + k * 2048, 8192, 1024);
          tc::mma_ss(tmem + d * BM, a, bp, IDESC_O, (it > 0 || k > 0) ? 1u : 0u);
        }
      }
      tc::commit(mbar_o);
    }
    alive = tc::mbar_wait_bounded(mbar_o, par, WAIT_LIMIT);
    tc::fence_after_sync();
    if (tid < BN) s_slot[(cur ^ 1) * BN + tid] = pending;
    if (__syncthreads_or(!alive)) break;
  }

  if (!alive) {
    if (tid == 0) atomicOr(p.err, ERR_TIMEOUT);
    // Give in-flight tensor-core work one more bounded wait before freeing TMEM.
    tc::mbar_wait_bounded(mbar_o, 0, WAIT_LIMIT);
    write_nan_rows(p, b, split, row0, tid);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc<TMEM_COLS>(tmem);
    return;
  }

  // ---- finish: row sums over all keys, LSE, normalised O.
  if (warp < 4) {
#pragma unroll
    for (int c = 0; c < BM; ++c) {
      float v = lpart[c];
#pragma unroll
      for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if ((c & 31) == lane) s_red[warp * BM + c] = v;
    }
  }
  __syncthreads();
  if (tid < BM) {
    const float l = s_red[tid] + s_red[BM + tid] + s_red[2 * BM + tid] + s_red[3 * BM + tid];
    s_l[tid] = l;
    const int gr = row0 + tid;
    if (gr < p.R) {
      const float lse = l > 0.f ? (s_mref[tid] + log2f(l)) * kLn2 : -INFINITY;
      if (p.nsplit == 1) p.lse[static_cast<size_t>(b) * p.R + gr] = lse;
      else p.ws_lse[(static_cast<size_t>(b) * p.nsplit + split) * p.R + gr] = lse;
    }
  }
  __syncthreads();
  {
    const int d0 = (warp >> 2) * 2;
    const int nrows = min(BM, p.R - row0);
#pragma unroll 1
    for (int d = d0; d < d0 + 2; ++d) {
      const int dim = d * 128 + quad * 32 + lane;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        uint32_t v[32];
        if (kb1 > kb0) {
          tc::tmem_ld32(tmem + (static_cast<uint32_t>(quad * 32) << 16) + d * BM + h * 32, v);
          tc::tmem_wait_ld();
        }
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int r = h * 32 + c;
          if (r >= nrows) continue;
          const float l = s_l[r];
          const float o = l > 0.f ? __uint_as_float(v[c]) / l : 0.f;
          const size_t row = static_cast<size_t>(b) * p.R + row0 + r;
          if (p.nsplit == 1) {
            if (p.out_bf16) {
              __nv_bfloat16 x = __float2bfloat16_rn(o);
              reinterpret_cast<__nv_bfloat16*>(p.out)[row * D_V + dim] = x;
            } else {
              reinterpret_cast<float*>(p.out)[row * D_V + dim] = o;
            }
          } else {
            p.ws_o[((static_cast<size_t>(b) * p.nsplit + split) * p.R + row0 + r) * D_V + dim] = o;
          }
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc<TMEM_COLS>(tmem);
}

}  // namespace

cudaError_t partial_tc_prepare() {
  return cudaFuncSetAttribute(partial_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              SMEM_TOTAL);
}

cudaError_t launch_partial_tc(const Params& p, cudaStream_t stream) {
  const dim3 grid(p.nsplit, (p.R + BM - 1) / BM, p.batch);
  partial_tc_kernel<<<grid, NTHREADS, SMEM_TOTAL, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mlav
