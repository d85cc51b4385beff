// Split-KV partial kernel on the sm_103a tensor cores (tcgen05 + TMEM),
// warp-specialised and pipelined.
//
// One CTA = one request b, one tile of 64 query rows (r = t*H + h), one key
// split: the KV-split "partial" half of the partial + reduce design in "The
// Decisive A/B: When Benchmarking Honesty Reveals the Real Bottleneck"
// (sections "The Context" and "What This Reveals About the Bottleneck": KV
// split for occupancy, 128-bit vector loads of scattered page_size=1 rows).
//
// The products are taken transposed so that every MMA has M = 128:
//     S^T[key, row] = K_block[128 x 576] . Q_tile[64 x 576]^T          (fp16)
//     O^T[dim, row] += V_block^T[512 x 128] . P^T[128 x 64]              (fp16)
// O^T lives in tensor memory for the whole split (4 tiles of 128 dims x 64
// rows = columns 0..255) and S^T in columns 256..319.  With one thread per
// key the softmax reduces each query row across the 128 TMEM lanes (a
// shuffle transpose-reduce per warp, shared memory across four warps).  The running row
// max is exact, so P <= 1 and the key holding the max has P = 1 exactly (a
// lazily moved max would round the dominant key's weight too, which doubles
// the worst-case output error on spiky keys); O^T columns are rescaled in
// TMEM only for the 32-row groups whose max moved.  P is fp16 and the values
// are fp16 (widened by the pack), because P in bf16 costs more than the 1e-2
// output tolerance allows.
//
// The key blocks come from the per-call pack (pack_kv.cu): 147456 contiguous
// bytes per 128-key block, already fp16 and already in the 128-byte-swizzled
// operand layout, so each chunk pair arrives with one 32 KB bulk copy.  The
// pack may still be running: the copy warp then waits for each block's
// ready flags (tagged with the call's epoch) instead of the whole pack grid,
// and the last CTA to finish advances the epoch.
//
// Roles (11 warps):
//   warps 0-7  softmax: one thread per (key of the block, half of the 64 query
//              rows); warps w and w+4 share TMEM lane quadrant w.  First they
//              load the Q tile (issued at entry) and widen it to fp16;
//   warp 8     issues the MMAs (one elected lane of the converged warp); it
//              owns the TMEM allocation;
//   warp 9     streams the packed blocks with cp.async.bulk (elected lane);
//   warps 9-10 instead, with no pack (one row tile per request), gather each
//              block's scattered rows themselves (16-byte cp.async), piece by
//              piece in the producer order below; the softmax warps widen
//              each piece in place while they wait for S^T.
// Pipeline over 128-key blocks k (mbarriers, all waits bounded):
//   producer: chunk pair d of block k+1 is copied as soon as O^T(k) tile d has
//             finished with it; the rope chunk (which holds P^T(k)) last;
//   MMA:      S^T(k) chunk pair by chunk pair as the pairs land, then, once
//             softmax(k) is done, O^T(k) tile by tile;
//   softmax:  after S^T(k): mask, max, P^T(k) into the rope chunk tile.
#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace mlav {
namespace {

constexpr int BM = 64;          // query rows per CTA: MMA N
constexpr int BN = 128;         // keys per block: MMA M of S^T
constexpr int NWARPS = 11;
constexpr int NTHREADS = NWARPS * 32;
constexpr int SOFTMAX_WARPS = 8, MMA_WARP = 8, COPY_WARP = 9;
constexpr int GATHER_WARPS = 2;   // direct mode: warps 9 and 10 gather keys 64w .. 64w+63 of each block
constexpr int HALF = BM / 2;    // query-row columns per softmax thread
constexpr int Q_CHUNK = BM * 128;   // one 64-dim chunk of the Q tile
constexpr int KV_CHUNK = BN * 128;  // one 64-dim chunk of the key block
constexpr int PACKED_BLOCK = 9 * KV_CHUNK;       // one packed 128-key block
constexpr int OFF_Q = 0;
constexpr int OFF_KV = OFF_Q + 9 * Q_CHUNK;
constexpr int OFF_P = OFF_KV + 8 * KV_CHUNK;   // rope chunk tile, reused for P^T
constexpr int OFF_RED = OFF_KV + 9 * KV_CHUNK;  // float [64][4] column max per quad; [4][64] sums
constexpr int OFF_MREF = OFF_RED + 4 * 64 * 4;  // float [64] final running row max (base 2)
constexpr int OFF_WARP = OFF_MREF + 64 * 4;     // float [8][2][32] per-warp row max / rescale factor
constexpr int OFF_L = OFF_WARP + 8 * 64 * 4;    // float [64] reciprocal of the final row sums (0: none)
constexpr int OFF_MASK = OFF_L + 64 * 4;        // uint32 [32] ancestor masks
constexpr int OFF_TOFR = OFF_MASK + MAX_T * 4;  // int [64] draft of each row, -1 past R
constexpr int NMBAR = 18;
constexpr int OFF_MBAR = OFF_TOFR + 64 * 4;     // uint64 [NMBAR] mbarriers
constexpr int OFF_MISC = OFF_MBAR + NMBAR * 8;  // tmem base, abort flag
constexpr int OFF_PAR = OFF_MISC + 16;          // int [32] draft parents
constexpr int OFF_SLOTK = OFF_PAR + MAX_T * 4;  // int [128] slots of the block being gathered (direct mode)
static_assert(GATHER_WARPS * 64 == BN, "each gather warp takes half of a block's keys");
constexpr int SMEM_TOTAL = OFF_SLOTK + BN * 4;
static_assert(SMEM_TOTAL <= 232448, "shared memory budget");
static_assert(OFF_KV % 1024 == 0 && OFF_P % 1024 == 0, "swizzled tiles need 1024-byte alignment");

// mbarrier indices
constexpr int MB_CHUNK = 0;   // [5] chunk pairs 0..3 and the rope chunk landed (copy bytes)
constexpr int MB_S = 5;       // S^T done (tcgen05.commit)
constexpr int MB_P = 6;       // P^T written, O^T rescaled (one arrival per softmax warp)
constexpr int MB_Q = 7;       // Q tile in fp16 (one arrival per softmax warp)
constexpr int MB_OT = 8;      // [4] O^T tile d done (tcgen05.commit)
constexpr int MB_DONE = 12;   // after an abort: every MMA the CTA issued is done
constexpr int MB_RAW = 13;    // [5] direct mode: piece g's rows landed (cp.async arrivals, bf16)

constexpr int TMEM_COLS = 512;
constexpr uint32_t TM_S = 256;                  // S^T columns; O^T tile d at d * 64
constexpr long long WAIT_LIMIT = 1LL << 31;     // cycles before a wait gives up

constexpr uint32_t IDESC_S = tc::idesc_f16(128, BM, 0, 0, 0);   // fp16, both K-major
constexpr uint32_t IDESC_O = tc::idesc_f16(128, BM, 0, 1, 1);   // fp16, both MN-major

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes));
}
__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(count) : "memory");
}

// Bounded wait; a timeout (or an earlier one anywhere in the CTA) sets the
// abort flag so every later wait returns at once.
__device__ __forceinline__ bool wait_phase(uint32_t mbar, uint32_t parity, volatile int* abort,
                                           int* err) {
  if (tc::mbar_test(mbar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (tc::mbar_try(mbar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > WAIT_LIMIT) {
      *abort = 1;
      atomicOr(err, ERR_TIMEOUT);
      return false;
    }
  }
}

// Warp-wide wait.  Every lane polls: measured faster here than one polling
// lane with the rest of the warp parked at __syncwarp.
__device__ __forceinline__ void wait_warp(uint32_t mbar, uint32_t parity, volatile int* abort,
                                          int* err) {
  wait_phase(mbar, parity, abort, err);
  __syncwarp();
}

// Bounded wait that ignores the abort flag: used to let this CTA's own
// copies land before it exits.
__device__ __forceinline__ void wait_drain(uint32_t mbar, uint32_t parity, int* err) {
  const long long t0 = clock64();
  while (!tc::mbar_try(mbar, parity)) {
    if (clock64() - t0 > WAIT_LIMIT) {
      atomicOr(err, ERR_TIMEOUT);
      return;
    }
  }
}

// Slot of key r of 128-key block kb, or -1 past the end of the request or
// when the table points outside the cache (reported when `report`).
__device__ __forceinline__ int block_slot(const Params& p, const Request& rq, int kb, int r,
                                          bool report) {
  const int j = kb * BN + r;
  if (j < rq.lo || j >= rq.hi) return -1;
  const long long s = key_slot(p, rq.ip0, j);
  if (s < 0 && report) atomicOr(p.err, ERR_SLOT);
  return static_cast<int>(s);
}

// Wait (bounded) until the pack kernel has published all 32 four-key units
// of block kb of request b for this call: lane l watches unit l's flag with
// acquire loads.  Whole warp; false on a timeout or an earlier abort.
__device__ __forceinline__ bool wait_packed(const Params& p, int b, int kb, unsigned long long tag,
                                            volatile int* abort, int* err) {
  const int lane = threadIdx.x & 31;
  const unsigned long long* flag =
      pack_flags(p.pack_sync) + 32 * (static_cast<size_t>(b) * p.packed_max_blocks + kb) + lane;
  const long long t0 = clock64();
  while (true) {   // every exit decision is warp-uniform
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];\n" : "=l"(v) : "l"(flag) : "memory");
    if (__all_sync(0xffffffffu, v == tag)) break;
    if (__any_sync(0xffffffffu, *abort != 0)) return false;
    if (__any_sync(0xffffffffu, clock64() - t0 > WAIT_LIMIT)) {
      if (lane == 0) {
        *abort = 1;
        atomicOr(err, ERR_TIMEOUT);
      }
      __syncwarp();
      return false;
    }
  }
  // The packed bytes were written through the generic proxy; the bulk copies
  // that follow read them through the async proxy.
  asm volatile("fence.proxy.async.global;\n" ::: "memory");
  return true;
}

// Every CTA takes one ticket when it is done; the last one of the grid
// advances the epoch, so the next call's pack kernel publishes a new tag.
// The 64-bit tag (epoch + 1) is never 0 -- the value of a flag no call has
// written -- and never repeats, so no flag left by an earlier call passes
// for this call's.
__device__ __forceinline__ void finish_call(const Params& p) {
  __threadfence();
  const unsigned total = gridDim.x * gridDim.y * gridDim.z;
  if (atomicAdd(p.pack_sync + PACK_SYNC_TICKET, 1u) == total - 1) {
    p.pack_sync[PACK_SYNC_TICKET] = 0;
    *reinterpret_cast<volatile unsigned long long*>(p.pack_sync) = pack_epoch(p.pack_sync) + 1ull;
  }
}

// Rows whose O^T columns one softmax warp rescales one by one (their loads
// overlapping the P computation); more moved rows take the whole-half pass.
constexpr int FEW_MOVED = 4;

// Column maxima of a warp's 32 x 32 tile (lane = key, v[c] = column c) in 31
// shuffles: each step halves the columns a lane holds and swaps the other
// half with the partner lane, so lane l ends with the maximum of column l
// over all 32 lanes in v[0].
__device__ __forceinline__ void transpose_max32(float (&v)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = upper ? v[i] : v[i + w];
      const float keep = upper ? v[i + w] : v[i];
      v[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, w));
    }
  }
}

__device__ __forceinline__ void write_nan_rows(const Params& p, int b, int split, int row0, int tid) {
  const float nan = __int_as_float(0x7fc00000);
  const size_t ws_row = ws_base(p, b, split);
  for (int i = tid; i < BM * D_V; i += static_cast<int>(blockDim.x)) {
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

// kDirect: no pack, the CTAs gather their own key blocks (p.direct_all).
// The two modes are separate instantiations so that neither's softmax loop
// is scheduled around the other's code: with the direct-mode widening in the
// same loop body the packed path measured ~15 % slower on one-block splits.
template <bool kDirect>
__global__ void __launch_bounds__(kDirect ? NTHREADS : NTHREADS - 32, 1) partial_tc_kernel(const Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int split = blockIdx.x, rt = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3;       // TMEM lanes 32*quad .. +32 are this warp's
  const int row0 = rt * BM;

  float* s_red = reinterpret_cast<float*>(smem + OFF_RED);
  float* s_mref = reinterpret_cast<float*>(smem + OFF_MREF);
  float* s_l = reinterpret_cast<float*>(smem + OFF_L);
  uint32_t* s_mask = reinterpret_cast<uint32_t*>(smem + OFF_MASK);
  int* s_tofr = reinterpret_cast<int*>(smem + OFF_TOFR);
  int* s_par = reinterpret_cast<int*>(smem + OFF_PAR);
  int* s_slotk = reinterpret_cast<int*>(smem + OFF_SLOTK);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + OFF_MISC + 12);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t mbar0 = sbase + OFF_MBAR;
  auto mbar = [&](int i) { return mbar0 + 8u * static_cast<uint32_t>(i); };

  // Q tile: 64 rows x 9 swizzled chunks (rows beyond R zero), loaded by the
  // softmax warps first -- its address needs nothing from the request, so
  // the load overlaps the request lookup.  Every exit drains it.
  if (warp < SOFTMAX_WARPS) {
    const uint16_t* qb = p.q + static_cast<size_t>(b) * p.R * D_QK;
#pragma unroll 1
    for (int e = tid; e < BM * ROW_CHUNKS; e += SOFTMAX_WARPS * 32) {
      const int r = e / ROW_CHUNKS, q = e - r * ROW_CHUNKS;
      const int gr = row0 + r;
      const bool in = gr < p.R;
      cp_async16(sbase + OFF_Q + (q >> 3) * Q_CHUNK + r * 128 + (((q & 7) ^ (r & 7)) << 4),
                 in ? qb + static_cast<size_t>(gr) * D_QK + q * 8 : p.q, in ? 16 : 0);
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
  }

  const Request rq = load_request(p, b);
  if (!rq.ok) {
    if (split == 0 && rt == 0 && tid == 0)
      atomicOr(p.err, (rq.n < p.T || rq.n > p.max_kv_len) ? ERR_LEN : ERR_INDPTR);
    write_nan_rows(p, b, split, row0, tid);
    if (tid == 0) finish_call(p);
    asm volatile("cp.async.wait_all;\n" ::: "memory");
    return;
  }
  if (sbase & 1023) {   // swizzled operand tiles need a 1024-byte aligned base
    if (tid == 0) {
      atomicOr(p.err, ERR_INTERNAL);
      finish_call(p);
    }
    write_nan_rows(p, b, split, row0, tid);
    asm volatile("cp.async.wait_all;\n" ::: "memory");
    return;
  }

  int kb0, kb1;
  split_blocks(rq, BN, split, p.nsplit, kb0, kb1);
  const int nb = kb1 - kb0;

  // Parents in one parallel load; the softmax warps walk the chains in
  // shared memory (a walk through global memory costs one round trip a step).
  if (tid < p.T) s_par[tid] = p.draft_parent[b * p.T + tid];
  if (tid < BM) s_tofr[tid] = row0 + tid < p.R ? (row0 + tid) / p.H : -1;
  if (tid == 0) {
    for (int i = 0; i < 5; ++i) {
      tc::mbar_init(mbar(MB_CHUNK + i), kDirect ? SOFTMAX_WARPS : 1);
      tc::mbar_init(mbar(MB_RAW + i), GATHER_WARPS * 32);
    }
    tc::mbar_init(mbar(MB_S), 1);
    tc::mbar_init(mbar(MB_P), SOFTMAX_WARPS);
    tc::mbar_init(mbar(MB_Q), SOFTMAX_WARPS);
    tc::mbar_init(mbar(MB_DONE), 1);
    for (int i = 0; i < 4; ++i) tc::mbar_init(mbar(MB_OT + i), 1);
    tc::mbar_fence_init();
    *s_abort = 0;
  }
  if (warp == MMA_WARP) tc::tmem_alloc<TMEM_COLS>(smem_u32(s_tmem));
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;

  if (kDirect && warp >= COPY_WARP) {
    // ===================== direct gather (no pack) ==========================
    // Gather warp w copies keys 64w .. 64w+63 of every block, in the packed
    // producer's order: chunk pair g of block k as soon as O^T(k-1) tile g
    // has read pair g of the previous block, the rope chunk (where P^T(k-1)
    // lived) last -- 16-byte cp.async of the scattered rows, zero-filled
    // past the request, each lane's copies arriving on the piece's MB_RAW
    // barrier when they land.  The softmax warps, idle until S^T(k), widen
    // each piece in place and release it to the MMA warp.
    const int gw = warp - COPY_WARP;
    int* wslot = s_slotk + 64 * gw;
    const int ka = 64 * gw + lane, kbk = ka + 32;   // the keys whose slots this lane looks up
    int sa = nb > 0 ? block_slot(p, rq, kb0, ka, false) : -1;
    int sb = nb > 0 ? block_slot(p, rq, kb0, kbk, false) : -1;
    // Exit decisions are warp-uniform (the abort flag is read lane by lane).
    auto aborted = [&]() { return __any_sync(0xffffffffu, *s_abort != 0); };
#pragma unroll 1
    for (int it = 0; it < nb && !aborted(); ++it) {
      __syncwarp();
      wslot[lane] = sa;
      wslot[32 + lane] = sb;
      __syncwarp();
      if (it + 1 < nb) {   // the next block's slots, in flight while this one is gathered
        sa = block_slot(p, rq, kb0 + it + 1, ka, false);
        sb = block_slot(p, rq, kb0 + it + 1, kbk, false);
      }
      const uint32_t prev = static_cast<uint32_t>((it - 1) & 1);
#pragma unroll 1
      for (int g = 0; g < 5; ++g) {
        if (it > 0 && g < 4) wait_warp(mbar(MB_OT + g), prev, s_abort, p.err);
        if (aborted()) break;
        // Lane l: granules l % 16 of chunk pair g of keys 2i + l / 16, or
        // granule l % 8 of the rope chunk of keys 4i + l / 8.
        const int n = g < 4 ? 32 : 16;
#pragma unroll 4
        for (int i = 0; i < n; ++i) {
          const int key = g < 4 ? 2 * i + (lane >> 4) : 4 * i + (lane >> 3);
          const int q = g < 4 ? 16 * g + (lane & 15) : 64 + (lane & 7);
          const int k = 64 * gw + key;
          const int sl = wslot[key];
          cp_async16(sbase + OFF_KV + (q >> 3) * KV_CHUNK + k * 128 + (((q & 7) ^ (k & 7)) << 4),
                     sl >= 0 ? p.kv + static_cast<size_t>(sl) * D_QK + q * 8 : p.kv, sl >= 0 ? 16 : 0);
        }
        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(mbar(MB_RAW + g)) : "memory");
      }
    }
    asm volatile("cp.async.wait_all;\n" ::: "memory");   // nothing in flight at exit
  } else if (warp == COPY_WARP) {
    // ======================= packed-block producer ==========================
    // The whole warp runs the loop; one elected lane issues each copy.
    const uint8_t* blocks = p.packed + static_cast<size_t>(b) * p.packed_max_blocks * PACKED_BLOCK;
    // The packed blocks come from the pack kernel just before this one on
    // the stream, which may still be running: with per-unit flags each block
    // is read once its 32 units carry this call's tag, else after the whole
    // pack grid (a no-op when launched without overlap).
    const unsigned long long tag = pack_epoch(p.pack_sync) + 1ull;
    if (!p.pack_flags) asm volatile("griddepcontrol.wait;\n" ::: "memory");
    int issued = 0;   // copies issued, in (block, g) order
#pragma unroll 1
    for (int it = 0; it < nb; ++it) {
      const uint8_t* src = blocks + static_cast<size_t>(kb0 + it) * PACKED_BLOCK;
      const uint32_t prev = static_cast<uint32_t>((it - 1) & 1);
      if (p.pack_flags && !wait_packed(p, b, kb0 + it, tag, s_abort, p.err)) break;
      for (int g = 0; g < 5; ++g) {
        // Pair g of this block overwrites pair g of the previous one (and
        // the rope chunk its P^T): wait until O^T(k-1) has read them.
        if (it > 0 && g < 4) wait_warp(mbar(MB_OT + g), prev, s_abort, p.err);
        if (*s_abort) break;
        const uint32_t bytes = g < 4 ? 2 * KV_CHUNK : KV_CHUNK;
        const uint32_t off = g < 4 ? 2 * g * KV_CHUNK : 8 * KV_CHUNK;
        tc::bulk_copy_expect(sbase + OFF_KV + off, src + off, bytes, mbar(MB_CHUNK + g));
        ++issued;
      }
      if (*s_abort) break;
    }
    // After an abort the last copy into each slot may still be in flight:
    // let it land before shared memory is reused or released.
    if (*s_abort) {
      for (int g = 0; g < 5 && g < issued; ++g)
        wait_drain(mbar(MB_CHUNK + g), static_cast<uint32_t>(((issued - 1 - g) / 5) & 1), p.err);
      __syncwarp();
    }
  } else if (warp == MMA_WARP) {
    // ============================ MMA issuer ===============================
    // The whole warp runs the loop (warp-uniform operands); one elected lane
    // issues each MMA and commit.
    if (nb > 0) {
      wait_warp(mbar(MB_Q), 0, s_abort, p.err);
      tc::fence_after_sync();
#pragma unroll 1
      for (int it = 0; it < nb; ++it) {
        const uint32_t par = static_cast<uint32_t>(it & 1);
        for (int g = 0; g < 5; ++g) {
          wait_warp(mbar(MB_CHUNK + g), par, s_abort, p.err);
          tc::fence_after_sync();
          const int k0 = g < 4 ? 8 * g : 32, k1 = g < 4 ? k0 + 8 : 36;
          for (int k = k0; k < k1; ++k) {
            const uint64_t a = tc::desc_sw128(sbase + OFF_KV + (k >> 2) * KV_CHUNK + (k & 3) * 32, 16, 1024);
            const uint64_t bq = tc::desc_sw128(sbase + OFF_Q + (k >> 2) * Q_CHUNK + (k & 3) * 32, 16, 1024);
            tc::mma_ss(tmem + TM_S, a, bq, IDESC_S, k > 0);
          }
        }
        tc::commit(mbar(MB_S));
        wait_warp(mbar(MB_P), par, s_abort, p.err);
        tc::fence_after_sync();
        for (int d = 0; d < 4; ++d) {
#pragma unroll
          for (int k = 0; k < BN / 16; ++k) {
            const uint64_t a = tc::desc_sw128(sbase + OFF_KV + 2 * d * KV_CHUNK + k * 2048, KV_CHUNK, 1024);
            const uint64_t bp = tc::desc_sw128(sbase + OFF_P + k * 2048, 8192, 1024);
            tc::mma_ss(tmem + d * BM, a, bp, IDESC_O, (it > 0 || k > 0) ? 1u : 0u);
          }
          tc::commit(mbar(MB_OT + d));
        }
      }
      // After an abort the waits above returned early and the softmax warps'
      // wait for the last O^T tile may not have covered every MMA: let them
      // all finish before TMEM is freed.
      if (__any_sync(0xffffffffu, *s_abort != 0)) {
        tc::commit(mbar(MB_DONE));
        wait_drain(mbar(MB_DONE), 0, p.err);
      }
    }
  } else if (warp < SOFTMAX_WARPS) {
    // ============================= softmax =================================
    // The Q tile (issued at entry) to fp16.  The ancestor masks are ready
    // after the barrier that follows the load.
    if (nb > 0) {
      if (tid < p.T) s_mask[tid] = ancestor_mask(s_par, tid, p.err);
      asm volatile("cp.async.wait_group 0;\n" ::: "memory");
      named_sync(1, SOFTMAX_WARPS * 32);
      bool bad = false;
#pragma unroll 1
      for (int e = tid; e < BM * ROW_CHUNKS; e += SOFTMAX_WARPS * 32) {
        uint4* ptr = reinterpret_cast<uint4*>(smem + OFF_Q + e * 16);
        *ptr = widen_bf16x8(*ptr, bad);
      }
      report_range(bad, p.err);
      tc::fence_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(mbar(MB_Q));
    } else {
      asm volatile("cp.async.wait_all;\n" ::: "memory");   // no key block: Q unused
    }
    const int j = quad * 32 + lane;     // key of this thread = TMEM lane
    const int hc = warp >> 2;           // query-row columns hc*32 .. +32
    const int c0 = hc * HALF;
    const bool all_rows = row0 + BM <= p.R;
    const float scale2 = p.scale_log2;
    float mrow = -INFINITY;             // running max (base 2) of row c0 + lane
    float* w_m = reinterpret_cast<float*>(smem + OFF_WARP) + warp * 64;   // [32] row max, fully masked -> 0
    float* w_a = w_m + 32;                                                // [32] rescale factor
    float lpart[HALF];                  // this key's share of its rows' sums
#pragma unroll
    for (int c = 0; c < HALF; ++c) lpart[c] = 0.f;
    // Direct mode: out-of-cache slots are reported here (else by the pack).
    constexpr bool direct = kDirect;
    int slot_next = nb > 0 ? block_slot(p, rq, kb0, j, direct) : -1;
    bool next_ok = slot_next >= 0;
#pragma unroll 1
    for (int it = 0; it < nb; ++it) {
      const int kb = kb0 + it;
      const uint32_t par = static_cast<uint32_t>(it & 1);
      const bool key_ok = next_ok;
      if (it + 1 < nb) next_ok = block_slot(p, rq, kb + 1, j, direct) >= 0;
      if (direct) {
        // Block kb's pieces as the gather warps' copies land: widen to fp16
        // in place (8 granules a thread per chunk pair, 4 of the rope chunk)
        // and release each to the MMA warp.
        bool bad = false;
#pragma unroll 1
        for (int g = 0; g < 5; ++g) {
          wait_warp(mbar(MB_RAW + g), par, s_abort, p.err);
          const int n = g < 4 ? 8 : 4;
#pragma unroll
          for (int i = 0; i < n; ++i) {
            const int e = tid + 256 * i;
            const int k = g < 4 ? e >> 4 : e >> 3;
            const int q = g < 4 ? 16 * g + (e & 15) : 64 + (e & 7);
            uint4* ptr = reinterpret_cast<uint4*>(smem + OFF_KV + (q >> 3) * KV_CHUNK + k * 128 +
                                                  (((q & 7) ^ (k & 7)) << 4));
            *ptr = widen_bf16x8(*ptr, bad);
          }
          tc::fence_async_smem();   // the tensor core reads the widened rows next
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(mbar(MB_CHUNK + g));
        }
        report_range(bad, p.err);
      }
      const int jg = kb * BN + j;
      // The half's rows that see this key (bit c: row c0 + c), decided
      // before the scores arrive: every row for a prefix key, the draft's
      // ancestors for a draft key, none past the request.
      uint32_t vis = 0;
      if (key_ok) {
        if (jg < rq.P && all_rows) {
          vis = 0xffffffffu;
        } else {
          const int di = jg - rq.P;   // draft index when >= 0
#pragma unroll
          for (int c = 0; c < HALF; ++c) {
            const int t = s_tofr[c0 + c];
            bool v = t >= 0;
            if (v && di >= 0) v = (s_mask[t] >> di) & 1u;
            vis |= (v ? 1u : 0u) << c;
          }
        }
      }
      wait_warp(mbar(MB_S), par, s_abort, p.err);
      tc::fence_after_sync();
      uint32_t sr[HALF];
      tc::tmem_ld32(tmem + (static_cast<uint32_t>(quad * 32) << 16) + TM_S + c0, sr);
      tc::tmem_wait_ld();
      float* s = reinterpret_cast<float*>(sr);   // scores overwrite the raw bits in place
      if (vis == 0xffffffffu) {
#pragma unroll
        for (int c = 0; c < HALF; ++c) s[c] = __uint_as_float(sr[c]) * scale2;
      } else {
#pragma unroll
        for (int c = 0; c < HALF; ++c) s[c] = (vis >> c) & 1u ? __uint_as_float(sr[c]) * scale2 : -INFINITY;
      }
      // Column (query row) max: over this warp's 32 keys (lane l ends with
      // column c0 + l), then over the four quads.  Lane l keeps the running
      // max of column c0 + l in a register.
      {
        float v[HALF];
#pragma unroll
        for (int c = 0; c < HALF; ++c) v[c] = s[c];
        transpose_max32(v, lane);
        s_red[(c0 + lane) * 4 + quad] = v[0];
      }
      named_sync(1, 256);
      bool moved;
      uint32_t moved_rows;
      {
        const float4 q4 = *reinterpret_cast<const float4*>(s_red + (c0 + lane) * 4);
        const float bm = fmaxf(fmaxf(q4.x, q4.y), fmaxf(q4.z, q4.w));
        float alpha = 1.f;
        if (bm > mrow) {
          if (mrow != -INFINITY) alpha = ex2(mrow - bm);
          mrow = bm;
        }
        moved_rows = __ballot_sync(0xffffffffu, alpha != 1.f);
        moved = moved_rows != 0;
        w_m[lane] = mrow == -INFINITY ? 0.f : mrow;   // a fully masked row: every p = ex2(-inf) = 0
        w_a[lane] = alpha;
        __syncwarp();
      }
      // Rescale of the O^T columns of this half's rows whose max moved
      // (O^T(k-1) is complete: S^T(k) finished after it on the in-order
      // tensor pipe).  A few rows: their columns of the four tiles are loaded
      // now, while P is computed, then scaled and stored; many: the whole
      // half after P.
      const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16) + c0;
      const int cnt = __popc(moved_rows);
      const bool few = moved && cnt <= FEW_MOVED;
      uint32_t rv[FEW_MOVED][4];
      uint32_t cols[FEW_MOVED];
      if (few) {
        uint32_t m = moved_rows;
#pragma unroll
        for (int i = 0; i < FEW_MOVED; ++i) {
          const int c = m ? __ffs(m) - 1 : 0;
          m &= m - 1;
          cols[i] = static_cast<uint32_t>(c);
          if (i < cnt)
#pragma unroll
            for (int d = 0; d < 4; ++d) rv[i][d] = tc::tmem_ld1(lane_base + d * BM + c);
        }
      }
      // This key's P^T entries for the half's 32 query rows as fp16 (four
      // 16-byte granules of the key's 128-byte swizzled row), into the rope
      // chunk tile (S^T(k) no longer reads it).
      uint32_t pk[HALF / 2];
      if (moved) {
#pragma unroll
        for (int c = 0; c < HALF; c += 2) {
          const float2 m = *reinterpret_cast<const float2*>(w_m + c);
          const float2 al = *reinterpret_cast<const float2*>(w_a + c);
          const float p0 = ex2(s[c] - m.x), p1 = ex2(s[c + 1] - m.y);
          lpart[c] = lpart[c] * al.x + p0;
          lpart[c + 1] = lpart[c + 1] * al.y + p1;
          __half2 h = __floats2half2_rn(p0, p1);
          pk[c >> 1] = *reinterpret_cast<uint32_t*>(&h);
        }
      } else {
#pragma unroll
        for (int c = 0; c < HALF; c += 2) {
          const float2 m = *reinterpret_cast<const float2*>(w_m + c);
          const float p0 = ex2(s[c] - m.x), p1 = ex2(s[c + 1] - m.y);
          lpart[c] += p0;
          lpart[c + 1] += p1;
          __half2 h = __floats2half2_rn(p0, p1);
          pk[c >> 1] = *reinterpret_cast<uint32_t*>(&h);
        }
      }
      uint8_t* prow = smem + OFF_P + j * 128;
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const int gg = hc * 4 + g;
        *reinterpret_cast<uint4*>(prow + ((gg ^ (j & 7)) << 4)) =
            make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
      }
      if (few) {
        tc::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < FEW_MOVED; ++i)
          if (i < cnt) {
            const float a = w_a[cols[i]];
#pragma unroll
            for (int d = 0; d < 4; ++d)
              tc::tmem_st1(lane_base + d * BM + cols[i], __float_as_uint(__uint_as_float(rv[i][d]) * a));
          }
        tc::tmem_wait_st();
      } else if (moved) {
#pragma unroll 1
        for (int d = 0; d < 4; d += 2) {
          const uint32_t ta = lane_base + d * BM;
          uint32_t v0[HALF], v1[HALF];
          tc::tmem_ld32(ta, v0);
          tc::tmem_ld32(ta + BM, v1);
          tc::tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < HALF; ++c) {
            const float a = w_a[c];
            v0[c] = __float_as_uint(__uint_as_float(v0[c]) * a);
            v1[c] = __float_as_uint(__uint_as_float(v1[c]) * a);
          }
          tc::tmem_st32(ta, v0);
          tc::tmem_st32(ta + BM, v1);
        }
        tc::tmem_wait_st();
      }
      tc::fence_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(mbar(MB_P));
    }
    if (nb > 0) {
      wait_warp(mbar(MB_OT + 3), static_cast<uint32_t>((nb - 1) & 1), s_abort, p.err);
      tc::fence_after_sync();
    }
    if (quad == 0) s_mref[c0 + lane] = mrow;
    // Row sums over all keys: this warp's 32 keys, then 4 quads.
#pragma unroll
    for (int c = 0; c < HALF; ++c) {
      float v = lpart[c];
#pragma unroll
      for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (c == lane) s_red[quad * BM + c0 + c] = v;
    }
    named_sync(1, 256);
    if (tid < BM) {
      const float l = s_red[tid] + s_red[BM + tid] + s_red[2 * BM + tid] + s_red[3 * BM + tid];
      s_l[tid] = l > 0.f ? 1.f / l : 0.f;
      const int gr = row0 + tid;
      if (gr < p.R) {
        const float lse = l > 0.f ? (s_mref[tid] + log2f(l)) * kLn2 : -INFINITY;
        if (p.nsplit == 1) p.lse[static_cast<size_t>(b) * p.R + gr] = lse;
        else p.ws_lse[ws_base(p, b, split) + gr] = lse;
      }
    }
  }

  // ---- normalised O out of TMEM (thread = value dim), staged row-major in
  // the idle key-block buffer, then one bulk store per row.
  tc::fence_before_sync();
  __syncthreads();
  // The combine may be scheduled now; it waits for this grid to complete.
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  tc::fence_after_sync();
  if (*s_abort != 0) {
    write_nan_rows(p, b, split, row0, tid);
  } else {
    const bool out16 = p.nsplit == 1 && p.out_bf16;
    const size_t ws_row = ws_base(p, b, split);
    if (warp < SOFTMAX_WARPS) {
      // Softmax warp (quad, half): the half's 32 rows of every O^T tile, two
      // tiles per TMEM wait, thread = value dim, stored straight from
      // registers: each warp store covers 32 consecutive dims of one row (128
      // contiguous bytes of fp32).  Staging the tile in shared memory for
      // bulk row stores measured ~3 us slower per CTA in the pair kernel.
      const int h = warp >> 2;
#pragma unroll 1
      for (int d = 0; d < 4; d += 2) {
        uint32_t v0[32], v1[32];
        if (nb > 0) {
          const uint32_t ta = tmem + (static_cast<uint32_t>(quad * 32) << 16) + d * BM + h * 32;
          tc::tmem_ld32(ta, v0);
          tc::tmem_ld32(ta + BM, v1);
          tc::tmem_wait_ld();
        }
        const int dim0 = d * 128 + quad * 32 + lane, dim1 = dim0 + 128;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int r = h * 32 + c, gr = row0 + r;
          if (gr >= p.R) continue;   // rows past R (warp-uniform)
          const float inv = s_l[r];
          const bool ok = inv > 0.f && nb > 0;
          const float o0 = ok ? __uint_as_float(v0[c]) * inv : 0.f;
          const float o1 = ok ? __uint_as_float(v1[c]) * inv : 0.f;
          if (p.nsplit > 1) {
            float* dst = p.ws_o + (ws_row + gr) * D_V;
            dst[dim0] = o0;
            dst[dim1] = o1;
          } else {
            const size_t e = (static_cast<size_t>(b) * p.R + gr) * D_V;
            if (out16) {
              reinterpret_cast<__nv_bfloat16*>(p.out)[e + dim0] = __float2bfloat16_rn(o0);
              reinterpret_cast<__nv_bfloat16*>(p.out)[e + dim1] = __float2bfloat16_rn(o1);
            } else {
              reinterpret_cast<float*>(p.out)[e + dim0] = o0;
              reinterpret_cast<float*>(p.out)[e + dim1] = o1;
            }
          }
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == MMA_WARP) tc::tmem_dealloc<TMEM_COLS>(tmem);
  if (tid == 0) finish_call(p);
}

}  // namespace

cudaError_t partial_tc_prepare() {
  for (auto fn : {partial_tc_kernel<false>, partial_tc_kernel<true>}) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_TOTAL);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_partial_tc(const Params& p, cudaStream_t stream, bool overlap) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.nsplit, (p.R + BM - 1) / BM, p.batch);
  // The second gather warp exists only when the CTAs gather their own keys.
  cfg.blockDim = dim3(p.direct_all ? NTHREADS : NTHREADS - 32);
  cfg.dynamicSmemBytes = SMEM_TOTAL;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  return p.direct_all ? cudaLaunchKernelEx(&cfg, partial_tc_kernel<true>, p)
                      : cudaLaunchKernelEx(&cfg, partial_tc_kernel<false>, p);
}

}  // namespace mlav
