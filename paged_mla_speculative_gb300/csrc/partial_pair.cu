// Split-KV partial kernel on a CTA pair (tcgen05 cta_group::2): the
// "partial" half of the partial + reduce design in "The Decisive A/B: When
// Benchmarking Honesty Reveals the Real Bottleneck" (section "The Context":
// KV split for occupancy, a fixed split count, one reduce), over the packed
// key blocks of pack_kv.cu.
//
// A cluster of two CTAs takes 128 query rows (r = t*H + h) of one request
// and one key split, and walks it in pair blocks of 256 keys: 128-key packed
// block 2i of the split for the even CTA, 2i+1 for the odd one.  Every MMA
// has M = 256 and N = 128 and is issued for both CTAs by one thread of the
// even CTA:
//     S^T[key, row] = K_pair[256 x 576] . Q_tile[128 x 576]^T
//         A: each CTA's own 128 keys, K-major, from its ring slots;
//         B: Q rows 0..63 from the even CTA, 64..127 from the odd one;
//         D: each CTA's TMEM holds the scores of its own keys for all 128
//            rows (two buffers of 128 columns, so S^T(i+1) runs while the
//            softmax warps work on S^T(i)).
//     O^T[dim, row] += V_pair^T[512 x 256] . P^T[256 x 128]   (two M tiles)
//         A: tile t, dims 256t .. 256t+127 from the even CTA, the next 128
//            from the odd one, for all 256 keys (both blocks' chunk pairs
//            are streamed to each CTA);
//         B: P^T rows 0..63 from the even CTA, 64..127 from the odd one, for
//            all 256 keys -- each CTA's softmax writes half of its keys' P^T
//            into the peer's shared memory;
//         D: each CTA holds its 256 value dims for all 128 rows in TMEM
//            columns 0..255 for the whole split.
// Per CTA the MMAs read 6 KB of shared memory per 64 cycles of tensor work
// (the single-CTA M128 N64 form reads 6 KB per 32), which is what lets the
// tensor pipe, not the shared-memory port, set the pace.
//
// The softmax is the one of partial_tc.cu (exact running max, P <= 1 with
// the maximum key's weight exactly 1, fp16 P, O^T rescaled in TMEM only for
// rows whose max moved), with the block max of each row combined across the
// pair through distributed shared memory.
//
// Roles (20 warps per CTA):
//   warps 0-15  softmax: thread = (key = TMEM lane 32*(w%4) + lane, 32 query
//               rows 32*(w/4) ..); they load and widen the CTA's Q half first;
//   warp 16     even CTA: issues every MMA (one elected lane); odd CTA: tells
//               the even CTA when its half of P^T is complete; in both it
//               allocates and frees the pair's TMEM;
//   warps 17-19 stream the packed chunk pairs into a ring of three 32 KB
//               slots, one warp per slot (and the rope chunk into its own
//               slot), with pair TMA loads: both CTAs' copies complete on the
//               even CTA's barrier.
// MMA order: S^T(0), S^T(1), O^T(0), S^T(2), O^T(1), .., O^T(n-1); the ring
// streams its chunk pairs in the same order (the value chunks of block i a
// second time for O^T(i)), and a slot is refilled as soon as its MMAs are done.
// Every wait is bounded.
//
// Cross-CTA signals carry their data or their bytes with them (pair TMA
// loads, st.async into the peer's shared memory, tcgen05.commit multicast):
// a release arrive at cluster scope, which waits for the SM's outstanding
// copies, measured microseconds on this path.
#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace mlav {
namespace {

constexpr int ROWS = 128;           // query rows per pair: MMA N
constexpr int HROWS = 64;           // rows of the B operands a CTA holds
constexpr int BN = 128;             // keys per CTA per pair block
constexpr int SOFTMAX_WARPS = 16, MMA_WARP = 16, COPY_WARP = 17;
constexpr int NCOPY = 3;            // copy warps: copy warp k fills ring slot k
constexpr int NWARPS = COPY_WARP + NCOPY;
constexpr int NTHREADS = NWARPS * 32;
constexpr int SM_THREADS = SOFTMAX_WARPS * 32;
constexpr int CHUNK = BN * 128;          // 16 KB: 128 keys x 64 dims fp16
constexpr int Q_CHUNK = HROWS * 128;     // 8 KB: 64 rows x 64 dims
constexpr int NSLOT = NCOPY;             // ring slots of one chunk pair (32 KB)
constexpr int OFF_Q = 0;
constexpr int OFF_P = OFF_Q + 9 * Q_CHUNK;            // P^T [key half][128 keys][64 rows] fp16
constexpr int OFF_RING = OFF_P + 2 * CHUNK;
constexpr int OFF_ROPE = OFF_RING + NSLOT * 2 * CHUNK;   // the rope chunk's own slot
constexpr int OFF_RING_END = OFF_ROPE + CHUNK;
constexpr int OFF_RED = OFF_RING_END;                 // float [128 rows][4 quads]
constexpr int OFF_XMAX = OFF_RED + ROWS * 4 * 4;      // float [2][128] the peer's block row max
constexpr int OFF_XSUM = OFF_XMAX + 2 * ROWS * 4;     // float [128] the peer's row sums
constexpr int OFF_M = OFF_XSUM + ROWS * 4;            // float [128] running row max (0: none yet)
constexpr int OFF_A = OFF_M + ROWS * 4;               // float [128] rescale factor of the step
constexpr int OFF_L = OFF_A + ROWS * 4;               // float [128] 1 / row sum (0: none)
constexpr int OFF_MREF = OFF_L + ROWS * 4;            // float [128] final row max (base 2)
constexpr int OFF_MASK = OFF_MREF + ROWS * 4;         // uint32 [32] ancestor masks
constexpr int OFF_TOFR = OFF_MASK + MAX_T * 4;        // int [128] draft of each row, -1 past R
constexpr int OFF_PAR = OFF_TOFR + ROWS * 4;          // int [32] draft parents
constexpr int OFF_MBAR = OFF_PAR + MAX_T * 4;         // uint64 [NMBAR]
constexpr int NMBAR = 20;
constexpr int OFF_MISC = OFF_MBAR + NMBAR * 8;        // tmem base, P-complete word, absent-unit word, abort flag
constexpr int SMEM_TOTAL = OFF_MISC + 16;
static_assert(SMEM_TOTAL <= 232448, "shared memory budget");
static_assert(OFF_P % 1024 == 0 && OFF_RING % 1024 == 0,
              "swizzled tiles need 1024-byte alignment");

// mbarrier indices (same offsets in both CTAs)
constexpr int MB_FULL = 0;     // [3] even CTA: ring slot landed in both CTAs (bytes of both)
constexpr int MB_EMPTY = 3;    // [3] ring slot read by its MMAs (commit to both CTAs)
constexpr int MB_RFULL = 6;    // even CTA: rope slot landed in both CTAs
constexpr int MB_REMPTY = 7;   // rope slot read
constexpr int MB_S = 8;        // [2] S^T buffer done
constexpr int MB_P = 10;       // this CTA's softmax warps wrote their P^T and rescaled O^T
constexpr int MB_PX = 11;      // the peer's half of this CTA's P^T landed (st.async bytes)
constexpr int MB_PF = 12;      // even CTA: the odd CTA's P^T is complete (st.async word)
constexpr int MB_OT = 13;      // O^T of a pair block done
constexpr int MB_Q = 14;       // even CTA: both Q halves in fp16, one arrival per softmax warp of the pair
constexpr int MB_X = 15;       // [2] the peer's block row max landed (st.async bytes)
constexpr int MB_XS = 17;      // the peer's row sums landed (st.async bytes)
constexpr int MB_DONE = 18;    // after an abort: every MMA issued is done

constexpr int TMEM_COLS = 512;
constexpr uint32_t TM_S = 256;                  // S^T buffer u at 256 + 128u; O^T tile t at 128t
constexpr long long WAIT_LIMIT = 1LL << 31;     // cycles before a wait gives up

constexpr uint32_t IDESC_S = tc::idesc_f16(256, ROWS, 0, 0, 0);   // fp16, both K-major
constexpr uint32_t IDESC_O = tc::idesc_f16(256, ROWS, 0, 1, 1);   // fp16, both MN-major

constexpr int FEW_MOVED = 4;
constexpr uint32_t ABSENT_BYTES = 4;   // the odd CTA's signal for a unit it has no block for

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes));
}
__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(count) : "memory");
}

// Bounded wait (acquire at cluster scope: some arrivals come from the peer
// CTA).  A timeout, or an earlier one in this CTA, returns false.
__device__ __forceinline__ bool wait_phase(uint32_t mbar, uint32_t parity, volatile int* abort, int* err) {
  if (tc::mbar_try_cluster(mbar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (tc::mbar_try_cluster(mbar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > WAIT_LIMIT) {
      *abort = 1;
      atomicOr(err, ERR_TIMEOUT);
      return false;
    }
  }
}
__device__ __forceinline__ void wait_warp(uint32_t mbar, uint32_t parity, volatile int* abort, int* err) {
  wait_phase(mbar, parity, abort, err);
  __syncwarp();
}
// Bounded wait that ignores the abort flag (own copies in flight at exit).
__device__ __forceinline__ void wait_drain(uint32_t mbar, uint32_t parity, int* err) {
  const long long t0 = clock64();
  while (!tc::mbar_try(mbar, parity)) {
    if (clock64() - t0 > WAIT_LIMIT) {
      atomicOr(err, ERR_TIMEOUT);
      return;
    }
  }
}

// Same as partial_tc.cu: wait (bounded) for the 32 ready flags of packed
// block kb of request b carrying this call's tag.  Whole warp.
__device__ __forceinline__ bool wait_packed(const Params& p, int b, int kb, unsigned long long tag,
                                            volatile int* abort, int* err) {
  const int lane = threadIdx.x & 31;
  const unsigned long long* flag =
      pack_flags(p.pack_sync) + 32 * (static_cast<size_t>(b) * p.packed_max_blocks + kb) + lane;
  const long long t0 = clock64();
  while (true) {
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
  asm volatile("fence.proxy.async.global;\n" ::: "memory");
  return true;
}

__device__ __forceinline__ void finish_call(const Params& p) {
  __threadfence();
  const unsigned total = gridDim.x * gridDim.y * gridDim.z;
  if (atomicAdd(p.pack_sync + PACK_SYNC_TICKET, 1u) == total - 1) {
    p.pack_sync[PACK_SYNC_TICKET] = 0;
    *reinterpret_cast<volatile unsigned long long*>(p.pack_sync) = pack_epoch(p.pack_sync) + 1ull;
  }
}

// Column maxima / sums of a warp's 32 x 32 tile (lane = key, v[c] = column
// c) in 31 shuffles: lane l ends with column l's result in v[0].
template <bool SUM>
__device__ __forceinline__ void transpose_reduce32(float (&v)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = upper ? v[i] : v[i + w];
      const float keep = upper ? v[i + w] : v[i];
      const float got = __shfl_xor_sync(0xffffffffu, send, w);
      v[i] = SUM ? keep + got : fmaxf(keep, got);
    }
  }
}

// Slot of key r of 128-key block kb, or -1 past the call's keys or when the
// table points outside the cache.
__device__ __forceinline__ int block_slot(const Params& p, const Request& rq, int kb, int r) {
  const int j = kb * BN + r;
  if (j < rq.lo || j >= rq.hi) return -1;
  return static_cast<int>(key_slot(p, rq.ip0, j));
}

// Ring unit order shared by the copy warps and the MMA warp.  Phase f of 2n:
// S(0), S(1), O(0), S(2), O(1), .., S(n-1), O(n-2), O(n-1); S(i) = the CTA's
// own block's chunk pairs 0..3 (and its rope chunk, into the rope slot),
// O(i) = for t in 0,1 and key half h in 0,1: chunk pair 2t + rank of block
// 2i + h.  Unit n goes to slot n % 3.
__device__ __forceinline__ void phase_of(int f, int n, bool& is_s, int& i) {
  if (f == 0) { is_s = true; i = 0; }
  else if (f == 2 * n - 1) { is_s = false; i = n - 1; }
  else if (f & 1) { is_s = true; i = (f + 1) >> 1; }
  else { is_s = false; i = (f >> 1) - 1; }
}

// Rows of this CTA's output: NaN (a request the kernel cannot serve).
__device__ __forceinline__ void write_nan_rows(const Params& p, int b, int split, int row0, uint32_t rank,
                                               int tid) {
  const float nan = __int_as_float(0x7fc00000);
  const size_t ws_row = ws_base(p, b, split);
  for (int i = tid; i < ROWS * 256; i += NTHREADS) {
    const int lr = i >> 8, dd = i & 255;
    const int d = (dd >> 7) * 256 + static_cast<int>(rank) * 128 + (dd & 127);
    const int gr = row0 + lr;
    if (gr >= p.R) continue;
    const bool lse_here = (dd == 0) && (lr >> 6) == static_cast<int>(rank);
    if (p.nsplit == 1) {
      const size_t o = (static_cast<size_t>(b) * p.R + gr) * D_V + d;
      if (p.out_bf16) reinterpret_cast<uint16_t*>(p.out)[o] = 0x7fc0;
      else reinterpret_cast<float*>(p.out)[o] = nan;
      if (lse_here) p.lse[static_cast<size_t>(b) * p.R + gr] = nan;
    } else {
      p.ws_o[(ws_row + gr) * D_V + d] = nan;
      if (lse_here) p.ws_lse[ws_row + gr] = nan;
    }
  }
}


// Spin about `cycles` (an abort path: lets copies and remote stores that
// are still in flight land before the pair leaves).
__device__ __forceinline__ void settle(long long cycles) {
  const long long t0 = clock64();
  while (clock64() - t0 < cycles) {
  }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS, 1)
    partial_pair_kernel(const Params p, const __grid_constant__ CUtensorMap tm_pair,
                        const __grid_constant__ CUtensorMap tm_chunk) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t rank = tc::cluster_rank();
  const uint32_t peer = rank ^ 1u;
  const int split = blockIdx.x >> 1, pt = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3;            // TMEM lanes 32*quad .. +32 are this warp's
  const int grp = warp >> 2;            // softmax: rows 32*grp .. +32
  const int row0 = pt * ROWS;

  float* s_red = reinterpret_cast<float*>(smem + OFF_RED);
  float* s_xmax = reinterpret_cast<float*>(smem + OFF_XMAX);
  float* s_xsum = reinterpret_cast<float*>(smem + OFF_XSUM);
  float* s_m = reinterpret_cast<float*>(smem + OFF_M);
  float* s_a = reinterpret_cast<float*>(smem + OFF_A);
  float* s_l = reinterpret_cast<float*>(smem + OFF_L);
  float* s_mref = reinterpret_cast<float*>(smem + OFF_MREF);
  uint32_t* s_mask = reinterpret_cast<uint32_t*>(smem + OFF_MASK);
  int* s_tofr = reinterpret_cast<int*>(smem + OFF_TOFR);
  int* s_par = reinterpret_cast<int*>(smem + OFF_PAR);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + OFF_MISC + 12);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t mbar0 = sbase + OFF_MBAR;
  auto mbar = [&](int i) { return mbar0 + 8u * static_cast<uint32_t>(i); };

  // This CTA's Q half: pair rows 64*rank .. +64, 9 swizzled chunks (rows
  // beyond R zero), loaded by the softmax warps first.
  if (warp < SOFTMAX_WARPS) {
    const uint16_t* qb = p.q + static_cast<size_t>(b) * p.R * D_QK;
#pragma unroll 1
    for (int e = tid; e < HROWS * ROW_CHUNKS; e += SM_THREADS) {
      const int r = e / ROW_CHUNKS, q = e - r * ROW_CHUNKS;
      const int gr = row0 + static_cast<int>(rank) * HROWS + r;
      const bool in = gr < p.R;
      cp_async16(sbase + OFF_Q + (q >> 3) * Q_CHUNK + r * 128 + (((q & 7) ^ (r & 7)) << 4),
                 in ? qb + static_cast<size_t>(gr) * D_QK + q * 8 : p.q, in ? 16 : 0);
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
  }

  // The draft parents load alongside the request lookup (independent
  // global loads, each a memory latency).
  if (tid < p.T) s_par[tid] = p.draft_parent[b * p.T + tid];
  // Both CTAs of the pair see the same request and take the same branches
  // up to the pair's first cluster barrier.
  const Request rq = load_request(p, b);
  if (!rq.ok || (sbase & 1023)) {
    if (!rq.ok && split == 0 && pt == 0 && rank == 0 && tid == 0)
      atomicOr(p.err, (rq.n < p.T || rq.n > p.max_kv_len) ? ERR_LEN : ERR_INDPTR);
    if (rq.ok && tid == 0) atomicOr(p.err, ERR_INTERNAL);
    write_nan_rows(p, b, split, row0, rank, tid);
    if (tid == 0) finish_call(p);
    asm volatile("cp.async.wait_all;\n" ::: "memory");
    return;
  }

  int kb0, kb1;
  split_range(p, rq, split, kb0, kb1);
  const int nb = (kb1 - kb0 + 1) >> 1;   // pair blocks; the last may hold one block

  if (tid < ROWS) s_tofr[tid] = row0 + tid < p.R ? (row0 + tid) / p.H : -1;
  if (tid == 0) {
    for (int i = 0; i < NSLOT; ++i) {
      tc::mbar_init(mbar(MB_FULL + i), 1);
      tc::mbar_init(mbar(MB_EMPTY + i), 1);
    }
    tc::mbar_init(mbar(MB_RFULL), 1);
    tc::mbar_init(mbar(MB_REMPTY), 1);
    tc::mbar_init(mbar(MB_S), 1);
    tc::mbar_init(mbar(MB_S + 1), 1);
    tc::mbar_init(mbar(MB_P), SOFTMAX_WARPS);
    tc::mbar_init(mbar(MB_PX), 1);
    tc::mbar_init(mbar(MB_PF), 1);
    tc::mbar_init(mbar(MB_OT), 1);
    tc::mbar_init(mbar(MB_Q), 2 * SOFTMAX_WARPS);
    tc::mbar_init(mbar(MB_X), 1);
    tc::mbar_init(mbar(MB_X + 1), 1);
    tc::mbar_init(mbar(MB_XS), 1);
    tc::mbar_init(mbar(MB_DONE), 1);
    tc::mbar_fence_init();
    *s_abort = 0;
  }
  if (warp == MMA_WARP) tc::tmem_alloc_pair<TMEM_COLS>(smem_u32(s_tmem));
  tc::fence_before_sync();
  __syncthreads();
  // The peer's barriers exist (their initialisation was published by
  // fence.mbarrier_init) and the pair's TMEM is allocated.  A release arrive
  // here would first wait for this CTA's Q loads, still in flight.
  tc::cluster_sync_relaxed();
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;
  const uint32_t even_mbar0 = tc::peer_addr(mbar0, 0);   // the even CTA's barriers
  const uint32_t peer_mbar0 = tc::peer_addr(mbar0, peer);
  auto even_mbar = [&](int i) { return even_mbar0 + 8u * static_cast<uint32_t>(i); };
  auto peer_mbar = [&](int i) { return peer_mbar0 + 8u * static_cast<uint32_t>(i); };
  auto present = [&](int i, int h) { return kb0 + 2 * i + h < kb1; };

  if (warp >= COPY_WARP) {
    // ========================= chunk producers ==============================
    // Copy warp k fills ring slot k (units k, k + 3, ..); the rope chunks
    // go with slot 2.  A warp's bulk copies complete one after another
    // (about 600 cycles each up to 32 KB), so each slot has its own warp.
    const int cw = warp - COPY_WARP;
    // Every unit completes with a signal from both CTAs' copy warps, each
    // sent after the warp's wait for the slot: for a block past the end of
    // the split (the odd CTA's, at the last pair block of an odd block
    // count) the odd CTA sends ABSENT_BYTES instead of the copy.  Otherwise
    // the even CTA's MMAs could consume units the odd CTA took no part in,
    // its slot barriers could run two phases ahead of its copy warp, and a
    // parity wait would then never end.
    const uint32_t absent_word = tc::peer_addr(smem_u32(s_tmem + 2), 0);
    // Row of the packed buffer (rows of 128 bytes) where chunk c of block kb
    // of request b starts.
    auto chunk_row = [&](int kb, int c) {
      return ((b * p.packed_max_blocks + kb) * 9 + c) * BN;
    };
    const unsigned long long tag = pack_epoch(p.pack_sync) + 1ull;
    if (!p.pack_flags) asm volatile("griddepcontrol.wait;\n" ::: "memory");
    int waited = kb0 - 1;   // highest block whose pack flags were seen
    auto ensure_packed = [&](int kb) {
      if (!p.pack_flags || kb <= waited) return true;
      for (int k = waited + 1; k <= kb; ++k)
        if (!wait_packed(p, b, k, tag, s_abort, p.err)) return false;
      waited = kb;
      return true;
    };
    int n = 0;   // units of the sequence so far
#pragma unroll 1
    for (int f = 0; f < 2 * nb && !*s_abort; ++f) {
      bool is_s;
      int i;
      phase_of(f, nb, is_s, i);
#pragma unroll 1
      for (int u = 0; u < 4; ++u, ++n) {
        const int slot = n % NSLOT;
        if (slot != cw) continue;
        // S units: the own block (the peer loads its own); O units: block
        // (i, h) in both CTAs.
        const int h = is_s ? static_cast<int>(rank) : (u & 1);
        const int pair_idx = is_s ? u : 2 * (u >> 1) + static_cast<int>(rank);
        const int kb = kb0 + 2 * i + h;
        const bool mine = kb < kb1;
        const bool peers = is_s ? present(i, static_cast<int>(peer)) : mine;
        // An overlapping pack's ready flags first: the acquire round trip
        // then overlaps the wait for the slot instead of following it.
        if (mine && !ensure_packed(kb)) break;
        if (n >= NSLOT) wait_warp(mbar(MB_EMPTY + slot), static_cast<uint32_t>((n / NSLOT - 1) & 1), s_abort, p.err);
        if (*s_abort) break;
        if (rank == 0) {
          if (lane == 0)
            tc::mbar_arrive_expect(mbar(MB_FULL + slot), (mine ? 2 * CHUNK : 0) + (peers ? 2 * CHUNK : ABSENT_BYTES));
          __syncwarp();
        }
        if (mine) {
          tc::tma_load_2d_pair(sbase + OFF_RING + slot * 2 * CHUNK, &tm_pair, 0, chunk_row(kb, 2 * pair_idx),
                               even_mbar(MB_FULL + slot));
        } else if (rank == 1) {
          if (lane == 0) tc::st_async_b32(absent_word, 0, even_mbar(MB_FULL + slot));
          __syncwarp();
        }
      }
      if (*s_abort) break;
      if (is_s && cw == NCOPY - 1) {
        // The rope chunk of the own block, once S^T(i-1) has read the last one.
        const int kb = kb0 + 2 * i + static_cast<int>(rank);
        const bool mine = kb < kb1, peers = present(i, static_cast<int>(peer));
        if (mine && !ensure_packed(kb)) break;
        if (i > 0) wait_warp(mbar(MB_REMPTY), static_cast<uint32_t>((i - 1) & 1), s_abort, p.err);
        if (*s_abort) break;
        if (rank == 0) {
          if (lane == 0) tc::mbar_arrive_expect(mbar(MB_RFULL), (mine ? CHUNK : 0) + (peers ? CHUNK : ABSENT_BYTES));
          __syncwarp();
        }
        if (mine) {
          tc::tma_load_2d_pair(sbase + OFF_ROPE, &tm_chunk, 0, chunk_row(kb, 8), even_mbar(MB_RFULL));
        } else if (rank == 1) {
          if (lane == 0) tc::st_async_b32(absent_word, 0, even_mbar(MB_RFULL));
          __syncwarp();
        }
      }
    }
    // After an abort, copies already issued (into this CTA, signalling the
    // even CTA) land within microseconds: wait far longer than that before
    // the pair's shared memory can be released.
    if (*s_abort) settle(1LL << 22);
  } else if (warp == MMA_WARP && rank == 1) {
    // =================== odd CTA: P^T complete -> even CTA ==================
    // This CTA's half of P^T(i) is its own softmax warps' stores (MB_P) plus
    // the even CTA's st.async bytes (MB_PX); when both are in, one st.async
    // word to the even CTA's MB_PF.
    uint32_t* s_word = s_tmem + 1;
    const uint32_t even_word = tc::peer_addr(smem_u32(s_word), 0);
#pragma unroll 1
    for (int i = 0; i < nb; ++i) {
      if (lane == 0) tc::mbar_arrive_expect(mbar(MB_PX), CHUNK);
      __syncwarp();
      wait_warp(mbar(MB_P), static_cast<uint32_t>(i & 1), s_abort, p.err);
      wait_warp(mbar(MB_PX), static_cast<uint32_t>(i & 1), s_abort, p.err);
      tc::fence_async_smem();   // the st.async bytes are read by the tensor core next
      if (lane == 0) tc::st_async_b32(even_word, static_cast<uint32_t>(i), even_mbar(MB_PF));
      __syncwarp();
    }
  } else if (warp == MMA_WARP) {
    // ======================= MMA issuer (even CTA) ==========================
    if (nb > 0) {
      wait_warp(mbar(MB_Q), 0, s_abort, p.err);
      tc::fence_after_sync();
      int n = 0;
#pragma unroll 1
      for (int f = 0; f < 2 * nb && !*s_abort; ++f) {
        bool is_s;
        int i;
        phase_of(f, nb, is_s, i);
        if (is_s) {
          const uint32_t d = tmem + TM_S + 128u * static_cast<uint32_t>(i & 1);
#pragma unroll 1
          for (int u = 0; u < 4; ++u, ++n) {
            const int slot = n % NSLOT;
            wait_warp(mbar(MB_FULL + slot), static_cast<uint32_t>((n / NSLOT) & 1), s_abort, p.err);
            tc::fence_after_sync();
            const uint32_t base = sbase + OFF_RING + slot * 2 * CHUNK;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const int k = 8 * u + kk;   // 16-dim step of the 576-dim contraction
              const uint64_t a = tc::desc_sw128(base + (kk >> 2) * CHUNK + (kk & 3) * 32, 16, 1024);
              const uint64_t bq = tc::desc_sw128(sbase + OFF_Q + (k >> 2) * Q_CHUNK + (k & 3) * 32, 16, 1024);
              tc::mma_pair(d, a, bq, IDESC_S, k > 0);
            }
            tc::commit_pair(mbar(MB_EMPTY + slot));
          }
          wait_warp(mbar(MB_RFULL), static_cast<uint32_t>(i & 1), s_abort, p.err);
          tc::fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t a = tc::desc_sw128(sbase + OFF_ROPE + kk * 32, 16, 1024);
            const uint64_t bq = tc::desc_sw128(sbase + OFF_Q + 8 * Q_CHUNK + kk * 32, 16, 1024);
            tc::mma_pair(d, a, bq, IDESC_S, 1);
          }
          tc::commit_pair(mbar(MB_REMPTY));
          tc::commit_pair(mbar(MB_S + (i & 1)));
        } else {
          // P^T(i): this CTA's softmax warps, the odd CTA's st.async bytes,
          // and the odd CTA's word that its own half is complete.
          if (lane == 0) {
            tc::mbar_arrive_expect(mbar(MB_PX), CHUNK);
            tc::mbar_arrive_expect(mbar(MB_PF), 4);
          }
          __syncwarp();
          wait_warp(mbar(MB_P), static_cast<uint32_t>(i & 1), s_abort, p.err);
          wait_warp(mbar(MB_PX), static_cast<uint32_t>(i & 1), s_abort, p.err);
          wait_warp(mbar(MB_PF), static_cast<uint32_t>(i & 1), s_abort, p.err);
          tc::fence_async_smem();
          tc::fence_after_sync();
#pragma unroll 1
          for (int u = 0; u < 4; ++u, ++n) {
            const int t = u >> 1, h = u & 1;
            const int slot = n % NSLOT;
            wait_warp(mbar(MB_FULL + slot), static_cast<uint32_t>((n / NSLOT) & 1), s_abort, p.err);
            tc::fence_after_sync();
            if (present(i, h)) {
              const uint32_t base = sbase + OFF_RING + slot * 2 * CHUNK;
#pragma unroll
              for (int kk = 0; kk < 8; ++kk) {   // 16-key steps of the key half
                const uint64_t a = tc::desc_sw128(base + kk * 2048, CHUNK, 1024);
                const uint64_t bp = tc::desc_sw128(sbase + OFF_P + h * CHUNK + kk * 2048, CHUNK, 1024);
                tc::mma_pair(tmem + 128u * static_cast<uint32_t>(t), a, bp, IDESC_O,
                             (i > 0 || h > 0 || kk > 0) ? 1u : 0u);
              }
            }
            tc::commit_pair(mbar(MB_EMPTY + slot));
          }
          tc::commit_pair(mbar(MB_OT));
        }
      }
      // After an abort: every MMA issued finishes before TMEM is freed.
      if (__any_sync(0xffffffffu, *s_abort != 0)) {
        tc::commit_pair(mbar(MB_DONE));
        wait_drain(mbar(MB_DONE), 0, p.err);
      }
    }
  } else if (warp < SOFTMAX_WARPS) {
    // ============================= softmax =================================
    if (nb > 0) {
      if (tid < p.T) s_mask[tid] = ancestor_mask(s_par, tid, p.err);
      asm volatile("cp.async.wait_group 0;\n" ::: "memory");
      named_sync(1, SM_THREADS);
      bool bad = false;
#pragma unroll 1
      for (int e = tid; e < HROWS * ROW_CHUNKS; e += SM_THREADS) {
        uint4* ptr = reinterpret_cast<uint4*>(smem + OFF_Q + e * 16);
        *ptr = widen_bf16x8(*ptr, bad);
      }
      report_range(bad, p.err);
      tc::fence_async_smem();
      __syncwarp();
      // Once per call: release at cluster scope (the odd CTA's Q half is read
      // by MMAs the even CTA issues).
      if (lane == 0) tc::mbar_arrive_cluster(even_mbar(MB_Q));
    } else {
      asm volatile("cp.async.wait_all;\n" ::: "memory");
    }
    const int j = quad * 32 + lane;     // key of this thread = TMEM lane
    const int c0 = grp * 32;            // pair rows c0 .. c0+31
    const bool all_rows = row0 + ROWS <= p.R;
    const float scale2 = p.scale_log2;
    const bool owner = quad == 0;       // lane l owns row c0 + l's running max
    float mrow = -INFINITY;
    float lrun = 0.f;                   // row c0 + lane's sum over this warp's keys so far
    // This key's P^T row (key half = rank) in the CTA that holds the group's
    // rows: a local store, or st.async into the peer with its MB_PX.
    const bool p_local = (grp >> 1) == static_cast<int>(rank);
    const uint32_t p_off = OFF_P + rank * CHUNK + j * 128;
    const uint32_t p_peer = tc::peer_addr(sbase + p_off, peer);
    const uint32_t xmax_peer = tc::peer_addr(sbase + OFF_XMAX, peer);
#pragma unroll 1
    for (int it = 0; it < nb; ++it) {
      const int kb = kb0 + 2 * it + static_cast<int>(rank);
      // Read while S^T(it) is still being computed.
      const bool key_ok = block_slot(p, rq, kb, j) >= 0;
      const int jg = kb * BN + j;
      // The group's rows that see this key (bit c: row c0 + c), decided
      // while S^T(it) is computed: every row for a prefix key, the draft's
      // ancestors for a draft key, none past the request.  (Applying the
      // tree mask row by row after the scores arrive cost ~3 us per pass on
      // the block that holds the drafts.)
      uint32_t vis = 0;
      if (key_ok) {
        if (jg < rq.P && all_rows) {
          vis = 0xffffffffu;
        } else {
          const int di = jg - rq.P;
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int t = s_tofr[c0 + c];
            bool v = t >= 0;
            if (v && di >= 0) v = (s_mask[t] >> di) & 1u;
            vis |= (v ? 1u : 0u) << c;
          }
        }
      }
      const uint32_t sb = static_cast<uint32_t>(it & 1);
      wait_warp(mbar(MB_S + sb), static_cast<uint32_t>((it >> 1) & 1), s_abort, p.err);
      tc::fence_after_sync();
      const uint32_t s_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + TM_S + 128u * sb + c0;
      float s[32];
      auto load_scores = [&]() { tc::tmem_ld32f(s_addr, s); };
      auto mask_scores = [&]() {
        if (vis == 0xffffffffu) {
#pragma unroll
          for (int c = 0; c < 32; ++c) s[c] *= scale2;
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) s[c] = (vis >> c) & 1u ? s[c] * scale2 : -INFINITY;
        }
      };
      load_scores();
      tc::tmem_wait_ld();
      mask_scores();
      transpose_reduce32<false>(s, lane);
      s_red[(c0 + lane) * 4 + quad] = s[0];
      named_sync(1, SM_THREADS);
      const uint32_t xb = static_cast<uint32_t>(it & 1);
      if (owner) {
        const float4 q4 = *reinterpret_cast<const float4*>(s_red + (c0 + lane) * 4);
        float bm = fmaxf(fmaxf(q4.x, q4.y), fmaxf(q4.z, q4.w));
        // The row max of the own keys to the peer (512 bytes from the four
        // owner warps), and the peer's into this CTA's MB_X.
        tc::st_async_b32(xmax_peer + (xb * ROWS + c0 + lane) * 4, __float_as_uint(bm), peer_mbar(MB_X + xb));
        if (tid == 0) tc::mbar_arrive_expect(mbar(MB_X + xb), ROWS * 4);
        wait_phase(mbar(MB_X + xb), static_cast<uint32_t>((it >> 1) & 1), s_abort, p.err);
        bm = fmaxf(bm, s_xmax[xb * ROWS + c0 + lane]);
        float alpha = 1.f;
        if (bm > mrow) {
          if (mrow != -INFINITY) alpha = ex2(mrow - bm);
          mrow = bm;
        }
        s_m[c0 + lane] = mrow == -INFINITY ? 0.f : mrow;   // a fully masked row: p = ex2(-inf) = 0
        s_a[c0 + lane] = alpha;
      }
      named_sync(1, SM_THREADS);
      // Rows whose max moved (the same mask in every lane).
      uint32_t moved_rows = 0;
#pragma unroll
      for (int c = 0; c < 32; c += 4) {
        const float4 a4 = *reinterpret_cast<const float4*>(s_a + c0 + c);
        moved_rows |= (a4.x != 1.f ? 1u : 0u) << c | (a4.y != 1.f ? 1u : 0u) << (c + 1) |
                      (a4.z != 1.f ? 1u : 0u) << (c + 2) | (a4.w != 1.f ? 1u : 0u) << (c + 3);
      }
      // O^T(it-1) done: the P^T buffers (here and in the peer) are free and
      // O^T can be rescaled.
      if (it > 0) {
        wait_warp(mbar(MB_OT), static_cast<uint32_t>((it - 1) & 1), s_abort, p.err);
        tc::fence_after_sync();
      }
      if (moved_rows != 0 && it > 0) {
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16) + c0;
        const int cnt = __popc(moved_rows);
        if (cnt <= FEW_MOVED) {
          uint32_t m = moved_rows;
          for (int k = 0; k < cnt; ++k) {
            const int c = __ffs(m) - 1;
            m &= m - 1;
            const float a = s_a[c0 + c];
            const uint32_t v0 = tc::tmem_ld1(lane_base + c);
            const uint32_t v1 = tc::tmem_ld1(lane_base + 128 + c);
            tc::tmem_wait_ld();
            tc::tmem_st1(lane_base + c, __float_as_uint(__uint_as_float(v0) * a));
            tc::tmem_st1(lane_base + 128 + c, __float_as_uint(__uint_as_float(v1) * a));
          }
        } else {
#pragma unroll 1
          for (int t = 0; t < 2; ++t) {
            uint32_t v[32];
            tc::tmem_ld32(lane_base + 128u * t, v);
            tc::tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * s_a[c0 + c]);
            tc::tmem_st32(lane_base + 128u * t, v);
          }
        }
        tc::tmem_wait_st();
      }
      load_scores();   // again, for P (registers were spent on the max)
      tc::tmem_wait_ld();
      mask_scores();
      // This key's P^T for the group's 32 rows, eight rows (one 16-byte
      // granule of the key's swizzled 128-byte row) at a time.
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const float4 m0 = *reinterpret_cast<const float4*>(s_m + c0 + 8 * g);
        const float4 m1 = *reinterpret_cast<const float4*>(s_m + c0 + 8 * g + 4);
        const float mm[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          const int c = 8 * g + e;
          const float p0 = ex2(s[c] - mm[e]), p1 = ex2(s[c + 1] - mm[e + 1]);
          s[c] = p0;
          s[c + 1] = p1;
          __half2 hh = __floats2half2_rn(p0, p1);
          pk[e >> 1] = *reinterpret_cast<uint32_t*>(&hh);
        }
        const uint32_t gran = static_cast<uint32_t>((((grp & 1) * 4 + g) ^ (j & 7)) << 4);
        const uint4 v = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        if (p_local) *reinterpret_cast<uint4*>(smem + p_off + gran) = v;
        else tc::st_async_v4(p_peer + gran, v, peer_mbar(MB_PX));
      }
      // The step's row sums over this warp's 32 keys (lane l: row c0 + l),
      // folded into the running sum after its rescale.
      transpose_reduce32<true>(s, lane);
      lrun = lrun * s_a[c0 + lane] + s[0];
      tc::fence_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(mbar(MB_P));
    }
    if (nb > 0) {
      wait_warp(mbar(MB_OT), static_cast<uint32_t>((nb - 1) & 1), s_abort, p.err);
      tc::fence_after_sync();
      // Row sums over the pair's keys: the four quads, then the peer's.
      s_red[(c0 + lane) * 4 + quad] = lrun;
      named_sync(1, SM_THREADS);
      if (owner) {
        const float4 q4 = *reinterpret_cast<const float4*>(s_red + (c0 + lane) * 4);
        const float ls = (q4.x + q4.y) + (q4.z + q4.w);
        tc::st_async_b32(tc::peer_addr(sbase + OFF_XSUM + (c0 + lane) * 4, peer), __float_as_uint(ls),
                         peer_mbar(MB_XS));
        if (tid == 0) tc::mbar_arrive_expect(mbar(MB_XS), ROWS * 4);
        wait_phase(mbar(MB_XS), 0, s_abort, p.err);
        // Both CTAs add the two halves in the same order.
        const float lo = rank == 0 ? ls : s_xsum[c0 + lane];
        const float hi = rank == 0 ? s_xsum[c0 + lane] : ls;
        const float l = lo + hi;
        const int r = c0 + lane;
        s_l[r] = l > 0.f ? 1.f / l : 0.f;
        s_mref[r] = mrow;
        const int gr = row0 + r;
        if (gr < p.R && (r >> 6) == static_cast<int>(rank)) {
          const float lse = l > 0.f ? (mrow + log2f(l)) * kLn2 : -INFINITY;
          if (p.nsplit == 1) p.lse[static_cast<size_t>(b) * p.R + gr] = lse;
          else p.ws_lse[ws_base(p, b, split) + gr] = lse;
        }
      }
    } else if (owner) {
      const int r = c0 + lane, gr = row0 + r;
      s_l[r] = 0.f;
      if (gr < p.R && (r >> 6) == static_cast<int>(rank)) {
        if (p.nsplit == 1) p.lse[static_cast<size_t>(b) * p.R + gr] = -INFINITY;
        else p.ws_lse[ws_base(p, b, split) + gr] = -INFINITY;
      }
    }
  }

  // ---- normalised O out of TMEM, thread = value dim, stored straight from
  // registers: each warp store covers 32 consecutive dims of one row (128
  // contiguous bytes of fp32).  Staging the tile in shared memory for 512-byte
  // bulk stores measured ~4 us per CTA, against ~1 us for these stores.
  tc::fence_before_sync();
  __syncthreads();
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  tc::fence_after_sync();
  if (*s_abort != 0) {
    write_nan_rows(p, b, split, row0, rank, tid);
  } else if (warp < SOFTMAX_WARPS) {
    const bool out16 = p.nsplit == 1 && p.out_bf16;
    const int c0 = grp * 32;
    const size_t ws_row = ws_base(p, b, split);
#pragma unroll 1
    for (int t = 0; t < 2; ++t) {
      uint32_t v[32];
      if (nb > 0) {
        tc::tmem_ld32(tmem + (static_cast<uint32_t>(quad * 32) << 16) + 128u * t + c0, v);
        tc::tmem_wait_ld();
      }
      const int dim = t * 256 + static_cast<int>(rank) * 128 + quad * 32 + lane;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const int r = c0 + c, gr = row0 + r;
        if (gr >= p.R) continue;   // rows past R (warp-uniform)
        const float inv = s_l[r];
        const float o = (inv > 0.f && nb > 0) ? __uint_as_float(v[c]) * inv : 0.f;
        if (p.nsplit > 1) {
          p.ws_o[(ws_row + gr) * D_V + dim] = o;
        } else {
          const size_t e = (static_cast<size_t>(b) * p.R + gr) * D_V + dim;
          if (out16) reinterpret_cast<__nv_bfloat16*>(p.out)[e] = __float2bfloat16_rn(o);
          else reinterpret_cast<float*>(p.out)[e] = o;
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  // Neither CTA leaves while the peer may still write into its shared
  // memory, signal its barriers or (even CTA) read its operands.
  tc::cluster_sync();
  tc::fence_after_sync();
  if (warp == MMA_WARP) tc::tmem_dealloc_pair<TMEM_COLS>(tmem);
  if (tid == 0) finish_call(p);
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

}  // namespace

cudaError_t make_pack_maps(PackMaps* maps, void* packed, size_t packed_bytes) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return e != cudaSuccess ? e : cudaErrorNotSupported;
  const EncodeTiled encode = reinterpret_cast<EncodeTiled>(fn);
  // The packed buffer as rows of 64 fp16 (128 bytes); its blocks are already
  // in the swizzled operand layout, so the copies do not swizzle.
  const cuuint64_t dims[2] = {64, packed_bytes / 128};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t estrides[2] = {1, 1};
  const cuuint32_t box_pair[2] = {64, 256}, box_chunk[2] = {64, 128};
  CUresult r = encode(&maps->pair, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, packed, dims, strides, box_pair, estrides,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r == CUDA_SUCCESS)
    r = encode(&maps->chunk, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, packed, dims, strides, box_chunk, estrides,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t partial_pair_prepare() {
  cudaError_t e = cudaFuncSetAttribute(partial_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SMEM_TOTAL);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(partial_pair_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                              cudaSharedmemCarveoutMaxShared);
}

cudaError_t launch_partial_pair(const Params& p, const PackMaps& maps, cudaStream_t stream, bool overlap) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * p.nsplit, (p.R + ROWS - 1) / ROWS, p.batch);
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = SMEM_TOTAL;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, partial_pair_kernel, p, maps.pair, maps.chunk);
}

}  // namespace mlav
