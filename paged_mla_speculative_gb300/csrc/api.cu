// C ABI of the verify-attention library: plan (workspace owner), argument
// checks, split planning and the capture-safe launch sequence.
//
// The launch path follows the capture-safety recipe of "The Decisive A/B:
// When Benchmarking Honesty Reveals the Real Bottleneck" (section "The
// Context"): a fixed split count, workspace allocated ahead of time, native
// buffer pointers, and no host synchronisation or device-memory read per
// call, so the whole call can be recorded in a CUDA graph.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <algorithm>
#include <new>

#include <cstdint>

#include "mla_verify.h"
#include "kernels.h"

using mlav::Params;

struct mla_verify_plan {
  int device;
  int max_batch, T, H, R, page_size;
  int64_t num_slots;
  int max_kv_len;
  int out_dtype;
  int num_sms;
  int forced_nsplit;      // 0 = choose per call
  int kernel;             // MLA_VERIFY_KERNEL_*
  long long ws_capacity;  // request-splits the workspace holds
  float* ws_o;
  float* ws_lse;
  int* err;
  size_t ws_bytes;
  // Device staging for mla_verify_attn_host.
  void* st_q;
  int32_t* st_idx;
  int32_t* st_indptr;
  int32_t* st_lens;
  int32_t* st_parent;
  void* st_out;
  float* st_lse;
  long long st_idx_cap;
  cudaEvent_t ev_after_pack;     // profiling: recorded after the pack kernel, or null
  cudaEvent_t ev_after_partial;  // profiling: recorded after the partial kernel, or null
  // Packed fp16 key blocks for the TC kernel: max_batch x pack_blocks blocks.
  void* packed;
  int pack_blocks;
  unsigned* pack_sync;    // epoch, ticket, per-unit ready flags (see Params)
  size_t pack_sync_bytes;
  // A call failed after its pack kernel was launched: its flags may carry
  // the tag the next call will use, so the next call clears them first.
  bool pack_flags_dirty;
  int fault;              // MLA_VERIFY_FAULT_* injected into the next call
  int pack_mode;          // MLA_VERIFY_PACK_* forced, or AUTO
  // mla_verify_get_error: an event recorded at the end of the last call made
  // outside capture, and a private stream to read the error word on.
  cudaEvent_t done_ev;
  bool done_recorded;
  cudaStream_t aux;
  // TMA descriptors of `packed` for the CTA-pair kernel.
  mlav::PackMaps pack_maps;
};

namespace {

constexpr int kRowsPerTile = 64;

// Keys one split step takes in each partial kernel: 64 (mma.sync), one
// 128-key block (TC), a 256-key pair block (PAIR).
int keys_per_block(int kernel) {
  return kernel == MLA_VERIFY_KERNEL_MMA ? 64 : kernel == MLA_VERIFY_KERNEL_PAIR ? 256 : 128;
}
// Query rows one unit of the grid (a CTA, or a CTA pair for PAIR) takes, and
// its CTAs.
int rows_per_unit(int kernel) { return kernel == MLA_VERIFY_KERNEL_PAIR ? 128 : kRowsPerTile; }
int ctas_per_unit(int kernel) { return kernel == MLA_VERIFY_KERNEL_PAIR ? 2 : 1; }
// Measured on GB300 (us): one split step (a 128-key block of a TC CTA, a
// 256-key pair block of a PAIR cluster) and a CTA's fixed cost (prologue,
// pipeline fill, epilogue), from the attention kernel's time over contexts
// of 1k to 93k keys.
double step_us(int kernel) { return kernel == MLA_VERIFY_KERNEL_PAIR ? 4.8 : 3.4; }
double fixed_us(int kernel) { return kernel == MLA_VERIFY_KERNEL_PAIR ? 20.0 : 16.0; }

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

constexpr long long kDirectMaxTiles = 1;   // 2 tiles measured slower (each block gathered twice)

// The attention CTAs gather their own key blocks (no pack): one row tile per
// request, or forced.
bool gathers_directly(const mla_verify_plan* pl) {
  return pl->pack_mode == MLA_VERIFY_PACK_NONE || ceil_div(pl->R, kRowsPerTile) <= kDirectMaxTiles;
}

// Pack schedule (see pack_kv.cu).  When the kernels may overlap and the
// attention grid leaves at least kMinPackSms SMs idle, the two-phase pack:
// `stay` = those idle SMs keep packing while the attention kernel runs, the
// others first pack the `wide` leading block positions of every split.
// `wide` is the fewest positions that keep the narrow phase ahead of the
// attention kernel, from rates measured on GB300: ~0.23 blocks/us per
// packing SM (the staged pack of pack_kv.cu, ~36 GB/s of rows alone on 24
// SMs, a little less beside a running attention kernel), one split step per
// step_us per attention unit, ~5 us before its first block.  When that needs more than half the positions, or
// otherwise, the whole pack runs first (stay = 0).
struct PackSchedule {
  int mode;       // MLA_VERIFY_PACK_WHOLE or _IDLE_SMS
  int wide, stay;
};
constexpr int kMinPackSms = 16;
PackSchedule pack_plan(const mla_verify_plan* pl, int fam, int batch, int nsplit, bool overlap,
                       int shards = 1) {
  const bool pairs = fam == MLA_VERIFY_KERNEL_PAIR;
  // Block positions per split (pairs of positions when splits take pairs).
  const long long shard_blocks = ceil_div(pl->pack_blocks, shards);
  const int positions = static_cast<int>(pairs ? 2 * ceil_div(ceil_div(shard_blocks, 2), nsplit)
                                               : ceil_div(shard_blocks, nsplit));
  const long long attn = 1LL * nsplit * ceil_div(pl->R, rows_per_unit(fam)) * batch * ctas_per_unit(fam);
  const long long idle = pl->num_sms - attn;
  const PackSchedule whole{MLA_VERIFY_PACK_WHOLE, positions, 0};
  if (!overlap || pl->pack_mode == MLA_VERIFY_PACK_WHOLE) return whole;
  const bool forced_idle = pl->pack_mode == MLA_VERIFY_PACK_IDLE_SMS;
  if (idle < (forced_idle ? 1 : kMinPackSms)) return whole;
  const double per_block_us = pairs ? step_us(fam) / 2 : step_us(fam), lead_us = 5.0,
               blocks_per_us_per_sm = 0.23;
  const double narrow_us = static_cast<double>(nsplit) * batch / (idle * blocks_per_us_per_sm);
  // Position q >= wide is ready after (q - wide + 1) narrow steps and needed
  // after lead + q attention steps; with narrow steps the slower, the last
  // position binds.
  int wide = 1;
  if (narrow_us > per_block_us)
    wide = static_cast<int>(std::ceil(positions - (lead_us + (positions - 1) * per_block_us) / narrow_us));
  wide = std::max(1, wide);
  if (2 * wide > positions && !forced_idle) return whole;
  return PackSchedule{MLA_VERIFY_PACK_IDLE_SMS, std::min(wide, positions), static_cast<int>(idle)};
}

// What the pack leaves on a call's critical path (us), at ~4.5 TB/s for a
// block's 1152-B rows read plus its 147 456 B written, plus ~3 us: the wide
// phase (`wide` block positions of every split) when it overlaps the
// attention kernel, else the whole gather of up to batch x max_kv_len rows;
// nothing when the attention CTAs gather directly.
double pack_us(const mla_verify_plan* pl, int fam, int batch, int nsplit, int shards) {
  if (fam == MLA_VERIFY_KERNEL_MMA || gathers_directly(pl)) return 0.0;
  const PackSchedule ps = pack_plan(pl, fam, batch, nsplit, true, shards);
  if (ps.mode != MLA_VERIFY_PACK_WHOLE)
    return 2.0 * 147456.0 * ps.wide * nsplit * batch / 4.5e12 * 1e6 + 3.0;
  return 2304.0 * batch * ceil_div(pl->max_kv_len, shards) / 4.5e12 * 1e6 + 3.0;
}

// Split steps run ~7 % slower beside the overlapping pack (its loads and
// stores share L2 and HBM with the attention kernel's copies): fitted on the
// 93k sweep point, 15 / 16 / 17 splits with the pack on 32 / 24 / 16 idle SMs
// at 142.6 / 145.5 / 152.4 us per call against 157.8 with 19 splits and the
// whole pack first.
constexpr double kBesidePack = 1.07;

// Keys a request can hold in a call covering one of `shards` shards: a
// shard takes at most ceil(nb / shards) of the request's nb 128-key blocks.
long long call_keys(const mla_verify_plan* pl, int shards) {
  return std::min<long long>(pl->max_kv_len, ceil_div(ceil_div(pl->max_kv_len, 128), shards) * 128);
}

// Split steps a request can have: pair blocks of a range with an odd block
// count may hold one block.
long long max_steps(const mla_verify_plan* pl, int kernel, int shards) {
  return kernel == MLA_VERIFY_KERNEL_PAIR ? ceil_div(ceil_div(call_keys(pl, shards), 128), 2)
                                          : ceil_div(call_keys(pl, shards), keys_per_block(kernel));
}

// Moving the split partials through the combine (us): a launch, and the
// partials' bytes (just written, in L2) at ~15 TB/s -- measured: 8.2 us for
// 2 splits and 10.2 us for 19 splits of 512 rows.
double combine_us(const mla_verify_plan* pl, int kernel, int batch, int ns) {
  if (ns <= 1) return 0.0;
  const double units = static_cast<double>(batch) * ceil_div(pl->R, rows_per_unit(kernel));
  return 3.4 + units * rows_per_unit(kernel) * ns * 4096.0 / 15e6;
}

// Estimated time (us) of a call of family `kernel` with `ns` splits: waves of
// units, each its fixed cost plus its split steps (slower beside an
// overlapping pack), then the combine and what the pack leaves on the
// critical path.
double split_call_us(const mla_verify_plan* pl, int kernel, int batch, int ns, int shards) {
  const long long units = static_cast<long long>(batch) * ceil_div(pl->R, rows_per_unit(kernel));
  const double waves = static_cast<double>(ceil_div(units * ns, pl->num_sms / ctas_per_unit(kernel)));
  const double steps = static_cast<double>(ceil_div(max_steps(pl, kernel, shards), ns));
  const bool beside = kernel != MLA_VERIFY_KERNEL_MMA && !gathers_directly(pl) &&
                      pack_plan(pl, kernel, batch, ns, true, shards).mode == MLA_VERIFY_PACK_IDLE_SMS;
  return waves * (fixed_us(kernel) + steps * step_us(kernel) * (beside ? kBesidePack : 1.0)) +
         combine_us(pl, kernel, batch, ns) + pack_us(pl, kernel, batch, ns, shards);
}

// Split count for `batch` requests: minimise (waves of units) x (steps per
// unit) plus the combine, in units of one split step.
int auto_nsplit(const mla_verify_plan* pl, int batch, int kernel, int shards = 1) {
  const long long units = static_cast<long long>(batch) * ceil_div(pl->R, rows_per_unit(kernel));
  const long long steps_max = max_steps(pl, kernel, shards);
  const int cap = static_cast<int>(std::min<long long>(mlav::MAX_NSPLIT, steps_max));
  const long long slots = pl->num_sms / ctas_per_unit(kernel);   // units resident at once
  const double st = step_us(kernel);
  auto best_split = [&](bool with_pack) {
    int best = 1;
    double best_cost = 1e300;
    for (int ns = 1; ns <= cap; ++ns) {
      const double waves = static_cast<double>(ceil_div(units * ns, slots));
      const double steps = static_cast<double>(ceil_div(steps_max, ns));
      double cost = waves * steps + combine_us(pl, kernel, batch, ns) / st;
      if (with_pack) cost += pack_us(pl, kernel, batch, ns, shards) / st;
      if (cost < best_cost - 1e-9) {
        best_cost = cost;
        best = ns;
      }
    }
    return best;
  };
  if (kernel == MLA_VERIFY_KERNEL_MMA || gathers_directly(pl)) return best_split(false);
  // Packed families: the split count whose whole call -- attention waves,
  // combine, and the pack schedule pack_plan picks for it -- is cheapest.
  // Fewer splits can leave enough SMs idle for the pack to run beside the
  // attention kernel instead of ahead of it (the 93k sweep point: 15 splits
  // and the overlapping pack, 142.6 us, against 19 and the whole pack first,
  // 157.8 us).
  int best = 1;
  double best_us = 1e300;
  for (int ns = 1; ns <= cap; ++ns) {
    const double us = split_call_us(pl, kernel, batch, ns, shards);
    if (us < best_us - 1e-9) {
      best_us = us;
      best = ns;
    }
  }
  return best;
}

// Forced counts are clamped to the number of split steps a request can have.
int family_nsplit(const mla_verify_plan* pl, int fam, int batch, int shards) {
  if (!pl->forced_nsplit) return auto_nsplit(pl, batch, fam, shards);
  return static_cast<int>(std::min<long long>(pl->forced_nsplit, max_steps(pl, fam, shards)));
}

// Estimated time (us) of a call of family `fam`: waves of units, each its
// fixed cost plus its split steps, then the combine and what the pack leaves
// on the critical path.
double call_estimate_us(const mla_verify_plan* pl, int fam, int batch, int shards) {
  return split_call_us(pl, fam, batch, family_nsplit(pl, fam, batch, shards), shards);
}

// The partial kernel a call launches.  One row tile per request, or no
// pack: the TC kernel's direct gather (PAIR always reads packed blocks).
// AUTO: the TC or PAIR kernel, whichever call_estimate_us expects faster
// (short contexts favour TC's smaller fixed cost, long ones PAIR's faster
// steps).
int call_family(const mla_verify_plan* pl, int batch, int shards = 1) {
  if (pl->kernel == MLA_VERIFY_KERNEL_MMA) return MLA_VERIFY_KERNEL_MMA;
  if (gathers_directly(pl)) return MLA_VERIFY_KERNEL_TC;
  if (pl->kernel != MLA_VERIFY_KERNEL_AUTO) return pl->kernel;
  return call_estimate_us(pl, MLA_VERIFY_KERNEL_TC, batch, shards) <=
                 call_estimate_us(pl, MLA_VERIFY_KERNEL_PAIR, batch, shards)
             ? MLA_VERIFY_KERNEL_TC
             : MLA_VERIFY_KERNEL_PAIR;
}

int effective_nsplit(const mla_verify_plan* pl, int batch, int shards = 1) {
  return family_nsplit(pl, call_family(pl, batch, shards), batch, shards);
}

PackSchedule pack_schedule(const mla_verify_plan* pl, const mlav::Params& p, bool overlap) {
  return pack_plan(pl, p.split_pairs ? MLA_VERIFY_KERNEL_PAIR : MLA_VERIFY_KERNEL_TC, p.batch, p.nsplit,
                   overlap, p.num_shards);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

void free_all(mla_verify_plan* p) {
  void* bufs[] = {p->ws_o, p->ws_lse, p->err, p->st_q, p->st_idx, p->st_indptr,
                  p->st_lens, p->st_parent, p->st_out, p->st_lse, p->packed, p->pack_sync};
  for (void* b : bufs)
    if (b) cudaFree(b);
}

// Mark the end of an eagerly launched call for mla_verify_get_error.  A call
// recorded into a graph is not tracked (the event would not fire on replay).
cudaError_t note_done(mla_verify_plan* pl, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cs);
  if (e != cudaSuccess) return e;
  if (cs != cudaStreamCaptureStatusNone) return cudaSuccess;
  e = cudaEventRecord(pl->done_ev, s);
  if (e == cudaSuccess) pl->done_recorded = true;
  return e;
}

// The device address of a page-locked host buffer mapped into the device's
// address space, or nullptr (pageable memory: the caller's copies go through
// DMA instead).  A cleared lookup error leaves no sticky state behind.
const void* device_view(const void* host) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

int check_device(const mla_verify_plan* pl) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_VERIFY_ERR_CUDA;
  return dev == pl->device ? MLA_VERIFY_OK : MLA_VERIFY_ERR_DEVICE;
}

}  // namespace

extern "C" {

int mla_verify_version(void) { return 100; }

const char* mla_verify_strerror(int status) {
  switch (status) {
    case MLA_VERIFY_OK: return "ok";
    case MLA_VERIFY_ERR_NULL: return "a required pointer is NULL";
    case MLA_VERIFY_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case MLA_VERIFY_ERR_SHAPE: return "unsupported shape, page size, dtype or split count";
    case MLA_VERIFY_ERR_BATCH: return "batch outside [1, max_batch]";
    case MLA_VERIFY_ERR_SCALE: return "scale is not finite";
    case MLA_VERIFY_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case MLA_VERIFY_ERR_DEVICE: return "the current CUDA device is not the plan's device";
    case MLA_VERIFY_ERR_OOM: return "device memory allocation failed";
    case MLA_VERIFY_ERR_ARG: return "invalid argument";
    case MLA_VERIFY_ERR_SCRATCH: return "the call needs more scratch than the static array holds";
    default: return "unknown status";
  }
}

int mla_verify_plan_create(mla_verify_plan** out, int max_batch, int num_drafts, int num_heads,
                           int page_size, int64_t num_slots, int max_kv_len, int out_dtype,
                           int device) {
  if (!out) return MLA_VERIFY_ERR_NULL;
  *out = nullptr;
  if (max_batch < 1 || num_drafts < 1 || num_drafts > mlav::MAX_T || num_heads < 1 ||
      static_cast<long long>(num_drafts) * num_heads > 4096 ||
      (page_size != 1 && page_size != mlav::PAGE) || num_slots < 1 || num_slots > INT32_MAX ||
      (page_size == mlav::PAGE && num_slots % mlav::PAGE) || max_kv_len < num_drafts ||
      (out_dtype != MLA_VERIFY_OUT_F32 && out_dtype != MLA_VERIFY_OUT_BF16))
    return MLA_VERIFY_ERR_SHAPE;
  if (cudaSetDevice(device) != cudaSuccess) return MLA_VERIFY_ERR_CUDA;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
    return MLA_VERIFY_ERR_CUDA;
  if (mlav::partial_mma_prepare() != cudaSuccess || mlav::partial_tc_prepare() != cudaSuccess ||
      mlav::partial_pair_prepare() != cudaSuccess || mlav::pack_kv_prepare() != cudaSuccess)
    return MLA_VERIFY_ERR_CUDA;

  mla_verify_plan* pl = new (std::nothrow) mla_verify_plan();
  if (!pl) return MLA_VERIFY_ERR_OOM;
  pl->device = device;
  pl->max_batch = max_batch;
  pl->T = num_drafts;
  pl->H = num_heads;
  pl->R = num_drafts * num_heads;
  pl->page_size = page_size;
  pl->num_slots = num_slots;
  pl->max_kv_len = max_kv_len;
  pl->out_dtype = out_dtype;
  pl->num_sms = sms;
  pl->kernel = MLA_VERIFY_KERNEL_AUTO;

  // Workspace capacity in request-splits: enough for the automatic choice at
  // every batch size, and for forced split counts up to a 64 MB floor.
  const long long max_blocks = ceil_div(max_kv_len, 64);
  long long cap = 0;
  for (int b = 1; b <= max_batch; ++b)
    for (int k : {MLA_VERIFY_KERNEL_MMA, MLA_VERIFY_KERNEL_TC, MLA_VERIFY_KERNEL_PAIR})
      cap = std::max<long long>(cap, 1LL * b * auto_nsplit(pl, b, k));
  const long long floor_rs = (64LL << 20) / (1LL * pl->R * (mlav::D_V + 1) * 4);
  cap = std::max(cap, std::min(1LL * max_batch * std::min<long long>(mlav::MAX_NSPLIT, max_blocks),
                               std::max(floor_rs, std::min<long long>(mlav::MAX_NSPLIT, max_blocks))));
  pl->ws_capacity = cap;
  const size_t rows = static_cast<size_t>(cap) * pl->R;
  const size_t out_elt = out_dtype == MLA_VERIFY_OUT_BF16 ? 2 : 4;
  const long long idx_per_req = page_size == 1 ? max_kv_len : ceil_div(max_kv_len, mlav::PAGE);
  pl->st_idx_cap = idx_per_req * max_batch;
  const size_t qrows = static_cast<size_t>(max_batch) * pl->R;

  bool ok = cudaMalloc(&pl->ws_o, rows * mlav::D_V * sizeof(float)) == cudaSuccess &&
            cudaMalloc(&pl->ws_lse, rows * sizeof(float)) == cudaSuccess &&
            cudaMalloc(&pl->err, 256) == cudaSuccess &&
            cudaMalloc(&pl->st_q, qrows * mlav::ROW_BYTES) == cudaSuccess &&
            cudaMalloc(&pl->st_idx, static_cast<size_t>(pl->st_idx_cap) * 4) == cudaSuccess &&
            cudaMalloc(&pl->st_indptr, static_cast<size_t>(max_batch + 1) * 4) == cudaSuccess &&
            cudaMalloc(&pl->st_lens, static_cast<size_t>(max_batch) * 4) == cudaSuccess &&
            cudaMalloc(&pl->st_parent, static_cast<size_t>(max_batch) * num_drafts * 4) == cudaSuccess &&
            cudaMalloc(&pl->st_out, qrows * mlav::D_V * out_elt) == cudaSuccess &&
            cudaMalloc(&pl->st_lse, qrows * sizeof(float)) == cudaSuccess;
  pl->pack_blocks = static_cast<int>(ceil_div(max_kv_len, 128));
  const size_t packed_bytes =
      static_cast<size_t>(max_batch) * pl->pack_blocks * mlav::packed_block_bytes();
  ok = ok && cudaMalloc(&pl->packed, packed_bytes) == cudaSuccess;
  ok = ok && mlav::make_pack_maps(&pl->pack_maps, pl->packed, packed_bytes) == cudaSuccess;
  const size_t sync_bytes =
      mlav::PACK_SYNC_HEADER * sizeof(unsigned) +
      static_cast<size_t>(max_batch) * pl->pack_blocks * 32 * sizeof(unsigned long long);
  ok = ok && cudaMalloc(&pl->pack_sync, sync_bytes) == cudaSuccess;
  pl->pack_sync_bytes = sync_bytes;
  if (!ok) {
    cudaGetLastError();
    free_all(pl);
    delete pl;
    return MLA_VERIFY_ERR_OOM;
  }
  pl->ws_bytes = rows * (mlav::D_V + 1) * sizeof(float) + 256 + packed_bytes + sync_bytes;
  if (cudaMemset(pl->err, 0, 256) != cudaSuccess || cudaMemset(pl->pack_sync, 0, sync_bytes) != cudaSuccess ||
      cudaEventCreateWithFlags(&pl->done_ev, cudaEventDisableTiming) != cudaSuccess ||
      cudaStreamCreateWithFlags(&pl->aux, cudaStreamNonBlocking) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    if (pl->done_ev) cudaEventDestroy(pl->done_ev);
    if (pl->aux) cudaStreamDestroy(pl->aux);
    free_all(pl);
    delete pl;
    return MLA_VERIFY_ERR_CUDA;
  }
  *out = pl;
  return MLA_VERIFY_OK;
}

void mla_verify_plan_destroy(mla_verify_plan* pl) {
  if (!pl) return;
  int prev = -1;
  cudaGetDevice(&prev);
  cudaSetDevice(pl->device);
  cudaDeviceSynchronize();
  if (pl->done_ev) cudaEventDestroy(pl->done_ev);
  if (pl->aux) cudaStreamDestroy(pl->aux);
  free_all(pl);
  if (prev >= 0) cudaSetDevice(prev);
  delete pl;
}

int mla_verify_plan_set_nsplit(mla_verify_plan* pl, int nsplit) {
  if (!pl) return MLA_VERIFY_ERR_NULL;
  if (nsplit < 0 || nsplit > mlav::MAX_NSPLIT) return MLA_VERIFY_ERR_SHAPE;
  pl->forced_nsplit = nsplit;
  return MLA_VERIFY_OK;
}

int mla_verify_plan_get_nsplit(const mla_verify_plan* pl, int batch) {
  if (!pl) return MLA_VERIFY_ERR_NULL;
  if (batch < 1 || batch > pl->max_batch) return MLA_VERIFY_ERR_BATCH;
  return effective_nsplit(pl, batch);
}

int mla_verify_plan_get_pack_schedule(const mla_verify_plan* pl, int batch, int* wide, int* stay) {
  if (!pl || !wide || !stay) return MLA_VERIFY_ERR_NULL;
  if (batch < 1 || batch > pl->max_batch) return MLA_VERIFY_ERR_BATCH;
  *wide = 0;
  *stay = 0;
  if (pl->kernel == MLA_VERIFY_KERNEL_MMA || gathers_directly(pl)) return MLA_VERIFY_OK;
  const int fam = call_family(pl, batch);
  const PackSchedule ps = pack_plan(pl, fam, batch, family_nsplit(pl, fam, batch, 1), true);
  *wide = ps.wide;
  *stay = ps.stay;
  return MLA_VERIFY_OK;
}

int mla_verify_plan_set_pack_schedule(mla_verify_plan* pl, int schedule) {
  if (!pl) return MLA_VERIFY_ERR_NULL;
  if (schedule != MLA_VERIFY_PACK_AUTO && schedule != MLA_VERIFY_PACK_WHOLE &&
      schedule != MLA_VERIFY_PACK_IDLE_SMS && schedule != MLA_VERIFY_PACK_NONE)
    return MLA_VERIFY_ERR_ARG;
  pl->pack_mode = schedule;
  return MLA_VERIFY_OK;
}

int mla_verify_plan_get_pack_mode(const mla_verify_plan* pl, int batch) {
  if (!pl) return MLA_VERIFY_ERR_NULL;
  if (batch < 1 || batch > pl->max_batch) return MLA_VERIFY_ERR_BATCH;
  if (pl->kernel == MLA_VERIFY_KERNEL_MMA || gathers_directly(pl)) return MLA_VERIFY_PACK_NONE;
  const int fam = call_family(pl, batch);
  return pack_plan(pl, fam, batch, family_nsplit(pl, fam, batch, 1), true).mode;
}

int mla_verify_plan_inject_fault(mla_verify_plan* pl, int fault) {
  if (!pl) return MLA_VERIFY_ERR_NULL;
  if (fault != MLA_VERIFY_FAULT_NONE && fault != MLA_VERIFY_FAULT_SKIP_PACK &&
      fault != MLA_VERIFY_FAULT_EPOCH_NEAR_WRAP)
    return MLA_VERIFY_ERR_ARG;
  pl->fault = fault;
  return MLA_VERIFY_OK;
}

int mla_verify_plan_set_kernel(mla_verify_plan* pl, int kernel) {
  if (!pl) return MLA_VERIFY_ERR_NULL;
  if (kernel != MLA_VERIFY_KERNEL_AUTO && kernel != MLA_VERIFY_KERNEL_MMA &&
      kernel != MLA_VERIFY_KERNEL_TC && kernel != MLA_VERIFY_KERNEL_PAIR)
    return MLA_VERIFY_ERR_ARG;
  pl->kernel = kernel;
  return MLA_VERIFY_OK;
}

int mla_verify_plan_get_kernel(const mla_verify_plan* pl) {
  if (!pl) return MLA_VERIFY_ERR_NULL;
  return pl->kernel;
}

int mla_verify_plan_get_call_kernel(const mla_verify_plan* pl, int batch) {
  if (!pl) return MLA_VERIFY_ERR_NULL;
  if (batch < 1 || batch > pl->max_batch) return MLA_VERIFY_ERR_BATCH;
  return call_family(pl, batch);
}

int mla_verify_plan_set_profile_events(mla_verify_plan* pl, void* after_pack, void* after_partial) {
  if (!pl) return MLA_VERIFY_ERR_NULL;
  pl->ev_after_pack = static_cast<cudaEvent_t>(after_pack);
  pl->ev_after_partial = static_cast<cudaEvent_t>(after_partial);
  return MLA_VERIFY_OK;
}

size_t mla_verify_plan_workspace_bytes(const mla_verify_plan* pl) { return pl ? pl->ws_bytes : 0; }

}  // extern "C"

namespace {

// One verify call (or one shard of it) on `s`: argument checks, the split
// count, then pack / partial / combine.  `out_bf16` is the output type.
int launch_call(mla_verify_plan* pl, int batch, const void* q, const void* kv_cache,
                const int32_t* kv_indices, const int32_t* kv_indptr, const int32_t* kv_lens,
                const int32_t* draft_parent, float scale, int shard, int num_shards, void* out,
                float* lse, bool out_bf16, cudaStream_t s) {
  if (!pl || !q || !kv_cache || !kv_indices || !kv_indptr || !kv_lens || !draft_parent || !out ||
      !lse)
    return MLA_VERIFY_ERR_NULL;
  if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(kv_indices) || !aligned16(kv_indptr) ||
      !aligned16(kv_lens) || !aligned16(draft_parent) || !aligned16(out) || !aligned16(lse))
    return MLA_VERIFY_ERR_ALIGN;
  if (batch < 1 || batch > pl->max_batch) return MLA_VERIFY_ERR_BATCH;
  if (!std::isfinite(scale)) return MLA_VERIFY_ERR_SCALE;
  if (num_shards < 1 || num_shards > mlav::MAX_NSPLIT || shard < 0 || shard >= num_shards)
    return MLA_VERIFY_ERR_ARG;
  const int dev_status = check_device(pl);
  if (dev_status != MLA_VERIFY_OK) return dev_status;
  const int fam = call_family(pl, batch, num_shards);
  const bool packs = fam != MLA_VERIFY_KERNEL_MMA;   // TC and PAIR read packed key blocks
  const int ns = family_nsplit(pl, fam, batch, num_shards);
  if (1LL * batch * ns > pl->ws_capacity) return MLA_VERIFY_ERR_SHAPE;

  Params p{};
  p.q = static_cast<const uint16_t*>(q);
  p.kv = static_cast<const uint16_t*>(kv_cache);
  p.kv_indices = kv_indices;
  p.kv_indptr = kv_indptr;
  p.kv_lens = kv_lens;
  p.draft_parent = draft_parent;
  p.scale_log2 = scale * mlav::kLog2e;
  p.batch = batch;
  p.T = pl->T;
  p.H = pl->H;
  p.R = pl->R;
  p.page_size = pl->page_size;
  p.num_slots = pl->num_slots;
  p.max_kv_len = pl->max_kv_len;
  p.nsplit = ns;
  p.shard = shard;
  p.num_shards = num_shards;
  p.ws_o = pl->ws_o;
  p.ws_lse = pl->ws_lse;
  p.ws_stride_b = 1LL * ns * pl->R;
  p.ws_stride_s = pl->R;
  p.out = out;
  p.lse = lse;
  p.out_bf16 = out_bf16 ? 1 : 0;
  p.err = pl->err;
  p.packed = static_cast<const uint8_t*>(pl->packed);
  p.packed_max_blocks = pl->pack_blocks;
  p.pack_sync = pl->pack_sync;
  p.split_pairs = fam == MLA_VERIFY_KERNEL_PAIR ? 1 : 0;
  // Each kernel may start while the one before it finishes (programmatic
  // dependent launch), except when profiling events sit between them: then
  // the kernels run back to back so that each event brackets one kernel.
  const bool overlap = !pl->ev_after_pack && !pl->ev_after_partial;
  cudaError_t le = cudaSuccess;
  if (packs && pl->pack_flags_dirty) {
    // Zero the flags and the ticket, keep the epoch: no tag is 0.
    const size_t head = mlav::PACK_SYNC_HEADER * sizeof(unsigned);
    le = cudaMemsetAsync(reinterpret_cast<uint8_t*>(pl->pack_sync) + head, 0, pl->pack_sync_bytes - head, s);
    if (le == cudaSuccess) le = cudaMemsetAsync(pl->pack_sync + mlav::PACK_SYNC_TICKET, 0, sizeof(unsigned), s);
    if (le == cudaSuccess) pl->pack_flags_dirty = false;
  }
  if (le == cudaSuccess && packs && pl->fault == MLA_VERIFY_FAULT_EPOCH_NEAR_WRAP) {
    // Testing: the tags of this call and the next cross 2^32, where 32-bit
    // tags would wrap (a pageable copy: the value is staged before
    // cudaMemcpyAsync returns).
    const unsigned long long near_wrap = 0xfffffffdull;
    le = cudaMemcpyAsync(pl->pack_sync, &near_wrap, sizeof(near_wrap), cudaMemcpyHostToDevice, s);
  }
  const bool skip_pack = pl->fault == MLA_VERIFY_FAULT_SKIP_PACK;
  pl->fault = MLA_VERIFY_FAULT_NONE;
  // One row tile per request: each key block is read by one attention CTA,
  // which gathers it itself instead of going through the pack (which writes
  // every block and reads it back).
  const bool direct = fam == MLA_VERIFY_KERNEL_TC && !skip_pack && gathers_directly(pl);
  bool attn_overlap = overlap;
  if (le == cudaSuccess && packs && skip_pack) {
    p.pack_flags = 1;   // injected: nothing sets the flags the attention kernel waits for
  } else if (le == cudaSuccess && direct) {
    p.direct_all = 1;
    attn_overlap = false;   // the first kernel of the call: no programmatic overlap with the last call
  } else if (le == cudaSuccess && packs) {
    const PackSchedule ps = pack_schedule(pl, p, overlap);
    p.pack_flags = ps.mode != MLA_VERIFY_PACK_WHOLE;
    le = ps.mode == MLA_VERIFY_PACK_IDLE_SMS
             ? mlav::launch_pack_kv_overlap(p, pl->packed, pl->pack_blocks, pl->num_sms, ps.wide, ps.stay, s)
             : mlav::launch_pack_kv(p, pl->packed, pl->pack_blocks, s);
  }
  const bool packed = le == cudaSuccess && packs && !skip_pack && !direct;
  if (le == cudaSuccess && pl->ev_after_pack) le = cudaEventRecord(pl->ev_after_pack, s);
  if (le == cudaSuccess)
    le = fam == MLA_VERIFY_KERNEL_MMA    ? mlav::launch_partial_mma(p, s)
         : fam == MLA_VERIFY_KERNEL_PAIR ? mlav::launch_partial_pair(p, pl->pack_maps, s, attn_overlap)
                                         : mlav::launch_partial_tc(p, s, attn_overlap);
  if (packed && le != cudaSuccess) pl->pack_flags_dirty = true;   // the epoch did not advance
  if (le == cudaSuccess && pl->ev_after_partial) le = cudaEventRecord(pl->ev_after_partial, s);
  if (le != cudaSuccess) return MLA_VERIFY_ERR_CUDA;
  if (ns > 1 && mlav::launch_combine(p, s, overlap) != cudaSuccess) return MLA_VERIFY_ERR_CUDA;
  if (note_done(pl, s) != cudaSuccess) return MLA_VERIFY_ERR_CUDA;
  return MLA_VERIFY_OK;
}

}  // namespace

extern "C" {

int mla_verify_attn(mla_verify_plan* pl, int batch, const void* q, const void* kv_cache,
                    const int32_t* kv_indices, const int32_t* kv_indptr, const int32_t* kv_lens,
                    const int32_t* draft_parent, float scale, void* out, float* lse,
                    void* stream) {
  if (!pl) return MLA_VERIFY_ERR_NULL;
  return launch_call(pl, batch, q, kv_cache, kv_indices, kv_indptr, kv_lens, draft_parent, scale, 0, 1,
                     out, lse, pl->out_dtype == MLA_VERIFY_OUT_BF16, static_cast<cudaStream_t>(stream));
}

int mla_verify_attn_partial(mla_verify_plan* pl, int batch, const void* q, const void* kv_cache,
                            const int32_t* kv_indices, const int32_t* kv_indptr,
                            const int32_t* kv_lens, const int32_t* draft_parent, float scale,
                            int shard, int num_shards, float* part_out, float* part_lse,
                            void* stream) {
  return launch_call(pl, batch, q, kv_cache, kv_indices, kv_indptr, kv_lens, draft_parent, scale, shard,
                     num_shards, part_out, part_lse, false, static_cast<cudaStream_t>(stream));
}

int mla_verify_combine_parts(mla_verify_plan* pl, int batch, int num_parts, const float* parts_out,
                             const float* parts_lse, void* out, float* lse, void* stream) {
  if (!pl || !parts_out || !parts_lse || !out || !lse) return MLA_VERIFY_ERR_NULL;
  if (!aligned16(parts_out) || !aligned16(parts_lse) || !aligned16(out) || !aligned16(lse))
    return MLA_VERIFY_ERR_ALIGN;
  if (batch < 1 || batch > pl->max_batch) return MLA_VERIFY_ERR_BATCH;
  if (num_parts < 1 || num_parts > mlav::MAX_NSPLIT) return MLA_VERIFY_ERR_ARG;
  const int dev_status = check_device(pl);
  if (dev_status != MLA_VERIFY_OK) return dev_status;
  Params p{};
  p.batch = batch;
  p.T = pl->T;
  p.H = pl->H;
  p.R = pl->R;
  p.nsplit = num_parts;
  p.shard = 0;
  p.num_shards = 1;
  // Part s of request b, row r: parts_out[((s * batch + b) * R + r) * 512].
  p.ws_o = const_cast<float*>(parts_out);
  p.ws_lse = const_cast<float*>(parts_lse);
  p.ws_stride_b = pl->R;
  p.ws_stride_s = 1LL * batch * pl->R;
  p.out = out;
  p.lse = lse;
  p.out_bf16 = pl->out_dtype == MLA_VERIFY_OUT_BF16;
  p.err = pl->err;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (mlav::launch_combine(p, s, false) != cudaSuccess || note_done(pl, s) != cudaSuccess)
    return MLA_VERIFY_ERR_CUDA;
  return MLA_VERIFY_OK;
}

int mla_verify_attn_host(mla_verify_plan* pl, int batch, const void* q_host, const void* kv_cache,
                         const int32_t* kv_indices_host, const int32_t* kv_indptr_host,
                         const int32_t* kv_lens_host, const int32_t* draft_parent_host,
                         float scale, void* out_host, float* lse_host, void* stream) {
  if (!pl || !q_host || !kv_cache || !kv_indices_host || !kv_indptr_host || !kv_lens_host ||
      !draft_parent_host || !out_host || !lse_host)
    return MLA_VERIFY_ERR_NULL;
  if (batch < 1 || batch > pl->max_batch) return MLA_VERIFY_ERR_BATCH;
  const long long nidx = kv_indptr_host[batch];
  if (nidx < 0 || nidx > pl->st_idx_cap || kv_indptr_host[0] < 0) return MLA_VERIFY_ERR_ARG;
  const int dev_status = check_device(pl);
  if (dev_status != MLA_VERIFY_OK) return dev_status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t rows = static_cast<size_t>(batch) * pl->R;
  const size_t out_elt = pl->out_dtype == MLA_VERIFY_OUT_BF16 ? 2 : 4;
  // Inputs: one copy kernel when every host array is mapped into the
  // device's address space (page-locked), else one DMA copy each.
  const void* in_host[5] = {q_host, kv_indices_host, kv_indptr_host, kv_lens_host, draft_parent_host};
  void* in_dev[5] = {pl->st_q, pl->st_idx, pl->st_indptr, pl->st_lens, pl->st_parent};
  const long long in_bytes[5] = {static_cast<long long>(rows * mlav::ROW_BYTES), nidx * 4, (batch + 1) * 4LL,
                                 batch * 4LL, static_cast<long long>(batch) * pl->T * 4};
  mlav::CopyRegions in{};
  bool mapped = true;
  for (int r = 0; r < 5 && mapped; ++r) {
    in.src[r] = device_view(in_host[r]);
    in.dst[r] = in_dev[r];
    in.bytes[r] = in_bytes[r];
    mapped = in.src[r] != nullptr;
  }
  in.n = 5;
  bool ok = true;
  if (mapped) {
    ok = mlav::launch_copy_regions(in, s) == cudaSuccess;
  } else {
    for (int r = 0; r < 5 && ok; ++r)
      ok = cudaMemcpyAsync(in_dev[r], in_host[r], static_cast<size_t>(in_bytes[r]), cudaMemcpyHostToDevice, s) ==
           cudaSuccess;
  }
  if (!ok) return MLA_VERIFY_ERR_CUDA;
  // Results: when the call ends in the split combine (plain stores) and both
  // output buffers are mapped, the combine writes them in host memory
  // directly; otherwise into the staging buffers, then copied back below.
  void* out_view = const_cast<void*>(device_view(out_host));
  void* lse_view = const_cast<void*>(device_view(lse_host));
  const bool direct_out = out_view && lse_view && aligned16(out_view) && aligned16(lse_view) &&
                          effective_nsplit(pl, batch) > 1;
  const int st = mla_verify_attn(pl, batch, pl->st_q, kv_cache, pl->st_idx, pl->st_indptr, pl->st_lens,
                                 pl->st_parent, scale, direct_out ? out_view : pl->st_out,
                                 direct_out ? static_cast<float*>(lse_view) : pl->st_lse, stream);
  if (st != MLA_VERIFY_OK) return st;
  if (direct_out) return cudaStreamSynchronize(s) == cudaSuccess ? MLA_VERIFY_OK : MLA_VERIFY_ERR_CUDA;
  void* out_dst[2] = {out_host, lse_host};
  const void* out_src[2] = {pl->st_out, pl->st_lse};
  const long long out_bytes[2] = {static_cast<long long>(rows * mlav::D_V * out_elt),
                                  static_cast<long long>(rows * sizeof(float))};
  mlav::CopyRegions out{};
  bool out_mapped = true;
  for (int r = 0; r < 2 && out_mapped; ++r) {
    out.src[r] = out_src[r];
    out.dst[r] = const_cast<void*>(device_view(out_dst[r]));
    out.bytes[r] = out_bytes[r];
    out_mapped = out.dst[r] != nullptr;
  }
  out.n = 2;
  if (out_mapped) {
    ok = mlav::launch_copy_regions(out, s) == cudaSuccess;
  } else {
    for (int r = 0; r < 2 && ok; ++r)
      ok = cudaMemcpyAsync(out_dst[r], out_src[r], static_cast<size_t>(out_bytes[r]), cudaMemcpyDeviceToHost, s) ==
           cudaSuccess;
  }
  ok = ok && cudaStreamSynchronize(s) == cudaSuccess;
  return ok ? MLA_VERIFY_OK : MLA_VERIFY_ERR_CUDA;
}

int mla_verify_build_indices(mla_verify_plan* pl, int batch, const int32_t* req_to_token,
                             int64_t stride, int pool_size, const int32_t* req_pool_indices,
                             const int32_t* prefix_lens, int32_t* kv_indices, int64_t capacity,
                             int32_t* kv_indptr, int32_t* kv_lens, void* stream) {
  if (!pl || !req_to_token || !req_pool_indices || !prefix_lens || !kv_indices || !kv_indptr ||
      !kv_lens)
    return MLA_VERIFY_ERR_NULL;
  if (!aligned16(req_to_token) || !aligned16(req_pool_indices) || !aligned16(prefix_lens) ||
      !aligned16(kv_indices) || !aligned16(kv_indptr) || !aligned16(kv_lens))
    return MLA_VERIFY_ERR_ALIGN;
  if (batch < 1 || batch > pl->max_batch) return MLA_VERIFY_ERR_BATCH;
  if (stride < pl->max_kv_len || pool_size < 1 || capacity < 0 || capacity > INT32_MAX)
    return MLA_VERIFY_ERR_ARG;
  const int dev_status = check_device(pl);
  if (dev_status != MLA_VERIFY_OK) return dev_status;
  mlav::IndexArgs a{};
  a.req_to_token = req_to_token;
  a.stride = stride;
  a.pool_size = pool_size;
  a.req_pool_indices = req_pool_indices;
  a.prefix_lens = prefix_lens;
  a.batch = batch;
  a.T = pl->T;
  a.page_size = pl->page_size;
  a.max_kv_len = pl->max_kv_len;
  a.capacity = capacity;
  a.kv_indices = kv_indices;
  a.kv_indptr = kv_indptr;
  a.kv_lens = kv_lens;
  a.err = pl->err;
  if (mlav::launch_build_indices(a, pl->max_kv_len, static_cast<cudaStream_t>(stream)) != cudaSuccess ||
      note_done(pl, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MLA_VERIFY_ERR_CUDA;
  return MLA_VERIFY_OK;
}

int mla_verify_compact_kv(mla_verify_plan* pl, int batch, const void* kv_src, int64_t src_slots,
                          const int32_t* kv_indices, const int32_t* kv_indptr,
                          const int32_t* kv_lens, const int32_t* free_pages,
                          int64_t num_free_pages, void* kv_dst, int64_t dst_slots,
                          int32_t* page_table, int32_t* page_indptr, void* stream) {
  if (!pl || !kv_src || !kv_indices || !kv_indptr || !kv_lens || !free_pages || !kv_dst ||
      !page_table || !page_indptr)
    return MLA_VERIFY_ERR_NULL;
  if (!aligned16(kv_src) || !aligned16(kv_indices) || !aligned16(kv_indptr) ||
      !aligned16(kv_lens) || !aligned16(free_pages) || !aligned16(kv_dst) ||
      !aligned16(page_table) || !aligned16(page_indptr))
    return MLA_VERIFY_ERR_ALIGN;
  if (batch < 1 || batch > pl->max_batch) return MLA_VERIFY_ERR_BATCH;
  if (src_slots < 0 || src_slots > INT32_MAX || num_free_pages < 0 ||
      num_free_pages > INT32_MAX || dst_slots <= 0 || dst_slots > INT32_MAX ||
      dst_slots % mlav::PAGE)
    return MLA_VERIFY_ERR_ARG;
  const int dev_status = check_device(pl);
  if (dev_status != MLA_VERIFY_OK) return dev_status;
  mlav::CompactArgs a{};
  a.kv_src = kv_src;
  a.src_slots = src_slots;
  a.kv_indices = kv_indices;
  a.kv_indptr = kv_indptr;
  a.kv_lens = kv_lens;
  a.free_pages = free_pages;
  a.num_free_pages = num_free_pages;
  a.kv_dst = kv_dst;
  a.dst_slots = dst_slots;
  a.page_table = page_table;
  a.page_indptr = page_indptr;
  a.batch = batch;
  a.max_kv_len = pl->max_kv_len;
  a.err = pl->err;
  if (mlav::launch_compact_kv(a, static_cast<cudaStream_t>(stream)) != cudaSuccess ||
      note_done(pl, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MLA_VERIFY_ERR_CUDA;
  return MLA_VERIFY_OK;
}

int mla_verify_get_error(mla_verify_plan* pl, int* device_status, int clear) {
  if (!pl || !device_status) return MLA_VERIFY_ERR_NULL;
  const int dev_status = check_device(pl);
  if (dev_status != MLA_VERIFY_OK) return dev_status;
  int v = 0;
  // The last eager call's kernels are done once its event is; the word is
  // then read (and cleared) on the plan's own stream only.
  if (pl->done_recorded && cudaEventSynchronize(pl->done_ev) != cudaSuccess) return MLA_VERIFY_ERR_CUDA;
  if (cudaMemcpyAsync(&v, pl->err, sizeof(int), cudaMemcpyDeviceToHost, pl->aux) != cudaSuccess)
    return MLA_VERIFY_ERR_CUDA;
  if (clear && cudaMemsetAsync(pl->err, 0, sizeof(int), pl->aux) != cudaSuccess) return MLA_VERIFY_ERR_CUDA;
  if (cudaStreamSynchronize(pl->aux) != cudaSuccess) return MLA_VERIFY_ERR_CUDA;
  *device_status = v;
  return MLA_VERIFY_OK;
}

}  // extern "C"
