/*
 * mla_verify.h - speculative-decoding verify attention for Multi-head Latent
 * Attention (MLA) over a paged KV cache, for NVIDIA GB300 (sm_103a).
 *
 * The operation.  "The Decisive A/B: When Benchmarking Honesty Reveals the
 * Real Bottleneck" (section "The Context") describes the verify step: the
 * drafter's speculative tokens attend to the target model's cached MLA
 * latent KV, stored with page_size=1 (one slot per token, rows scattered
 * through the cache), computed by a KV-split "partial" kernel plus a
 * "reduce" kernel, with a fixed split count, pre-allocated workspace and no
 * host synchronisation so the call can be captured in a CUDA graph.  "The
 * Moment of Truth: Benchmarking a Custom sm_120 Verify Kernel Against
 * Triton" (sections "The Raw Numbers" and "The CUDA Graph Dilemma") names
 * the tree ("kdtree") verify and the static-buffer requirement.
 *
 * For request b with n_b = kv_lens[b] cached rows (the last T rows are the
 * drafts' own rows, P_b = n_b - T is the prefix), draft t, head h:
 *
 *     s_j  = scale * dot(q[b,t,h,0:576], k_j[0:576])
 *     key j is visible iff j < P_b, or j - P_b is t or an ancestor of t
 *     lse  = log(sum over visible j of exp(s_j))              (natural log)
 *     out  = sum over visible j of exp(s_j - lse) * k_j[0:512]
 *
 * k_j is the cache row of logical key j: slot kv_indices[kv_indptr[b] + j]
 * when page_size == 1, or row j % 64 of page kv_indices[kv_indptr[b] + j/64]
 * when page_size == 64.  Values are the first 512 (latent) dims of each row;
 * the last 64 (rope) dims enter the scores only.
 *
 * Layouts (all row-major, contiguous):
 *     q            bf16  [B, T, H, 576]          (query row r = t*H + h)
 *     kv_cache     bf16  [num_slots, 576]        (1152-byte rows)
 *     kv_indices   int32 [kv_indptr[B]]          slot ids (ps 1) or page ids (ps 64)
 *     kv_indptr    int32 [B + 1]                 non-decreasing, kv_indptr[0] >= 0
 *     kv_lens      int32 [B]                     n_b = P_b + T, T <= n_b <= max_kv_len
 *     draft_parent int32 [B, T]                  -1 (hangs off the prefix) or an earlier draft
 *     out          fp32 or bf16 [B, T, H, 512]   (plan's out_dtype)
 *     lse          fp32  [B, T, H]
 * Every device pointer must be 16-byte aligned.
 *
 * Numerics: both products run on the tensor cores in fp16 with fp32
 * accumulation; the bf16 inputs are widened to fp16, which is exact for |x|
 * in [2^-14, 65504] (smaller magnitudes keep an absolute error below 2^-25).
 * A gathered key or query value of magnitude 65536 or more (or NaN) has no
 * fp16 counterpart: the kernel that widens it sets MLA_VERIFY_DEV_RANGE and
 * the rows that read it come out inf or NaN.  The softmax runs in fp32.
 *
 * Ownership: the caller owns every tensor.  The plan owns its workspace
 * (split partials), a device error word and, for mla_verify_attn_host, its
 * device staging buffers; all are allocated by mla_verify_plan_create and
 * freed by mla_verify_plan_destroy.
 *
 * Errors: functions return MLA_VERIFY_OK (0) or a negative status for
 * problems visible on the host (null or misaligned pointer, sizes beyond the
 * plan, unsupported shape, CUDA launch failure).  Problems only visible in
 * device data (slot or page id out of range, a kv_len outside [T,
 * max_kv_len], indptr inconsistent with kv_lens, a parent that is not an
 * earlier draft) never fault: the kernels set a sticky bit in the plan's
 * device error word, mask the offending key (bad slot), treat the parent as
 * -1 (bad parent) or write NaN for the whole request (bad length/indptr),
 * and carry on.  Read and clear the word with mla_verify_get_error.
 */
#ifndef MLA_VERIFY_H_
#define MLA_VERIFY_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define MLA_VERIFY_OK                 0
#define MLA_VERIFY_ERR_NULL          -1   /* a required pointer is NULL            */
#define MLA_VERIFY_ERR_ALIGN         -2   /* a pointer is not 16-byte aligned      */
#define MLA_VERIFY_ERR_SHAPE         -3   /* unsupported T/H/page_size/dtype/sizes */
#define MLA_VERIFY_ERR_BATCH         -4   /* batch < 1 or > plan's max_batch       */
#define MLA_VERIFY_ERR_SCALE         -5   /* scale not finite                      */
#define MLA_VERIFY_ERR_CUDA          -6   /* a CUDA runtime call or launch failed  */
#define MLA_VERIFY_ERR_DEVICE        -7   /* current device is not the plan's      */
#define MLA_VERIFY_ERR_OOM           -8   /* device or pinned allocation failed    */
#define MLA_VERIFY_ERR_ARG           -9   /* other invalid argument                */
#define MLA_VERIFY_ERR_SCRATCH      -10   /* call needs more than the static scratch */

/* Bits of the device error word (mla_verify_get_error). */
#define MLA_VERIFY_DEV_BAD_SLOT       1   /* slot or page id outside the cache     */
#define MLA_VERIFY_DEV_BAD_LEN        2   /* kv_len < T or > max_kv_len            */
#define MLA_VERIFY_DEV_BAD_PARENT     4   /* draft_parent[i] not in {-1} U [0, i)  */
#define MLA_VERIFY_DEV_BAD_INDPTR     8   /* indptr range does not match kv_len    */
#define MLA_VERIFY_DEV_TIMEOUT       16   /* a bounded device wait gave up         */
#define MLA_VERIFY_DEV_INTERNAL      32   /* an internal layout invariant failed   */
#define MLA_VERIFY_DEV_BAD_POOL      64   /* index builder: pool row / prefix / length out of range */
#define MLA_VERIFY_DEV_CAPACITY     128   /* index builder: kv_indices capacity exceeded */
#define MLA_VERIFY_DEV_RANGE        256   /* a q or key value is outside the fp16 range
                                             (|x| >= 65536, or NaN): rows that used it
                                             are not reliable */

/* Output element type. */
#define MLA_VERIFY_OUT_F32            0
#define MLA_VERIFY_OUT_BF16           1

/* Kernel family for the partial (split-KV) step.  AUTO picks TC or PAIR per
 * call from the plan's shape and the batch (TC's smaller fixed cost for short
 * contexts, PAIR's faster steps for long ones). */
#define MLA_VERIFY_KERNEL_AUTO        0
#define MLA_VERIFY_KERNEL_MMA         1   /* warp-level mma.sync, O in registers   */
#define MLA_VERIFY_KERNEL_TC          2   /* tcgen05 MMAs on one SM, 64 query rows
                                             per CTA, O^T in tensor memory; key
                                             rows gathered once per call by a pack
                                             kernel, streamed by bulk copies (or,
                                             with one 64-row tile per request,
                                             gathered by the attention CTAs)     */
#define MLA_VERIFY_KERNEL_PAIR        3   /* tcgen05 MMAs on a pair of SMs (one
                                             cluster, cta_group::2), 128 query rows
                                             per pair, 256 keys per step, O^T split
                                             by value dim across the two SMs' tensor
                                             memory; packed keys as TC.  With one
                                             64-row tile per request (T*H <= 64) or
                                             the pack schedule forced to NONE, calls
                                             run the TC family's direct gather.  */

typedef struct mla_verify_plan mla_verify_plan;

/*
 * Create a plan for calls with batch <= max_batch on CUDA device `device`.
 * num_drafts (T) in [1, 32]; num_heads (H) >= 1 with T*H <= 4096;
 * page_size 1 or 64; 1 <= num_slots < 2^31 (a multiple of 64 when page_size is 64);
 * 1 <= max_kv_len; out_dtype MLA_VERIFY_OUT_F32 or _BF16.
 * Allocates all device memory the plan will ever use (cudaMalloc) and sets
 * kernel attributes; makes `device` current on the calling thread.
 * On success *plan receives the handle.  Not to be called during capture.
 */
int mla_verify_plan_create(mla_verify_plan** plan, int max_batch, int num_drafts,
                           int num_heads, int page_size, int64_t num_slots,
                           int max_kv_len, int out_dtype, int device);

/* Release everything the plan owns (synchronises the plan's device). */
void mla_verify_plan_destroy(mla_verify_plan* plan);

/*
 * Fix the split count used by later calls (1..MLA_VERIFY_MAX_NSPLIT), or 0
 * to choose it from the batch, the plan's max_kv_len and the SM count.
 * A count above the number of key blocks in max_kv_len (64 keys for the
 * MMA family, 128 for the TC family) is clamped to it.
 * A call whose batch x split count exceeds the workspace the plan sized
 * (the automatic choice at every batch, or at least 64 MB) returns
 * MLA_VERIFY_ERR_SHAPE.
 */
#define MLA_VERIFY_MAX_NSPLIT 32
int mla_verify_plan_set_nsplit(mla_verify_plan* plan, int nsplit);

/* The split count a call with `batch` requests will use (>= 1), or < 0. */
int mla_verify_plan_get_nsplit(const mla_verify_plan* plan, int batch);

/*
 * The key-pack schedule of the TC family for a call with `batch` requests
 * and no profiling events.  *stay > 0: the pack overlaps the attention
 * kernel -- every SM but *stay packs the first *wide 128-key blocks of every
 * split, then *stay pack CTAs keep packing the rest on the SMs the attention
 * grid leaves idle while it runs.  *stay = 0: the whole pack runs before the
 * attention kernel starts (*wide = all positions).  Both 0: no pack -- the
 * MMA family, or T*H <= 64 (one row tile per request), where each attention
 * CTA gathers its own key blocks from the cache.  MLA_VERIFY_OK, or < 0
 * (NULL pointer, bad batch).
 */
int mla_verify_plan_get_pack_schedule(const mla_verify_plan* plan, int batch, int* wide, int* stay);

/*
 * Key-pack schedule of the TC family, for tuning and tests (the automatic
 * choice otherwise).  WHOLE: the whole pack runs first.  IDLE_SMS: the
 * two-phase pack above on the SMs the attention grid leaves idle (WHOLE when
 * it leaves none).  NONE: no pack -- every attention CTA gathers its own key
 * blocks from the cache (the automatic choice with one row tile per
 * request).  Calls with profiling events pack WHOLE unless NONE applies.  MLA_VERIFY_ERR_ARG for an
 * unknown schedule.  mla_verify_plan_get_pack_mode returns the schedule a
 * call with `batch` requests uses (MLA_VERIFY_PACK_NONE when it packs
 * nothing), or < 0.
 */
#define MLA_VERIFY_PACK_AUTO          0
#define MLA_VERIFY_PACK_WHOLE         1
#define MLA_VERIFY_PACK_IDLE_SMS      2
#define MLA_VERIFY_PACK_NONE          4
int mla_verify_plan_set_pack_schedule(mla_verify_plan* plan, int schedule);
int mla_verify_plan_get_pack_mode(const mla_verify_plan* plan, int batch);

/* Select the partial-kernel family (MLA_VERIFY_KERNEL_*; the default is AUTO). */
int mla_verify_plan_set_kernel(mla_verify_plan* plan, int kernel);

/* The kernel family selected (possibly AUTO), or < 0.  The kernel a call
 * actually launches is reported by mla_verify_plan_get_call_kernel. */
int mla_verify_plan_get_kernel(const mla_verify_plan* plan);
/* The partial kernel a call with `batch` requests launches: MLA_VERIFY_KERNEL_
 * MMA, TC or PAIR, or < 0 (null plan, batch outside [1, max_batch]). */
int mla_verify_plan_get_call_kernel(const mla_verify_plan* plan, int batch);

/*
 * Profiling hook.  Later mla_verify_attn calls record `after_pack` (if not
 * NULL) on the call's stream right after the key-gather/pack kernel (right
 * at the start for the MMA family, which has none) and `after_partial` (if
 * not NULL) right after the split-KV partial kernel.  With events recorded
 * just before and just after the call, the differences time the pack, the
 * partial kernel and the combine separately.  Both must be cudaEvent_t
 * created with timing enabled; the records are ordinary stream operations and
 * are captured into graphs like the kernels.  Pass NULLs to stop.  Without
 * events each kernel of a call may start while the previous one runs
 * (programmatic dependent launch; the TC partial kernel streams each packed
 * block as soon as the pack kernel has published it); with events they run
 * back to back, so the split times each kernel alone and the call as a whole
 * is slower.
 */
int mla_verify_plan_set_profile_events(mla_verify_plan* plan, void* after_pack,
                                       void* after_partial);

/*
 * Testing hook: a fault injected on the host into the plan's next call (then
 * cleared).  MLA_VERIFY_FAULT_SKIP_PACK (TC family): the call launches the
 * attention kernel waiting for per-block ready flags but not the pack kernel
 * that sets them, so every block wait runs out after its cycle limit (about
 * a second): the rows come out NaN, the device status word gets
 * MLA_VERIFY_DEV_TIMEOUT and the context stays usable.
 * MLA_VERIFY_FAULT_EPOCH_NEAR_WRAP (a call that packs its keys): before the
 * call, the pack hand-off epoch is set to 2^32 - 3, so the calls from there
 * on use the tags 2^32 - 2, 2^32 - 1, 2^32, .. (the epoch and the tags are
 * 64-bit: they do not wrap); every result must stay exact.  The value is
 * written by a pageable host copy: not for a call under stream capture.
 * MLA_VERIFY_OK, or MLA_VERIFY_ERR_ARG for an unknown fault.
 */
#define MLA_VERIFY_FAULT_NONE         0
#define MLA_VERIFY_FAULT_SKIP_PACK    1
#define MLA_VERIFY_FAULT_EPOCH_NEAR_WRAP 2
int mla_verify_plan_inject_fault(mla_verify_plan* plan, int fault);

/* Bytes of device workspace the plan holds (partials, packed key blocks,
 * pack hand-off flags, error word). */
size_t mla_verify_plan_workspace_bytes(const mla_verify_plan* plan);

/*
 * The verify attention, all pointers on the plan's device (layouts above).
 * Enqueues its kernels on `stream` (a cudaStream_t; NULL = legacy default
 * stream) and returns: no allocation, no synchronisation, no device-memory
 * read on the host, and the launch grid depends only on `batch` and the plan,
 * so the call may be captured into a CUDA graph and replayed with new data
 * in the same buffers.  Calls sharing one plan must not overlap on the GPU
 * (they share the workspace); use one plan per concurrent stream.
 */
int mla_verify_attn(mla_verify_plan* plan, int batch, const void* q,
                    const void* kv_cache, const int32_t* kv_indices,
                    const int32_t* kv_indptr, const int32_t* kv_lens,
                    const int32_t* draft_parent, float scale, void* out,
                    float* lse, void* stream);

/*
 * The same operation with q, kv_indices, kv_indptr, kv_lens, draft_parent,
 * out and lse in HOST memory (pinned memory gives the fastest copies) and
 * kv_cache on the device (the cache is resident model state).  Copies the
 * inputs into the plan's device staging buffers on `stream`, runs
 * mla_verify_attn, copies out/lse back and synchronises `stream` before
 * returning.  When all five inputs are page-locked and mapped into the
 * device's address space (cudaHostAlloc / pinned tensors on a unified-
 * address system) one copy kernel moves them; otherwise one DMA copy per
 * array.  The results likewise; when both output buffers are mapped and the
 * call ends in the split combine, the combine kernel writes them in place.
 * kv_indptr[batch] entries of kv_indices are copied; that count must not
 * exceed max_batch * max_kv_len.  Not capturable.
 */
int mla_verify_attn_host(mla_verify_plan* plan, int batch, const void* q_host,
                         const void* kv_cache, const int32_t* kv_indices_host,
                         const int32_t* kv_indptr_host, const int32_t* kv_lens_host,
                         const int32_t* draft_parent_host, float scale,
                         void* out_host, float* lse_host, void* stream);

/*
 * Context-parallel split of one call over several GPUs (or several calls):
 * the KV split with a reduce step of "The Decisive A/B: When Benchmarking
 * Honesty Reveals the Real Bottleneck" (section "The Context"), taken one
 * level up -- each rank computes the partial of its shard of every request's
 * keys, the ranks exchange the partials (an all-gather), and each rank
 * merges them with mla_verify_combine_parts.
 *
 * Shards: request b's ceil(n_b / 128) blocks of 128 consecutive logical keys
 * are dealt out evenly -- shard s of S takes blocks floor(s * nb / S) ..
 * floor((s+1) * nb / S) - 1, clipped to n_b -- so the shards are disjoint
 * and cover every key.  A shard may be empty for short requests.
 *
 * mla_verify_attn_partial: the verify attention restricted to shard `shard`
 * of `num_shards` (0 <= shard < num_shards <= MLA_VERIFY_MAX_NSPLIT), with
 * the inputs of mla_verify_attn.  A key counts iff it is in the shard and
 * visible as usual.  Writes part_out fp32 [B, T, H, 512], normalised over the
 * counted keys, and part_lse fp32 [B, T, H], their log-sum-exp (natural log);
 * a row with no counted key gets part_lse = -inf and part_out = 0 (weight 0
 * in the merge).  Same rules as mla_verify_attn otherwise (capturable, no
 * allocation or synchronisation; device-side errors set the sticky bits).
 * MLA_VERIFY_ERR_ARG for a bad shard / num_shards.
 *
 * mla_verify_combine_parts: merges num_parts (1..MLA_VERIFY_MAX_NSPLIT)
 * partials of the same batch, laid out shard-major as an all-gather leaves
 * them: parts_out fp32 [num_parts, B, T, H, 512], parts_lse fp32
 * [num_parts, B, T, H].  lse = log sum_s exp(lse_s), out = sum_s
 * exp(lse_s - lse) * out_s, written in the plan's out_dtype; partials with
 * lse_s = -inf have weight 0, a NaN lse_s makes the row NaN.  With the parts
 * of shards 0 .. S-1 of one set of inputs this equals mla_verify_attn on
 * those inputs (up to rounding).  Capturable; allocates nothing.
 */
int mla_verify_attn_partial(mla_verify_plan* plan, int batch, const void* q,
                            const void* kv_cache, const int32_t* kv_indices,
                            const int32_t* kv_indptr, const int32_t* kv_lens,
                            const int32_t* draft_parent, float scale, int shard,
                            int num_shards, float* part_out, float* part_lse, void* stream);
int mla_verify_combine_parts(mla_verify_plan* plan, int batch, int num_parts,
                             const float* parts_out, const float* parts_lse, void* out,
                             float* lse, void* stream);

/*
 * Read the sticky device error word (MLA_VERIFY_DEV_* bits) into
 * *device_status; clear it when `clear` is nonzero.  Waits for the plan's
 * last eagerly launched call (an event the plan records at the end of every
 * mla_verify_attn, mla_verify_build_indices and mla_verify_compact_kv call
 * made outside stream capture), then reads and clears the word on a private
 * stream of the plan: other streams and devices are not synchronised.  Work
 * replayed from a CUDA graph is not tracked: synchronise the replay stream
 * first.  Call outside graph capture.
 */
int mla_verify_get_error(mla_verify_plan* plan, int* device_status, int clear);

/*
 * Per-step index builder: fills kv_lens, kv_indptr and kv_indices for a
 * verify step on the GPU, in `stream`, from the serving stack's
 * request-to-token table -- the "marshaling" work the pages see dominate at
 * short context when it runs on the host per layer, with a kernel on the GPU
 * named as one remedy ("The Moment of Truth: Benchmarking a Custom sm_120
 * Verify Kernel Against Triton", sections "Interpreting the Crossover: The
 * Marshaling Tax" and "Assumptions and Their Validity").  The outputs feed
 * mla_verify_attn directly; both calls can be captured into one graph.
 *
 *   req_to_token      int32 [pool_size][stride]: cache slot of each token
 *                     position of the request held in that pool row; stride
 *                     >= the plan's max_kv_len.  For page_size 64 whole pages
 *                     are allocated: a page's 64 positions hold 64 consecutive
 *                     slots starting at a multiple of 64, and only the first
 *                     slot of each page is read.
 *   req_pool_indices  int32 [batch]: pool row of request b.
 *   prefix_lens       int32 [batch]: prefix length P_b; the step reads
 *                     positions 0 .. P_b + T - 1 (the last T are the drafts').
 *   kv_indices        int32 [capacity] out: slots (page_size 1) or page ids.
 *   kv_indptr         int32 [batch + 1] out, kv_lens int32 [batch] out.
 *
 * kv_lens[b] = P_b + T; kv_indptr is the exclusive prefix sum of each
 * request's entry count (P_b + T slots, or ceil((P_b + T) / 64) pages).
 * Device-side problems set sticky bits (mla_verify_get_error) and never fault:
 * a pool row outside [0, pool_size), a negative prefix or P_b + T > max_kv_len
 * gives kv_lens[b] = 0 and no entries (MLA_VERIFY_DEV_BAD_POOL; the attention
 * then rejects the request); when the entries exceed `capacity` the longest
 * leading run of requests that fits keeps them and every later request gets
 * kv_lens 0 (MLA_VERIFY_DEV_CAPACITY); a page whose first slot is negative or
 * not a multiple of 64 gets page id -1 (MLA_VERIFY_DEV_BAD_SLOT).  Host-side
 * errors as for mla_verify_attn (null or misaligned pointers, batch outside
 * [1, max_batch], stride < max_kv_len, pool_size < 1 or capacity outside
 * [0, 2^31) give MLA_VERIFY_ERR_ARG).  Allocates nothing and does not
 * synchronise.
 */
int mla_verify_build_indices(mla_verify_plan* plan, int batch, const int32_t* req_to_token,
                             int64_t stride, int pool_size, const int32_t* req_pool_indices,
                             const int32_t* prefix_lens, int32_t* kv_indices, int64_t capacity,
                             int32_t* kv_indptr, int32_t* kv_lens, void* stream);

/*
 * KV compaction: copies each request's page_size 1 rows, in logical order,
 * into fresh 64-row pages of `kv_dst` taken in order from `free_pages`, and
 * writes the page_size 64 table of the same requests -- the defragmentation
 * the pages name as a step after the custom verify kernel ("The Moment of
 * Truth: Benchmarking a Custom sm_120 Verify Kernel Against Triton", section
 * "The Broader Context: From Kernel to System"), so that later verify steps
 * of those requests can run with page_size 64 over contiguous pages.
 *
 *   kv_src        bf16 [src_slots][576], the page_size 1 cache.
 *   kv_indices, kv_indptr [batch + 1], kv_lens [batch]: the requests' page_size
 *                 1 slot table (as for mla_verify_attn).
 *   free_pages    int32 [num_free_pages]: destination page ids, used in order.
 *   kv_dst        bf16 [dst_slots][576], dst_slots a multiple of 64.  It may be
 *                 kv_src itself when no destination page holds a row that a
 *                 request of this call reads.
 *   page_table    int32 [num_free_pages] out: the consumed prefix of free_pages.
 *   page_indptr   int32 [batch + 1] out: request b's pages are
 *                 page_table[page_indptr[b] .. page_indptr[b+1]).
 *
 * Row j of request b goes to slot page_table[page_indptr[b] + j / 64] * 64 +
 * j % 64; the rest of a request's last page is left unchanged; kv_lens stays
 * valid for the new table.  Device-side problems set sticky bits and never
 * fault: a length outside [0, max_kv_len] or an indptr range that does not
 * hold kv_lens[b] slots inside [0, kv_indptr[batch]) gives the request no
 * pages (MLA_VERIFY_DEV_BAD_LEN / BAD_INDPTR); when the free pages run out
 * the longest leading run of requests that fits keeps its pages, every later
 * request gets none (MLA_VERIFY_DEV_CAPACITY); a source slot outside kv_src
 * is copied as a zero row and a page outside kv_dst is not written
 * (MLA_VERIFY_DEV_BAD_SLOT).  Host-side errors as for mla_verify_attn (null or
 * misaligned pointers, batch outside [1, max_batch]; src_slots or
 * num_free_pages outside [0, 2^31), dst_slots not a positive multiple of 64
 * below 2^31 give MLA_VERIFY_ERR_ARG).  Allocates nothing, does not
 * synchronise.
 */
int mla_verify_compact_kv(mla_verify_plan* plan, int batch, const void* kv_src, int64_t src_slots,
                          const int32_t* kv_indices, const int32_t* kv_indptr,
                          const int32_t* kv_lens, const int32_t* free_pages,
                          int64_t num_free_pages, void* kv_dst, int64_t dst_slots,
                          int32_t* page_table, int32_t* page_indptr, void* stream);

/*
 * Allocation-free verify attention, for callers that cannot allocate device
 * memory: code running inside a memory pool that owns the whole device, a
 * serving loop that must not allocate after start-up, or a layer that is only
 * handed pointers by an outer framework.  The pages have no counterpart; it
 * is an integration convenience.
 *
 * Runs the MMA family (mma.sync partial kernel + LSE combine, out in fp32)
 * with `nsplit` key splits (1..MLA_VERIFY_MAX_NSPLIT, no automatic choice).
 * The split partials live in a file-scope device array of
 * MLA_VERIFY_STATIC_SCRATCH_BYTES held by every GPU that loads the library
 * until the process exits; a call needing more (batch * nsplit * T * H * 2052
 * bytes + 256 when nsplit > 1) returns MLA_VERIFY_ERR_SCRATCH.  Arguments,
 * layouts and device-side error behaviour are those of mla_verify_attn, with
 * the shape given per call; `device_status` is an optional device int the
 * kernels OR their MLA_VERIFY_DEV_* bits into (the caller clears it); when it
 * is NULL the bits go to a word inside the array, cleared at every call and
 * not readable.  Calls nothing that allocates (no cudaMalloc or cudaFree).
 *
 * The first call on each device looks up the array's device address and sets
 * a kernel attribute for that device: make it before any stream capture.
 * When a CUDA call of this entry fails (for example after cudaDeviceReset,
 * which discards the device context the cached address belongs to), the call
 * returns MLA_VERIFY_ERR_CUDA and the next call on that device repeats the
 * set-up.
 * Every call on a device shares the one array, so calls that overlap on the
 * GPU (different streams, or different host threads without ordering) race
 * on it and corrupt each other's results; serialise them.
 */
#define MLA_VERIFY_STATIC_SCRATCH_BYTES (32u << 20)
int mla_verify_attn_static(int batch, int num_drafts, int num_heads, int page_size,
                           int64_t num_slots, int max_kv_len, int nsplit, const void* q,
                           const void* kv_cache, const int32_t* kv_indices,
                           const int32_t* kv_indptr, const int32_t* kv_lens,
                           const int32_t* draft_parent, float scale, float* out, float* lse,
                           int* device_status, void* stream);

/* Static text for a status code. */
const char* mla_verify_strerror(int status);

/* Library ABI version (major * 100 + minor). */
int mla_verify_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_VERIFY_H_ */
