/*
 * moe.h -- C ABI of the routed-expert FFN layer over a fixed GPU expert-slot
 * pool, for NVIDIA GB300 (sm_103a).
 *
 * One routed mixture-of-experts FFN layer: router logits -> top-k and a
 * softmax over the selected experts -> tokens grouped by expert -> each
 * selected expert looked up in a (layer, expert) -> slot map, misses copied
 * from pinned host memory into evicted slots -> per expert gate and up
 * projections, SwiGLU, down projection on MXFP4 weights used in their native
 * format -> outputs summed with the routing weights.
 *
 * Sources of the operations (page title, section):
 *   [R1] tinyserve README, "Performance": GPT-OSS-20B, 24 layers x 32
 *        experts, top_k=4.
 *   [R2] tinyserve README, "How it works" item 1: expert weights are raw
 *        quantised bytes in pinned CPU memory, not dequantised at load.
 *   [R3] tinyserve README, "How it works" item 2: fused dequant+matmul in the
 *        native quantised format; an expert is gate, up and down.
 *   [R4] tinyserve README, "How it works" item 3: expert cache keyed by
 *        (layer, expert_id) with a GPU slot map; "Configuration":
 *        cache_policy lru.
 *   [R5] tinyserve README, "How it works" item 6: batched prefill groups
 *        tokens by expert and loads each unique expert once.
 *   [P1] llama.cpp discussion "fixed GPU expert working set with Native CPU
 *        miss execution", main post: a fixed subset of packed experts is
 *        materialised in a GPU pool; selected IDs are split into resident
 *        hits and misses; outputs are merged with the routing weights.
 *   [X1] "Expert Offloading" topic page, replay-semantics study: cache
 *        events are fused per (layer, step), not replayed per access.
 *   [MX] OCP Microscaling Formats (MX) v1.0: E2M1 elements with block-32
 *        E8M0 scales (MXFP4), E4M3 elements (MXFP8).
 *
 * Conventions for every call:
 *   - Return value: MOE_OK or a negative MOE_ERR_* status; nothing aborts.
 *     Arguments are validated before anything is launched; on
 *     MOE_ERR_INVALID nothing was enqueued.  On MOE_ERR_CUDA,
 *     moe_last_cuda_error() gives the CUDA runtime error code.
 *   - All buffers are owned by the caller.  "device" pointers must be
 *     device-accessible memory of the current CUDA device; "host" pointers
 *     are ordinary host memory; "pinned" pointers are page-locked host
 *     memory (cudaHostAlloc / cudaHostRegister).  The library keeps host
 *     metadata only and allocates no device memory.
 *   - moe_stream_t is a cudaStream_t passed as an opaque pointer (NULL is
 *     the legacy default stream).  Work is enqueued asynchronously.  The
 *     calls that wait on the host are: moe_pool_stage and
 *     moe_prefill_staged (for the work enqueued so far on their compute
 *     stream, polling at most timeout_ms), moe_ffn_status (for the work
 *     enqueued so far on its stream, polling at most 10 s),
 *     moe_pool_device_attach and moe_pool_device_detach (for their state
 *     copies, polling at most timeout_ms) and moe_pool_create with preload
 *     (synchronous copies of the preloaded experts); no other call waits.
 *   - Tensors are dense row-major.  T tokens, E experts, k top_k,
 *     H hidden size, I expert intermediate size, A = T*k assignments,
 *     assignment a = t*k + j is the j-th ranked expert of token t.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_OK 0
#define MOE_ERR_INVALID (-1)     /* bad argument; nothing enqueued          */
#define MOE_ERR_CUDA (-2)        /* a CUDA runtime call failed              */
#define MOE_ERR_CAPACITY (-3)    /* unique routed experts exceed the slots  */
#define MOE_ERR_TIMEOUT (-4)     /* a bounded host wait ran out             */
#define MOE_ERR_STATE (-5)       /* object in the wrong state for the call  */
#define MOE_ERR_UNSUPPORTED (-6) /* shape or device the kernels do not handle */

#define MOE_MAX_EXPERTS 256
#define MOE_MAX_TOPK 32

/* moe_expert_ffn path selection */
#define MOE_PATH_AUTO 0          /* decode when A <= MOE_DECODE_MAX_ASSIGN   */
#define MOE_PATH_DECODE 1        /* bf16 activations, CUDA-core GEMV         */
#define MOE_PATH_PREFILL 2       /* MXFP8 activations, tcgen05 grouped GEMM  */
#define MOE_DECODE_MAX_ASSIGN 64
/* OR-ed into moe_expert_ffn's path: out is added to (out += the layer's
 * output, as a residual stream takes it) instead of overwritten. */
#define MOE_FFN_ACCUMULATE 0x100
/* OR-ed into moe_expert_ffn's path (decode only): assignments whose
 * expert's slot_of entry is -1 (any negative value) are not served -- they
 * add nothing and get no work -- instead of yielding NaN.  With two calls
 * over complementary slot maps (the second with MOE_FFN_ACCUMULATE) a layer
 * is computed in two parts, e.g. resident experts while missed ones are
 * still being copied (moe_pool_stage_device). */
#define MOE_FFN_SKIP_ABSENT 0x200

typedef void* moe_stream_t;

/* Threads: the stateless calls (routing, expert FFN, combine, quantiser,
 * packing) may be made from several host threads at once, each with its
 * own workspace (moe_route_plan_noalloc excepted: its calls share one
 * device array).  A pool keeps host state (slot maps, policy stamps,
 * counters): calls on one pool must not overlap in time; different pools
 * are independent. */

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

/* Text of a status code (static string, never NULL). */
MOE_API const char* moe_status_str(int status);

/* CUDA runtime error code of the last MOE_ERR_CUDA on this thread (0 if
 * none). */
MOE_API int moe_last_cuda_error(void);

/* Number of CUDA devices the library sees (0 without a GPU); never fails. */
MOE_API int moe_device_count(void);

/* ------------------------------------------------------------------------ */
/* Weights [R2][R3][MX]                                                      */
/* ------------------------------------------------------------------------ */

/* Bytes one expert occupies in the GPU-native packed layout (the unit of a
 * pool slot and of one miss copy).  hidden and inter must be positive
 * multiples of 64.  Errors: MOE_ERR_INVALID. */
MOE_API int moe_expert_bytes(int hidden, int inter, size_t* out_bytes);

/* Convert one expert from the canonical MXFP4 layout into the GPU-native
 * layout, on the host, once, outside any timed region.
 *   gate_codes, up_codes   host [inter][hidden/2]  E2M1 pairs, element 2i in
 *                          the low nibble of byte i
 *   gate_scales, up_scales host [inter][hidden/32] E8M0 bytes, one per block
 *                          of 32 along hidden
 *   down_codes             host [hidden][inter/2]
 *   down_scales            host [hidden][inter/32]
 *   dst                    host, moe_expert_bytes() bytes, written fully
 * The native layout keeps each row's codes followed by its scales (rows
 * padded to 32 bytes) and interleaves gate and up rows in chunks of 32 (gate rows
 * 32c..32c+31, then up rows 32c..32c+31) so one tile of the fused gate/up
 * product holds matching gate and up rows.  After the row-major down
 * matrix it also keeps a column-blocked copy of down for the decode path:
 * for each block of 16 columns, every row's 8 code bytes of those columns,
 * then every row's scale byte of the 32-block they lie in (so one decode
 * work item, 16 elements of h, reads its down weights contiguously).
 * Errors: MOE_ERR_INVALID. */
MOE_API int moe_pack_expert(const uint8_t* gate_codes, const uint8_t* gate_scales,
                    const uint8_t* up_codes, const uint8_t* up_scales,
                    const uint8_t* down_codes, const uint8_t* down_scales,
                    int hidden, int inter, void* dst);

/* ------------------------------------------------------------------------ */
/* Routing and grouping [R1][R5][P1]                                         */
/* ------------------------------------------------------------------------ */

/* Scratch bytes moe_route_plan needs for T tokens, E experts, top-k. */
MOE_API int moe_route_workspace_bytes(int T, int E, int k, size_t* out_bytes);

/* Top-k + softmax + per-expert histogram + stable permutation, one call.
 *   logits      device fp32 [T][E]
 *   ids         device int32 [T][k]  out: selected experts, larger logit
 *               first, equal logits by lower id (NaN ranks last)
 *   w           device fp32 [T][k]   out: softmax over the k selected logits,
 *               evaluated in float-float (about 48 bits) and rounded once
 *               to fp32: within 2 ulp of the fp64 value
 *   counts      device int32 [E]     out: assignments per expert
 *   offsets     device int32 [E+1]   out: exclusive prefix sum of counts
 *   perm        device int32 [A]     out: assignment indices grouped by
 *               expert (ascending), ascending a inside a group
 *   inv         device int32 [A]     out: inv[perm[p]] = p
 *   counts_host pinned int32 [E] or NULL: when given, counts are copied
 *               there asynchronously on the same stream
 *   workspace   device, >= moe_route_workspace_bytes(), 16-byte aligned
 * Limits: 1 <= E <= MOE_MAX_EXPERTS, 1 <= k <= min(E, MOE_MAX_TOPK),
 * T >= 0 (T = 0 writes zero counts).  Errors: MOE_ERR_INVALID, MOE_ERR_CUDA. */
MOE_API int moe_route_plan(const float* logits, int T, int E, int k,
                   int32_t* ids, float* w, int32_t* counts, int32_t* offsets,
                   int32_t* perm, int32_t* inv, int32_t* counts_host,
                   void* workspace, size_t ws_bytes, moe_stream_t stream);

/* moe_route_plan without a workspace argument.  The pages have no
 * counterpart: this entry exists for callers that cannot allocate device
 * memory where they route -- engines whose device memory is carved up in
 * advance by their own allocator under a fixed budget (there is nothing left
 * to hand out, and allocating behind that allocator breaks its accounting),
 * and latency-bound decode loops that must never call into the driver's
 * allocator, whose calls can block or synchronise the device.  The per-tile
 * histograms use a 64 KB array that the library keeps in device memory
 * (every GPU that loads the library holds it until exit); nothing is
 * allocated per call, and no cudaMalloc/cudaFree is ever made.
 *   Arguments, outputs and results are those of moe_route_plan.
 *   Limit: T <= 16384 tokens (64 tiles of 256); larger T returns
 *   MOE_ERR_INVALID before anything is enqueued.
 *   The first call on a device resolves the array's device address for that
 *   device (a runtime symbol lookup, made with that device current) and keeps
 *   it for the life of the process; do not call this entry again after the
 *   device has been reset (cudaDeviceReset) in the same process.  Each call clears the part of the array it uses with an
 *   asynchronous memset on `stream` (no allocation) before counting into
 *   it; all calls share the array, so calls that can overlap on the GPU
 *   race.
 * Errors: MOE_ERR_INVALID, MOE_ERR_CUDA. */
MOE_API int moe_route_plan_noalloc(const float* logits, int T, int E, int k,
                                   int32_t* ids, float* w, int32_t* counts, int32_t* offsets,
                                   int32_t* perm, int32_t* inv, int32_t* counts_host,
                                   moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Expert-slot pool [R2][R4][P1][X1]                                         */
/* ------------------------------------------------------------------------ */

typedef struct moe_pool moe_pool_t;

/* Eviction policies of the slot pool (tinyserve README, "Configuration":
 * cache_policy lru, lfru, slru, lfu, fifo; "How it works" item 3:
 * frequency-recency eviction).  The pages name them without defining them;
 * the readings implemented (per fused event; a miss evicts a resident
 * expert that is not routed in the same event):
 *   LRU   victim: least recently routed.
 *   FIFO  victim: loaded earliest (routing does not refresh).
 *   LFU   victim: fewest events routed since loaded, ties by lower id.
 *   LFRU  victim: fewest events routed since loaded, ties by least recent.
 *   SLRU  segmented LRU: a routed probationary expert becomes protected
 *         (at most S/2, at least 1; the least recent protected one drops back
 *         to probation); victim: least recent probationary, else least
 *         recent protected. */
#define MOE_POLICY_LRU  0
#define MOE_POLICY_FIFO 1
#define MOE_POLICY_LFU  2
#define MOE_POLICY_LFRU 3
#define MOE_POLICY_SLRU 4

/* Which parts of a packed expert the pool copies in (moe_pool_desc). */
#define MOE_STAGE_WHOLE  0
#define MOE_STAGE_DECODE 1

typedef struct {
    int layers;            /* L >= 1                                         */
    int experts;           /* E, 1..MOE_MAX_EXPERTS                          */
    int slots_per_layer;   /* S, 1..E                                        */
    int hidden, inter;     /* H, I (multiples of 64)                         */
    void* host_experts;    /* pinned [L][E][expert_bytes] packed experts;
                              NULL only in dry-run mode                      */
    void* dev_slots;       /* device [L][S][expert_bytes]; NULL only in
                              dry-run mode                                   */
    int preload;           /* 1: at create, slot s of every layer is filled
                              with expert s (s < S), copied synchronously    */
    int dry_run;           /* 1: policy only -- no CUDA call is ever made;
                              stage updates the map and counters and reports
                              the copies it would issue                      */
    int policy;            /* MOE_POLICY_*: which resident expert a miss
                              evicts (0 = LRU)                               */
    int stage_parts;       /* MOE_STAGE_WHOLE (0): a miss copies the whole
                              packed expert.  MOE_STAGE_DECODE: only what
                              the fused decode kernel reads (gate/up rows and
                              the column-blocked down copy, about 3/4 of the
                              bytes); moe_expert_ffn then refuses the prefill
                              path and decode shapes the fused kernel cannot
                              take (MOE_ERR_UNSUPPORTED)                     */
} moe_pool_desc;

typedef struct {
    uint64_t hits;         /* unique routed experts found resident           */
    uint64_t misses;       /* unique routed experts copied in                */
    uint64_t evictions;    /* resident experts displaced by a miss           */
    uint64_t h2d_bytes;    /* bytes copied host -> device by stage           */
    uint64_t errors;       /* stage calls that failed and were rolled back   */
    uint64_t events;       /* staging events served (one per moe_pool_stage  */
                           /* call, one per window of moe_prefill_staged)    */
    uint64_t prefetches;   /* experts copied in by moe_pool_prefetch         */
    uint64_t prefetch_hits;/* of those, routed before being evicted          */
} moe_counters;

/* Create a pool.  Stores a copy of *desc; the buffers stay caller-owned and
 * must outlive the pool.  With preload, the initial copies are issued on
 * the legacy stream and waited for before returning.
 * Errors: MOE_ERR_INVALID, MOE_ERR_CUDA. */
MOE_API int moe_pool_create(const moe_pool_desc* desc, moe_pool_t** out_pool);

/* One fused cache event for (layer, this step) [X1]:
 *   1. waits (polling, at most timeout_ms; <= 0 means 10 s) until all work
 *      enqueued so far on `compute` is done, so counts_host is valid;
 *   2. U = {e : counts_host[e] > 0}.  Every resident e in U is a hit and is
 *      touched; every absent e in U, ascending, takes the lowest free slot,
 *      else evicts the resident expert not in U that the pool's policy
 *      names (the least recently used one under MOE_POLICY_LRU);
 *   3. issues one cudaMemcpyAsync (pinned host -> slot) per miss on `copy`,
 *      records an event there and makes `compute` wait on it;
 *   4. copies the layer's slot map (int32 [E], -1 = absent) to slot_of_dev
 *      on `compute` (skipped when slot_of_dev is NULL).
 *   counts_host  pinned int32 [E] (typically from moe_route_plan)
 *   slot_of_dev  device int32 [E] or NULL
 * If |U| > S nothing changes and MOE_ERR_CAPACITY is returned.  If a copy
 * fails to enqueue, the event is rolled back (map, stamps and counters as
 * before the call, errors += 1) and MOE_ERR_CUDA is returned.  The wait
 * returns MOE_ERR_TIMEOUT without changing any state.
 * Errors: MOE_ERR_INVALID, MOE_ERR_CAPACITY, MOE_ERR_TIMEOUT, MOE_ERR_CUDA. */
MOE_API int moe_pool_stage(moe_pool_t* pool, int layer, const int32_t* counts_host,
                   int32_t* slot_of_dev, moe_stream_t compute, moe_stream_t copy,
                   int timeout_ms);

/* Prefill of one layer through a pool whose slots may be fewer than the
 * layer's routed experts: per-layer unique-expert staging in windows, each
 * unique expert loaded at most once per call [R3][P2].
 *   1. waits (as moe_pool_stage, at most timeout_ms) until all work enqueued
 *      so far on `compute` is done, so counts_host is final;
 *   2. on `compute`: zeroes out and quantises every token's x once into its
 *      k grouped rows (as moe_expert_ffn, MOE_PATH_PREFILL);
 *   3. cuts U = {e : counts_host[e] > 0}, ascending, into windows of at most
 *      `window` experts.  Window i is one staging event (as moe_pool_stage,
 *      step 2, over the window's experts) whose victims are never the
 *      previous window's experts; its miss copies go on `copy` after the
 *      GEMMs of window i - 2 (which may have read the evicted slots) and
 *      overlap the GEMMs of window i - 1; `compute` then waits for them and
 *      runs the window's grouped gate/up and down GEMMs, the down GEMM
 *      adding w * y into out.  No host wait after step 1.
 *   x_bf16, ids, w, offsets, perm, inv, workspace, out: as moe_expert_ffn
 *            on the prefill path (workspace >= moe_ffn_workspace_bytes(...,
 *            MOE_PATH_PREFILL)); out is complete once `compute` reaches the
 *            end of the call's work
 *   counts_host  pinned int32 [E] from the same moe_route_plan call (sum
 *            T * k)
 *   window   1 <= window <= S / 2 (a window and its predecessor are
 *            resident together)
 * A dry-run pool performs steps 1 and 3's bookkeeping only (no device
 * pointers are read).  Pools staging decode parts only (MOE_STAGE_DECODE)
 * lack the row-major down matrix: MOE_ERR_UNSUPPORTED.  If a window's
 * staging fails, MOE_ERR_CUDA is returned as moe_pool_stage does, earlier
 * windows' work stays enqueued and out is incomplete.
 * Errors: MOE_ERR_INVALID, MOE_ERR_UNSUPPORTED, MOE_ERR_TIMEOUT, MOE_ERR_CUDA. */
MOE_API int moe_prefill_staged(moe_pool_t* pool, int layer, const void* x_bf16, int T, int k,
                               const int32_t* ids, const float* w, const int32_t* offsets,
                               const int32_t* perm, const int32_t* inv, const int32_t* counts_host,
                               int window, void* workspace, size_t ws_bytes, float* out,
                               moe_stream_t compute, moe_stream_t copy, int timeout_ms);

/* Speculative staging of `layer` ahead of its routing (next-layer
 * prefetch) [X3]: the layer's non-resident experts that were routed in at
 * least one earlier event, most often routed first (ties: lower id), are
 * copied in one by one, at most max_loads of them, each into the lowest
 * free slot, else into the slot of the resident expert the pool's policy
 * names as victim (never one loaded by this call), but only while that
 * victim was routed in fewer events than the candidate; the first
 * candidate that finds no such slot ends the call.  A prefetched expert is
 * loaded as a miss would be (policy state, h2d_bytes, evictions), counts in
 * `prefetches`, and counts in `prefetch_hits` when an event routes it
 * before it is evicted.  The copies go on `copy` after all work enqueued so
 * far on `compute` (which may still read the evicted slots); nothing waits
 * for them here: the layer's next moe_pool_stage, moe_prefill_staged or
 * moe_pool_prefetch makes its streams wait first.  No host wait.
 *   loaded   host int, out: experts copied (may be NULL)
 * A dry-run pool updates its state only.
 * Errors: MOE_ERR_INVALID, MOE_ERR_CUDA (state as after the copies that
 * were enqueued). */
MOE_API int moe_pool_prefetch(moe_pool_t* pool, int layer, int max_loads, moe_stream_t compute,
                              moe_stream_t copy, int* loaded);

/* Device-planned staging [R2][X1]: the same staging events as
 * moe_pool_stage (the planning code is shared, so every hit, miss, victim,
 * stamp and counter comes out the same under every policy), with the
 * pool's state for all layers kept in a caller-provided device buffer while
 * attached, each event planned on the GPU from the routing counts in
 * device memory, and the missed experts copied by the SMs straight out of
 * the pinned host store through its device address (Grace hosts: the same
 * link rate as the copy engines).  A layer's routing, staging and FFN are
 * then three enqueues on one stream with no host wait or round trip
 * between them (tinyserve README, "How it works" items 3 and 4).
 *
 * moe_pool_device_state_bytes: size of the device buffer (L records).
 *
 * moe_pool_device_attach: uploads the pool's state into dev_state (device,
 *   16-byte aligned, >= moe_pool_device_state_bytes; caller-owned, must stay
 *   untouched while attached) on `stream`, orders `stream` after the pool's
 *   prefetch copies still in flight, and waits (polling, at most timeout_ms;
 *   <= 0 means 10 s) for the upload.  The host store must be mapped into the
 *   device's address space (cudaHostAlloc, or cudaHostRegister with
 *   cudaHostRegisterMapped): MOE_ERR_UNSUPPORTED otherwise.  Work the caller
 *   enqueued on other streams that reads the slots must be ordered before
 *   `stream` by the caller.  Dry-run pools and attached pools: MOE_ERR_STATE.
 *
 * moe_pool_stage_device: enqueues one event of `layer`: the planner on
 *   `compute`, then the copy of the misses' bytes (the whole packed expert,
 *   or the decode parts with MOE_STAGE_DECODE) host -> slot by a kernel on
 *   `copy` after the planner (on `compute` itself when copy is NULL or the
 *   same stream).
 *   counts_dev  device int32 [E] (moe_route_plan's counts), read on the GPU
 *   slot_of_dev device int32 [E], written: the layer's slot map after the
 *               event (-1 = absent)
 *   split_dev   device int32 [2][E] or NULL, written: row 0 the slots of the
 *               event's hits, row 1 the slots of its loads, -1 elsewhere --
 *               the maps of two moe_expert_ffn calls with
 *               MOE_FFN_SKIP_ABSENT: the hits' part on `compute` while the
 *               copies run, then moe_pool_device_join, then the loads' part
 *               with MOE_FFN_ACCUMULATE (tinyserve README, "How it works"
 *               item 4: H2D overlapped with compute).  Or the loads' part
 *               on `copy` right behind the copy kernel (which is launched
 *               with programmatic stream serialisation, so the FFN launches
 *               while it runs and waits for it), both parts with
 *               MOE_FFN_ACCUMULATE into a zeroed or residual `out` and with
 *               workspaces of their own, and `compute` made to wait for
 *               `copy` (an event) before `out` is read.
 *   An event with a negative count or more than S routed experts changes
 *   nothing (no copies; slot_of_dev gets the current map, row 0 of
 *   split_dev slot S -- out of range, so NaN -- for routed experts without
 *   a slot) and is reported by moe_pool_device_detach.  Nothing waits on
 *   the host; the call may be captured in a CUDA graph (with `copy` forked
 *   from and joined back to `compute` inside the capture).  Copy-failure
 *   injection does not apply.
 *
 * moe_pool_route_stage_device: moe_route_plan of T tokens (T * k <= 32, the
 *   decode shapes; MOE_ERR_UNSUPPORTED above) followed by
 *   moe_pool_stage_device on its counts, with the routing and the planning
 *   in one launch on `compute` (the routing warp ranks the tokens while the
 *   other warps load the layer's record; the counts reach the planner in
 *   shared memory).  logits, ids, w, counts, offsets, perm and inv are
 *   moe_route_plan's (device, same layouts; E = the pool's experts) and get
 *   the same values; slot_of_dev, split_dev, compute and copy are
 *   moe_pool_stage_device's.  Validation happens before anything is
 *   enqueued.
 *
 * moe_pool_device_join: makes `compute` wait for the copies of `layer`'s
 *   last event enqueued on a separate copy stream (no-op otherwise).  The
 *   layer's next moe_pool_stage_device / moe_pool_route_stage_device and
 *   moe_pool_device_detach join by themselves.
 *
 * moe_pool_device_detach: downloads the state into the pool on `stream`
 *   (polling, at most timeout_ms) after the work enqueued so far; the
 *   counters, slot maps, last loads and checkpoints then read as after the
 *   same events staged by moe_pool_stage.  Returns MOE_ERR_INVALID if an
 *   event saw a negative count, MOE_ERR_CAPACITY if one routed more than S
 *   experts (the state is detached either way), MOE_ERR_TIMEOUT if the wait
 *   ran out (still attached).
 *
 * While attached, moe_pool_stage, moe_prefill_staged, moe_pool_prefetch,
 * moe_pool_counters, moe_pool_slot_map, moe_pool_last_loads, moe_pool_save
 * and moe_pool_load return MOE_ERR_STATE.
 * Errors: MOE_ERR_INVALID, MOE_ERR_STATE, MOE_ERR_UNSUPPORTED,
 * MOE_ERR_CAPACITY, MOE_ERR_TIMEOUT, MOE_ERR_CUDA. */
MOE_API int moe_pool_device_state_bytes(const moe_pool_t* pool, size_t* out_bytes);
MOE_API int moe_pool_device_attach(moe_pool_t* pool, void* dev_state, size_t bytes, moe_stream_t stream,
                                   int timeout_ms);
MOE_API int moe_pool_stage_device(moe_pool_t* pool, int layer, const int32_t* counts_dev,
                                  int32_t* slot_of_dev, int32_t* split_dev, moe_stream_t compute,
                                  moe_stream_t copy);
MOE_API int moe_pool_route_stage_device(moe_pool_t* pool, int layer, const float* logits, int T, int k,
                                        int32_t* ids, float* w, int32_t* counts, int32_t* offsets, int32_t* perm,
                                        int32_t* inv, int32_t* slot_of_dev, int32_t* split_dev,
                                        moe_stream_t compute, moe_stream_t copy);
MOE_API int moe_pool_device_join(moe_pool_t* pool, int layer, moe_stream_t compute);
MOE_API int moe_pool_device_detach(moe_pool_t* pool, moe_stream_t stream, int timeout_ms);

/* Counters of one layer, or summed over all layers with layer = -1. */
MOE_API int moe_pool_counters(const moe_pool_t* pool, int layer, moe_counters* out);

/* The layer's expert -> slot map, host int32 [E] (-1 = absent). */
MOE_API int moe_pool_slot_map(const moe_pool_t* pool, int layer, int32_t* slot_of_host);

/* Copies issued by the last successful stage call of a layer, in issue
 * order: load_expert/load_slot host int32 [S]; *n_loads <= S. */
MOE_API int moe_pool_last_loads(const moe_pool_t* pool, int layer, int32_t* load_expert,
                        int32_t* load_slot, int* n_loads);

/* Checkpoint / resume of the pool's host state (slot maps, recency stamps,
 * counters) -- not the slot contents.  moe_pool_state_bytes gives the size;
 * save writes it to a host buffer; load restores it into a pool created with
 * the same desc (MOE_ERR_STATE otherwise).  After a load the caller must
 * refill the device slots (e.g. by re-creating with preload or copying). */
MOE_API int moe_pool_state_bytes(const moe_pool_t* pool, size_t* out_bytes);
MOE_API int moe_pool_save(const moe_pool_t* pool, void* buf, size_t bytes);
MOE_API int moe_pool_load(moe_pool_t* pool, const void* buf, size_t bytes);

/* Host-side fault injection for tests: the next n miss copies of stage
 * report failure before being enqueued (no GPU work is affected). */
MOE_API int moe_pool_inject_copy_failures(moe_pool_t* pool, int n);

MOE_API void moe_pool_destroy(moe_pool_t* pool);

/* ------------------------------------------------------------------------ */
/* Expert FFN and combine [R3][R5][P1][MX]                                   */
/* ------------------------------------------------------------------------ */

/* Scratch bytes moe_expert_ffn needs (path as passed to moe_expert_ffn). */
MOE_API int moe_ffn_workspace_bytes(int T, int k, int hidden, int inter, int path,
                            size_t* out_bytes);

/* The routed experts of one layer, combined:
 *   out[t] = sum_j w[t][j] * down_e(bf16(silu(gate_e x_t) * up_e x_t)),
 *   e = ids[t][j], summed in fp32.  Both paths fold the k terms (and the
 *   decode path also the partial down sums) into out with fp32 atomics, so
 *   the order of those additions, and with it the last bits of out, varies
 *   between runs.
 *   pool      the pool whose dev_slots hold the layer's experts
 *   x_bf16    device bf16 [T][H]
 *   ids, w    device, from moe_route_plan
 *   offsets, perm, inv  device, from moe_route_plan (prefill path only;
 *             may be NULL for the decode path)
 *   slot_of   device int32 [E]: slot of each expert in this layer; every
 *             routed expert must be resident (moe_pool_stage ensures it),
 *             except with MOE_FFN_SKIP_ABSENT: entries < 0 then mark the
 *             assignments this call leaves out
 *   path      MOE_PATH_DECODE: bf16 activations times fp32-dequantised
 *             MXFP4 on CUDA cores, fp32 accumulation, SwiGLU output rounded
 *             to bf16.  MOE_PATH_PREFILL: activations and the SwiGLU output
 *             quantised to MXFP8 (E4M3, block-32 E8M0 scale
 *             2^(floor(log2 amax) - 8), RNE, satfinite) and multiplied on
 *             tcgen05 block-scaled tensor cores, fp32 accumulation.
 *             MOE_PATH_AUTO: decode when T*k <= MOE_DECODE_MAX_ASSIGN.
 *             With MOE_FFN_ACCUMULATE or-ed in, out += the result; the
 *             decode path then needs no completion pass and prefill no
 *             zeroing of out.  With MOE_FFN_SKIP_ABSENT or-ed in (decode
 *             path with the one-launch kernel only, else
 *             MOE_ERR_UNSUPPORTED) the result sums only the assignments
 *             whose expert has slot_of >= 0, their work spread over all
 *             CTAs (a token none of whose assignments is served gets 0).
 *   workspace device, >= moe_ffn_workspace_bytes(), 256-byte aligned.
 *             On the decode path it holds a completion counter and an fp32
 *             [T][H] accumulator that must be zero when the workspace is
 *             first used (allocate it zero-filled); the library leaves them
 *             zero after every call.  One workspace must not be used by two
 *             calls that can run at the same time.
 *   out       device fp32 [T][H], 16-byte aligned, fully overwritten (added
 *             to with MOE_FFN_ACCUMULATE)
 * Errors: MOE_ERR_INVALID, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA. */
MOE_API int moe_expert_ffn(const moe_pool_t* pool, int layer, const void* x_bf16, int T, int k,
                   const int32_t* ids, const float* w, const int32_t* offsets,
                   const int32_t* perm, const int32_t* inv, const int32_t* slot_of,
                   int path, void* workspace, size_t ws_bytes, float* out,
                   moe_stream_t stream);

/* One decode step of one layer in a single launch: moe_route_plan followed
 * by moe_expert_ffn on the decode path, fused [R1][R3][P1].  For small
 * batches on a pool whose routed experts are resident (no staging between
 * routing and the experts).  Every CTA ranks the logits itself; the routing
 * outputs (ids, w, counts, offsets, perm, inv, as moe_route_plan defines
 * them) are written too.  Results equal moe_route_plan + moe_expert_ffn
 * (MOE_PATH_DECODE) on the same inputs, up to fp32 rounding order: the
 * down sums and the combine are folded across CTAs with fp32 atomics.
 *   logits   device fp32 [T][E]; x_bf16 device bf16 [T][H]
 *   slot_of  device int32 [E]: every routed expert must be resident
 *   workspace as moe_expert_ffn, MOE_PATH_DECODE (zero-filled before first
 *            use)
 *   out      device fp32 [T][H], 16-byte aligned, fully overwritten
 * Limits: T*k <= 32.  Errors: MOE_ERR_INVALID, MOE_ERR_STATE,
 * MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA. */
MOE_API int moe_decode_layer(const moe_pool_t* pool, int layer, const float* logits,
                             const void* x_bf16, int T, int k, int32_t* ids, float* w,
                             int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                             const int32_t* slot_of, void* workspace, size_t ws_bytes,
                             float* out, moe_stream_t stream);

/* moe_decode_layer with out += the layer's output (a residual stream)
 * instead of out = ...: the CTAs add their partial sums into out directly,
 * so the launch has no completion pass.  Same arguments and errors. */
MOE_API int moe_decode_layer_acc(const moe_pool_t* pool, int layer, const float* logits,
                                 const void* x_bf16, int T, int k, int32_t* ids, float* w,
                                 int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                                 const int32_t* slot_of, void* workspace, size_t ws_bytes,
                                 float* out, moe_stream_t stream);

/* Device-side status of the work done with `workspace` (path: the layout it
 * was sized for, MOE_PATH_DECODE or MOE_PATH_PREFILL): every wait inside the
 * kernels is bounded (about a second); one that runs out sets a bit here and
 * the launch finishes with NaN where its data was missing, instead of
 * hanging or faulting.  Waits (polling, at most 10 s) for all work enqueued
 * so far on `stream`, returns the bits in *bits (0: nothing ran out) and
 * clears them; MOE_ERR_TIMEOUT if the stream's work does not finish in time
 * (the bits are then neither read nor cleared).
 * Decode bits: 4 copy producer, 8 consumers (data not landed).  Prefill
 * bits: 1 TMA producer, 2 MMA issuer, 4 invalid slot, 8 epilogue, 16
 * teardown, 32 misaligned output, 64 scale-factor feeders.
 * Errors: MOE_ERR_INVALID, MOE_ERR_TIMEOUT, MOE_ERR_CUDA. */
MOE_API int moe_ffn_status(void* workspace, int path, moe_stream_t stream, uint32_t* bits);

/* Test hook for the failure path above: the next n fused decode launches
 * leave their first work item's copies unissued, so the waits on it run
 * out and set status bits; nothing faults and the context stays usable.
 * Errors: MOE_ERR_INVALID (n < 0). */
MOE_API int moe_debug_stall_next_decode(int n);

/* Weighted combine of per-assignment expert outputs held in grouped order:
 *   out[t][h] = sum_j w[t][j] * y_perm[inv[t*k+j]][h], j ascending, fp32.
 *   y_perm device fp32 [A][H]; w device fp32 [T][k]; inv device int32 [A];
 *   out device fp32 [T][H].  Errors: MOE_ERR_INVALID, MOE_ERR_CUDA. */
MOE_API int moe_combine(const float* y_perm, const float* w, const int32_t* inv,
                int T, int k, int H, float* out, moe_stream_t stream);

/* MXFP8 quantisation of bf16 rows, optionally gathered by a permutation:
 * output row p quantises x[perm[p] / k] (or x[p] when perm is NULL).
 *   x_bf16 device [*][K]; q device uint8 [rows][K] E4M3 codes;
 *   scales device uint8 [rows][scale_stride] E8M0 bytes (the first K/32 of
 *   each row are written); K a multiple of 32; scale_stride >= K/32.
 * Errors: MOE_ERR_INVALID, MOE_ERR_CUDA. */
MOE_API int moe_quant_mxfp8(const void* x_bf16, int K, const int32_t* perm, int k, int rows,
                    uint8_t* q, uint8_t* scales, int scale_stride, moe_stream_t stream);

/* MXFP4 quantisation of bf16 rows [MX] (OCP MX v1.0: E2M1 elements, shared
 * exponent floor(log2(amax)) - 2 per block of 32, E8M0 byte clamped to
 * [0, 254], 0 for an all-zero block; round to nearest even, finite overflow
 * saturated to +-6), for MXFP4 activations:
 *   x_bf16 device [rows][K] (16-byte aligned); q device uint8 [rows][K/2],
 *   element 2i in the low nibble of byte i (16-byte aligned); scales device
 *   uint8 [rows][scale_stride], the first K/32 of each row written;
 *   K a multiple of 32.
 * Errors: MOE_ERR_INVALID, MOE_ERR_CUDA. */
MOE_API int moe_quant_mxfp4(const void* x_bf16, int K, int rows, uint8_t* q, uint8_t* scales,
                            int scale_stride, moe_stream_t stream);


/* ------------------------------------------------------------------------ */
/* Decode on GGUF expert weights [R3]                                        */
/* ------------------------------------------------------------------------ */

/* GGUF block formats of the experts (tinyserve README, "How it works" item
 * 2 and "Supported models", Formats, run experts in their native GGUF
 * quantisation; the block layouts are the published GGUF / ggml ones):
 *   Q8_0  per 32 elements, 34 bytes: binary16 d (little-endian), 32 int8 q;
 *         element = d * q.
 *   Q4_K  per 256 elements, 144 bytes: binary16 d and dmin, 12 bytes packing
 *         eight 6-bit scales sc and mins m (sub-blocks 0-3 in the low 6 bits
 *         of bytes j and j+4; 4-7 split over the nibbles of byte j+4 and the
 *         top 2 bits of bytes j-4 and j), 128 bytes of 4-bit values q
 *         (sub-blocks 2g and 2g+1 in the low and high nibbles of the same 32
 *         bytes); element = d*sc*q - dmin*m. */
#define MOE_GGUF_Q8_0 0
#define MOE_GGUF_Q4_K 1

/* Bytes of one GGUF expert slot: [gate I rows][up I rows][down H rows],
 * each row the format's blocks back to back (gate and up rows of H
 * elements, down rows of I elements), the total rounded up to 256 bytes.
 * Q8_0 needs hidden and inter multiples of 64, Q4_K multiples of 256.
 * Errors: MOE_ERR_INVALID. */
MOE_API int moe_gguf_expert_bytes(int fmt, int hidden, int inter, size_t* out_bytes);

/* Workspace bytes of moe_expert_ffn_gguf and moe_decode_layer_gguf: a
 * 256-byte control block (word 2: the status bits moe_ffn_status reads
 * with MOE_PATH_DECODE), bf16 h [T*k][inter] at byte 256, then fp32 y
 * [T*k][hidden] at 256 + round_up(T*k*inter*2, 256) (each assignment's down
 * output before the combine, on the three-launch path).  Allocate it
 * zero-filled: the single-launch kernel keeps cross-CTA counters in the
 * control block and leaves them zero after every call. */
MOE_API int moe_gguf_workspace_bytes(int T, int k, int hidden, int inter, size_t* out_bytes);

/* The routed experts of one layer on GGUF weights read in place, the
 * decode path's arithmetic: out[t] = sum_j w[t][j] * down_e(h), h =
 * bf16(silu(gate_e x_t) * up_e x_t), e = ids[t][j]; bf16 activations times
 * the exactly dequantised weights, fp32 sums (each block summed in its own
 * factors: d * sum(q x), or d*sc * sum(q x) - dmin*m * sum(x) per 32),
 * the k terms summed in rank order, no floating-point atomics.  Calls of
 * at most 32 assignments whose GGUF rows are multiples of 16 bytes (and x
 * 16-byte aligned) run as one cooperative launch: one CTA per SM streams
 * its gate/up rows through shared memory with bulk copies and fetches the
 * down rows of its output rows early; it forms its output rows for all k
 * ranks of their token, once (a bounded wait: about a second, then status
 * bit 16 and NaN output) the other CTAs have written all of h of those
 * assignments.  Other calls take three launches (gate/up with SwiGLU;
 * down per assignment; the combine).
 *   fmt       MOE_GGUF_Q8_0 or MOE_GGUF_Q4_K
 *   slots     device [n_slots][moe_gguf_expert_bytes()] GGUF experts, 256-byte
 *             aligned
 *   x_bf16    device bf16 [T][hidden]
 *   ids, w    device, from moe_route_plan ([T][k])
 *   slot_of   device int32 [E]: slot of each expert; a routed expert without
 *             a valid slot makes its token's output NaN
 *   workspace device, >= moe_gguf_workspace_bytes(), 256-byte aligned
 *   out       device fp32 [T][hidden]; accumulate != 0: out += result
 * Limits: 1 <= E <= MOE_MAX_EXPERTS, 1 <= k <= MOE_MAX_TOPK, T >= 0, the
 * shapes above, hidden and inter at most 11,000 (one fp32 staged copy per
 * CTA).  Errors: MOE_ERR_INVALID, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA. */
MOE_API int moe_expert_ffn_gguf(int fmt, const void* slots, int n_slots, int hidden, int inter,
                                const void* x_bf16, int T, int k, const int32_t* ids, const float* w,
                                const int32_t* slot_of, int E, void* workspace, size_t ws_bytes, float* out,
                                int accumulate, moe_stream_t stream);

/* One decode step of one layer on GGUF experts in a single launch: the
 * routing of moe_route_plan fused with moe_expert_ffn_gguf, the way
 * moe_decode_layer fuses it for MXFP4 pools [R1][R3].  Every CTA ranks the
 * logits itself (larger logit first, equal logits by lower id, NaN last;
 * softmax over the k selected); CTA 0 writes the routing outputs (ids, w,
 * counts, offsets, perm, inv, as moe_route_plan defines them).  Results
 * equal moe_route_plan + moe_expert_ffn_gguf on the same inputs.
 *   logits    device fp32 [T][E]
 *   x_bf16    device bf16 [T][hidden], 16-byte aligned
 *   other arguments as moe_expert_ffn_gguf and moe_route_plan
 * Limits: T*k <= 32, k <= E; the shape must take the single-launch kernel
 * (MOE_ERR_UNSUPPORTED otherwise: GGUF rows not multiples of 16 bytes, or
 * more shared memory than the GPU has).  Errors: MOE_ERR_INVALID,
 * MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA. */
MOE_API int moe_decode_layer_gguf(int fmt, const void* slots, int n_slots, int hidden, int inter,
                                  const float* logits, const void* x_bf16, int T, int k, int32_t* ids, float* w,
                                  int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                                  const int32_t* slot_of, int E, void* workspace, size_t ws_bytes, float* out,
                                  int accumulate, moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Measurement                                                               */
/* ------------------------------------------------------------------------ */

/* Peak-rate probe of the tensor-core instruction the prefill GEMMs issue
 * (tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X, M 128,
 * N 256, K 32; E4M3 A and E2M1 B operands in shared memory, E8M0 scale
 * factors in tensor memory).  The pages have no counterpart: it gives the
 * roofline denominator of the prefill path.  One CTA per SM issues
 * stages x 4 such MMAs back to back on operands that stay in shared memory
 * (no global reads), so the launch's duration, timed by the caller with
 * CUDA events on `stream`, gives the instruction's rate:
 *   FLOPs per launch = ctas * stages * 4 * 2 * 128 * 256 * 32.
 *   stages      1 .. 2^16 (a launch of 2^16 stages lasts some tens of
 *               milliseconds, well inside the bounded wait)
 *   status_dev  device uint32, bit 1 set if the bounded completion wait
 *               ran out (caller zeroes it; read it after the launch)
 *   ctas        host int, out: CTAs launched (one per SM); may be NULL
 * Errors: MOE_ERR_INVALID, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA. */
MOE_API int moe_probe_mxf8f6f4(int stages, uint32_t* status_dev, int* ctas, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
