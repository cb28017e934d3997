/*
 * moe_slot_cache — decode-time routed-MoE layer with an HBM expert slot cache
 * (GB300 / sm_103a).  C ABI.
 *
 * The method (web page "GLM 5.3 Testing: HBM Expert Allocation", section
 * "What the slot cache is"): every routed expert of every MoE layer lives in
 * pinned host memory; each layer owns a fixed ring of S HBM slots.  Before the
 * expert computation the router's top-k expert ids are mapped to slot ids on
 * the device; a missing expert's weight row and scale row are copied into the
 * least-recently-used slot, then the map is updated; the expert kernel reads
 * the same bytes it would read if every expert were in HBM, only the index
 * changes.  Fixed addresses and fixed shapes make a decode round replayable as
 * a CUDA graph.  Steps with more than 16 rows (prefill) bypass the cache, so
 * no expert is ever unreachable: each expert they use is read once from host
 * memory, staged into HBM a chunk at a time (or read zero-copy, by option).
 *
 * Conventions
 *  - Every function returns MOE_OK (0) or a negative MOE_ERR_* code; nothing
 *    throws across the ABI.  moe_cache_strerror() names a code.
 *  - "host" pointers are CPU addresses, "device" pointers are CUDA device
 *    addresses on the device that was current at moe_cache_create.
 *  - A handle is used from one host thread at a time; calls are not
 *    thread-safe.  All device work of a handle goes to the stream passed to
 *    moe_cache_step, which must be the same stream (or a stream ordered after
 *    it) for every step of the handle.
 *  - Device-side anomalies (non-finite router logits, a device wait that gave
 *    up) never trap: they set sticky bits in moe_cache_stats_t.error_flags and
 *    the step still completes with defined (possibly meaningless) output.
 */
#ifndef MOE_SLOT_CACHE_H
#define MOE_SLOT_CACHE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ----------------------------------------------------------------- codes */
#define MOE_OK 0
#define MOE_ERR_ARG (-1)         /* bad argument, shape or pointer */
#define MOE_ERR_NOT_PINNED (-2)  /* host backing is not device-accessible pinned memory */
#define MOE_ERR_OOM (-3)         /* device or pinned host allocation failed */
#define MOE_ERR_CUDA (-4)        /* a CUDA runtime call or kernel launch failed */
#define MOE_ERR_UNSUPPORTED (-5) /* shape outside the compiled limits below */

/* sticky device flags (moe_cache_stats_t.error_flags) */
#define MOE_FLAG_NONFINITE_LOGIT 0x1u /* a router logit was NaN or +-inf */
#define MOE_FLAG_WAIT_TIMEOUT 0x2u    /* a kernel's bounded wait on its own copies gave up */
#define MOE_FLAG_BAD_PLAN 0x4u        /* a kernel found an out-of-range index in the step's plan
                                         and skipped that access (output undefined) */

/* limits */
#define MOE_MAX_EXPERTS 1024
#define MOE_MAX_TOPK 16
#define MOE_MAX_CACHED_ROWS 16                       /* rows of one cached step */
#define MOE_MAX_PICKS (MOE_MAX_CACHED_ROWS * MOE_MAX_TOPK)
#define MOE_MAX_DIM 8192                             /* hidden and inter */

/* copy backends (moe_cache_opts_t.copy_backend) */
#define MOE_COPY_SM 0 /* SM kernel, 16-byte loads from pinned host memory; graph-capturable */

/* --------------------------------------------------------------- types */

typedef struct moe_cache moe_cache_t; /* opaque, library-owned */

/* One layer's backing store, caller-owned (the library never frees it; it must
 * outlive the handle).  Expert e's bytes:
 *   w + e*Bw, Bw = 3*hidden*inter/2 bytes of E2M1 codes, two per byte, element
 *     2i in the low nibble of byte i.  Rows in order: gate [inter][hidden/2],
 *     up [inter][hidden/2], down [hidden][inter/2].
 *   s + e*Bs, Bs = 3*hidden*inter/16 bytes of E4M3 block scales, one per 16
 *     consecutive elements of a row, same row order: [rows][K/16].
 *   gscale[3*e .. 3*e+2]: fp32 global scales (gate, up, down).
 * The weight of row r, element i is e2m1(code) * e4m3(scale) * gscale.
 * Block scales are non-negative: every scale byte must be a finite E4M3 code
 * with the sign bit clear (0x00 .. 0x7E; the tensor-core path reads them as
 * unsigned E4M3).  moe_cache_create reads the scale banks once and returns
 * MOE_ERR_ARG if a byte has the sign bit set or is the NaN code 0x7F; the
 * contents must therefore be in place at create and must not change while
 * the handle lives.
 * w and s must be pinned, mapped host memory (e.g. from moe_host_alloc or
 * cudaHostAlloc with cudaHostAllocMapped), 16-byte aligned, of at least
 * experts*Bw and experts*Bs bytes.  gscale is ordinary host memory, read once
 * at create. */
typedef struct {
  const void* w;
  const void* s;
  const float* gscale;
} moe_host_layer_t;

typedef struct {
  int copy_backend;   /* MOE_COPY_SM (default) */
  int bypass_rows;    /* steps with more rows bypass the cache; default and max 16 */
  int all_resident;   /* 1: every expert lives in HBM (S = experts, loaded at create);
                         same kernels, used to check that caching changes no output bit */
  int trace_capacity; /* per-layer ring of moe_step_record_t for cached steps (0 = off) */
  int max_rows;       /* largest rows of any step (sizes the multi-row and bypass
                         workspaces); raised to bypass_rows if smaller.  Default (0):
                         bypass_rows, a decode-only handle: steps with more rows return
                         MOE_ERR_UNSUPPORTED and no prefill staging is allocated.  Set it
                         to the largest prefill chunk to take bypass steps */
  int prefill_chunk;  /* bypass steps: experts staged into HBM per chunk, two chunks held at
                         once (a 2 * prefill_chunk expert staging area, allocated at create
                         when max_rows > bypass_rows); 0: default 32; -1: no staging, the
                         grouped kernels read host memory directly */
  int batch_invariant; /* 1: one-row steps take the grouped tensor-core path of multi-row
                          rounds, so every row's output is bit-identical whether it is
                          stepped alone or inside a round of up to 16 rows (exact verify
                          rows for speculative decoding); 0 (default): one-row steps take
                          the faster CUDA-core decode path */
  const int32_t* slots_per_layer; /* NULL: every layer has `slots` slots; else host int32
                                     [layers], layer l's ring size (top_k <= S_l <= experts,
                                     e.g. from moe_policy_size_layers), read at create only;
                                     ignored with all_resident */
} moe_cache_opts_t;

typedef struct {
  uint64_t steps;        /* moe_cache_step calls on the layer(s) */
  uint64_t picks;        /* routed picks of cached steps (rows * top_k) */
  uint64_t hits;         /* picks whose expert was resident at step start */
  uint64_t misses;       /* unique missing experts (one copy each) */
  uint64_t evictions;    /* misses that replaced a resident expert */
  uint64_t bytes_copied; /* host->HBM bytes moved by miss copies */
  uint64_t bypass_calls; /* steps that bypassed the cache */
  uint32_t error_flags;  /* MOE_FLAG_* (sticky) */
  uint32_t reserved;
} moe_cache_stats_t;

/* One cached layer-step, for checking the cache trace against a reference. */
typedef struct {
  uint32_t clock;  /* layer's LRU clock after the step (advances on cached steps only) */
  int32_t rows;
  int32_t n_union; /* distinct experts over all rows */
  int32_t n_miss;
  int32_t bypass;  /* 1: union larger than S, step read host memory, cache untouched */
  int32_t ids[MOE_MAX_PICKS];       /* rank order per row, row-major [rows][top_k] */
  float weights[MOE_MAX_PICKS];
  int32_t slot[MOE_MAX_PICKS];      /* slot read by each pick (-1 on bypass) */
  int32_t hit[MOE_MAX_PICKS];       /* resident at step start */
  int32_t miss_expert[MOE_MAX_PICKS]; /* ascending expert id */
  int32_t miss_slot[MOE_MAX_PICKS];
  int32_t miss_evicted[MOE_MAX_PICKS]; /* previous owner, -1 if the slot was empty */
} moe_step_record_t;

/* --------------------------------------------------------------- cache */

/* Build a slot cache of `layers` MoE layers, each with `experts` routed experts
 * of shape (hidden, inter), top_k routing and `slots` HBM slots.  Allocates all
 * device state (slots, maps, stamps, counters, workspaces) once; addresses never
 * change afterwards.  Caches start empty.  host_backing has `layers` entries.
 * opts may be NULL (defaults).  Limits: experts <= MOE_MAX_EXPERTS,
 * top_k <= min(experts, MOE_MAX_TOPK), top_k <= slots <= experts,
 * hidden and inter multiples of 128 and <= MOE_MAX_DIM, inter / 32 a multiple
 * or a divisor of 32 (the one-row down pass spreads a W2 row's 32-element
 * blocks over a warp's lanes).  Errors: MOE_ERR_ARG, MOE_ERR_NOT_PINNED, MOE_ERR_OOM, MOE_ERR_CUDA,
 * MOE_ERR_UNSUPPORTED.  On error *out is NULL and nothing leaks. */
int moe_cache_create(moe_cache_t** out, int layers, int experts, int slots, int hidden,
                     int inter, int top_k, const moe_host_layer_t* host_backing,
                     const moe_cache_opts_t* opts);

/* One layer-step for `rows` tokens:
 *   router_logits: device fp32 [rows][experts]
 *   x:             device bf16 bits [rows][hidden], 16-byte aligned
 *   out:           device fp32 [rows][hidden] (written, not accumulated),
 *                  16-byte aligned
 *   stream:        cudaStream_t (NULL = legacy default stream)
 * rows <= bypass_rows: route (top-k by logit, ties to the lower id; weights =
 * softmax of the k selected logits), map ids to slots, copy misses host->slot,
 * run gate/up -> SwiGLU -> down on slot-resident bytes and combine with the
 * router weights.  rows > bypass_rows: same result, experts read from host
 * memory, cache untouched.  Enqueues kernels only (no host sync, no
 * allocation); capturable into a CUDA graph.  Buffers must keep their
 * addresses across graph replays.  Errors: MOE_ERR_ARG, MOE_ERR_UNSUPPORTED,
 * MOE_ERR_CUDA (launch failure). */
int moe_cache_step(moe_cache_t* h, int layer, int rows, const float* router_logits,
                   const uint16_t* x, float* out, void* stream);

/* The same layer-step with host buffers: router_logits (fp32 [rows][experts])
 * and x (bf16 bits [rows][hidden]) are moved host -> device into the handle's
 * staging, the step runs, and out (fp32 [rows][hidden]) is moved device ->
 * host, all enqueued on `stream` in that order.  Returns without waiting: the
 * host buffers must stay valid and unchanged until the stream has passed the
 * step.  Page-locked buffers are read and written by two small kernels through
 * their device addresses (asynchronous); pageable ones go through copies
 * (synchronous for the host).  rows <= max_rows.  One-row steps replay a CUDA graph of the
 * step over the staging buffers, captured for each layer on its second
 * one-row call (never with timing events set, which take the eager path); the
 * handle's addresses never change, so a graph stays valid until
 * moe_cache_destroy.  Steps on one handle must be ordered on one stream, as for
 * moe_cache_step.  Errors: as moe_cache_step; MOE_ERR_ARG for rows > max_rows. */
int moe_cache_step_host(moe_cache_t* h, int layer, int rows, const float* router_logits,
                        const uint16_t* x, float* out, void* stream);

/* Counters of one layer (layer >= 0) or summed over all layers (layer == -1;
 * error_flags OR-ed).  The counts follow how the pages account for the cache
 * ("GB300 GLM 5.3 Testing": the September 14 correction counts misses per
 * layer-step; the September 7 E0/E1/E5 window history takes the hit rate over
 * the routed picks of an engine step, rows * top_k): hit rate = hits / picks,
 * misses are unique experts fetched per layer-step.  Waits for all device work
 * (device synchronize). */
int moe_cache_stats(const moe_cache_t* h, int layer, moe_cache_stats_t* out);

/* The ring's owner table ("GLM 5.3 Testing: HBM Expert Allocation", "What the
 * slot cache is": the router asks by expert id and the cache answers with a
 * slot; this is the reverse view, which expert each slot holds).
 * expert_of_slot: host int32 [layer's ring size]; -1 = empty.  Device
 * synchronize. */
int moe_cache_slot_map(const moe_cache_t* h, int layer, int32_t* expert_of_slot);

/* *slots = the ring size of `layer`. */
int moe_cache_layer_slots(const moe_cache_t* h, int layer, int* slots);

/* Copy one slot's resident bytes to host memory (w_dst: Bw bytes, s_dst: Bs
 * bytes; either may be NULL).  Device synchronize. */
int moe_cache_slot_bytes(const moe_cache_t* h, int layer, int slot, void* w_dst, void* s_dst);

/* Copy up to max_recs of the layer's most recent step records, oldest first,
 * into recs (host); *n_recs receives the count.  Requires trace_capacity > 0.
 * Device synchronize. */
int moe_cache_trace(const moe_cache_t* h, int layer, moe_step_record_t* recs, int max_recs,
                    int* n_recs);

/* Empty every ring, zero counters, flags and traces (all_resident: reload
 * identity map): the state at create.  The cache state is a function of the
 * routing history alone (exact LRU with stamps, "What the slot cache is"), so
 * reset + replaying a routing history reproduces any earlier state; the pages
 * have no further checkpoint for it.  Device synchronize. */
int moe_cache_reset(moe_cache_t* h);

/* Failure-detection hook (for tests of the timeout path; production code
 * leaves the default).  Every device wait in the library is bounded; this sets
 * the limit of the one-row expert kernels' waits for their own weight copies
 * to `microseconds` (0: the default, about 2 s) for the steps enqueued after
 * the call.  A wait that runs out sets MOE_FLAG_WAIT_TIMEOUT, and the kernel
 * finishes the step on whatever bytes arrived (output undefined; a missed
 * expert's slot may be left incomplete, so moe_cache_reset before relying on
 * the cache again).  Copies still in flight are always drained under the
 * default limit before a kernel exits.  Synchronous (device synchronize).
 * Errors: MOE_ERR_ARG (microseconds < 0), MOE_ERR_CUDA. */
int moe_cache_set_wait_timeout(moe_cache_t* h, int microseconds);

/* Free everything the handle owns (not the host backing).  NULL is a no-op.
 * Handle lifetime is the library's own; the pages have no counterpart. */
int moe_cache_destroy(moe_cache_t* h);

/* A static string naming a MOE_OK / MOE_ERR_* code (the library's own; the
 * pages have no counterpart). */
const char* moe_cache_strerror(int code);

/* Byte sizes of one expert's codes (Bw) and scales (Bs) for (hidden, inter). */
int moe_expert_bytes(int hidden, int inter, uint64_t* Bw, uint64_t* Bs);

/* ---------------------------------------------------------- host memory */

/* Exact-size pinned host allocation, portable and mapped, with its device view
 * checked to be the same address (UVA).  ("GLM 5.3 Testing: HBM Expert
 * Allocation", "Five launches, four failures": allocators that round pinned
 * blocks up to powers of two wasted a third of host memory; allocate exactly.)
 * Errors: MOE_ERR_ARG, MOE_ERR_OOM, MOE_ERR_NOT_PINNED (no UVA view). */
int moe_host_alloc(void** out, size_t bytes);
int moe_host_free(void* p);

/* --------------------------------------------------------- measurement */

/* Host->HBM read bandwidth over the host link, measured with the same SM copy
 * the miss path uses (method 0) or cudaMemcpyAsync (method 1): copies `bytes`
 * from pinned host_src to device dev_dst `iters` times and returns the best
 * GB/s (1e9 bytes/s).  Synchronous.  Both pointers 16-byte aligned. */
int moe_probe_host_link(const void* host_src, void* dev_dst, size_t bytes, int method,
                        int iters, double* best_gbps);

/* Per-kernel timing hook: events points at MOE_TIMING_EVENTS cudaEvent_t
 * (created by the caller, timing enabled).  While set, every moe_cache_step
 * records them (also inside a CUDA-graph capture, where they become
 * event-record nodes):
 *   0 before route/remap, 1 after it (caller's stream);
 *   one-row steps, the library's second stream: 2 before the missed picks'
 *     read-through pass (host -> slot with gate/up and down on the way in),
 *     3 and 4 after it;
 *   multi-row steps, the caller's stream: 2 after the miss copy, 3 after the
 *     grouped gate/up, 4 after the grouped down;
 *   5 after the resident picks' gate/up, 6 after their down (one-row steps;
 *     multi-row: same points as 3 and 4);
 *   7 end of the step (after the combine).
 * NULL stops recording.  The library does not own the events. */
#define MOE_TIMING_EVENTS 8
int moe_cache_set_timing_events(moe_cache_t* h, void* const* events);

/* Step-input feeder (a device step cursor).  A decode round is captured once
 * as a CUDA graph over fixed input buffers ("GLM 5.3 Testing: HBM Expert
 * Allocation", "What the slot cache is": fixed addresses and shapes make a
 * round replayable as a graph).  Put this call first in the captured round and
 * one graph replays over fresh inputs: each call copies entry
 * t = cursor[0] mod steps of two device-resident input traces into the fixed
 * buffers the round's steps read, then adds one to cursor[0].
 *   logits_trace: device, steps entries of logits_bytes each (e.g. fp32
 *     [layers][rows][experts] per round);
 *   x_trace: device, steps entries of x_bytes each (e.g. bf16 bits
 *     [layers][rows][hidden]); NULL with x_bytes == 0 copies logits only
 *     (and the reverse);
 *   logits_dst, x_dst: device buffers of one entry each, the addresses the
 *     captured steps read;
 *   cursor: device uint32 [2], caller-owned, zero before the first call;
 *     cursor[0] counts the entries fed (set it to restart the trace at an
 *     entry), cursor[1] is the launch's own count and must stay zero between
 *     calls.
 * Byte counts multiples of 16; every pointer 16-byte aligned (cursor 4-byte).
 * Enqueues one kernel on `stream` (capturable); calls on one cursor must be
 * ordered on the device.  Errors: MOE_ERR_ARG, MOE_ERR_CUDA. */
int moe_feed_inputs(const void* logits_trace, const void* x_trace, size_t logits_bytes,
                    size_t x_bytes, int steps, void* logits_dst, void* x_dst, uint32_t* cursor,
                    void* stream);

/* --------------------------------------------------- offline slot policy */

/* Slot policies evaluated on a routing trace, host only (no GPU, no handle).
 * The pages compare the cache's LRU with a hindsight-static pin of the
 * hottest experts and with hybrids, on recorded routing traces, and size each
 * layer's ring from its trace ("GB300 GLM 5.3 Testing", LRU vs static and
 * hybrid hit rates; "GLM 5.3 Testing: HBM Expert Allocation", per-layer slot
 * budgets).
 *   trace: host int32 [steps][picks], one layer's expert ids per layer-step
 *          (picks = rows * top_k, row-major), each in [0, experts).
 * LRU follows the cache exactly: a pick hits if its expert was resident when
 * the step began; each missing expert of the step's union is fetched once; a
 * union larger than the ring bypasses it (read from host memory, ring and
 * clock untouched).  Errors: MOE_ERR_ARG (bad sizes or an id out of range). */
typedef struct {
  uint64_t steps;        /* layer-steps in the trace */
  uint64_t picks;        /* picks of the steps that did not bypass */
  uint64_t hits;         /* of those, picks served from HBM (resident or pinned) */
  uint64_t misses;       /* experts fetched into the ring */
  uint64_t evictions;    /* fetches that replaced a resident expert */
  uint64_t bypass_steps; /* steps whose (unpinned) union exceeded the ring */
  uint64_t host_experts; /* experts read over the host link: fetches, bypassed
                            unions, and unpinned experts under a static pin */
} moe_policy_result_t;

/* LRU ring of `slots` slots (1 <= slots <= experts). */
int moe_policy_lru(const int32_t* trace, int steps, int picks, int experts, int slots,
                   moe_policy_result_t* out);
/* Hindsight static: the `slots` most picked experts of the whole trace (ties
 * to the lower id) are always resident; every other expert a step uses is
 * read from host memory each time (host_experts counts it once per step).
 * 0 <= slots <= experts; misses and evictions are 0. */
int moe_policy_static(const int32_t* trace, int steps, int picks, int experts, int slots,
                      moe_policy_result_t* out);
/* Hybrid: the `pinned` hottest experts are always resident and the other
 * slots - pinned slots run LRU for the rest (pinned == 0: LRU; pinned ==
 * slots: static).  0 <= pinned <= slots <= experts. */
int moe_policy_hybrid(const int32_t* trace, int steps, int picks, int experts, int slots,
                      int pinned, moe_policy_result_t* out);
/* host_experts[S - 1] of an S-slot LRU ring for S = 1 .. max_slots. */
int moe_policy_lru_curve(const int32_t* trace, int steps, int picks, int experts, int max_slots,
                         uint64_t* host_experts);
/* Per-layer ring sizes for a total slot budget: given each layer's LRU curve
 * (host_experts: host [layers][max_slots], row l from moe_policy_lru_curve on
 * layer l's trace), choose slots_out[l] in [min_slots, max_slots] with
 * sum <= budget minimising the summed host-link experts (exact dynamic
 * programme).  slots_out: host int32 [layers]. */
int moe_policy_size_layers(const uint64_t* host_experts, int layers, int max_slots, int budget,
                           int min_slots, int32_t* slots_out);

/* ------------------------------------------------------ no-allocation pass */

/* The one-row expert pass (gate/up -> SwiGLU -> down -> combine with the
 * router weights) over k experts already resident in device memory, for
 * callers that cannot allocate device memory: e.g. a serving engine that has
 * reserved all free HBM for its own pools and owns every further byte, or a
 * decode loop that cannot afford an allocation's implicit synchronisation.
 * The pages have no counterpart: it is the library's own addition.
 *   expert_w[j], expert_s[j]: host arrays of k device addresses of expert j's
 *     codes (Bw bytes) and scales (Bs bytes), storage layout as in
 *     moe_host_layer_t, 16-byte aligned;
 *   gscale: host [k][3]; weights: host [k] (router weights, rank order);
 *   x: device bf16 [hidden]; out: device fp32 [hidden] (written); both
 *     16-byte aligned;
 *   flags_out: device uint32, 4-byte aligned, or NULL: receives the call's
 *     MOE_FLAG_* bits once its kernels are done (0: clean; MOE_FLAG_WAIT_TIMEOUT:
 *     a wait for the call's own weight copies gave up, MOE_FLAG_BAD_PLAN: a
 *     plan check failed; either leaves out undefined).
 * Allocates nothing: its scratch (about 1.1 MB: plan, h, per-expert partial
 * outputs, tile tickets) is one file-scope device array, fixed in size for
 * k <= MOE_MAX_TOPK and hidden, inter <= MOE_MAX_DIM, held by every GPU that
 * loads the library until the process exits; larger sizes return
 * MOE_ERR_UNSUPPORTED.  The first call on a device looks up the array's device
 * address (make it before any stream capture) and keeps it for the life of
 * the process: do not use the pass on a device after cudaDeviceReset.  All
 * calls share the array and it keeps the last call's contents (each call
 * clears what must start at zero): calls whose work overlaps on the GPU race
 * and must be ordered by the caller.
 * Errors: MOE_ERR_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA. */
int moe_expert_pass_noalloc(int k, int hidden, int inter, const void* const* expert_w,
                            const void* const* expert_s, const float* gscale,
                            const float* weights, const uint16_t* x, float* out,
                            uint32_t* flags_out, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_SLOT_CACHE_H */
