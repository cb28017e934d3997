// Internal definitions shared by the library's translation units (not installed).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "../../include/moe_slot_cache.h"

namespace moe {

// ------------------------------------------------------------------ state

// Per-layer device counters; summed/OR-ed by moe_cache_stats.
struct DevStats {
  unsigned long long steps, picks, hits, misses, evictions, bytes_copied, bypass_calls;
  unsigned int flags;
  unsigned int pad;
};

// Everything the remap kernel needs about one layer (passed by value).
struct LayerDev {
  int32_t* map;           // [E]  expert -> slot or -1
  int32_t* owner;         // [S]  slot -> expert or -1
  uint32_t* stamp;        // [S]  last-use step, 0 = never
  uint32_t* clock;        // [1]  cached steps so far
  uint8_t* slot_w;        // [S][Bw]
  uint8_t* slot_s;        // [S][Bs]
  const uint8_t* host_w;  // [E][Bw] pinned host (device-visible address)
  const uint8_t* host_s;  // [E][Bs]
  const float* gscale;    // [E][3] device copy
  DevStats* stats;
  moe_step_record_t* trace;  // [trace_cap] or null
  uint32_t* trace_head;      // records written so far
  uint32_t trace_cap;
  uint32_t* step_ctr = nullptr;  // the handle's one-row step counters: route/remap clears
                                 // the read-through's (work and h counts) for the step
};

// The per-step plan written by the remap kernel and read by the copy and
// expert kernels.  One per handle: steps run in order on one stream.
struct Plan {
  int32_t rows, npicks, n_union, n_miss, bypass;
  int32_t n_hit;   // picks resident at step start (one-row steps)
  uint32_t wait_us;  // not written by the steps (moe_cache_set_wait_timeout sets it): the
                     // one-row expert kernels' waits for their stages give up after this
                     // many microseconds (0: the default limit); waits that drain copies
                     // in flight keep the default
  int32_t pad;
  int32_t order[MOE_MAX_PICKS];  // picks, hits first, each part in rank order
  int32_t ids[MOE_MAX_PICKS];
  float wts[MOE_MAX_PICKS];
  int32_t miss_e[MOE_MAX_PICKS];
  int32_t miss_v[MOE_MAX_PICKS];
  const uint8_t* wptr[MOE_MAX_PICKS];  // expert codes this pick reads (slot or host)
  const uint8_t* sptr[MOE_MAX_PICKS];  // expert scales
  const uint8_t* hwptr[MOE_MAX_PICKS]; // the expert's host backing (read-through of a miss)
  const uint8_t* hsptr[MOE_MAX_PICKS];
  float gs[MOE_MAX_PICKS][4];          // (gate, up, down, unused) global scales
};

// Multi-row steps: picks grouped by expert so each expert's bytes are read
// once for all rows that chose it ("TensorFold GLM-5.3 explained": a round
// fetches the union of its rows' experts once).  Groups are in ascending
// expert id, members (pick indices p = row * k + rank) ascending within a
// group, jobs = (group, tile of kRowsPerJob members).  Sized at create for the
// largest step (P = max_rows * top_k picks).
constexpr int kLevels = 6;       // residual NVFP4 levels of the activations
constexpr int kRowsPerJob = 5;   // members per MMA N-tile (5 * 6 = 30 of 32 columns)
// Groups list the experts resident at step start (hits) first, then the rest,
// each part in ascending expert id, so a step can run the hit groups while the
// misses copy.  kHitGroups as a launch's g0 or g1 stands for n_hit_groups;
// miss_part(p, P) for the first miss group of part p of P: the miss groups
// [n_hit_groups, n_groups) cut at n_hit_groups + (n_groups - n_hit_groups) * p / P
// (p = P: n_groups).  Part p's groups are the misses of part p of the plan's
// miss list (also ascending expert id), so a step can compute the misses of
// one part while the next part copies.  P < 16.
constexpr int kHitGroups = -1;
__host__ __device__ constexpr int miss_part(int p, int P) { return -(64 + 16 * p + P); }
struct GroupPlan {
  int32_t n_groups, n_jobs, rows, npicks;
  int32_t n_hit_groups;    // groups [0, n_hit_groups) need no copy this step
  int32_t* g_expert;       // [G]
  int32_t* g_start;        // [G] first member
  int32_t* g_count;        // [G]
  const uint8_t** g_wptr;  // [G] expert codes (slot, or host memory on a bypass)
  const uint8_t** g_sptr;  // [G]
  float* g_gs;             // [G][3]
  int32_t* members;        // [P] pick indices grouped
  int32_t* jobs;           // [J] (group << 8) | tile
  float* wts;              // [P] router weights by pick
  int32_t* g_job;          // [G + 1] first job of each group; [n_groups] = n_jobs
};

// Activations in residual NVFP4: codes [rows][kLevels][K/2], scales
// [rows][kLevels][K/16] (UE4M3), level scales [rows][kLevels] (fp32).
struct QuantBuf {
  uint8_t* codes;
  uint8_t* scales;
  float* gl;
};

// ------------------------------------------------------------ launchers

// route + remap/LRU for rows <= MOE_MAX_CACHED_ROWS (one CTA); gp != null
// also emits the expert groups of a multi-row step.
cudaError_t launch_route_remap(cudaStream_t st, const float* logits, int rows, int E, int k,
                               int S, long long Bw, long long Bs, const LayerDev& L, Plan* plan,
                               int all_resident, GroupPlan* gp);
// bypass steps: route every row, group picks by expert over host backing.
cudaError_t launch_route_rows(cudaStream_t st, const float* logits, int rows, int E, int k,
                              int32_t* ids, GroupPlan* gp, const LayerDev& L, long long Bw,
                              long long Bs);
// activations (bf16 or fp32 rows of K) -> residual NVFP4 levels.
cudaError_t launch_quantize_rows(cudaStream_t st, const void* src, bool bf16_in, int rows, int K,
                                 const QuantBuf& q);
// Tensor maps (the 128 opaque bytes cuTensorMapEncodeTiled writes) over a
// device region of n experts, codes [n][Bw] and scales [n][Bs], each viewed
// as 2-D row arrays for the grouped MMA's weight tiles: w13 (rows of H/2
// bytes; expert v's W13 = rows [3I v, 3I v + 2I)), w2 (rows of I/2 bytes;
// its W2 = rows [3H v + 2H, 3H (v + 1))), and the matching scale views s13
// (rows of H/16 bytes) and s2 (rows of I/16 bytes).  ok is false when the
// shape has no such views (H or I not a multiple of 256) or encoding failed;
// the grouped MMA then stages its operands with cp.async.
struct alignas(64) TmaMap {
  unsigned char b[128];
};
struct TmaSource {
  TmaMap w13, w2, s13, s2;
  const uint8_t* base_w = nullptr;
  const uint8_t* base_s = nullptr;
  unsigned long long n = 0;
  int grid = 0;  // persistent CTAs (one per SM)
  bool ok = false;
};
bool make_tma_source(const uint8_t* w, const uint8_t* s, unsigned long long n, int H, int I,
                     long long Bw, long long Bs, int num_sms, TmaSource* out);

// grouped tcgen05 expert matmuls: gate/up + SwiGLU -> h [P][I], or down -> y [P][H].
// Jobs of groups [g0, g1) (all groups: g0 = 0, g1 = INT_MAX).  With tma (ok)
// the weight tiles of experts in its region come by TMA and a persistent grid
// takes the (job, tile) items; experts elsewhere (host memory) are staged with
// cp.async by grid_x CTAs per weight tile, launched too when tma is null or
// maybe_host says the step may read host memory (a device-side bypass).  Both
// kernels give the same bits.
bool mma_supported(int H, int I);
cudaError_t launch_grouped_mma(cudaStream_t st, const GroupPlan* gp, int grid_x, bool gate_up,
                               int H, int I, int k, const QuantBuf& act, float* out,
                               uint32_t* flags, int g0 = 0, int g1 = 0x7FFFFFFF,
                               const TmaSource* tma = nullptr, bool maybe_host = false);
// residual-NVFP4 quantisation of the rows of src named by the members of groups [g0, g1)
cudaError_t launch_quantize_members(cudaStream_t st, const float* src, int K, const GroupPlan* gp,
                                    int g0, int g1, const QuantBuf& q, int grid);
// staged prefill: copy the experts of groups [q*C, q*C + C) host -> staging half (q & 1) and
// point the groups' weight pointers at the staged bytes
cudaError_t launch_stage_copy(cudaStream_t st, GroupPlan* gp, int q, int C, const LayerDev& L,
                              uint8_t* stage_w, uint8_t* stage_s, long long Bw, long long Bs,
                              int grid);
// out[m] = sum_j w[m,j] y[m*k+j], rank order.
cudaError_t launch_combine(cudaStream_t st, const GroupPlan* gp, const float* y, float* out,
                           int rows, int H, int k);

// miss copy host -> slot, SM kernel; reads the miss list from the plan and copies
// part `part` of `parts` of it (misses n * part / parts .. n * (part + 1) / parts).
cudaError_t launch_miss_copy(cudaStream_t st, const Plan* plan, const uint8_t* host_w,
                             const uint8_t* host_s, uint8_t* slot_w, uint8_t* slot_s,
                             long long Bw, long long Bs, int grid, int part = 0, int parts = 1);
cudaError_t launch_link_probe(cudaStream_t st, const void* src, void* dst, size_t bytes,
                              int grid);
// A step's host-buffer inputs and output moved by kernels over page-locked
// host memory's device-side addresses (lg_h, x_h, out_h); the set_* calls
// point a captured graph's nodes of those kernels at another call's buffers.
cudaError_t launch_host_in(cudaStream_t st, const float* lg_h, const uint16_t* x_h, float* lg_d,
                           uint16_t* x_d, int nl, int nx);
cudaError_t launch_host_out(cudaStream_t st, const float* out_d, float* out_h, int n);
bool is_host_in_node(const void* func);
bool is_host_out_node(const void* func);
cudaError_t set_host_in_node(cudaGraphExec_t ex, cudaGraphNode_t node, const float* lg_h,
                             const uint16_t* x_h, float* lg_d, uint16_t* x_d, int nl, int nx);
cudaError_t set_host_out_node(cudaGraphExec_t ex, cudaGraphNode_t node, const float* out_d,
                              float* out_h, int n);

// M = 1 expert path: gate/up + SwiGLU -> hbuf [k][I]; down + combine -> out [H].
struct GemvWorkspace {
  float* hbuf;        // [MOE_MAX_PICKS][I]
  float* ypart;       // [MOE_MAX_TOPK][H]
  uint32_t* tile_cnt; // step counters (kStepCounterWords words, laid out below)
  uint32_t* flags;    // error flags word for waits (per layer stats flags)
};
// Pick subsets of a one-row step: the picks resident at step start, the
// missed picks, or all picks.
enum PickSubset { kPicksHit = 0, kPicksMiss = 1, kPicksAll = 2 };
// Where a one-row step's expert pointers may point: expert i of the layer's
// host bank is host_w + i*Bw (and host_s + i*Bs), i < host_n; slot v of its
// ring is slot_w + v*Bw, v < slot_n.  The kernels check every pointer the plan
// hands them against these before they address memory (MOE_FLAG_BAD_PLAN and
// no access on a failure).  A null slot_w / host_w leaves that range
// unchecked (the no-allocation pass, whose experts are the caller's).
struct PickBounds {
  const uint8_t* slot_w = nullptr;
  const uint8_t* slot_s = nullptr;
  const uint8_t* host_w = nullptr;
  const uint8_t* host_s = nullptr;
  unsigned long long slot_n = 0, host_n = 0;
  long long Bw = 0, Bs = 0;
};
struct GemvLaunch {
  int subset;      // PickSubset
  bool from_host;  // read-through launch only: the picks come from host memory
  int grid;        // CTAs (0: the kernel's default, a full persistent grid)
  int stages;      // units in flight per CTA (0: as many as fit)
  bool pdl = false;  // gate/up and down launches: programmatic dependent launch
                     // on the previous kernel of their stream (see pdl_wait)
  PickBounds bounds{};
};
// Counters of a one-row step:
//   [kWorkCtr] read-through units taken,
//   [kBlockCtr + b] (pick, row) pairs whose y'_j row of output block b
//   (kOutBlockRows rows) is written: zero between steps, reset by the CTA that
//   combines the block,
//   [kHCtr + jl] gate/up units of missed pick jl whose h rows are written
//   (read-through).
// The work and h counters are cleared by the step's route/remap (clear_link_ctr),
// which completes before the read-through starts.
constexpr int kOutBlockRows = 32;
constexpr int kWorkCtr = 0;
constexpr int kBlockCtr = 1;
constexpr int kHCtr = 1 + MOE_MAX_DIM / kOutBlockRows;
constexpr int kStepCounterWords = kHCtr + MOE_MAX_TOPK;
cudaError_t launch_gemv_gateup(cudaStream_t st, const Plan* plan, const uint16_t* x, int H, int I,
                               int k, const GemvWorkspace& ws, uint32_t* flags, int num_sms,
                               const GemvLaunch& how);
// The missed picks' host-link pass (subset kPicksMiss, from_host): each
// missed expert read once from host memory and written through to its slot;
// gate/up + SwiGLU computed on its W13 rows on the way in -> ws.hbuf, then
// its W2 rows reduced on the way in -> ws.ypart, counted for their output
// blocks (combined into out by whichever launch completes a block).  Takes
// its work from ctr[kWorkCtr]; the step's route/remap has cleared that and the h
// counters.
cudaError_t launch_gemv_readthrough(cudaStream_t st, const Plan* plan, const uint16_t* x, int H,
                                    int I, int k, const GemvWorkspace& ws, uint32_t* flags,
                                    int num_sms, const GemvLaunch& how, float* out, uint32_t* ctr);
int gemv_readthrough_grid(int I, int k, int num_sms, const GemvLaunch& how);
// y'_j = gscale_j * w_j * (W2_j h_j) for the subset's picks -> ws.ypart [k][H], a unit
// being kOutBlockRows rows of one pick.  Each finished unit is counted in ctr[2 + b] for
// its output block b; the CTA that completes a block's count (all the step's picks, from
// this launch or the step's other down launch) adds out = sum_j y'_j over the block's rows
// in rank order and resets the count.  ctr: kStepCounterWords words, zero.
cudaError_t launch_gemv_down(cudaStream_t st, const Plan* plan, int H, int I, int k,
                             const GemvWorkspace& ws, uint32_t* flags, int num_sms,
                             const GemvLaunch& how, float* out, uint32_t* ctr);
int gemv_down_grid(int H, int num_sms, const GemvLaunch& how);
// Shapes the M = 1 expert kernels handle (dims % 128 == 0, inter / 32 a multiple or a
// divisor of 32).
bool gemv_supported(int H, int I, int k);

// Every kernel of a step asks for the maximum shared-memory carveout, so an SM
// never has to drain to re-partition L1/shared memory between kernels, and the
// step's concurrent kernels (miss copy beside the resident picks' GEMVs) can
// share SMs.  Call once per kernel function before its first launch.
template <class F>
inline cudaError_t prefer_max_shared(F* func) {
  return cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout,
                              cudaSharedmemCarveoutMaxShared);
}

// Launch with programmatic stream serialisation: the kernel may be scheduled
// while the previous kernel of the stream finishes; it must call pdl_wait()
// before touching anything that kernel writes.
template <class... KArgs, class... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ------------------------------------------------------- device helpers

#ifdef __CUDACC__

// Waits until the grid this one depends on (launch_pdl) has completed and its
// writes are visible; returns at once for a normal launch.
// Thread t of a route/remap launch: clears one of the read-through's counters
// of the step (0 <= t <= MOE_MAX_TOPK; any other t does nothing).
__device__ __forceinline__ void clear_link_ctr(uint32_t* ctr, int t) {
  if (!ctr || t < 0 || t > MOE_MAX_TOPK) return;
  if (t == 0)
    ctr[kWorkCtr] = 0u;
  else
    ctr[kHCtr + t - 1] = 0u;
}

__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lets the next kernel of the stream, if launched with launch_pdl, be
// scheduled once every CTA of this grid has started; its pdl_wait() still
// waits for this grid to complete.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;");
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Plain arrival (count one) on an mbarrier, release at CTA scope.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Waits on an mbarrier phase for at most limit_ns (default ~2 s); on timeout
// sets MOE_FLAG_WAIT_TIMEOUT in *flags and returns false (never traps).
constexpr uint64_t kWaitLimitNs = 2000000000ull;
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint32_t* flags,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) {
      atomicOr(flags, MOE_FLAG_WAIT_TIMEOUT);
      return false;
    }
    __nanosleep(64);
  }
}

// Waits on an mbarrier phase until it completes (true), the CTA's abort word
// is set, or the default limit runs out (MOE_FLAG_WAIT_TIMEOUT); false in both
// of the latter cases.
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t* bar, uint32_t parity,
                                                   const volatile int* abort_word,
                                                   uint32_t* flags) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_word) return false;
    if (global_ns() - t0 > kWaitLimitNs) {
      atomicOr(flags, MOE_FLAG_WAIT_TIMEOUT);
      return false;
    }
    __nanosleep(64);
  }
}

// A plan's wait limit in nanoseconds (Plan::wait_us; 0: the default).
__device__ __forceinline__ uint64_t plan_wait_ns(const Plan* plan) {
  const uint32_t us = plan->wait_us;
  return us ? (uint64_t)us * 1000ull : kWaitLimitNs;
}

// Index check on plan data one kernel hands to the next: false (and the sticky
// MOE_FLAG_BAD_PLAN set in *flags) when cond fails, so the caller skips the
// access instead of touching memory outside its buffers.
__device__ __forceinline__ bool plan_ok(bool cond, uint32_t* flags) {
  if (!cond) {
    if (flags) atomicOr(flags, MOE_FLAG_BAD_PLAN);
    __threadfence_system();
  }
  return cond;
}

// Waits (acquire, at most limit_ns, default ~2 s) until the global counter
// *ctr reaches target; on timeout sets MOE_FLAG_WAIT_TIMEOUT in *flags and
// returns false.
__device__ __forceinline__ bool count_wait_bounded(const uint32_t* ctr, uint32_t target,
                                                   uint32_t* flags,
                                                   uint64_t limit_ns = kWaitLimitNs) {
  const uint64_t t0 = global_ns();
  while (true) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v >= target) return true;
    if (global_ns() - t0 > limit_ns) {
      atomicOr(flags, MOE_FLAG_WAIT_TIMEOUT);
      return false;
    }
    __nanosleep(128);
  }
}

// 1-D bulk copy global -> this CTA's shared memory, completion counted on bar.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// 16-byte streaming load that does not allocate in L1 (host or device memory).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Two E2M1 codes (element 2i in the low nibble) -> two floats, exact.
__device__ __forceinline__ float2 e2m1x2_to_float2(uint32_t byte) {
  __half2_raw r = __nv_cvt_fp4x2_to_halfraw2(static_cast<__nv_fp4x2_storage_t>(byte), __NV_E2M1);
  __half2 h = *reinterpret_cast<__half2*>(&r);
  return __half22float2(h);
}

// Two E4M3 bytes (first in the low byte) -> two floats, exact.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two) {
  __half2_raw r =
      __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two & 0xFFFFu), __NV_E4M3);
  __half2 h = *reinterpret_cast<__half2*>(&r);
  return __half22float2(h);
}

// Expert pointer check: p == base + i * stride for some i < n (base null:
// unchecked).
__device__ __forceinline__ bool expert_ptr_ok(const uint8_t* p, const uint8_t* base,
                                              unsigned long long n, long long stride) {
  if (!base) return p != nullptr;
  if (p < base || stride <= 0) return false;
  const unsigned long long off = (unsigned long long)(p - base);
  return off % (unsigned long long)stride == 0 && off / (unsigned long long)stride < n;
}

// One pick's plan entries for a one-row kernel: j indexes the step's picks,
// its slot pointers lie in the ring and (host) its backing pointers in the bank.
__device__ __forceinline__ bool pick_ok_v(int j, int npicks, const uint8_t* w, const uint8_t* s,
                                          const uint8_t* hw, const uint8_t* hs,
                                          const PickBounds& b, bool host) {
  if (j < 0 || j >= npicks || j >= MOE_MAX_TOPK) return false;
  if (!expert_ptr_ok(w, b.slot_w, b.slot_n, b.Bw) || !expert_ptr_ok(s, b.slot_s, b.slot_n, b.Bs))
    return false;
  return !host || (expert_ptr_ok(hw, b.host_w, b.host_n, b.Bw) &&
                   expert_ptr_ok(hs, b.host_s, b.host_n, b.Bs));
}

__device__ __forceinline__ bool pick_ok(const Plan* plan, int j, int npicks,
                                        const PickBounds& b, bool host) {
  if (j < 0 || j >= npicks || j >= MOE_MAX_TOPK) return false;
  return pick_ok_v(j, npicks, plan->wptr[j], plan->sptr[j], host ? plan->hwptr[j] : nullptr,
                   host ? plan->hsptr[j] : nullptr, b, host);
}

// A launch's group bound g (a group index, kHitGroups or miss_part(p, P)) for a
// step with nh hit groups of ng: a group index in [0, ng] (or above ng for "all").
__device__ __forceinline__ int resolve_group(int g, int nh, int ng) {
  if (g == kHitGroups) return nh;
  if (g <= -64) {
    const int v = -g - 64, p = v / 16, P = v % 16;
    return P > 0 ? nh + (int)((long long)(ng - nh) * p / P) : ng;
  }
  return g < 0 ? 0 : g;
}

// The subset's pick range of a one-row plan, checked: 0 <= n_hit <= npicks <=
// MOE_MAX_TOPK.  False (and no picks) when the plan fails the check.
__device__ __forceinline__ bool subset_range_v(int npicks, int n_hit, int subset, int& pbeg,
                                               int& pcnt) {
  pbeg = 0;
  pcnt = 0;
  if (npicks < 0 || npicks > MOE_MAX_TOPK || n_hit < 0 || n_hit > npicks) return false;
  pcnt = npicks;
  if (subset == kPicksHit) pcnt = n_hit;
  if (subset == kPicksMiss) {
    pbeg = n_hit;
    pcnt = npicks - n_hit;
  }
  return true;
}

__device__ __forceinline__ bool subset_range(const Plan* plan, int subset, int& pbeg, int& pcnt) {
  return subset_range_v(plan->npicks, plan->n_hit, subset, pbeg, pcnt);
}

// A one-row kernel's picks of `subset`, read by one warp in a single round of
// independent loads (every lane < MOE_MAX_TOPK loads entry `lane` of each plan
// array; the subset's picks are then gathered by shuffles) and checked.  Lane l
// < pcnt returns pick j and its entries; ok is warp-uniform and false (pcnt 0)
// when any check fails.  host: the backing pointers are loaded and checked too.
struct WarpPicks {
  int pcnt, npicks, j;
  bool ok;
  const uint8_t *w, *s, *hw, *hs;
  float gs0, gs1, gs2, wt;
};
__device__ __forceinline__ WarpPicks warp_picks(const Plan* plan, int subset,
                                                const PickBounds& b, bool host, int lane) {
  WarpPicks p;
  const int np_raw = plan->npicks, nh_raw = plan->n_hit;
  const bool in = lane < MOE_MAX_TOPK;
  const int ol = in ? plan->order[lane] : 0;
  const uint8_t* wl = in ? plan->wptr[lane] : nullptr;
  const uint8_t* sl = in ? plan->sptr[lane] : nullptr;
  const uint8_t* hwl = (in && host) ? plan->hwptr[lane] : nullptr;
  const uint8_t* hsl = (in && host) ? plan->hsptr[lane] : nullptr;
  const float g0 = in ? plan->gs[lane][0] : 0.f, g1 = in ? plan->gs[lane][1] : 0.f;
  const float g2 = in ? plan->gs[lane][2] : 0.f, wt = in ? plan->wts[lane] : 0.f;
  int pbeg = 0, pcnt = 0;
  bool ok = subset_range_v(np_raw, nh_raw, subset, pbeg, pcnt);
  p.npicks = ok ? np_raw : 0;
  const int oi = pbeg + lane;
  const int oj = __shfl_sync(0xFFFFFFFFu, ol, oi < MOE_MAX_TOPK ? oi : 0);
  int j = 0;
  if (lane < pcnt) j = subset == kPicksAll ? lane : oj;
  const int src = (j >= 0 && j < MOE_MAX_TOPK) ? j : 0;
  p.w = reinterpret_cast<const uint8_t*>(
      __shfl_sync(0xFFFFFFFFu, reinterpret_cast<unsigned long long>(wl), src));
  p.s = reinterpret_cast<const uint8_t*>(
      __shfl_sync(0xFFFFFFFFu, reinterpret_cast<unsigned long long>(sl), src));
  p.hw = reinterpret_cast<const uint8_t*>(
      __shfl_sync(0xFFFFFFFFu, reinterpret_cast<unsigned long long>(hwl), src));
  p.hs = reinterpret_cast<const uint8_t*>(
      __shfl_sync(0xFFFFFFFFu, reinterpret_cast<unsigned long long>(hsl), src));
  p.gs0 = __shfl_sync(0xFFFFFFFFu, g0, src);
  p.gs1 = __shfl_sync(0xFFFFFFFFu, g1, src);
  p.gs2 = __shfl_sync(0xFFFFFFFFu, g2, src);
  p.wt = __shfl_sync(0xFFFFFFFFu, wt, src);
  if (lane < pcnt) ok = ok && pick_ok_v(j, p.npicks, p.w, p.s, p.hw, p.hs, b, host);
  p.ok = __all_sync(0xFFFFFFFFu, ok);
  p.pcnt = p.ok ? pcnt : 0;
  p.j = j;
  return p;
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits) {
  return __uint_as_float(bits << 16);
}

#endif  // __CUDACC__

}  // namespace moe
