// Router top-k + slot remap / LRU victim selection for one cached layer-step.
//
// One CTA does the whole step (the pages fuse all bookkeeping into a single
// kernel: "GLM 5.3 Testing: HBM Expert Allocation", "The build, measured ...":
// remap, miss detection and LRU in one launch instead of a dozen tiny ops).
// The layer's map, owners, last-use stamps, clock and trace head are read in
// one coalesced pass at the start (the picks' global scales as soon as the
// picks are known), all decisions are taken in shared memory, only what
// changed is written back and the counters take fire-and-forget atomics, so
// the kernel costs about one global round trip.
//
// Router ("What the slot cache is": the router chooses top-8 expert ids before
// the expert kernel; "TensorFold GLM-5.3 explained": ties break by a stable
// expert order): the E logits are ranked by (logit desc, id asc) with NaN below
// every number, as distinct 64-bit keys.  Several rows: one warp per row, k
// rounds of a warp max.  One row: the whole CTA; the k-th largest of the
// warps' maxima is a lower bound T of the k-th largest key (those maxima are k
// distinct keys), so only keys >= T can be selected, and each candidate's rank
// is its count of larger candidates.  Weights are the softmax over the k
// selected logits, the same code either way.
//
// Remap/LRU ("What the slot cache is": a miss fills an LRU-victim slot, then
// the map is updated; "TensorFold GLM-5.3 explained": the union of a round's
// experts is fetched once): U = union of all picks; resident ids are hits and
// their slots are stamped with this step's clock t; missing ids, in ascending
// expert id, take the slots not used this step with the smallest
// (stamp, slot id); |U| > S bypasses the cache (expert pointers go to host
// memory, state untouched).  The i-th miss gets the i-th smallest unused slot,
// which equals filling the misses one at a time.
//
// Indices derived from the step's own data (expert ids, group ranks, member
// and job slots) are checked before they address memory; a failed check sets
// MOE_FLAG_BAD_PLAN and skips the access.
#include "internal.cuh"
#include "router.cuh"

namespace moe {
namespace {

constexpr int kThreads = 512;
constexpr int kWords = MOE_MAX_EXPERTS / 32;

// Multi-row steps: group the picks by expert for the grouped tensor-core pass.
// Groups are the union's experts resident at step start (hits) in ascending
// id, then the others (misses) in ascending id, so the hit groups can run
// while the misses copy; members are pick indices in ascending order, jobs
// are tiles of kRowsPerJob members.  s_hpre / s_mpre: hits / misses of the
// union before each 32-expert word; n_hitu: hits in the union.  Called by
// every thread of the CTA.
__device__ void emit_groups(GroupPlan* gp, int rows, int npicks, int n_union, int n_hitu,
                            const int32_t* s_ids, const float* s_wts,
                            const uint8_t* const* s_wp, const uint8_t* const* s_sp,
                            const uint32_t* s_union, const uint32_t* s_missmask,
                            const int32_t* s_hpre, const int32_t* s_mpre, int32_t* s_pgroup,
                            int32_t* s_gcount, int32_t* s_gstart, int32_t* s_jstart,
                            const float* gscale, int E, uint32_t* fl) {
  const int tid = threadIdx.x;
  for (int g = tid; g < n_union; g += kThreads) s_gcount[g] = 0;
  __syncthreads();
  for (int p = tid; p < npicks; p += kThreads) {
    const int e = s_ids[p];
    if (!plan_ok(e >= 0 && e < E, fl)) continue;
    const uint32_t below = (1u << (e & 31)) - 1u, mw = s_missmask[e >> 5];
    const int g = ((mw >> (e & 31)) & 1u)
                      ? n_hitu + s_mpre[e >> 5] + __popc(mw & below)
                      : s_hpre[e >> 5] + __popc(s_union[e >> 5] & ~mw & below);
    if (!plan_ok(g >= 0 && g < n_union, fl)) continue;
    s_pgroup[p] = g;
    atomicAdd(&s_gcount[g], 1);
    gp->wts[p] = s_wts[p];
  }
  __syncthreads();
  if (tid == 0) {
    int m = 0, j = 0;
    for (int g = 0; g < n_union; ++g) {
      s_gstart[g] = m;
      s_jstart[g] = j;
      m += s_gcount[g];
      j += (s_gcount[g] + kRowsPerJob - 1) / kRowsPerJob;
    }
    gp->n_groups = n_union;
    gp->n_hit_groups = n_hitu;
    gp->n_jobs = j;
    gp->rows = rows;
    gp->npicks = npicks;
  }
  __syncthreads();
  for (int g = tid; g < n_union; g += kThreads) {
    int idx = 0, first = -1;
    for (int p = 0; p < npicks; ++p) {
      if (s_pgroup[p] != g) continue;
      if (plan_ok(s_gstart[g] + idx < npicks, fl)) gp->members[s_gstart[g] + idx] = p;
      ++idx;
      if (first < 0) first = p;
    }
    if (!plan_ok(first >= 0, fl)) continue;
    const int e = s_ids[first];
    if (!plan_ok(e >= 0 && e < E, fl)) continue;
    gp->g_expert[g] = e;
    gp->g_start[g] = s_gstart[g];
    gp->g_count[g] = s_gcount[g];
    gp->g_wptr[g] = s_wp[first];
    gp->g_sptr[g] = s_sp[first];
    gp->g_gs[3 * g + 0] = gscale[3 * e + 0];
    gp->g_gs[3 * g + 1] = gscale[3 * e + 1];
    gp->g_gs[3 * g + 2] = gscale[3 * e + 2];
    const int nj = (s_gcount[g] + kRowsPerJob - 1) / kRowsPerJob;
    for (int t = 0; t < nj; ++t)
      if (plan_ok(s_jstart[g] + t < npicks, fl)) gp->jobs[s_jstart[g] + t] = (g << 8) | t;
    gp->g_job[g] = s_jstart[g];
  }
  if (tid == 0 && plan_ok(n_union <= npicks, fl)) gp->g_job[n_union] = gp->n_jobs;
}

// KPL = keys per lane = ceil(E / 32) rounded up to a power of two.
template <int KPL>
__global__ void __launch_bounds__(kThreads, 1)
route_remap_kernel(const float* __restrict__ logits, int rows, int E, int k, int S, long long Bw,
                   long long Bs, LayerDev L, Plan* __restrict__ plan, int all_resident,
                   GroupPlan* __restrict__ gp) {
  __shared__ int32_t s_ids[MOE_MAX_PICKS];
  __shared__ float s_wts[MOE_MAX_PICKS];
  __shared__ int32_t s_hit[MOE_MAX_PICKS];
  __shared__ int32_t s_miss_e[MOE_MAX_PICKS];
  __shared__ int32_t s_victim[MOE_MAX_PICKS];
  __shared__ int32_t s_evicted[MOE_MAX_PICKS];
  __shared__ int32_t s_map[MOE_MAX_EXPERTS];               // expert -> slot
  __shared__ int32_t s_owner[MOE_MAX_EXPERTS];             // slot -> expert
  __shared__ unsigned long long s_key[MOE_MAX_EXPERTS];    // (stamp, slot); ~0 = used now
  __shared__ uint32_t s_union[kWords];
  __shared__ uint32_t s_missmask[kWords];
  __shared__ int32_t s_upre[kWords];                   // union ranks before each word
  __shared__ int32_t s_hpre[kWords], s_mpre[kWords];   // hits / misses of the union before it
  __shared__ const uint8_t* s_wp[MOE_MAX_PICKS];       // bytes each pick reads
  __shared__ const uint8_t* s_sp[MOE_MAX_PICKS];
  __shared__ int32_t s_pgroup[MOE_MAX_PICKS], s_gcount[MOE_MAX_PICKS];
  __shared__ int32_t s_gstart[MOE_MAX_PICKS], s_jstart[MOE_MAX_PICKS];
  __shared__ int32_t s_n_union, s_n_miss, s_n_hits, s_n_evict;
  __shared__ uint32_t s_flags, s_clock, s_trace_head;
  // one-row router
  __shared__ float s_logit[MOE_MAX_EXPERTS];
  __shared__ unsigned long long s_cand[MOE_MAX_EXPERTS];
  __shared__ unsigned long long s_gmax[kThreads / 32], s_T;
  __shared__ float s_lsel[MOE_MAX_TOPK];
  __shared__ int32_t s_ncand;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int npicks = rows * k;
  uint32_t* const fl = &L.stats->flags;  // plan index checks report here

  // the next kernel of the stream may be scheduled now (it waits for this one)
  asm volatile("griddepcontrol.launch_dependents;");
  clear_link_ctr(L.step_ctr, tid - (kThreads - 1 - MOE_MAX_TOPK));  // the last 17 threads

  // ---- state into shared memory: every global load in flight at once
  constexpr int KPT = (MOE_MAX_EXPERTS + kThreads - 1) / kThreads;
  int32_t r_map[KPT], r_owner[KPT];
  uint32_t r_stamp[KPT];
  float r_logit[KPT];
#pragma unroll
  for (int q = 0; q < KPT; ++q) {
    const int e = tid + q * kThreads;
    r_map[q] = e < E ? L.map[e] : -1;
    r_owner[q] = e < S ? L.owner[e] : -1;
    r_stamp[q] = e < S ? L.stamp[e] : 0u;
    r_logit[q] = (rows == 1 && e < E) ? logits[e] : 0.f;
  }
  const uint32_t r_clock = tid == 0 ? *L.clock : 0u;
  const uint32_t r_head = (tid == 0 && L.trace_cap) ? *L.trace_head : 0u;
  if (tid < kWords) {
    s_union[tid] = 0;
    s_missmask[tid] = 0;
  }
  if (tid == 0) {
    s_flags = 0;
    s_n_hits = 0;
    s_n_evict = 0;
    s_ncand = 0;
    s_clock = r_clock;
    s_trace_head = r_head;
  }
#pragma unroll
  for (int q = 0; q < KPT; ++q) {
    const int e = tid + q * kThreads;
    if (e < E) s_map[e] = r_map[q];
    if (e < S) {
      s_owner[e] = r_owner[q];
      s_key[e] = ((unsigned long long)r_stamp[q] << 32) | (unsigned)e;
    }
  }

  // ---- router
  if (rows == 1) {
    unsigned long long key[KPT];
    bool bad = false;
#pragma unroll
    for (int q = 0; q < KPT; ++q) {
      const int e = tid + q * kThreads;
      key[q] = 0ull;
      if (e < E) {
        const float f = r_logit[q];
        bad |= !isfinite(f);
        key[q] = route_key(f, e);
        s_logit[e] = f;
      }
    }
    unsigned long long m = key[0];
#pragma unroll
    for (int q = 1; q < KPT; ++q) m = umax64(m, key[q]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = umax64(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (lane == 0) s_gmax[warp] = m;
    if (__syncthreads_or(bad) && tid == 0) s_flags |= MOE_FLAG_NONFINITE_LOGIT;
    if (warp == 0) {  // T = k-th largest warp maximum (1: every key, if fewer warps have keys)
      const int G = min(kThreads / 32, (E + 31) / 32);
      const unsigned long long g = lane < G ? s_gmax[lane] : 0ull;
      int r = 0;
      for (int u = 0; u < G; ++u) r += s_gmax[u] > g;
      if (lane < G && r == k - 1) s_T = g;
      if (lane == 0 && G < k) s_T = 1ull;
    }
    __syncthreads();
    const unsigned long long T = s_T;
#pragma unroll
    for (int q = 0; q < KPT; ++q)
      if (key[q] >= T) s_cand[atomicAdd(&s_ncand, 1)] = key[q];
    __syncthreads();
    const int nc = s_ncand;
    for (int i = tid; i < nc; i += kThreads) {
      const unsigned long long kk = s_cand[i];
      int r = 0;
      for (int u = 0; u < nc; ++u) r += s_cand[u] > kk;
      if (r < k) {
        const int e = (int)(0xFFFFFFFFu - (uint32_t)(kk & 0xFFFFFFFFull));
        s_ids[r] = e;
        s_lsel[r] = s_logit[e];
      }
    }
    __syncthreads();
    if (warp == 0) route_weights(lane < k ? s_lsel[lane] : 0.f, k, lane, s_wts);
  } else {  // warp per row
    for (int m = warp; m < rows; m += kThreads / 32) {
      const bool bad =
          route_row<KPL>(logits + (size_t)m * E, E, k, lane, s_ids + m * k, s_wts + m * k, fl);
      if (bad && lane == 0) atomicOr(&s_flags, MOE_FLAG_NONFINITE_LOGIT);
    }
  }
  __syncthreads();
  // the picks' global scales, in flight while the remap decisions are taken
  float gs0 = 0.f, gs1 = 0.f, gs2 = 0.f;
  if (tid < npicks && plan_ok(s_ids[tid] >= 0 && s_ids[tid] < E, fl)) {
    const int e = s_ids[tid];
    gs0 = L.gscale[3 * e + 0];
    gs1 = L.gscale[3 * e + 1];
    gs2 = L.gscale[3 * e + 2];
  }

  // ---- union, hits (slot marked used), missing ids
  for (int p = tid; p < npicks; p += kThreads) {
    const int e = s_ids[p];
    if (!plan_ok(e >= 0 && e < E, fl)) continue;
    atomicOr(&s_union[e >> 5], 1u << (e & 31));
    const int v = s_map[e];
    s_hit[p] = v >= 0;
    if (v >= 0 && !plan_ok(v < S, fl)) continue;
    if (v >= 0) {
      s_key[v] = ~0ull;
      atomicAdd(&s_n_hits, 1);
    } else {
      atomicOr(&s_missmask[e >> 5], 1u << (e & 31));
    }
  }
  __syncthreads();
  if (warp == 0) {
    const int nu = __popc(s_union[lane]);
    const uint32_t mm = s_missmask[lane];
    const int nm = __popc(mm);
    int incl = nm, tot_u = nu, uincl = nu;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      const int b = __shfl_up_sync(0xFFFFFFFFu, uincl, o);
      if (lane >= o) {
        incl += a;
        uincl += b;
      }
    }
    s_upre[lane] = uincl - nu;
    s_mpre[lane] = incl - nm;
    s_hpre[lane] = (uincl - nu) - (incl - nm);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot_u += __shfl_xor_sync(0xFFFFFFFFu, tot_u, o);
    int i = incl - nm;
    uint32_t bits = mm;
    while (bits) {  // misses in ascending expert id
      const int b = __ffs(bits) - 1;
      if (plan_ok(i < MOE_MAX_PICKS, fl)) s_miss_e[i] = 32 * lane + b;
      ++i;
      bits &= bits - 1;
    }
    if (lane == 31) s_n_miss = incl;
    if (lane == 0) s_n_union = tot_u;
  }
  __syncthreads();
  const int n_union = s_n_union;
  const int n_miss = s_n_miss;
  DevStats* st = L.stats;

  if (!all_resident && n_union > S) {
    // read every expert from host memory; cache state untouched
    for (int p = tid; p < npicks; p += kThreads) {
      const int e = s_ids[p];
      if (!plan_ok(e >= 0 && e < E, fl)) continue;
      plan->ids[p] = e;
      plan->wts[p] = s_wts[p];
      plan->wptr[p] = L.host_w + (long long)e * Bw;
      plan->sptr[p] = L.host_s + (long long)e * Bs;
      s_wp[p] = plan->wptr[p];
      s_sp[p] = plan->sptr[p];
      plan->gs[p][0] = gs0;  // p == tid: npicks <= kThreads
      plan->gs[p][1] = gs1;
      plan->gs[p][2] = gs2;
      if (L.trace_cap) {
        moe_step_record_t* r = L.trace + (s_trace_head % L.trace_cap);
        r->ids[p] = e;
        r->weights[p] = s_wts[p];
        r->slot[p] = -1;
        r->hit[p] = s_hit[p];
      }
    }
    __syncthreads();
    if (gp)
      emit_groups(gp, rows, npicks, n_union, n_union - n_miss, s_ids, s_wts, s_wp, s_sp, s_union,
                  s_missmask, s_hpre, s_mpre, s_pgroup,
                  s_gcount, s_gstart, s_jstart, L.gscale, E, fl);
    if (tid == 0) {
      plan->rows = rows;
      plan->npicks = npicks;
      plan->n_union = n_union;
      plan->n_miss = 0;
      plan->bypass = 1;
      atomicAdd(&st->steps, 1ull);
      atomicAdd(&st->bypass_calls, 1ull);
      if (s_flags) atomicOr(&st->flags, s_flags);
      if (L.trace_cap) {
        moe_step_record_t* r = L.trace + (s_trace_head % L.trace_cap);
        r->clock = s_clock;
        r->rows = rows;
        r->n_union = n_union;
        r->n_miss = 0;
        r->bypass = 1;
        *L.trace_head = s_trace_head + 1u;
      }
    }
    return;
  }

  const uint32_t t = s_clock + 1u;

  // ---- victims: the n_miss smallest (stamp, slot) among slots unused this step
  if (n_miss > 0) {
    for (int v = tid; v < S; v += kThreads) {
      const unsigned long long kv = s_key[v];
      if (kv == ~0ull) continue;
      int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
      int u = 0;
      for (; u + 4 <= S; u += 4) {
        r0 += s_key[u] < kv;
        r1 += s_key[u + 1] < kv;
        r2 += s_key[u + 2] < kv;
        r3 += s_key[u + 3] < kv;
      }
      for (; u < S; ++u) r0 += s_key[u] < kv;
      const int r = r0 + r1 + r2 + r3;
      if (r < n_miss) s_victim[r] = v;
    }
  }
  __syncthreads();

  // ---- fill: evict the previous owner, then map the missing expert
  for (int i = tid; i < n_miss; i += kThreads) {
    const int e = s_miss_e[i], v = s_victim[i];
    const int ev = s_owner[v];
    if (ev >= 0) {
      L.map[ev] = -1;
      atomicAdd(&s_n_evict, 1);
    }
    L.map[e] = v;
    L.owner[v] = e;
    L.stamp[v] = t;
    s_map[e] = v;
    s_evicted[i] = ev;
    plan->miss_e[i] = e;
    plan->miss_v[i] = v;
  }
  for (int v = tid; v < S; v += kThreads)
    if (s_key[v] == ~0ull) L.stamp[v] = t;
  __syncthreads();

  // ---- per pick: the slot it reads
  moe_step_record_t* r = L.trace_cap ? L.trace + (s_trace_head % L.trace_cap) : nullptr;
  for (int p = tid; p < npicks; p += kThreads) {
    const int e = s_ids[p];
    const int v = s_map[e];
    plan->ids[p] = e;
    plan->wts[p] = s_wts[p];
    plan->wptr[p] = L.slot_w + (long long)v * Bw;
    plan->sptr[p] = L.slot_s + (long long)v * Bs;
    plan->hwptr[p] = L.host_w + (long long)e * Bw;
    plan->hsptr[p] = L.host_s + (long long)e * Bs;
    s_wp[p] = plan->wptr[p];
    s_sp[p] = plan->sptr[p];
    plan->gs[p][0] = gs0;  // p == tid: npicks <= kThreads
    plan->gs[p][1] = gs1;
    plan->gs[p][2] = gs2;
    if (r) {
      r->ids[p] = e;
      r->weights[p] = s_wts[p];
      r->slot[p] = v;
      r->hit[p] = s_hit[p];
    }
  }
  if (r) {
    for (int i = tid; i < n_miss; i += kThreads) {
      r->miss_expert[i] = s_miss_e[i];
      r->miss_slot[i] = s_victim[i];
      r->miss_evicted[i] = s_evicted[i];
    }
  }
  __syncthreads();
  if (gp)
    emit_groups(gp, rows, npicks, n_union, n_union - n_miss, s_ids, s_wts, s_wp, s_sp, s_union,
                  s_missmask, s_hpre, s_mpre, s_pgroup,
                s_gcount, s_gstart, s_jstart, L.gscale, E, fl);
  if (rows == 1 && warp == 0) {  // hits first, then misses, each in rank order (npicks <= 32)
    const bool in = lane < npicks;
    const bool hit = in && s_hit[lane];
    const uint32_t hb = __ballot_sync(0xFFFFFFFFu, hit);
    const uint32_t mb = __ballot_sync(0xFFFFFFFFu, in && !hit);
    const uint32_t below = (1u << lane) - 1u;
    if (hit) plan->order[__popc(hb & below)] = lane;
    if (in && !hit) plan->order[__popc(hb) + __popc(mb & below)] = lane;
    if (lane == 0) plan->n_hit = __popc(hb);
  }
  // bookkeeping spread over warps so no thread carries a serial tail
  if (tid == 0) {
    plan->rows = rows;
    plan->npicks = npicks;
    plan->n_union = n_union;
    plan->n_miss = n_miss;
    plan->bypass = 0;
    *L.clock = t;
  } else if (tid >= 32 && tid < 39) {
    const int c = tid - 32;
    if (c == 0) atomicAdd(&st->steps, 1ull);
    if (c == 1) atomicAdd(&st->picks, (unsigned long long)npicks);
    if (c == 2) atomicAdd(&st->hits, (unsigned long long)s_n_hits);
    if (c == 3) atomicAdd(&st->misses, (unsigned long long)n_miss);
    if (c == 4) atomicAdd(&st->evictions, (unsigned long long)s_n_evict);
    if (c == 5) atomicAdd(&st->bytes_copied, (unsigned long long)n_miss * (unsigned long long)(Bw + Bs));
    if (c == 6 && s_flags) atomicOr(&st->flags, s_flags);
  } else if (tid == 64 && r) {
    r->clock = t;
    r->rows = rows;
    r->n_union = n_union;
    r->n_miss = n_miss;
    r->bypass = 0;
    *L.trace_head = s_trace_head + 1u;
  }
}

// One row, one warp: the same decisions as route_remap_kernel's one-row path,
// without a CTA barrier.  Launched as a programmatic dependent: its launch
// overlaps the kernel before it, whose completion it waits for before any
// access.  Every global load is then issued before any is used; the top-k
// takes k rounds of a warp max (the rounds of route_row, each a pair of 32-bit
// warp reductions over the key's high and low words) and reads each selected
// logit back from its key; hits, misses (ascending id) and victims (k rounds
// at most of a warp min over the unused slots' (stamp, slot) keys, likewise)
// come from ballots and warp reductions; the bookkeeping is spread over lanes.
template <int KPL>  // keys per lane >= ceil(max(E, S) / 32)
__global__ void __launch_bounds__(32, 1)
route_one_kernel(const float* __restrict__ logits, int E, int k, int S, long long Bw, long long Bs,
                 LayerDev L, Plan* __restrict__ plan) {
  __shared__ int32_t s_map[MOE_MAX_EXPERTS];
  __shared__ int32_t s_owner[MOE_MAX_EXPERTS];
  __shared__ unsigned long long s_skey[MOE_MAX_EXPERTS];  // (stamp, slot); ~0: used this step
  __shared__ int32_t s_ids[MOE_MAX_TOPK];
  __shared__ float s_wts[MOE_MAX_TOPK];
  __shared__ int32_t s_miss_e[MOE_MAX_TOPK], s_victim[MOE_MAX_TOPK];
  asm volatile("griddepcontrol.launch_dependents;");
  // launched programmatically: nothing is read or written before the kernel
  // before this one has completed
  pdl_wait();
  const int lane = threadIdx.x;
  const unsigned full = 0xFFFFFFFFu;
  clear_link_ctr(L.step_ctr, lane - (32 - 1 - MOE_MAX_TOPK));  // lanes 15..31
  uint32_t* const fl = &L.stats->flags;
  if (lane < MOE_MAX_TOPK) {  // in range even where a failed plan check skips a write
    s_ids[lane] = 0;
    s_miss_e[lane] = 0;
    s_victim[lane] = 0;
  }
  __syncwarp();

  // ---- every global load in flight at once
  float lg[KPL];
  int32_t mp[KPL], ow[KPL];
  uint32_t sp[KPL];
#pragma unroll
  for (int q = 0; q < KPL; ++q) {
    const int e = lane + 32 * q;
    lg[q] = e < E ? logits[e] : 0.f;
    mp[q] = e < E ? L.map[e] : -1;
    ow[q] = e < S ? L.owner[e] : -1;
    sp[q] = e < S ? L.stamp[e] : 0u;
  }
  const uint32_t clk = *L.clock;
  const uint32_t head = L.trace_cap ? *L.trace_head : 0u;
#pragma unroll
  for (int q = 0; q < KPL; ++q) {
    const int e = lane + 32 * q;
    if (e < E) s_map[e] = mp[q];
    if (e < S) {
      s_owner[e] = ow[q];
      s_skey[e] = ((unsigned long long)sp[q] << 32) | (unsigned)e;
    }
  }

  // ---- router: (logit desc, id asc), k rounds of a warp max
  unsigned long long key[KPL];
  bool bad = false;
#pragma unroll
  for (int q = 0; q < KPL; ++q) {
    const int e = lane + 32 * q;
    key[q] = 0ull;
    if (e < E) {
      bad |= !isfinite(lg[q]);
      key[q] = route_key(lg[q], e);
    }
  }
  unsigned long long best = 0ull;
#pragma unroll
  for (int q = 0; q < KPL; ++q) best = umax64(best, key[q]);
  float lsel = 0.f;  // lane j < k: the j-th selected logit
  for (int j = 0; j < k; ++j) {
    // the warp's largest key: the largest high word, then the largest low
    // word among the keys that carry it (two 32-bit warp reductions)
    const uint32_t bh = (uint32_t)(best >> 32);
    const uint32_t mh = __reduce_max_sync(full, bh);
    const uint32_t ml = __reduce_max_sync(full, bh == mh ? (uint32_t)best : 0u);
    const unsigned long long w = ((unsigned long long)mh << 32) | ml;
    const int e = (int)(0xFFFFFFFFu - ml);
    if ((e & 31) == lane) {  // the owning lane drops the winner and rescans
      best = 0ull;
#pragma unroll
      for (int q = 0; q < KPL; ++q) {
        if (lane + 32 * q == e) key[q] = 0ull;
        best = umax64(best, key[q]);
      }
    }
    if (lane == 0 && plan_ok(e >= 0 && e < E, fl)) s_ids[j] = e;
    if (lane == j) lsel = key_logit(w);
  }
  route_weights(lsel, k, lane, s_wts);
  const bool any_bad = __any_sync(full, bad) != 0;
  __syncwarp();

  // the picks' global scales, in flight while the remap decisions are taken
  const int e_me = lane < k ? s_ids[lane] : 0;
  float gs0 = 0.f, gs1 = 0.f, gs2 = 0.f;
  if (lane < k && plan_ok(e_me >= 0 && e_me < E, fl)) {
    gs0 = L.gscale[3 * e_me + 0];
    gs1 = L.gscale[3 * e_me + 1];
    gs2 = L.gscale[3 * e_me + 2];
  }

  // ---- hits (slot marked used) and misses in ascending expert id
  const int v_me = lane < k ? s_map[e_me] : -1;
  const bool hit = lane < k && v_me >= 0 && plan_ok(v_me < S, fl);
  const bool miss = lane < k && v_me < 0;
  const uint32_t hitmask = __ballot_sync(full, hit), missmask = __ballot_sync(full, miss);
  if (hit) s_skey[v_me] = ~0ull;
  const int n_hits = __popc(hitmask), n_miss = __popc(missmask);
  int mrank = 0;
  for (int q = 0; q < k; ++q) {
    const int eq = __shfl_sync(full, e_me, q);
    mrank += ((missmask >> q) & 1u) && eq < e_me;
  }
  if (miss) s_miss_e[mrank] = e_me;
  __syncwarp();

  // ---- victims: the n_miss smallest (stamp, slot) among slots unused this step
  const uint32_t t = clk + 1u;
  for (int r = 0; r < n_miss; ++r) {
    unsigned long long m = ~0ull;
#pragma unroll
    for (int q = 0; q < KPL; ++q) {
      const int v = lane + 32 * q;
      if (v < S) m = umin64(m, s_skey[v]);
    }
    {  // the warp's smallest key, high word first (two 32-bit warp reductions)
      const uint32_t mh = __reduce_min_sync(full, (uint32_t)(m >> 32));
      const uint32_t ml = __reduce_min_sync(full, (uint32_t)(m >> 32) == mh ? (uint32_t)m : ~0u);
      m = ((unsigned long long)mh << 32) | ml;
    }
    const int v = (int)(m & 0xFFFFFFFFull);
    if (lane == 0 && plan_ok(m != ~0ull && v < S, fl)) {
      s_victim[r] = v;
      s_skey[v] = ~0ull;
    }
    __syncwarp();
  }

  // ---- fill: evict the previous owner, then map the missing expert
  int ev = -1;
  if (lane < n_miss) {
    const int e = s_miss_e[lane], v = s_victim[lane];
    ev = s_owner[v];
    if (ev >= 0) L.map[ev] = -1;
    L.map[e] = v;
    L.owner[v] = e;
    L.stamp[v] = t;
    s_map[e] = v;
    plan->miss_e[lane] = e;
    plan->miss_v[lane] = v;
  }
  const int n_evict = __popc(__ballot_sync(full, lane < n_miss && ev >= 0));
  if (hit) L.stamp[v_me] = t;
  __syncwarp();

  // ---- per pick: the slot it reads, the trace, the order (hits, then misses)
  moe_step_record_t* rec = L.trace_cap ? L.trace + (head % L.trace_cap) : nullptr;
  if (lane < k) {
    const int v = s_map[e_me];
    plan->ids[lane] = e_me;
    plan->wts[lane] = s_wts[lane];
    plan->wptr[lane] = L.slot_w + (long long)v * Bw;
    plan->sptr[lane] = L.slot_s + (long long)v * Bs;
    plan->hwptr[lane] = L.host_w + (long long)e_me * Bw;
    plan->hsptr[lane] = L.host_s + (long long)e_me * Bs;
    plan->gs[lane][0] = gs0;
    plan->gs[lane][1] = gs1;
    plan->gs[lane][2] = gs2;
    const uint32_t below = (1u << lane) - 1u;
    plan->order[hit ? __popc(hitmask & below) : n_hits + __popc(missmask & below)] = lane;
    if (rec) {
      rec->ids[lane] = e_me;
      rec->weights[lane] = s_wts[lane];
      rec->slot[lane] = v;
      rec->hit[lane] = hit ? 1 : 0;
    }
  }
  if (rec && lane < n_miss) {
    rec->miss_expert[lane] = s_miss_e[lane];
    rec->miss_slot[lane] = s_victim[lane];
    rec->miss_evicted[lane] = ev;
  }
  DevStats* st = L.stats;
  if (lane == 0) {
    plan->rows = 1;
    plan->npicks = k;
    plan->n_union = k;
    plan->n_miss = n_miss;
    plan->bypass = 0;
    plan->n_hit = n_hits;
    *L.clock = t;
  } else if (lane == 1) {
    atomicAdd(&st->steps, 1ull);
  } else if (lane == 2) {
    atomicAdd(&st->picks, (unsigned long long)k);
  } else if (lane == 3) {
    atomicAdd(&st->hits, (unsigned long long)n_hits);
  } else if (lane == 4) {
    atomicAdd(&st->misses, (unsigned long long)n_miss);
  } else if (lane == 5) {
    atomicAdd(&st->evictions, (unsigned long long)n_evict);
  } else if (lane == 6) {
    atomicAdd(&st->bytes_copied, (unsigned long long)n_miss * (unsigned long long)(Bw + Bs));
  } else if (lane == 7 && any_bad) {
    atomicOr(&st->flags, MOE_FLAG_NONFINITE_LOGIT);
  } else if (lane == 8 && rec) {
    rec->clock = t;
    rec->rows = 1;
    rec->n_union = k;
    rec->n_miss = n_miss;
    rec->bypass = 0;
    *L.trace_head = head + 1u;
  }
}

}  // namespace

cudaError_t launch_route_remap(cudaStream_t st, const float* logits, int rows, int E, int k,
                               int S, long long Bw, long long Bs, const LayerDev& L, Plan* plan,
                               int all_resident, GroupPlan* gp) {
  const int kpl = (E + 31) / 32;
  if (rows == 1 && !gp && k <= 32 && S <= E) {  // one row: the one-warp kernel
#define RO(N)                                                                                   \
    if (kpl <= N) {                                                                            \
      return launch_pdl(route_one_kernel<N>, dim3(1), dim3(32), 0, st, logits, E, k, S, Bw, Bs, \
                        L, plan);                                                              \
    }
    RO(1) RO(2) RO(4) RO(8) RO(16) RO(32)
#undef RO
  }
#define RR(N)                                                                                   \
  if (kpl <= N) {                                                                              \
    static bool once = false;                                                                  \
    if (!once) {                                                                               \
      cudaError_t e = prefer_max_shared(route_remap_kernel<N>);                                \
      if (e != cudaSuccess) return e;                                                          \
      once = true;                                                                             \
    }                                                                                          \
    route_remap_kernel<N><<<1, kThreads, 0, st>>>(logits, rows, E, k, S, Bw, Bs, L, plan,      \
                                                  all_resident, gp);                           \
    return cudaGetLastError();                                                                 \
  }
  RR(1) RR(2) RR(4) RR(8) RR(16) RR(32)
#undef RR
  return cudaErrorInvalidValue;
}

}  // namespace moe
