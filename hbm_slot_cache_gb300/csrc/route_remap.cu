// Router top-k + slot remap / LRU victim selection for one cached layer-step.
//
// One CTA does the whole step (the pages fuse all bookkeeping into a single
// kernel: "GLM 5.3 Testing: HBM Expert Allocation", "The build, measured ...":
// remap, miss detection and LRU in one launch instead of a dozen tiny ops).
//
// Router ("What the slot cache is": the router chooses top-8 expert ids before
// the expert kernel; "TensorFold GLM-5.3 explained": ties break by a stable
// expert order): one warp per row ranks the E logits by (logit desc, id asc)
// with NaN below every number, in k rounds of a warp max over 64-bit keys.
// Weights are the softmax over the k selected logits.
//
// Remap/LRU ("What the slot cache is": a miss fills an LRU-victim slot, then
// the map is updated; "TensorFold GLM-5.3 explained": the union of a round's
// experts is fetched once): U = union of all picks; resident ids are hits and
// their slots are stamped with this step's clock t; missing ids, in ascending
// expert id, take the slots not used this step with the smallest
// (stamp, slot id); |U| > S bypasses the cache (expert pointers go to host
// memory, state untouched).  The i-th miss gets the i-th smallest unused slot,
// which equals filling the misses one at a time.
#include "internal.cuh"

namespace moe {
namespace {

constexpr int kThreads = 512;

__device__ __forceinline__ uint32_t rank_key(float f) {
  if (isnan(f)) return 0u;                       // below -inf
  uint32_t u = __float_as_uint(f == 0.0f ? 0.0f : f);  // -0 ranks as +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(kThreads, 1)
route_remap_kernel(const float* __restrict__ logits, int rows, int E, int k, int S, long long Bw,
                   long long Bs, LayerDev L, Plan* __restrict__ plan, int all_resident) {
  __shared__ int32_t s_ids[MOE_MAX_PICKS];
  __shared__ float s_wts[MOE_MAX_PICKS];
  __shared__ int32_t s_hit[MOE_MAX_PICKS];
  __shared__ int32_t s_miss_e[MOE_MAX_PICKS];
  __shared__ int32_t s_victim[MOE_MAX_PICKS];
  __shared__ int32_t s_evicted[MOE_MAX_PICKS];
  __shared__ uint32_t s_union[MOE_MAX_EXPERTS / 32];
  __shared__ uint32_t s_missmask[MOE_MAX_EXPERTS / 32];
  __shared__ int32_t s_misspre[MOE_MAX_EXPERTS / 32];
  __shared__ unsigned long long s_key[MOE_MAX_EXPERTS];
  __shared__ int32_t s_n_union, s_n_miss, s_n_hits, s_n_evict;
  __shared__ uint32_t s_flags;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int npicks = rows * k;

  if (tid == 0) {
    s_flags = 0;
    s_n_hits = 0;
    s_n_evict = 0;
  }
  if (tid < MOE_MAX_EXPERTS / 32) {
    s_union[tid] = 0;
    s_missmask[tid] = 0;
  }
  __syncthreads();

  // ---- router: warp per row
  for (int m = warp; m < rows; m += kThreads / 32) {
    const float* lr = logits + (size_t)m * E;
    unsigned long long key[MOE_MAX_EXPERTS / 32];
    bool bad = false;
#pragma unroll
    for (int i = 0; i < MOE_MAX_EXPERTS / 32; ++i) {
      const int e = lane + 32 * i;
      key[i] = 0ull;
      if (e < E) {
        const float f = lr[e];
        bad |= !isfinite(f);
        key[i] = ((unsigned long long)rank_key(f) << 32) | (0xFFFFFFFFu - (uint32_t)e);
      }
    }
    if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) atomicOr(&s_flags, MOE_FLAG_NONFINITE_LOGIT);
    for (int j = 0; j < k; ++j) {
      unsigned long long best = 0ull;
#pragma unroll
      for (int i = 0; i < MOE_MAX_EXPERTS / 32; ++i) best = key[i] > best ? key[i] : best;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, best, o);
        best = other > best ? other : best;
      }
      const int e = (int)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull));
#pragma unroll
      for (int i = 0; i < MOE_MAX_EXPERTS / 32; ++i)
        if (lane + 32 * i == e) key[i] = 0ull;
      if (lane == 0) s_ids[m * k + j] = e;
    }
    __syncwarp();
    if (lane == 0) {
      // softmax over the k selected logits; NaN counts as -inf; a logit equal
      // to the maximum contributes exactly 1
      float lmax = -INFINITY;
      for (int j = 0; j < k; ++j) {
        float l = lr[s_ids[m * k + j]];
        if (isnan(l)) l = -INFINITY;
        lmax = fmaxf(lmax, l);
      }
      float sum = 0.0f;
      for (int j = 0; j < k; ++j) {
        float l = lr[s_ids[m * k + j]];
        if (isnan(l)) l = -INFINITY;
        const float ej = (l == lmax) ? 1.0f : expf(l - lmax);
        s_wts[m * k + j] = ej;
        sum += ej;
      }
      for (int j = 0; j < k; ++j) s_wts[m * k + j] = s_wts[m * k + j] / sum;
    }
  }
  __syncthreads();

  // ---- union of the picks
  for (int p = tid; p < npicks; p += kThreads) {
    const int e = s_ids[p];
    atomicOr(&s_union[e >> 5], 1u << (e & 31));
  }
  __syncthreads();
  if (warp == 0) {
    int c = 0;
    for (int w = lane; w < MOE_MAX_EXPERTS / 32; w += 32) c += __popc(s_union[w]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
    if (lane == 0) s_n_union = c;
  }
  __syncthreads();
  const int n_union = s_n_union;
  const bool bypass = (!all_resident) && (n_union > S);

  if (bypass) {
    // read every expert from host memory; cache state untouched
    for (int p = tid; p < npicks; p += kThreads) {
      const int e = s_ids[p];
      s_hit[p] = L.map[e] >= 0;
      plan->ids[p] = e;
      plan->wts[p] = s_wts[p];
      plan->wptr[p] = L.host_w + (long long)e * Bw;
      plan->sptr[p] = L.host_s + (long long)e * Bs;
      plan->gs[p][0] = L.gscale[3 * e + 0];
      plan->gs[p][1] = L.gscale[3 * e + 1];
      plan->gs[p][2] = L.gscale[3 * e + 2];
    }
    if (tid == 0) {
      plan->rows = rows;
      plan->npicks = npicks;
      plan->n_union = n_union;
      plan->n_miss = 0;
      plan->bypass = 1;
      DevStats* st = L.stats;
      st->steps += 1;
      st->bypass_calls += 1;
      if (s_flags) atomicOr(&st->flags, s_flags);
    }
    __syncthreads();
    if (L.trace_cap && tid == 0) {
      moe_step_record_t* r = L.trace + (*L.trace_head % L.trace_cap);
      r->clock = *L.clock;
      r->rows = rows;
      r->n_union = n_union;
      r->n_miss = 0;
      r->bypass = 1;
      for (int p = 0; p < npicks; ++p) {
        r->ids[p] = s_ids[p];
        r->weights[p] = s_wts[p];
        r->slot[p] = -1;
        r->hit[p] = s_hit[p];
      }
      *L.trace_head += 1;
    }
    return;
  }

  const uint32_t t = *L.clock + 1u;

  // ---- hits: mark their slots used this step; collect missing ids
  for (int v = tid; v < S; v += kThreads)
    s_key[v] = ((unsigned long long)L.stamp[v] << 32) | (unsigned)v;
  __syncthreads();
  for (int p = tid; p < npicks; p += kThreads) {
    const int e = s_ids[p];
    const int v = L.map[e];
    s_hit[p] = v >= 0;
    if (v >= 0) {
      s_key[v] = ~0ull;  // used this step: never a victim
      atomicAdd(&s_n_hits, 1);
    } else {
      atomicOr(&s_missmask[e >> 5], 1u << (e & 31));
    }
  }
  __syncthreads();
  if (tid == 0) {
    int c = 0;
    for (int w = 0; w < MOE_MAX_EXPERTS / 32; ++w) {
      s_misspre[w] = c;
      c += __popc(s_missmask[w]);
    }
    s_n_miss = c;
  }
  __syncthreads();
  const int n_miss = s_n_miss;

  // ---- misses in ascending expert id
  for (int w = tid; w < MOE_MAX_EXPERTS / 32; w += kThreads) {
    uint32_t bits = s_missmask[w];
    int i = s_misspre[w];
    while (bits) {
      const int b = __ffs(bits) - 1;
      s_miss_e[i++] = 32 * w + b;
      bits &= bits - 1;
    }
  }
  // ---- victims: the n_miss smallest (stamp, slot) among unused slots
  if (n_miss > 0) {
    for (int v = tid; v < S; v += kThreads) {
      const unsigned long long kv = s_key[v];
      if (kv == ~0ull) continue;
      int r = 0;
      for (int u = 0; u < S; ++u) r += s_key[u] < kv;
      if (r < n_miss) s_victim[r] = v;
    }
  }
  __syncthreads();

  // ---- fill: evict the previous owner, then map the missing expert
  for (int i = tid; i < n_miss; i += kThreads) {
    const int e = s_miss_e[i], v = s_victim[i];
    const int ev = L.owner[v];
    if (ev >= 0) {
      L.map[ev] = -1;
      atomicAdd(&s_n_evict, 1);
    }
    L.map[e] = v;
    L.owner[v] = e;
    L.stamp[v] = t;
    s_evicted[i] = ev;
    plan->miss_e[i] = e;
    plan->miss_v[i] = v;
  }
  for (int v = tid; v < S; v += kThreads)
    if (s_key[v] == ~0ull) L.stamp[v] = t;
  __syncthreads();

  // ---- per pick: the slot it reads
  for (int p = tid; p < npicks; p += kThreads) {
    const int e = s_ids[p];
    const int v = L.map[e];
    plan->ids[p] = e;
    plan->wts[p] = s_wts[p];
    plan->wptr[p] = L.slot_w + (long long)v * Bw;
    plan->sptr[p] = L.slot_s + (long long)v * Bs;
    plan->gs[p][0] = L.gscale[3 * e + 0];
    plan->gs[p][1] = L.gscale[3 * e + 1];
    plan->gs[p][2] = L.gscale[3 * e + 2];
    if (L.trace_cap) {
      moe_step_record_t* r = L.trace + (*L.trace_head % L.trace_cap);
      r->ids[p] = e;
      r->weights[p] = s_wts[p];
      r->slot[p] = v;
      r->hit[p] = s_hit[p];
    }
  }
  if (L.trace_cap) {
    moe_step_record_t* r = L.trace + (*L.trace_head % L.trace_cap);
    for (int i = tid; i < n_miss; i += kThreads) {
      r->miss_expert[i] = s_miss_e[i];
      r->miss_slot[i] = s_victim[i];
      r->miss_evicted[i] = s_evicted[i];
    }
  }
  __syncthreads();
  if (tid == 0) {
    plan->rows = rows;
    plan->npicks = npicks;
    plan->n_union = n_union;
    plan->n_miss = n_miss;
    plan->bypass = 0;
    *L.clock = t;
    DevStats* st = L.stats;
    st->steps += 1;
    st->picks += (unsigned long long)npicks;
    st->hits += (unsigned long long)s_n_hits;
    st->misses += (unsigned long long)n_miss;
    st->evictions += (unsigned long long)s_n_evict;
    st->bytes_copied += (unsigned long long)n_miss * (unsigned long long)(Bw + Bs);
    if (s_flags) atomicOr(&st->flags, s_flags);
    if (L.trace_cap) {
      moe_step_record_t* r = L.trace + (*L.trace_head % L.trace_cap);
      r->clock = t;
      r->rows = rows;
      r->n_union = n_union;
      r->n_miss = n_miss;
      r->bypass = 0;
      *L.trace_head += 1;
    }
  }
}

}  // namespace

cudaError_t launch_route_remap(cudaStream_t st, const float* logits, int rows, int E, int k,
                               int S, long long Bw, long long Bs, const LayerDev& L, Plan* plan,
                               int all_resident) {
  route_remap_kernel<<<1, kThreads, 0, st>>>(logits, rows, E, k, S, Bw, Bs, L, plan,
                                             all_resident);
  return cudaGetLastError();
}

}  // namespace moe
