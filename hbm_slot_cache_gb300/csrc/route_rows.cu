// Routing and expert grouping for steps with more rows than the cache serves
// (prefill).  "GLM 5.3 Testing: HBM Expert Allocation", "What the slot cache
// is": prefill with M > 16 tokens bypasses to the plain UVA kernel, so no
// expert is ever unreachable because a slot set is too small.  The cache is
// not touched: every group points at the expert's host backing and the
// grouped tensor-core pass reads it zero-copy over the host link, each expert
// once for all rows that chose it.
//
// route_rows_kernel: one warp per row, the same router as cached steps.
// group_rows_kernel: one CTA builds the group plan by counting sort over the
// expert ids (groups in ascending id, members in ascending pick index).
#include "internal.cuh"
#include "router.cuh"

namespace moe {
namespace {

constexpr int kRouteThreads = 512;
constexpr int kGroupThreads = 1024;

template <int KPL>
__global__ void __launch_bounds__(kRouteThreads)
route_rows_kernel(const float* __restrict__ logits, int rows, int E, int k,
                  int32_t* __restrict__ ids, GroupPlan* __restrict__ gp, DevStats* st) {
  const int lane = threadIdx.x & 31;
  const int m = blockIdx.x * (kRouteThreads / 32) + (threadIdx.x >> 5);
  if (m >= rows) return;
  const bool bad =
      route_row<KPL>(logits + (size_t)m * E, E, k, lane, ids + (size_t)m * k, gp->wts + (size_t)m * k,
                     &st->flags);
  if (bad && lane == 0) atomicOr(&st->flags, MOE_FLAG_NONFINITE_LOGIT);
}

// Exclusive scan over the CTA (one value per thread); returns the total.
__device__ int block_exclusive_scan(int v, int* excl_out, int* s_warp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += a;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int w = lane < nw ? s_warp[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xFFFFFFFFu, wi, o);
      if (lane >= o) wi += a;
    }
    if (lane < nw) s_warp[lane] = wi - w;  // exclusive warp offsets
    if (lane == 31) s_warp[32] = wi;       // total
  }
  __syncthreads();
  *excl_out = s_warp[warp] + incl - v;
  const int total = s_warp[32];
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(kGroupThreads)
group_rows_kernel(const int32_t* __restrict__ ids, int rows, int E, int k, long long Bw,
                  long long Bs, LayerDev L, GroupPlan* __restrict__ gp) {
  extern __shared__ uint16_t s_ids[];  // [npicks]
  __shared__ int s_count[MOE_MAX_EXPERTS];
  __shared__ int s_warp[33];
  const int tid = threadIdx.x;
  const int npicks = rows * k;
  for (int e = tid; e < MOE_MAX_EXPERTS; e += blockDim.x) s_count[e] = 0;
  __syncthreads();
  for (int p = tid; p < npicks; p += blockDim.x) {
    const int e = ids[p];
    s_ids[p] = (uint16_t)e;
    atomicAdd(&s_count[e], 1);
  }
  __syncthreads();
  // one thread per expert (E <= 1024 = blockDim)
  const int e = tid;
  const int cnt = e < E ? s_count[e] : 0;
  int gidx, mstart, jstart;
  const int n_groups = block_exclusive_scan(cnt > 0 ? 1 : 0, &gidx, s_warp);
  block_exclusive_scan(cnt, &mstart, s_warp);
  const int nj = (cnt + kRowsPerJob - 1) / kRowsPerJob;
  const int n_jobs = block_exclusive_scan(nj, &jstart, s_warp);
  if (cnt > 0) {
    int idx = 0;
    for (int p = 0; p < npicks; ++p)
      if (s_ids[p] == e) gp->members[mstart + idx++] = p;
    gp->g_expert[gidx] = e;
    gp->g_start[gidx] = mstart;
    gp->g_count[gidx] = cnt;
    gp->g_wptr[gidx] = L.host_w + (long long)e * Bw;
    gp->g_sptr[gidx] = L.host_s + (long long)e * Bs;
    gp->g_gs[3 * gidx + 0] = L.gscale[3 * e + 0];
    gp->g_gs[3 * gidx + 1] = L.gscale[3 * e + 1];
    gp->g_gs[3 * gidx + 2] = L.gscale[3 * e + 2];
    for (int t = 0; t < nj; ++t) gp->jobs[jstart + t] = (gidx << 8) | t;
    gp->g_job[gidx] = jstart;
  }
  if (tid == 0) {
    gp->g_job[n_groups] = n_jobs;
    gp->n_groups = n_groups;
    gp->n_hit_groups = n_groups;  // a bypass copies nothing
    gp->n_jobs = n_jobs;
    gp->rows = rows;
    gp->npicks = npicks;
    L.stats->steps += 1;
    L.stats->bypass_calls += 1;
  }
}

}  // namespace

cudaError_t launch_route_rows(cudaStream_t st, const float* logits, int rows, int E, int k,
                              int32_t* ids, GroupPlan* gp, const LayerDev& L, long long Bw,
                              long long Bs) {
  const int per = kRouteThreads / 32;
  const int grid = (rows + per - 1) / per;
  const int kpl = (E + 31) / 32;
  cudaError_t e = cudaErrorInvalidValue;
#define RR(N)                                                                             \
  if (e == cudaErrorInvalidValue && kpl <= N) {                                           \
    route_rows_kernel<N><<<grid, kRouteThreads, 0, st>>>(logits, rows, E, k, ids, gp,     \
                                                         L.stats);                        \
    e = cudaGetLastError();                                                               \
  }
  RR(1) RR(2) RR(4) RR(8) RR(16) RR(32)
#undef RR
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(uint16_t) * (size_t)rows * k;
  static size_t smem_set = 0;
  if (smem > 48 * 1024 && smem > smem_set) {
    e = cudaFuncSetAttribute(group_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    smem_set = smem;
  }
  group_rows_kernel<<<1, kGroupThreads, smem, st>>>(ids, rows, E, k, Bw, Bs, L, gp);
  return cudaGetLastError();
}

}  // namespace moe
