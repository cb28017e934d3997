// Decode expert kernels for one row (M = 1): the grouped NVFP4
// gate/up -> SwiGLU -> down pass over the k routed experts, reading only the
// bytes the plan points at (a slot, or host memory on a bypassed step).
// ("GLM 5.3 Testing: HBM Expert Allocation", "What the slot cache is": the
// expert kernel reads the same bytes as in the all-HBM case, only the index
// changes; "A correction first": 0.041 ms for the all-HBM layer under graphs.)
//
// Design (HBM-bound GEMV, ~3.6 flop/byte):
//  - persistent grid, one CTA per SM; work is cut into units of whole weight
//    rows and handed out round-robin;
//  - each unit's code rows and scale rows are contiguous in the slot and are
//    staged into shared memory by 1-D TMA bulk copies (cp.async.bulk) on an
//    mbarrier, NS stages deep (~220 KB in flight per SM);
//  - a thread owns one 16-element block (8 code bytes + 1 scale byte) of every
//    row it touches and keeps the matching 16 activations in registers, so
//    shared memory carries each code byte once; E2M1 and E4M3 decode with the
//    hardware conversions (exact), products accumulate in fp32;
//  - row sums reduce across the row's threads with a reduce-scatter butterfly
//    of warp shuffles, then across warps in shared memory, in a fixed order.
// Gate/up unit: R row pairs of one pick (gate rows r.., up rows I+r..), whose
// epilogue writes h = silu(gate) * up.  Down unit: R2 output rows of one pick,
// writing y_j = W2_j h_j; the last of a row tile's k units (atomic ticket)
// combines out = sum_j w_j y_j in rank order.  Every order is fixed, so a
// cached step and an all-resident step give the same bits.
#include "internal.cuh"

namespace moe {
namespace {

constexpr int kMaxThreads = 512;
constexpr int kGateUpRows = 8;   // row pairs per gate/up unit
constexpr int kDownRows = 32;    // output rows per down unit
constexpr int kSmemBudget = 227 * 1024;

// 16 E2M1 codes (8 bytes, element 2i in the low nibble) times 16 fp32 values.
__device__ __forceinline__ float dot16(uint2 codes, const float* __restrict__ v) {
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const float2 f = e2m1x2_to_float2((codes.x >> (8 * b)) & 0xFFu);
    s0 = fmaf(f.x, v[2 * b], s0);
    s1 = fmaf(f.y, v[2 * b + 1], s1);
  }
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const float2 f = e2m1x2_to_float2((codes.y >> (8 * b)) & 0xFFu);
    s0 = fmaf(f.x, v[8 + 2 * b], s0);
    s1 = fmaf(f.y, v[8 + 2 * b + 1], s1);
  }
  return s0 + s1;
}

__device__ __forceinline__ float e4m3_to_float(uint32_t byte) {
  return e4m3x2_to_float2(byte & 0xFFu).x;
}

// Reduce-scatter V values across the 32 lanes: afterwards lane l holds in a[0]
// the warp sum of value (l >> (5 - log2 V)) & (V - 1).
template <int V>
__device__ __forceinline__ float warp_reduce_scatter(float (&a)[V], int lane) {
#pragma unroll
  for (int s = 0; s < 5; ++s) {
    const int o = 16 >> s;
    const int n = (V >> s) > 1 ? (V >> s) : 1;
    if (n > 1) {
      const int h = n / 2;
      const bool upper = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < h; ++i) {
        const float send = upper ? a[i] : a[i + h];
        const float keep = upper ? a[i + h] : a[i];
        a[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, o);
      }
    } else {
      a[0] += __shfl_xor_sync(0xFFFFFFFFu, a[0], o);
    }
  }
  return a[0];
}

constexpr int ilog2(int v) { return v <= 1 ? 0 : 1 + ilog2(v / 2); }

// Writes the per-thread partials `a` of row group g to `red` so that
// sum_partial(g, i) can add them in a fixed order.
template <int V, bool WARP_RED>
__device__ __forceinline__ void stash_partials(float (&a)[V], float* red, int g, int c, int C,
                                               int lane) {
  if constexpr (WARP_RED) {
    const int W = C / 32;
    const float s = warp_reduce_scatter<V>(a, lane);
    constexpr int sh = 5 - ilog2(V);
    if ((lane & ((1 << sh) - 1)) == 0) red[(g * W + (c >> 5)) * V + (lane >> sh)] = s;
  } else {
#pragma unroll
    for (int i = 0; i < V; ++i) red[(g * C + c) * V + i] = a[i];
  }
}

template <int V, bool WARP_RED>
__device__ __forceinline__ float sum_partial(const float* red, int g, int i, int C) {
  const int n = WARP_RED ? C / 32 : C;
  float s = 0.f;
  for (int w = 0; w < n; ++w) s += red[(g * n + w) * V + i];
  return s;
}

struct Stages {
  uint8_t* base;
  uint64_t* full;
  float* red;
  int* abort_flag;
};

__device__ __forceinline__ Stages carve(uint8_t* smem, int NS, int stage_bytes) {
  Stages s;
  s.base = smem;
  s.full = reinterpret_cast<uint64_t*>(smem + (size_t)NS * stage_bytes);
  s.abort_flag = reinterpret_cast<int*>(s.full + NS);
  s.red = reinterpret_cast<float*>(s.full + NS + 1);
  return s;
}

// After a timed-out wait: wait (bounded) for the fills still in flight into
// this CTA's shared memory, so none lands after the CTA exits.
__device__ void drain_fills(const Stages& S, int i, int NS, int my_units, uint32_t* flags) {
  if (threadIdx.x != 0) return;
  for (int ii = i; ii < i + NS && ii < my_units; ++ii)
    if (!mbar_wait_bounded(&S.full[ii % NS], (uint32_t)((ii / NS) & 1), flags)) return;
}

// ----------------------------------------------------------- gate / up

template <int RPT, bool WARP_RED>
__global__ void __launch_bounds__(kMaxThreads, 1)
gemv_gateup_kernel(const Plan* __restrict__ plan, const uint16_t* __restrict__ x,
                   float* __restrict__ hbuf, int H, int I, int RL, int NS, uint32_t* flags) {
  constexpr int V = 2 * RPT;
  constexpr int R = kGateUpRows;
  extern __shared__ __align__(128) uint8_t smem[];
  const int C = H / 16;
  const int tid = threadIdx.x, lane = tid & 31;
  const int g = tid / C, c = tid - g * C;
  const int cb = R * H / 2, sb = R * H / 16;
  const int stage_bytes = 2 * cb + 2 * sb;
  Stages S = carve(smem, NS, stage_bytes);

  const int upp = I / R;  // units per pick
  const int nunits = plan->npicks * upp;
  const int my_units = nunits > (int)blockIdx.x ? (nunits - 1 - (int)blockIdx.x) / gridDim.x + 1 : 0;

  auto issue = [&](int unit, int stage) {
    const int j = unit / upp, rb = unit - j * upp;
    const uint8_t* w = plan->wptr[j];
    const uint8_t* s = plan->sptr[j];
    uint8_t* dst = S.base + (size_t)stage * stage_bytes;
    mbar_arrive_expect_tx(&S.full[stage], (uint32_t)stage_bytes);
    bulk_g2s(dst, w + (size_t)rb * R * (H / 2), cb, &S.full[stage]);
    bulk_g2s(dst + cb, w + (size_t)(I + rb * R) * (H / 2), cb, &S.full[stage]);
    bulk_g2s(dst + 2 * cb, s + (size_t)rb * R * (H / 16), sb, &S.full[stage]);
    bulk_g2s(dst + 2 * cb + sb, s + (size_t)(I + rb * R) * (H / 16), sb, &S.full[stage]);
  };

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&S.full[s], 1);
    fence_mbar_init();
    *S.abort_flag = 0;
  }
  __syncthreads();
  if (tid == 0)
    for (int s = 0; s < NS && s < my_units; ++s) issue(blockIdx.x + s * gridDim.x, s);

  // this thread's 16 activations
  float xv[16];
  {
    const uint4* xp = reinterpret_cast<const uint4*>(x + c * 16);
    const uint4 a = __ldg(xp), b = __ldg(xp + 1);
    const uint32_t wds[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      xv[2 * i] = bf16_bits_to_float(wds[i] & 0xFFFFu);
      xv[2 * i + 1] = bf16_bits_to_float(wds[i] >> 16);
    }
  }

  for (int i = 0; i < my_units; ++i) {
    const int unit = blockIdx.x + i * gridDim.x;
    const int stage = i % NS;
    if (!mbar_wait_bounded(&S.full[stage], (uint32_t)((i / NS) & 1), flags)) *S.abort_flag = 1;
    __syncthreads();
    if (*S.abort_flag) {
      drain_fills(S, i, NS, my_units, flags);
      return;
    }
    const uint8_t* st = S.base + (size_t)stage * stage_bytes;
    float a[V];
#pragma unroll
    for (int q = 0; q < RPT; ++q) {
      const int r = g + q * RL;
      const uint2 cg = *reinterpret_cast<const uint2*>(st + r * (H / 2) + c * 8);
      const uint2 cu = *reinterpret_cast<const uint2*>(st + cb + r * (H / 2) + c * 8);
      const uint32_t sg = st[2 * cb + r * (H / 16) + c];
      const uint32_t su = st[2 * cb + sb + r * (H / 16) + c];
      a[q] = dot16(cg, xv) * e4m3_to_float(sg);
      a[RPT + q] = dot16(cu, xv) * e4m3_to_float(su);
    }
    stash_partials<V, WARP_RED>(a, S.red, g, c, C, lane);
    __syncthreads();
    if (tid == 0 && i + NS < my_units) issue(unit + NS * gridDim.x, stage);
    if (tid < RL * RPT) {
      const int gg = tid / RPT, q = tid - gg * RPT;
      const int j = unit / upp, rb = unit - j * upp;
      const float gate = plan->gs[j][0] * sum_partial<V, WARP_RED>(S.red, gg, q, C);
      const float up = plan->gs[j][1] * sum_partial<V, WARP_RED>(S.red, gg, RPT + q, C);
      const float h = gate / (1.0f + expf(-gate)) * up;
      hbuf[(size_t)j * I + rb * R + gg + q * RL] = h;
    }
  }
}

// ---------------------------------------------------------- down + combine

template <int RPT, bool WARP_RED>
__global__ void __launch_bounds__(kMaxThreads, 1)
gemv_down_kernel(const Plan* __restrict__ plan, const float* __restrict__ hbuf,
                 float* __restrict__ ypart, uint32_t* __restrict__ tile_cnt,
                 float* __restrict__ out, int H, int I, int RL, int NS, uint32_t* flags) {
  constexpr int V = RPT;
  constexpr int R = kDownRows;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_last;
  const int C = I / 16;
  const int tid = threadIdx.x, lane = tid & 31;
  const int g = tid / C, c = tid - g * C;
  const int cb = R * I / 2, sb = R * I / 16;
  const int stage_bytes = cb + sb;
  Stages S = carve(smem, NS, stage_bytes);

  const int k = plan->npicks;
  const int nunits = (H / R) * k;
  const int my_units = nunits > (int)blockIdx.x ? (nunits - 1 - (int)blockIdx.x) / gridDim.x + 1 : 0;
  const size_t w2_codes = (size_t)I * H;        // 2I rows of H/2 bytes precede W2
  const size_t w2_scales = (size_t)I * H / 8;   // 2I rows of H/16 bytes

  auto issue = [&](int unit, int stage) {
    const int tile = unit / k, j = unit - tile * k;
    uint8_t* dst = S.base + (size_t)stage * stage_bytes;
    mbar_arrive_expect_tx(&S.full[stage], (uint32_t)stage_bytes);
    bulk_g2s(dst, plan->wptr[j] + w2_codes + (size_t)tile * R * (I / 2), cb, &S.full[stage]);
    bulk_g2s(dst + cb, plan->sptr[j] + w2_scales + (size_t)tile * R * (I / 16), sb,
             &S.full[stage]);
  };

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&S.full[s], 1);
    fence_mbar_init();
    *S.abort_flag = 0;
  }
  __syncthreads();
  if (tid == 0)
    for (int s = 0; s < NS && s < my_units; ++s) issue(blockIdx.x + s * gridDim.x, s);

  for (int i = 0; i < my_units; ++i) {
    const int unit = blockIdx.x + i * gridDim.x;
    const int tile = unit / k, j = unit - tile * k;
    const int stage = i % NS;
    // h_j for this thread's 16 inputs (written by the gate/up kernel)
    float hv[16];
    {
      const float4* hp = reinterpret_cast<const float4*>(hbuf + (size_t)j * I + c * 16);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 v = __ldg(hp + q);
        hv[4 * q] = v.x;
        hv[4 * q + 1] = v.y;
        hv[4 * q + 2] = v.z;
        hv[4 * q + 3] = v.w;
      }
    }
    if (!mbar_wait_bounded(&S.full[stage], (uint32_t)((i / NS) & 1), flags)) *S.abort_flag = 1;
    __syncthreads();
    if (*S.abort_flag) {
      drain_fills(S, i, NS, my_units, flags);
      return;
    }
    const uint8_t* st = S.base + (size_t)stage * stage_bytes;
    float a[V];
#pragma unroll
    for (int q = 0; q < RPT; ++q) {
      const int r = g + q * RL;
      const uint2 cw = *reinterpret_cast<const uint2*>(st + r * (I / 2) + c * 8);
      const uint32_t sw = st[cb + r * (I / 16) + c];
      a[q] = dot16(cw, hv) * e4m3_to_float(sw);
    }
    stash_partials<V, WARP_RED>(a, S.red, g, c, C, lane);
    __syncthreads();
    if (tid == 0 && i + NS < my_units) issue(unit + NS * gridDim.x, stage);
    if (tid < RL * RPT) {
      const int gg = tid / RPT, q = tid - gg * RPT;
      const int row = tile * R + gg + q * RL;
      ypart[(size_t)j * H + row] = plan->gs[j][2] * sum_partial<V, WARP_RED>(S.red, gg, q, C);
      __threadfence();
    }
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(&tile_cnt[tile], 1u) == (uint32_t)(k - 1);
    __syncthreads();
    if (s_last) {
      __threadfence();
      for (int t = tid; t < R; t += blockDim.x) {
        const int row = tile * R + t;
        float acc = 0.f;
        for (int jj = 0; jj < k; ++jj) acc = fmaf(plan->wts[jj], __ldcg(ypart + (size_t)jj * H + row), acc);
        out[row] = acc;
      }
      if (tid == 0) tile_cnt[tile] = 0;
    }
  }
}

// ------------------------------------------------------------- dispatch

struct Shape {
  int C, RL, RPT, NT, NS, smem;
  bool warp_red;
};

int pow2_floor(int v) {
  int p = 1;
  while (p * 2 <= v) p *= 2;
  return p;
}

// K = inner dimension, R = rows (or row pairs) per unit, vals = partials per row
Shape plan_shape(int K, int R, int rows_per_unit_factor, int stage_bytes) {
  Shape s;
  s.C = K / 16;
  int lim = 256 / s.C;
  if (lim < 1) lim = 1;
  if (lim > R) lim = R;
  s.RL = pow2_floor(lim);
  s.RPT = R / s.RL;
  s.NT = s.C * s.RL;
  s.warp_red = (s.C % 32) == 0;
  const int V = rows_per_unit_factor * s.RPT;
  const int red_floats = s.warp_red ? s.RL * (s.C / 32) * V : s.NT * V;
  const int fixed = 16 + 8 + red_floats * 4 + 128;
  int ns = (kSmemBudget - fixed) / stage_bytes;
  if (ns > 4) ns = 4;
  s.NS = ns;
  s.smem = ns * stage_bytes + 8 * ns + 8 + red_floats * 4;
  return s;
}

template <int RPT, bool WR>
cudaError_t run_gateup(cudaStream_t st, int grid, const Shape& s, const Plan* plan,
                       const uint16_t* x, float* hbuf, int H, int I, uint32_t* flags) {
  auto kern = gemv_gateup_kernel<RPT, WR>;
  static int smem_set = 0;  // raise the opt-in limit once per size (not a stream operation)
  if (s.smem > smem_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, s.smem);
    if (e != cudaSuccess) return e;
    smem_set = s.smem;
  }
  kern<<<grid, s.NT, s.smem, st>>>(plan, x, hbuf, H, I, s.RL, s.NS, flags);
  return cudaGetLastError();
}

template <int RPT, bool WR>
cudaError_t run_down(cudaStream_t st, int grid, const Shape& s, const Plan* plan,
                     const float* hbuf, float* ypart, uint32_t* cnt, float* out, int H, int I,
                     uint32_t* flags) {
  auto kern = gemv_down_kernel<RPT, WR>;
  static int smem_set = 0;
  if (s.smem > smem_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, s.smem);
    if (e != cudaSuccess) return e;
    smem_set = s.smem;
  }
  kern<<<grid, s.NT, s.smem, st>>>(plan, hbuf, ypart, cnt, out, H, I, s.RL, s.NS, flags);
  return cudaGetLastError();
}

}  // namespace

int gemv_down_tile_rows(int H, int I) {
  (void)H;
  (void)I;
  return kDownRows;
}

cudaError_t launch_gemv_gateup(cudaStream_t st, const Plan* plan, const uint16_t* x, int H, int I,
                               int k, const GemvWorkspace& ws, uint32_t* flags, int num_sms) {
  const int R = kGateUpRows;
  const Shape s = plan_shape(H, R, 2, R * H + R * H / 8);
  if (s.NS < 2 || s.NT > kMaxThreads) return cudaErrorInvalidConfiguration;
  const int nunits = k * (I / R);
  const int grid = nunits < num_sms ? nunits : num_sms;
#define GU(N)                                                                            \
  if (s.RPT == N)                                                                        \
    return s.warp_red ? run_gateup<N, true>(st, grid, s, plan, x, ws.hbuf, H, I, flags) \
                      : run_gateup<N, false>(st, grid, s, plan, x, ws.hbuf, H, I, flags);
  GU(1) GU(2) GU(4) GU(8)
#undef GU
  return cudaErrorInvalidConfiguration;
}

cudaError_t launch_gemv_down(cudaStream_t st, const Plan* plan, int H, int I, int k,
                             const GemvWorkspace& ws, float* out, uint32_t* flags, int num_sms) {
  const int R = kDownRows;
  const Shape s = plan_shape(I, R, 1, R * I / 2 + R * I / 16);
  if (s.NS < 2 || s.NT > kMaxThreads) return cudaErrorInvalidConfiguration;
  const int nunits = (H / R) * k;
  const int grid = nunits < num_sms ? nunits : num_sms;
#define DN(N)                                                                              \
  if (s.RPT == N)                                                                          \
    return s.warp_red                                                                      \
               ? run_down<N, true>(st, grid, s, plan, ws.hbuf, ws.ypart, ws.tile_cnt, out, \
                                   H, I, flags)                                            \
               : run_down<N, false>(st, grid, s, plan, ws.hbuf, ws.ypart, ws.tile_cnt, out, \
                                    H, I, flags);
  DN(1) DN(2) DN(4) DN(8) DN(16) DN(32)
#undef DN
  return cudaErrorInvalidConfiguration;
}

}  // namespace moe
