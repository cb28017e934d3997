// Decode expert kernels for one row (M = 1): the grouped NVFP4
// gate/up -> SwiGLU -> down pass over the k routed experts, reading only the
// bytes the plan points at (a slot, or host memory on a bypassed step).
// ("GLM 5.3 Testing: HBM Expert Allocation", "What the slot cache is": the
// expert kernel reads the same bytes as in the all-HBM case, only the index
// changes; "A correction first": 0.041 ms for the all-HBM layer under graphs.)
//
// Both kernels are HBM-bound GEMVs (~3.6 flop per weight byte) whose limit on
// CUDA cores is the instruction issue rate of FP4 decode, so the inner loops
// are built around the cheapest exact decode: the hardware E2M1x2 -> f16x2
// conversion, then products into fp32 accumulators.
//
// gate/up + SwiGLU: persistent grid, 2 CTAs per SM.  A unit is R row pairs of
// one pick (gate rows r.., up rows I+r..), contiguous in the slot; its code
// and scale rows are staged into shared memory by 1-D TMA bulk copies
// (cp.async.bulk on an mbarrier), NS units in flight per CTA.  A thread owns a
// 16-element block of every row it touches and keeps the matching 16
// activations in registers as f16 (the row is prescaled by a power of two so
// no activation overflows f16; bf16 -> f16 is then exact apart from f16
// subnormals), so each product is one mixed-precision fma.rn.f32.f16.  Row
// sums: reduce-scatter butterfly of shuffles, then a fixed-order sum across
// warps.  The epilogue writes h = silu(gate) * up in fp32.
//
// down: persistent grid, 1 CTA per SM.  A thread owns one (pick j, 32-element
// block of I) pair and keeps gscale_j * w_j * h_j for it in registers for the
// whole kernel; a unit is R2 output rows of the launch's picks, reduced per
// pick (shuffles within the pick's lanes, then its warps) into the weighted
// output y'_j.  combine: out = sum_j y'_j in rank order.
//
// Both GEMVs take a subset of the step's picks (the resident ones, the missed
// ones, or all), so a step can run the resident picks while the missed picks'
// bytes are still being copied.  A pick's computation and reduction order do
// not depend on the subset it runs in, so a cached step and an all-resident
// step give the same bits.
#include "internal.cuh"

namespace moe {
namespace {

constexpr int kGateUpRows = 4;     // row pairs per gate/up unit
constexpr int kGateUpThreads = 512;
constexpr int kDownRows = 4;       // output rows per down unit
constexpr int kDownThreads = 512;
constexpr int kSmemPerSm = 227 * 1024;

// Four E2M1 pairs of one 32-bit word -> four f16x2 (element 2i in the low half).
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t w, uint32_t& h0, uint32_t& h1,
                                                uint32_t& h2, uint32_t& h3) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
      : "r"(w));
}

// s0 += lo(c) * lo(x), s1 += hi(c) * hi(x): f16 operands, fp32 fma.
__device__ __forceinline__ void fma_f16x2_f32(uint32_t c, uint32_t x, float& s0, float& s1) {
  asm("{\n\t.reg .b16 cl, ch, xl, xh;\n\t"
      "mov.b32 {cl, ch}, %2;\n\t"
      "mov.b32 {xl, xh}, %3;\n\t"
      "fma.rn.f32.f16 %0, cl, xl, %0;\n\t"
      "fma.rn.f32.f16 %1, ch, xh, %1;\n\t}"
      : "+f"(s0), "+f"(s1)
      : "r"(c), "r"(x));
}

// 16 codes (8 bytes) times 16 f16 activations (8 f16x2 words).
__device__ __forceinline__ float dot16_f16(uint2 codes, const uint32_t* __restrict__ xh) {
  uint32_t h[8];
  e2m1x8_to_f16x8(codes.x, h[0], h[1], h[2], h[3]);
  e2m1x8_to_f16x8(codes.y, h[4], h[5], h[6], h[7]);
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int b = 0; b < 8; ++b) fma_f16x2_f32(h[b], xh[b], s0, s1);
  return s0 + s1;
}

// 16 codes (8 bytes) times 16 fp32 values.
__device__ __forceinline__ float dot16_f32(uint32_t lo, uint32_t hi, const float* __restrict__ v) {
  uint32_t h[8];
  e2m1x8_to_f16x8(lo, h[0], h[1], h[2], h[3]);
  e2m1x8_to_f16x8(hi, h[4], h[5], h[6], h[7]);
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[b]));
    s0 = fmaf(f.x, v[2 * b], s0);
    s1 = fmaf(f.y, v[2 * b + 1], s1);
  }
  return s0 + s1;
}

__device__ __forceinline__ float e4m3_to_float(uint32_t byte) {
  return e4m3x2_to_float2(byte & 0xFFu).x;
}

// Reduce-scatter V values across the 32 lanes: afterwards lane l holds the
// warp sum of value (l >> (5 - log2 V)) & (V - 1).
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

__host__ __device__ constexpr int ilog2(int v) { return v <= 1 ? 0 : 1 + ilog2(v / 2); }

// Partials of row group g (C threads) to shared memory; sum_partial adds them
// in a fixed order.
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

__device__ __forceinline__ int units_of_block(int nunits) {
  return nunits > (int)blockIdx.x ? (nunits - 1 - (int)blockIdx.x) / gridDim.x + 1 : 0;
}

// ----------------------------------------------------------- gate / up

template <int RPT, bool WARP_RED>
__global__ void __launch_bounds__(kGateUpThreads, 2)
gemv_gateup_kernel(const Plan* __restrict__ plan, const uint16_t* __restrict__ x,
                   float* __restrict__ hbuf, int H, int I, int RL, int NS, uint32_t* flags,
                   int subset) {
  constexpr int V = 2 * RPT;
  constexpr int R = kGateUpRows;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float s_xmax[kGateUpThreads / 32];
  const int C = H / 16;
  const int tid = threadIdx.x, lane = tid & 31;
  const int g = tid / C, c = tid - g * C;
  const int cb = R * H / 2, sb = R * H / 16;
  const int stage_bytes = 2 * cb + 2 * sb;
  Stages S = carve(smem, NS, stage_bytes);

  // the picks this launch covers
  int pbeg = 0, pcnt = plan->npicks;
  if (subset == kPicksHit) pcnt = plan->n_hit;
  if (subset == kPicksMiss) {
    pbeg = plan->n_hit;
    pcnt = plan->npicks - plan->n_hit;
  }
  auto pick_of = [&](int jl) { return subset == kPicksAll ? jl : plan->order[pbeg + jl]; };
  const int upp = I / R;  // units per pick
  const int nunits = pcnt * upp;
  const int my_units = units_of_block(nunits);

  auto issue = [&](int unit, int stage) {
    const int jl = unit / upp, rb = unit - jl * upp;
    const int j = pick_of(jl);
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

  // this thread's 16 activations, as f16 after a power-of-two prescale of the
  // whole row that keeps max |x| below 2^15
  float xf[16];
  float amax = 0.f;
  {
    const uint4* xp = reinterpret_cast<const uint4*>(x + c * 16);
    const uint4 a = __ldg(xp), b = __ldg(xp + 1);
    const uint32_t wds[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      xf[2 * i] = bf16_bits_to_float(wds[i] & 0xFFFFu);
      xf[2 * i + 1] = bf16_bits_to_float(wds[i] >> 16);
      amax = fmaxf(amax, fmaxf(fabsf(xf[2 * i]), fabsf(xf[2 * i + 1])));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  if (lane == 0) s_xmax[tid >> 5] = amax;
  __syncthreads();
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) amax = fmaxf(amax, s_xmax[w]);
  int e2 = 0;
  frexpf(amax, &e2);                    // amax < 2^e2
  const int xshift = e2 > 15 ? e2 - 15 : 0;
  const float xdown = ldexpf(1.0f, -xshift), xup = ldexpf(1.0f, xshift);
  uint32_t xh[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const __half2 p = __floats2half2_rn(xf[2 * i] * xdown, xf[2 * i + 1] * xdown);
    xh[i] = *reinterpret_cast<const uint32_t*>(&p);
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
      a[q] = dot16_f16(cg, xh) * e4m3_to_float(sg);
      a[RPT + q] = dot16_f16(cu, xh) * e4m3_to_float(su);
    }
    stash_partials<V, WARP_RED>(a, S.red, g, c, C, lane);
    __syncthreads();
    if (tid == 0 && i + NS < my_units) issue(unit + NS * gridDim.x, stage);
    if (tid < RL * RPT) {
      const int gg = tid / RPT, q = tid - gg * RPT;
      const int jl = unit / upp, rb = unit - jl * upp;
      const int j = pick_of(jl);
      const float gate = plan->gs[j][0] * xup * sum_partial<V, WARP_RED>(S.red, gg, q, C);
      const float up = plan->gs[j][1] * xup * sum_partial<V, WARP_RED>(S.red, gg, RPT + q, C);
      const float h = gate / (1.0f + expf(-gate)) * up;
      hbuf[(size_t)j * I + rb * R + gg + q * RL] = h;
    }
  }
}

// ---------------------------------------------------------- down + combine

template <int R2>
__global__ void __launch_bounds__(kDownThreads, 1)
gemv_down_kernel(const Plan* __restrict__ plan, const float* __restrict__ hbuf,
                 float* __restrict__ ypart, int H, int I, int NS, uint32_t* flags, int subset) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int C = I / 32;  // 32-element blocks per h row; C divides 32 or is a multiple of it
  const int kmax = plan->npicks;
  int pbeg = 0, pcnt = kmax;
  if (subset == kPicksHit) pcnt = plan->n_hit;
  if (subset == kPicksMiss) {
    pbeg = plan->n_hit;
    pcnt = kmax - plan->n_hit;
  }
  auto pick_of = [&](int jl) { return subset == kPicksAll ? jl : plan->order[pbeg + jl]; };
  // Few picks: spread each unit's rows over RL row groups so the CTA stays
  // busy (thread = (row group g, pick jl, 32-block c)); RL * pcnt <= kmax keeps
  // a stage within the room sized for all picks.
  int RL = 1;
  while (pcnt > 0 && 2 * RL * pcnt <= kmax && 2 * RL * pcnt * C <= (int)blockDim.x) RL *= 2;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per_g = pcnt * C;
  const bool active = tid < RL * per_g;
  const int g = active ? tid / per_g : 0;
  const int rem = tid - g * per_g;
  const int jl = active ? rem / C : 0, c = active ? rem - jl * C : 0;
  const int j = active ? pick_of(jl) : 0;
  const int UR = R2 * RL;                           // rows per unit
  const int cb = UR * I / 2, sb = UR * I / 16;      // per pick
  const int stage_stride = kmax * R2 * (I / 2 + I / 16);
  const int stage_bytes = pcnt * (cb + sb);
  Stages S = carve(smem, NS, stage_stride);

  const int nunits = pcnt > 0 ? H / UR : 0;
  const int my_units = units_of_block(nunits);
  const size_t w2_codes = (size_t)I * H;        // 2I rows of H/2 bytes precede W2
  const size_t w2_scales = (size_t)I * H / 8;   // 2I rows of H/16 bytes

  auto issue = [&](int unit, int stage) {
    uint8_t* dst = S.base + (size_t)stage * stage_stride;
    mbar_arrive_expect_tx(&S.full[stage], (uint32_t)stage_bytes);
    for (int q = 0; q < pcnt; ++q) {
      const int jj = pick_of(q);
      bulk_g2s(dst + q * cb, plan->wptr[jj] + w2_codes + (size_t)unit * cb, cb, &S.full[stage]);
      bulk_g2s(dst + pcnt * cb + q * sb, plan->sptr[jj] + w2_scales + (size_t)unit * sb, sb,
               &S.full[stage]);
    }
  };

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&S.full[s], 1);
    fence_mbar_init();
    *S.abort_flag = 0;
  }
  __syncthreads();
  if (tid == 0)
    for (int s = 0; s < NS && s < my_units; ++s) issue(blockIdx.x + s * gridDim.x, s);

  // gscale_j * w_j * h_j for this thread's 32 inputs, for the whole kernel
  float hv[32];
  {
    const float f = active ? plan->gs[j][2] * plan->wts[j] : 0.f;
    const float4* hp = reinterpret_cast<const float4*>(hbuf + (size_t)j * I + c * 32);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 v = active ? __ldg(hp + q) : make_float4(0.f, 0.f, 0.f, 0.f);
      hv[4 * q] = f * v.x;
      hv[4 * q + 1] = f * v.y;
      hv[4 * q + 2] = f * v.z;
      hv[4 * q + 3] = f * v.w;
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
    const uint8_t* st = S.base + (size_t)stage * stage_stride;
    float a[R2];
#pragma unroll
    for (int r = 0; r < R2; ++r) {
      a[r] = 0.f;
      if (active) {
        const int row = g + RL * r;
        const uint4 cw = *reinterpret_cast<const uint4*>(st + jl * cb + row * (I / 2) + c * 16);
        const uint32_t s2 = *reinterpret_cast<const uint16_t*>(st + pcnt * cb + jl * sb +
                                                               row * (I / 16) + c * 2);
        const float2 sc = e4m3x2_to_float2(s2);
        a[r] = dot16_f32(cw.x, cw.y, hv) * sc.x + dot16_f32(cw.z, cw.w, hv + 16) * sc.y;
      }
    }
    if (C >= 32) {
      // a (row group, pick) spans C/32 whole warps: butterfly per warp, then its warps
      const float s = warp_reduce_scatter<R2>(a, lane);
      constexpr int sh = 5 - ilog2(R2);
      if ((lane & ((1 << sh) - 1)) == 0) S.red[warp * R2 + (lane >> sh)] = s;
      __syncthreads();
      if (tid == 0 && i + NS < my_units) issue(unit + NS * gridDim.x, stage);
      if (tid < RL * pcnt * R2) {
        const int gq = tid / R2, r = tid - gq * R2;  // gq = g * pcnt + q
        const int gg = gq / pcnt, q = gq - gg * pcnt, wp = C / 32;
        float y = 0.f;
        for (int w = 0; w < wp; ++w) y += S.red[(gq * wp + w) * R2 + r];
        ypart[(size_t)pick_of(q) * H + unit * UR + gg + RL * r] = y;
      }
    } else {
      // several (row group, pick) pairs per warp: reduce within each aligned group of C lanes
#pragma unroll
      for (int r = 0; r < R2; ++r)
        for (int o = C / 2; o > 0; o >>= 1) a[r] += __shfl_xor_sync(0xFFFFFFFFu, a[r], o);
      if (active && c == 0)
#pragma unroll
        for (int r = 0; r < R2; ++r) ypart[(size_t)j * H + unit * UR + g + RL * r] = a[r];
      __syncthreads();
      if (tid == 0 && i + NS < my_units) issue(unit + NS * gridDim.x, stage);
    }
  }
}

// out[o] = sum_j y'_j[o], j in rank order.
__global__ void gemv_combine_kernel(const float* __restrict__ ypart, float* __restrict__ out, int H,
                                    int k) {
  const int o = blockIdx.x * blockDim.x + threadIdx.x;
  if (o >= H) return;
  float acc = 0.f;
  for (int j = 0; j < k; ++j) acc += ypart[(size_t)j * H + o];
  out[o] = acc;
}

// ------------------------------------------------------------- dispatch

int pow2_floor(int v) {
  int p = 1;
  while (p * 2 <= v) p *= 2;
  return p;
}

struct GateUpShape {
  int C, RL, RPT, NT, NS, smem;
  bool warp_red;
};

GateUpShape gateup_shape(int H) {
  GateUpShape s;
  const int R = kGateUpRows;
  s.C = H / 16;
  int lim = kGateUpThreads / s.C;
  if (lim < 1) lim = 1;
  if (lim > R) lim = R;
  s.RL = pow2_floor(lim);
  s.RPT = R / s.RL;
  s.NT = s.C * s.RL;
  s.warp_red = (s.C % 32) == 0;
  const int V = 2 * s.RPT;
  const int red_floats = s.warp_red ? s.RL * (s.C / 32) * V : s.NT * V;
  const int stage = 2 * R * H / 2 + 2 * R * H / 16;
  const int per_cta = kSmemPerSm / 2 - 1024;  // two CTAs per SM
  int ns = (per_cta - 16 - red_floats * 4) / stage;
  if (ns > 6) ns = 6;
  s.NS = ns;
  s.smem = ns * stage + 8 * ns + 8 + red_floats * 4;
  return s;
}

template <int RPT, bool WR>
cudaError_t run_gateup(cudaStream_t st, int grid, const GateUpShape& s, const Plan* plan,
                       const uint16_t* x, float* hbuf, int H, int I, uint32_t* flags,
                       int subset) {
  auto kern = gemv_gateup_kernel<RPT, WR>;
  static int smem_set = 0;  // raise the opt-in limit once per size (not a stream operation)
  if (s.smem > smem_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, s.smem);
    if (e == cudaSuccess) e = prefer_max_shared(kern);
    if (e != cudaSuccess) return e;
    smem_set = s.smem;
  }
  kern<<<grid, s.NT, s.smem, st>>>(plan, x, hbuf, H, I, s.RL, s.NS, flags, subset);
  return cudaGetLastError();
}

}  // namespace

bool gemv_supported(int H, int I, int k) {
  const int C = I / 32;  // a pick's threads in the down kernel: whole warps or part of one
  return H % 128 == 0 && I % 128 == 0 && H <= MOE_MAX_DIM && I <= MOE_MAX_DIM &&
         k * C <= kDownThreads && (C % 32 == 0 || 32 % C == 0) &&
         H / 16 <= kGateUpThreads * kGateUpRows;
}

int gemv_down_tile_rows(int H, int I) {
  (void)H;
  (void)I;
  return kDownRows;
}

cudaError_t launch_gemv_gateup(cudaStream_t st, const Plan* plan, const uint16_t* x, int H, int I,
                               int k, const GemvWorkspace& ws, uint32_t* flags, int num_sms,
                               int subset) {
  const GateUpShape s = gateup_shape(H);
  if (s.NS < 2 || s.NT > kGateUpThreads) return cudaErrorInvalidConfiguration;
  const int nunits = k * (I / kGateUpRows);
  const int grid = nunits < 2 * num_sms ? nunits : 2 * num_sms;
#define GU(N)                                                                                    \
  if (s.RPT == N)                                                                                \
    return s.warp_red ? run_gateup<N, true>(st, grid, s, plan, x, ws.hbuf, H, I, flags, subset) \
                      : run_gateup<N, false>(st, grid, s, plan, x, ws.hbuf, H, I, flags, subset);
  GU(1) GU(2) GU(4)
#undef GU
  return cudaErrorInvalidConfiguration;
}

cudaError_t launch_gemv_down(cudaStream_t st, const Plan* plan, int H, int I, int k,
                             const GemvWorkspace& ws, uint32_t* flags, int num_sms, int subset) {
  constexpr int R2 = kDownRows;
  if (k * (I / 32) > kDownThreads) return cudaErrorInvalidConfiguration;
  const int stage = k * (R2 * I / 2 + R2 * I / 16);
  const int red_floats = (kDownThreads / 32) * R2;
  int ns = (kSmemPerSm - 1024 - 16 - red_floats * 4) / stage;
  if (ns > 8) ns = 8;
  if (ns < 2) return cudaErrorInvalidConfiguration;
  const int smem = ns * stage + 8 * ns + 8 + red_floats * 4;
  const int nunits = H / R2;
  const int grid = nunits < num_sms ? nunits : num_sms;
  int nt = ((k * (I / 32) + 31) / 32) * 32;
  auto kern = gemv_down_kernel<R2>;
  static int smem_set = 0;
  if (smem > smem_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) e = prefer_max_shared(kern);
    if (e != cudaSuccess) return e;
    smem_set = smem;
  }
  kern<<<grid, nt, smem, st>>>(plan, ws.hbuf, ws.ypart, H, I, ns, flags, subset);
  return cudaGetLastError();
}

cudaError_t launch_gemv_combine(cudaStream_t st, const float* ypart, float* out, int H, int k) {
  static bool once = false;
  if (!once) {
    cudaError_t e = prefer_max_shared(gemv_combine_kernel);
    if (e != cudaSuccess) return e;
    once = true;
  }
  gemv_combine_kernel<<<(H + 255) / 256, 256, 0, st>>>(ypart, out, H, k);
  return cudaGetLastError();
}

}  // namespace moe
