// Decode expert kernels for one row (M = 1): the grouped NVFP4
// gate/up -> SwiGLU -> down pass over the k routed experts.
// ("GLM 5.3 Testing: HBM Expert Allocation", "What the slot cache is": the
// expert kernel reads the same bytes as in the all-HBM case, only the index
// changes; "A correction first": 0.041 ms for the all-HBM layer under graphs.)
//
// Both kernels are HBM-bound GEMVs (~3.6 flop per weight byte) whose limit on
// CUDA cores is the instruction issue rate of FP4 decode, so the inner loops
// are built around the cheapest exact decode: the hardware E2M1x2 -> f16x2
// conversion, then products into fp32 accumulators.
//
// gate/up + SwiGLU: persistent grid.  A unit is R row pairs of one pick (gate
// rows r.., up rows I+r..), contiguous in the expert's bytes; its code and
// scale rows are staged into shared memory NS units ahead.  A thread owns a
// 16-element block of every row it touches and keeps the matching 16
// activations in registers as f16 (the row is prescaled by a power of two so
// no activation overflows f16; bf16 -> f16 is then exact apart from f16
// subnormals), so each product is one mixed-precision fma.rn.f32.f16.  Row
// sums: reduce-scatter butterfly of shuffles, then a fixed-order sum across
// warps.  The epilogue writes h = silu(gate) * up in fp32.
//
// down: persistent grid.  A thread owns one (pick j, 32-element block of I)
// pair and keeps gscale_j * w_j * h_j for it in registers for the whole
// kernel; a unit is a few output rows of the launch's picks, reduced per pick
// (shuffles within the pick's lanes, then its warps) into the weighted output
// y'_j.  The last CTA of the step's down launches to finish adds
// out = sum_j y'_j in rank order.
//
// Both GEMVs run on a subset of the step's picks (the resident ones, the
// missed ones, or all) and stage slot bytes from HBM with 1-D TMA bulk copies
// (cp.async.bulk) on an mbarrier.
//
// read-through: the missed picks take one launch that reads each missed
// expert once over the host link and uses it on the way in.  Every thread
// stages 16-byte pieces from host memory with cp.async, an mbarrier counts
// the threads' completions, and after use each stage is written through to
// the pick's victim slot.  Phase A is the gate/up kernel above on the W13
// rows; each finished unit is counted per pick.  Phase B takes the pick's W2
// rows (prefetched from the launch's start, so the link never idles): once
// the pick's count shows all its h is written, a warp per row computes y'_j,
// with the per-thread blocks and reduction tree of the down kernel.
//
// A pick's computation and reduction order do not depend on the subset, the
// source or the kernel it runs in, so a cached step and an all-resident step
// give the same bits.  Every launch that writes y'_j counts its CTAs in a
// step counter; the CTA that completes the count adds out = sum_j y'_j in
// rank order and resets the counters.
#include "internal.cuh"

namespace moe {
namespace {

constexpr int kGateUpRows = 4;     // row pairs per gate/up unit
constexpr int kGateUpThreads = 512;
constexpr int kDownUnitRows = 32;  // W2 rows per down unit (each warp takes two)
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

// 16 codes (8 bytes) times 16 fp32 values v(0..15): even elements into s0,
// odd ones into s1 (both rn fp32 FMAs, done as one packed f32x2 FMA), then
// s0 + s1.
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

template <class Get>
__device__ __forceinline__ float dot16_f32(uint32_t lo, uint32_t hi, Get v) {
  uint32_t h[8];
  e2m1x8_to_f16x8(lo, h[0], h[1], h[2], h[3]);
  e2m1x8_to_f16x8(hi, h[4], h[5], h[6], h[7]);
  uint64_t acc = 0ull;  // (s0, s1) = (+0, +0)
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[b]));
    asm("fma.rn.f32x2 %0, %1, %2, %0;"
        : "+l"(acc)
        : "l"(pack_f32x2(f.x, f.y)), "l"(pack_f32x2(v(2 * b), v(2 * b + 1))));
  }
  float s0, s1;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(s0), "=f"(s1) : "l"(acc));
  return s0 + s1;
}

// One 32-element block of a W2 row: 16 code bytes, 2 scale bytes, and the 32
// values v(0..31) of gscale * w * h.  Roundings are pinned so every kernel
// gets the same bits.
template <class Get>
__device__ __forceinline__ float w2_block(uint4 cw, uint32_t s2, Get v) {
  const float2 sc = e4m3x2_to_float2(s2);
  const float d0 = dot16_f32(cw.x, cw.y, v);
  const float d1 = dot16_f32(cw.z, cw.w, [&](int i) { return v(16 + i); });
  return __fmaf_rn(d0, sc.x, __fmul_rn(d1, sc.y));
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
// this CTA's shared memory, so none lands after the CTA is done with it.
template <bool FROM_HOST>
__device__ void drain_fills(const Stages& S, int i, int NS, int my_units, uint32_t* flags) {
  if constexpr (FROM_HOST) {
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else {
    if (threadIdx.x != 0) return;
    for (int ii = i; ii < i + NS && ii < my_units; ++ii)
      if (!mbar_wait_bounded(&S.full[ii % NS], (uint32_t)((ii / NS) & 1), flags)) return;
  }
}

__device__ __forceinline__ int units_of_block(int nunits) {
  return nunits > (int)blockIdx.x ? (nunits - 1 - (int)blockIdx.x) / gridDim.x + 1 : 0;
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}

// The mbarrier receives one arrival when all of this thread's earlier
// cp.async copies have landed (its expected count is the thread count).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

// A stage made of consecutive byte segments: segment i is n[i] bytes copied
// from src[i] (and, on write-through, to dst[i]).  Sizes are multiples of 16.
template <int NSEG>
struct Segs {
  const uint8_t* src[NSEG];
  uint8_t* dst[NSEG];
  int n[NSEG];
};

// All threads: stage the segments piece by piece (16 B) with cp.async.
template <int NSEG>
__device__ __forceinline__ void stage_from_host(uint8_t* stage, const Segs<NSEG>& sg, int nseg,
                                                uint64_t* bar) {
  int base = 0;
  for (int s = 0; s < nseg; ++s) {
    for (int off = threadIdx.x * 16; off < sg.n[s]; off += blockDim.x * 16)
      cp_async16(stage + base + off, sg.src[s] + off);
    base += sg.n[s];
  }
  cp_async_arrive(bar);
}

// All threads: write the staged segments through to their destinations.
template <int NSEG>
__device__ __forceinline__ void write_through(const uint8_t* stage, const Segs<NSEG>& sg, int nseg) {
  int base = 0;
  for (int s = 0; s < nseg; ++s) {
    for (int off = threadIdx.x * 16; off < sg.n[s]; off += blockDim.x * 16)
      *reinterpret_cast<uint4*>(sg.dst[s] + off) =
          *reinterpret_cast<const uint4*>(stage + base + off);
    base += sg.n[s];
  }
}

// Counters of one step (a small array, zero between steps):
//   [0]             CTAs of the step's y'_j launches that have finished
//   [kWorkCtr]      W2 units taken by the read-through launch
//   [kPickCtr + jl] gate/up units done for pick jl of the read-through launch
constexpr int kWorkCtr = 1;   // phase-B units taken by the read-through launch
constexpr int kPickCtr = 2;
constexpr int kMaxStagesB = 8;

// Tail of every launch that writes y'_j: count this CTA; the CTA that brings
// the count to total_ctas adds out = sum_j y'_j in rank order and resets the
// counters for the next step.
__device__ void finish_step(const Plan* __restrict__ plan, const float* __restrict__ ypart,
                            float* __restrict__ out, int H, uint32_t* ctr, int total_ctas,
                            int* s_last) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) *s_last = atomicAdd(ctr, 1u) == (uint32_t)(total_ctas - 1);
  __syncthreads();
  if (*s_last) {
    __threadfence();
    // four outputs a thread, eight picks' loads in flight at once
    const int kmax = plan->npicks;
    const int H4 = H / 4;
    const float4* __restrict__ y4 = reinterpret_cast<const float4*>(ypart);
    for (int o = threadIdx.x; o < H4; o += blockDim.x) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int j0 = 0; j0 < kmax; j0 += 8) {
        float4 v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (j0 + q < kmax) v[q] = __ldcg(y4 + (size_t)(j0 + q) * H4 + o);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (j0 + q < kmax) {
            acc.x += v[q].x;
            acc.y += v[q].y;
            acc.z += v[q].z;
            acc.w += v[q].w;
          }
      }
      reinterpret_cast<float4*>(out)[o] = acc;
    }
    if (threadIdx.x == 0) {
      ctr[0] = 0u;
      ctr[kWorkCtr] = 0u;
      for (int jj = 0; jj < kmax; ++jj) ctr[kPickCtr + jj] = 0u;
    }
  }
}

// One W2 row, one warp: y = sum over the row's 32-element blocks c, each the
// partial w2_block computes, reduced in a fixed order: a butterfly over 32
// consecutive blocks, then those sums in order (I/32 >= 32); or a butterfly
// within groups of I/32 < 32 lanes.  get(m, i) returns element i of block
// lane + 32 m of gscale * w * h (block lane when I/32 < 32); nb = blocks per
// lane.  Every caller uses this function, so a pick gets the same bits in
// every kernel.
template <class Get>
__device__ __forceinline__ float w2_row_warp_g(const uint8_t* __restrict__ cw,
                                               const uint8_t* __restrict__ sc, int C, int nb,
                                               int lane, Get get) {
  if (C >= 32) {
    float y = 0.f;
#pragma unroll
    for (int m = 0; m < nb; ++m) {
      const int c = lane + 32 * m;
      float p = w2_block(*reinterpret_cast<const uint4*>(cw + c * 16),
                         *reinterpret_cast<const uint16_t*>(sc + c * 2),
                         [&](int i) { return get(m, i); });
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) p += __shfl_xor_sync(0xFFFFFFFFu, p, o);
      y += p;
    }
    return y;
  }
  float p = 0.f;
  if (lane < C)
    p = w2_block(*reinterpret_cast<const uint4*>(cw + lane * 16),
                 *reinterpret_cast<const uint16_t*>(sc + lane * 2),
                 [&](int i) { return get(0, i); });
  for (int o = C / 2; o > 0; o >>= 1) p += __shfl_xor_sync(0xFFFFFFFFu, p, o);
  return p;
}

// The same with gscale * w * h transposed in shared memory (element c*32+i at
// i*C + c, so a warp's lanes read distinct banks).
__device__ __forceinline__ float w2_row_warp(const uint8_t* __restrict__ cw,
                                             const uint8_t* __restrict__ sc,
                                             const float* __restrict__ hs, int I, int lane) {
  const int C = I / 32;
  return w2_row_warp_g(cw, sc, C, C >= 32 ? C / 32 : 1, lane,
                       [&](int m, int i) { return hs[i * C + lane + 32 * m]; });
}

// Extra arguments of the read-through launch.
struct RtArgs {
  float* ypart;     // [k][H] weighted outputs y'_j
  float* out;       // [H]
  uint32_t* ctr;    // step counters (see kPickCtr)
  int total_ctas;   // CTAs of all the step's y'_j launches
  int URB;          // W2 rows per phase-B unit
  int NSB;          // phase-B stages
  int b_off;        // byte offset of the phase-B region in dynamic shared memory
};

// ----------------------------------------------------------- gate / up

template <int RPT, bool WARP_RED, bool FROM_HOST>
__global__ void __launch_bounds__(kGateUpThreads, 2)
gemv_gateup_kernel(const Plan* __restrict__ plan, const uint16_t* __restrict__ x,
                   float* __restrict__ hbuf, int H, int I, int RL, int NS, uint32_t* flags,
                   int subset, RtArgs rt) {
  constexpr int V = 2 * RPT;
  constexpr int R = kGateUpRows;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float s_xmax[kGateUpThreads / 32];
  __shared__ int s_last;
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

  // a unit's four segments: gate codes, up codes, gate scales, up scales
  auto segs = [&](int unit) {
    const int jl = unit / upp, rb = unit - jl * upp;
    const int j = pick_of(jl);
    const uint8_t* w = FROM_HOST ? plan->hwptr[j] : plan->wptr[j];
    const uint8_t* s = FROM_HOST ? plan->hsptr[j] : plan->sptr[j];
    const size_t og = (size_t)rb * R, ou = (size_t)I + (size_t)rb * R;
    Segs<4> sg;
    sg.src[0] = w + og * (H / 2);
    sg.src[1] = w + ou * (H / 2);
    sg.src[2] = s + og * (H / 16);
    sg.src[3] = s + ou * (H / 16);
    uint8_t* dw = const_cast<uint8_t*>(plan->wptr[j]);
    uint8_t* ds = const_cast<uint8_t*>(plan->sptr[j]);
    sg.dst[0] = dw + og * (H / 2);
    sg.dst[1] = dw + ou * (H / 2);
    sg.dst[2] = ds + og * (H / 16);
    sg.dst[3] = ds + ou * (H / 16);
    sg.n[0] = sg.n[1] = cb;
    sg.n[2] = sg.n[3] = sb;
    return sg;
  };
  auto issue = [&](int unit, int stage) {  // FROM_HOST: every thread; else thread 0
    uint8_t* dst = S.base + (size_t)stage * stage_bytes;
    const Segs<4> sg = segs(unit);
    if constexpr (FROM_HOST) {
      stage_from_host(dst, sg, 4, &S.full[stage]);
    } else {
      mbar_arrive_expect_tx(&S.full[stage], (uint32_t)stage_bytes);
      int base = 0;
      for (int q = 0; q < 4; ++q) {
        bulk_g2s(dst + base, sg.src[q], sg.n[q], &S.full[stage]);
        base += sg.n[q];
      }
    }
  };

  // phase B (read-through only): W2 rows of the missed picks, URB rows a unit.
  // Units are taken in ascending order from the step's work counter, so CTAs
  // that finish phase A early take more.  Stages: NSB of its own from the
  // start (none by default: the link serves phase A first), then NSA more in
  // the phase-A stage memory once phase A is done.
  const int URB = FROM_HOST ? rt.URB : 1, NSB = FROM_HOST ? rt.NSB : 0;
  const int stage_b = URB * (I / 2 + I / 16);
  const int NSA = FROM_HOST ? min(kMaxStagesB - NSB, NS * stage_bytes / stage_b) : 0;
  const int NST = NSB + NSA;
  uint8_t* stB = smem + rt.b_off;
  uint64_t* barB = reinterpret_cast<uint64_t*>(stB + (size_t)NSB * stage_b);
  float* hs = reinterpret_cast<float*>(barB + kMaxStagesB);
  const int uppb = H / URB;
  const int nb = FROM_HOST ? pcnt * uppb : 0;
  auto stage_ptr = [&](int s) {
    return s < NSB ? stB + (size_t)s * stage_b : S.base + (size_t)(s - NSB) * stage_b;
  };
  __shared__ int s_unitB[kMaxStagesB];  // unit staged in each phase-B stage, -1: none
  __shared__ int s_nextB[2];            // by iteration parity: read after the writer moved on
  auto segs_b = [&](int unit) {
    const int jl = unit / uppb, rb = unit - jl * uppb;
    const int j = pick_of(jl);
    const size_t oc = (size_t)I * H + (size_t)rb * URB * (I / 2);
    const size_t os = (size_t)I * H / 8 + (size_t)rb * URB * (I / 16);
    Segs<2> sg;
    sg.src[0] = plan->hwptr[j] + oc;
    sg.src[1] = plan->hsptr[j] + os;
    sg.dst[0] = const_cast<uint8_t*>(plan->wptr[j]) + oc;
    sg.dst[1] = const_cast<uint8_t*>(plan->sptr[j]) + os;
    sg.n[0] = URB * (I / 2);
    sg.n[1] = URB * (I / 16);
    return sg;
  };

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&S.full[s], FROM_HOST ? blockDim.x : 1);
    for (int s = 0; s < NST; ++s) mbar_init(&barB[s], blockDim.x);
    fence_mbar_init();
    *S.abort_flag = 0;
    if (FROM_HOST) {  // this CTA's first phase-B units
      const int u0 = (int)atomicAdd(&rt.ctr[kWorkCtr], (uint32_t)NSB);
      for (int s = 0; s < kMaxStagesB; ++s) s_unitB[s] = (s < NSB && u0 + s < nb) ? u0 + s : -1;
    }
  }
  __syncthreads();
  if (FROM_HOST || tid == 0)
    for (int s = 0; s < NS && s < my_units; ++s) issue(blockIdx.x + s * gridDim.x, s);
  if constexpr (FROM_HOST)
    for (int s = 0; s < NSB; ++s)
      if (s_unitB[s] >= 0) stage_from_host(stage_ptr(s), segs_b(s_unitB[s]), 2, &barB[s]);

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

  // ---- phase A: gate/up + SwiGLU
  bool failed = false;
  for (int i = 0; i < my_units; ++i) {
    const int unit = blockIdx.x + i * gridDim.x;
    const int stage = i % NS;
    if (!mbar_wait_bounded(&S.full[stage], (uint32_t)((i / NS) & 1), flags)) *S.abort_flag = 1;
    __syncthreads();
    // read-through: the previous unit's h is written and fenced; count it for its pick
    if (FROM_HOST && tid == 0 && i > 0)
      atomicAdd(&rt.ctr[kPickCtr + (unit - gridDim.x) / upp], 1u);
    if (*S.abort_flag) {
      drain_fills<FROM_HOST>(S, i, NS, my_units, flags);
      if constexpr (!FROM_HOST) return;
      failed = true;
      break;
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
    if constexpr (FROM_HOST) write_through(st, segs(unit), 4);
    stash_partials<V, WARP_RED>(a, S.red, g, c, C, lane);
    __syncthreads();
    if ((FROM_HOST || tid == 0) && i + NS < my_units) issue(unit + NS * gridDim.x, stage);
    if (tid < RL * RPT) {
      const int gg = tid / RPT, q = tid - gg * RPT;
      const int jl = unit / upp, rb = unit - jl * upp;
      const int j = pick_of(jl);
      const float gate = plan->gs[j][0] * xup * sum_partial<V, WARP_RED>(S.red, gg, q, C);
      const float up = plan->gs[j][1] * xup * sum_partial<V, WARP_RED>(S.red, gg, RPT + q, C);
      const float h = gate / (1.0f + expf(-gate)) * up;
      hbuf[(size_t)j * I + rb * R + gg + q * RL] = h;
      if constexpr (FROM_HOST) __threadfence();
    }
  }
  if constexpr (FROM_HOST) {
  // ---- phase B (read-through): the missed picks' W2 rows -> y'_j
  __syncthreads();
  if (tid == 0 && !failed && my_units > 0)
    atomicAdd(&rt.ctr[kPickCtr + (blockIdx.x + (my_units - 1) * gridDim.x) / upp], 1u);
  if (failed) {
    // let the other CTAs' phase B run (on garbage, flagged) instead of timing out
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (tid == 0)
      for (int jl = 0; jl < pcnt; ++jl) atomicAdd(&rt.ctr[kPickCtr + jl], (uint32_t)upp);
  } else {
    // phase-A stage memory is free now: stage NSA more units there
    if (tid == 0 && NSA > 0) {
      const int u0 = (int)atomicAdd(&rt.ctr[kWorkCtr], (uint32_t)NSA);
      for (int s = NSB; s < NST; ++s) s_unitB[s] = u0 + (s - NSB) < nb ? u0 + (s - NSB) : -1;
    }
    __syncthreads();
    for (int s = NSB; s < NST; ++s)
      if (s_unitB[s] >= 0) stage_from_host(stage_ptr(s), segs_b(s_unitB[s]), 2, &barB[s]);
    const int warp = tid >> 5, nwarps = blockDim.x >> 5;
    int cur = -1;
    for (int i = 0;; ++i) {
      const int stage = i % NST;
      const int unit = s_unitB[stage];
      if (unit < 0) break;  // units are taken in order: none left for this CTA
      // the unit that refills this stage: taken now, its value used at the end
      const int taken = tid == 0 ? (int)atomicAdd(&rt.ctr[kWorkCtr], 1u) : 0;
      const int jl = unit / uppb, rb = unit - jl * uppb;
      const int j = pick_of(jl);
      if (j != cur) {  // wait until all of h_j is written, then stage gscale * w * h_j
        if (tid == 0 && !count_wait_bounded(&rt.ctr[kPickCtr + jl], (uint32_t)upp, flags))
          *S.abort_flag = 1;
        __syncthreads();
        if (*S.abort_flag) {
          asm volatile("cp.async.wait_all;" ::: "memory");
          break;
        }
        const float f = __fmul_rn(plan->gs[j][2], plan->wts[j]);
        for (int e = tid; e < I; e += blockDim.x)  // transposed: lanes read distinct banks
          hs[(e & 31) * (I / 32) + (e >> 5)] = __fmul_rn(f, __ldcg(hbuf + (size_t)j * I + e));
        cur = j;
      }
      if (!mbar_wait_bounded(&barB[stage], (uint32_t)((i / NST) & 1), flags)) *S.abort_flag = 1;
      __syncthreads();
      if (*S.abort_flag) {
        asm volatile("cp.async.wait_all;" ::: "memory");
        break;
      }
      const uint8_t* st = stage_ptr(stage);
      for (int r = warp; r < URB; r += nwarps) {
        const float y = w2_row_warp(st + r * (I / 2), st + URB * (I / 2) + r * (I / 16), hs, I, lane);
        if (lane == 0) rt.ypart[(size_t)j * H + rb * URB + r] = y;
      }
      write_through(st, segs_b(unit), 2);
      if (tid == 0) s_nextB[i & 1] = taken < nb ? taken : -1;
      __syncthreads();
      const int nxt = s_nextB[i & 1];
      if (tid == 0) s_unitB[stage] = nxt;
      if (nxt >= 0) stage_from_host(stage_ptr(stage), segs_b(nxt), 2, &barB[stage]);
    }
  }
  finish_step(plan, rt.ypart, rt.out, H, rt.ctr, rt.total_ctas, &s_last);
  }
}

// ---------------------------------------------------------------- down

// Each CTA serves one pick (CTAs b, b + pcnt, ... share pick b % pcnt), keeps
// gscale * w * h of that pick in shared memory (transposed), and walks units
// of kDownUnitRows W2 rows, a warp per row with w2_row_warp.  A unit's code and
// scale rows are contiguous in the slot and arrive by two 1-D TMA bulk copies.
template <int MB>  // h blocks a lane keeps in registers (0: read them from shared memory)
__global__ void __launch_bounds__(kDownThreads, 1)
gemv_down_kernel(const Plan* __restrict__ plan, const float* __restrict__ hbuf,
                 float* __restrict__ ypart, int H, int I, int NS, uint32_t* flags, int subset,
                 float* __restrict__ out, uint32_t* __restrict__ done, int total_ctas) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_last, s_abort;
  constexpr int UR = kDownUnitRows;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  int pbeg = 0, pcnt = plan->npicks;
  if (subset == kPicksHit) pcnt = plan->n_hit;
  if (subset == kPicksMiss) {
    pbeg = plan->n_hit;
    pcnt = plan->npicks - plan->n_hit;
  }
  const int row_b = I / 2 + I / 16;
  const int stage_b = UR * row_b;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)NS * stage_b);
  float* hs = reinterpret_cast<float*>(full + NS);
  // this CTA's pick and its share of the pick's row units
  const int jl = pcnt > 0 ? (int)blockIdx.x % pcnt : 0;
  const int q = pcnt > 0 ? (int)blockIdx.x / pcnt : 0;
  const int nq = pcnt > 0 ? ((int)gridDim.x - jl + pcnt - 1) / pcnt : 0;
  const int units = H / UR;
  const int my_units = (pcnt > 0 && q < units) ? (units - 1 - q) / nq + 1 : 0;
  const int j = pcnt > 0 ? (subset == kPicksAll ? jl : plan->order[pbeg + jl]) : 0;
  const uint8_t* wsrc = plan->wptr[j] + (size_t)I * H;     // W2 codes
  const uint8_t* ssrc = plan->sptr[j] + (size_t)I * H / 8; // W2 scales
  auto issue = [&](int i, int stage) {  // thread 0
    const int rb = q + i * nq;
    uint8_t* dst = smem + (size_t)stage * stage_b;
    mbar_arrive_expect_tx(&full[stage], (uint32_t)stage_b);
    bulk_g2s(dst, wsrc + (size_t)rb * UR * (I / 2), UR * (I / 2), &full[stage]);
    bulk_g2s(dst + UR * (I / 2), ssrc + (size_t)rb * UR * (I / 16), UR * (I / 16), &full[stage]);
  };
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
    s_abort = 0;
    for (int s = 0; s < NS && s < my_units; ++s) issue(s, s);
  }
  if (my_units > 0) {  // uniform
    const float f = __fmul_rn(plan->gs[j][2], plan->wts[j]);
    for (int e = tid; e < I; e += blockDim.x)  // transposed: lanes read distinct banks
      hs[(e & 31) * (I / 32) + (e >> 5)] = __fmul_rn(f, __ldg(hbuf + (size_t)j * I + e));
  }
  __syncthreads();
  // this lane's blocks of the pick's h, kept in registers for the whole kernel
  const int C = I / 32;
  float hv[MB > 0 ? MB : 1][32];
  if constexpr (MB > 0) {
#pragma unroll
    for (int m = 0; m < MB; ++m)
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int c = lane + 32 * m;
        hv[m][e] = (my_units > 0 && c < C) ? hs[e * C + c] : 0.f;
      }
  }
  for (int i = 0; i < my_units; ++i) {
    const int stage = i % NS;
    if (!mbar_wait_bounded(&full[stage], (uint32_t)((i / NS) & 1), flags)) s_abort = 1;
    __syncthreads();
    if (s_abort) {
      drain_fills<false>(Stages{smem, full, nullptr, nullptr}, i, NS, my_units, flags);
      break;  // still counted below, so the step's combine happens
    }
    const uint8_t* st = smem + (size_t)stage * stage_b;
    const int rb = q + i * nq;
    for (int r = warp; r < UR; r += nwarps) {
      const uint8_t* cw = st + r * (I / 2);
      const uint8_t* sc = st + UR * (I / 2) + r * (I / 16);
      float y;
      if constexpr (MB > 0)
        y = w2_row_warp_g(cw, sc, C, MB, lane, [&](int m, int e) { return hv[m][e]; });
      else
        y = w2_row_warp(cw, sc, hs, I, lane);
      if (lane == 0) ypart[(size_t)j * H + rb * UR + r] = y;
    }
    __syncthreads();
    if (tid == 0 && i + NS < my_units) issue(i + NS, stage);
  }
  finish_step(plan, ypart, out, H, done, total_ctas, &s_last);
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

GateUpShape gateup_shape(int H, int stages) {
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
  if (stages > 0 && stages < ns) ns = stages;
  s.NS = ns;
  s.smem = ns * stage + 8 * ns + 8 + red_floats * 4;
  return s;
}

// Phase-B shape of the read-through launch: W2 rows per unit (about 20 KB a
// stage), no stages of its own (the W2 stages use phase A's stage memory once
// phase A is done, so phase A has the host link to itself until then), then
// gscale * w * h of one pick in shared memory.
struct RtShape {
  int URB, NSB, b_off, smem;
};

RtShape rt_shape(const GateUpShape& s, int I) {
  RtShape r;
  const int row = I / 2 + I / 16;
  int urb = 16;
  while (urb > 4 && urb * row > 20 * 1024) urb /= 2;
  r.URB = urb;
  r.NSB = 0;
  r.b_off = (s.smem + 127) / 128 * 128;
  r.smem = r.b_off + r.NSB * urb * row + 8 * kMaxStagesB + I * 4;
  return r;
}

template <int RPT, bool WR, bool FH>
cudaError_t run_gateup(cudaStream_t st, int grid, const GateUpShape& s, int smem, const Plan* plan,
                       const uint16_t* x, float* hbuf, int H, int I, uint32_t* flags,
                       int subset, const RtArgs& rt) {
  auto kern = gemv_gateup_kernel<RPT, WR, FH>;
  static int smem_set = 0;  // raise the opt-in limit once per size (not a stream operation)
  if (smem > smem_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) e = prefer_max_shared(kern);
    if (e != cudaSuccess) return e;
    smem_set = smem;
  }
  kern<<<grid, s.NT, smem, st>>>(plan, x, hbuf, H, I, s.RL, s.NS, flags, subset, rt);
  return cudaGetLastError();
}

int gateup_grid(int I, int k, int num_sms, const GemvLaunch& how) {
  const int nunits = k * (I / kGateUpRows);
  const int grid = how.grid > 0 ? how.grid : 2 * num_sms;
  return grid < nunits ? grid : nunits;
}

template <bool FH>
cudaError_t dispatch_gateup(cudaStream_t st, int grid, const GateUpShape& s, int smem,
                            const Plan* plan, const uint16_t* x, float* hbuf, int H, int I,
                            uint32_t* flags, int subset, const RtArgs& rt) {
#define GU(N)                                                                                   \
  if (s.RPT == N)                                                                               \
    return s.warp_red                                                                           \
               ? run_gateup<N, true, FH>(st, grid, s, smem, plan, x, hbuf, H, I, flags, subset, rt) \
               : run_gateup<N, false, FH>(st, grid, s, smem, plan, x, hbuf, H, I, flags, subset, rt);
  GU(1) GU(2) GU(4)
#undef GU
  return cudaErrorInvalidConfiguration;
}

struct DownShape {
  int NS, smem, stage;
};

DownShape down_shape(int I, int stages) {
  DownShape d;
  d.stage = kDownUnitRows * (I / 2 + I / 16);
  const int per_cta = kSmemPerSm / 2 - 1024;  // room for one more CTA of another kernel
  int ns = (per_cta - I * 4 - 8 * 8) / d.stage;
  if (ns < 2) ns = (kSmemPerSm - 1024 - I * 4 - 8 * 8) / d.stage;  // large I
  if (ns > 8) ns = 8;
  if (stages > 0 && stages < ns) ns = stages;
  d.NS = ns;
  d.smem = ns * d.stage + 8 * ns + I * 4;
  return d;
}

template <int MB>
cudaError_t run_down(cudaStream_t st, int grid, const DownShape& d, const Plan* plan,
                     const GemvWorkspace& ws, int H, int I, uint32_t* flags, int subset,
                     float* out, uint32_t* done, int total_ctas) {
  auto kern = gemv_down_kernel<MB>;
  static int smem_set = 0;
  if (d.smem > smem_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, d.smem);
    if (e == cudaSuccess) e = prefer_max_shared(kern);
    if (e != cudaSuccess) return e;
    smem_set = d.smem;
  }
  kern<<<grid, kDownThreads, d.smem, st>>>(plan, ws.hbuf, ws.ypart, H, I, d.NS, flags, subset,
                                           out, done, total_ctas);
  return cudaGetLastError();
}

}  // namespace

bool gemv_supported(int H, int I, int k) {
  const int C = I / 32;  // 32-element blocks of a W2 row: whole warps of them or part of one
  return H % 128 == 0 && I % 128 == 0 && H <= MOE_MAX_DIM && I <= MOE_MAX_DIM && k >= 1 &&
         (C % 32 == 0 || 32 % C == 0) && H / 16 <= kGateUpThreads * kGateUpRows &&
         gateup_shape(H, 0).NT % 32 == 0 && down_shape(I, 0).NS >= 1;
}

cudaError_t launch_gemv_gateup(cudaStream_t st, const Plan* plan, const uint16_t* x, int H, int I,
                               int k, const GemvWorkspace& ws, uint32_t* flags, int num_sms,
                               const GemvLaunch& how) {
  const GateUpShape s = gateup_shape(H, how.stages);
  if (s.NS < 1 || s.NT > kGateUpThreads || how.from_host) return cudaErrorInvalidConfiguration;
  return dispatch_gateup<false>(st, gateup_grid(I, k, num_sms, how), s, s.smem, plan, x, ws.hbuf,
                                H, I, flags, how.subset, RtArgs{});
}

int gemv_readthrough_grid(int I, int k, int num_sms, const GemvLaunch& how) {
  return gateup_grid(I, k, num_sms, how);
}

cudaError_t launch_gemv_readthrough(cudaStream_t st, const Plan* plan, const uint16_t* x, int H,
                                    int I, int k, const GemvWorkspace& ws, uint32_t* flags,
                                    int num_sms, const GemvLaunch& how, float* out, uint32_t* ctr,
                                    int total_ctas) {
  const GateUpShape s = gateup_shape(H, how.stages);
  if (s.NS < 1 || s.NT > kGateUpThreads || !how.from_host || how.subset != kPicksMiss)
    return cudaErrorInvalidConfiguration;
  const RtShape r = rt_shape(s, I);
  RtArgs rt;
  rt.ypart = ws.ypart;
  rt.out = out;
  rt.ctr = ctr;
  rt.total_ctas = total_ctas;
  rt.URB = r.URB;
  rt.NSB = r.NSB;
  rt.b_off = r.b_off;
  return dispatch_gateup<true>(st, gemv_readthrough_grid(I, k, num_sms, how), s, r.smem, plan, x,
                               ws.hbuf, H, I, flags, how.subset, rt);
}

int gemv_down_grid(int H, int num_sms, const GemvLaunch& how) {
  (void)H;
  const int grid = how.grid > 0 ? how.grid : num_sms;
  return grid > MOE_MAX_TOPK ? grid : MOE_MAX_TOPK;  // at least one CTA per pick
}

cudaError_t launch_gemv_down(cudaStream_t st, const Plan* plan, int H, int I, int k,
                             const GemvWorkspace& ws, uint32_t* flags, int num_sms,
                             const GemvLaunch& how, float* out, uint32_t* done, int total_ctas) {
  (void)k;
  const DownShape d = down_shape(I, how.stages);
  if (d.NS < 1 || how.from_host) return cudaErrorInvalidConfiguration;  // slot bytes only
  const int grid = gemv_down_grid(H, num_sms, how);
  const int C = I / 32;  // h blocks per W2 row: in registers up to two per lane
  if (C <= 32)
    return run_down<1>(st, grid, d, plan, ws, H, I, flags, how.subset, out, done, total_ctas);
  if (C == 64)
    return run_down<2>(st, grid, d, plan, ws, H, I, flags, how.subset, out, done, total_ctas);
  return run_down<0>(st, grid, d, plan, ws, H, I, flags, how.subset, out, done, total_ctas);
}

}  // namespace moe
