// Decode expert kernels for one row (M = 1): the grouped NVFP4
// gate/up -> SwiGLU -> down pass over the k routed experts.
// ("GLM 5.3 Testing: HBM Expert Allocation", "What the slot cache is": the
// expert kernel reads the same bytes as in the all-HBM case, only the index
// changes; "A correction first": 0.041 ms for the all-HBM layer under graphs.)
//
// Both passes are GEMVs (~3.6 flop per weight byte) whose limit on CUDA cores
// is the instruction issue rate of FP4 decode, so the inner loops are built
// around the cheapest exact decode: the hardware E2M1x2 -> f16x2 conversion,
// then products into fp32 accumulators.
//
// gate/up + SwiGLU (resident picks): persistent grid, warp-specialised.  A
// unit is kGateUpRows row pairs of one pick (gate rows r.., up rows I+r..);
// its four segments (gate codes, up codes, gate scales, up scales) arrive by
// 1-D TMA bulk copies on the stage's mbarrier.  A compute thread owns 32
// columns of every row it touches and keeps the matching activations in
// registers as f16 (the row prescaled by a power of two so none overflows;
// bf16 -> f16 is then exact apart from f16 subnormals), so each product is
// one mixed-precision fma.rn.f32.f16.  Row sums: a reduce-scatter butterfly of
// shuffles, then a fixed-order sum across warps.  Compute warps count
// themselves in on a per-stage mbarrier without waiting; a control warp
// refills the stage and writes h = silu(gate) * up in fp32.
//
// down (resident picks): one CTA per SM serves one pick; each warp
// owns a ring of 2-row stages (TMA bulk copies) and reduces each W2 row with
// w2_row_warp_g against gscale_j * w_j * h_j held in registers, writing the
// weighted output y'_j.  At exit a CTA counts its 32-row output blocks; the CTA
// that completes a block's count over all the step's picks adds that block of
// out = sum_j y'_j in rank order.
//
// read-through (missed picks): one launch reads each missed expert once over
// the host link.  Its work list (units taken one at a time from a step
// counter) holds each missed pick's gate/up units, computed on arrival with
// the functions the resident gate/up uses, then the pick's W2 bytes as copy
// units, each reduced on arrival against the pick's h; every unit is written
// through to the pick's victim slot.  Every thread stages 16-byte pieces from
// host memory with cp.async and an mbarrier counts the threads' completions.
//
// A pick's computation and reduction order do not depend on the subset, the
// source or the kernel it runs in, so a cached step and an all-resident step
// give the same bits.
#include "internal.cuh"

namespace moe {
namespace {

constexpr int kGateUpRows = 4;     // row pairs per gate/up unit
constexpr int kGateUpThreads = 512;
constexpr int kDownUnitRows = kOutBlockRows;  // W2 rows per down unit
constexpr int kDownItemRows = 2;              // W2 rows a down warp takes at a time
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

constexpr int kMaxStages = 8;  // gate/up stages at most

// The plan, h and the partial outputs y' are written by a grid that may still
// be running when a kernel here reads them (a programmatic launch reads them
// after its dependency wait; the per-block combine reads other CTAs' y'), so
// they carry no __restrict__: with it the compiler may read them through the
// non-coherent path or move a load ahead of the wait.

// Output blocks are combined by whoever finishes them.  Each block of
// kOutBlockRows output rows has a counter of finished (pick, row) pairs; a
// kernel that has written y'_j for some rows of a block adds their number, and
// the CTA whose addition brings the count to npicks * kOutBlockRows adds that
// block's out = sum_j y'_j in rank order and resets the count.  The one-row
// down pass finishes whole blocks of a pick; the read-through pass finishes
// the rows of its W2 units, which may straddle blocks.

// True when adding `rows` finished rows to block b completed it.
__device__ __forceinline__ bool add_block_rows(uint32_t* ctr, int b, uint32_t rows, int npicks) {
  const uint32_t total = (uint32_t)npicks * kOutBlockRows;
  return atomicAdd(&ctr[kBlockCtr + b], rows) + rows == total;
}

// Every thread of the CTA: the nl blocks listed in s_lastb were completed by
// this CTA; one warp per block (a lane per row) adds out for it.
__device__ __forceinline__ void combine_blocks(int npicks, const float* ypart,
                                               float* __restrict__ out, int H, uint32_t* ctr,
                                               const int* s_lastb, int nl) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  if (nl == 0) return;
  __threadfence();
  for (int t = warp; t < nl; t += nwarps) {  // a lane per row of the block
    const int b = s_lastb[t];
    const int row = b * kOutBlockRows + lane;
    float v[MOE_MAX_TOPK];
#pragma unroll
    for (int j = 0; j < MOE_MAX_TOPK; ++j)
      if (j < npicks) v[j] = __ldcg(ypart + (size_t)j * H + row);
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < MOE_MAX_TOPK; ++j)
      if (j < npicks) acc += v[j];
    out[row] = acc;
    if (lane == 0) ctr[kBlockCtr + b] = 0u;
  }
}

// Every thread of a down CTA, once all its units' rows are written: count
// each unit (this CTA's pick, output blocks b0, b0 + db, ...) as a whole block
// of one pick, then combine the blocks this CTA completed.  s_lastb: room for
// nunits ints.
__device__ __forceinline__ void count_blocks(const Plan* plan, const float* ypart,
                                             float* __restrict__ out, int H, uint32_t* ctr,
                                             int b0, int db, int nunits, int* s_lastb,
                                             int* s_nlast) {
  const int npicks = plan->npicks;
  __threadfence();
  if (threadIdx.x == 0) *s_nlast = 0;
  __syncthreads();
  for (int u = threadIdx.x; u < nunits; u += blockDim.x) {
    const int b = b0 + u * db;
    if (add_block_rows(ctr, b, kOutBlockRows, npicks)) s_lastb[atomicAdd(s_nlast, 1)] = b;
  }
  __syncthreads();
  combine_blocks(npicks, ypart, out, H, ctr, s_lastb, *s_nlast);
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

// ----------------------------------------------------------- gate / up

// This thread's 32 activations (elements 32c .. 32c + 31 of the row) as
// f16, after a power-of-two prescale of the whole row that keeps max |x|
// below 2^15; returns the factor that undoes the prescale.  Every thread of
// the CTA calls it (one barrier); the CTA's threads cover the whole row.
__device__ __forceinline__ float load_x_f16(const uint16_t* __restrict__ x, int c, float* s_xmax,
                                            uint32_t (&xh)[16]) {
  const int tid = threadIdx.x, lane = tid & 31;
  float xf[32];
  float amax = 0.f;
  {
    const uint4* xp = reinterpret_cast<const uint4*>(x + c * 32);
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const uint4 a = __ldg(xp + v);
      const uint32_t wds[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        xf[8 * v + 2 * i] = bf16_bits_to_float(wds[i] & 0xFFFFu);
        xf[8 * v + 2 * i + 1] = bf16_bits_to_float(wds[i] >> 16);
        amax = fmaxf(amax, fmaxf(fabsf(xf[8 * v + 2 * i]), fabsf(xf[8 * v + 2 * i + 1])));
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  if (lane == 0) s_xmax[tid >> 5] = amax;
  __syncthreads();
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) amax = fmaxf(amax, s_xmax[w]);
  int e2 = 0;
  frexpf(amax, &e2);  // amax < 2^e2
  const int xshift = e2 > 15 ? e2 - 15 : 0;
  const float xdown = ldexpf(1.0f, -xshift);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const __half2 p = __floats2half2_rn(xf[2 * i] * xdown, xf[2 * i + 1] * xdown);
    xh[i] = *reinterpret_cast<const uint32_t*>(&p);
  }
  return ldexpf(1.0f, xshift);
}

// Partial dot products of one staged gate/up unit (kGateUpRows row pairs laid
// out as gate codes, up codes, gate scales, up scales) over this thread's 32
// columns 32c .. 32c + 31 (two 16-element scale blocks) of rows g, g + RL, ...:
// a[q] gate rows, a[RPT + q] up rows.
template <int RPT>
__device__ __forceinline__ void gateup_partials(const uint8_t* __restrict__ st, int H, int RL,
                                                int g, int c, const uint32_t (&xh)[16],
                                                float (&a)[2 * RPT]) {
  const int cb = kGateUpRows * H / 2, sb = kGateUpRows * H / 16;
#pragma unroll
  for (int q = 0; q < RPT; ++q) {
    const int r = g + q * RL;
#pragma unroll
    for (int u = 0; u < 2; ++u) {  // gate, up
      const uint4 cw = *reinterpret_cast<const uint4*>(st + u * cb + r * (H / 2) + c * 16);
      const float2 sc = e4m3x2_to_float2(
          *reinterpret_cast<const uint16_t*>(st + 2 * cb + u * sb + r * (H / 16) + c * 2));
      const float d0 = dot16_f16(make_uint2(cw.x, cw.y), &xh[0]);
      const float d1 = dot16_f16(make_uint2(cw.z, cw.w), &xh[8]);
      a[u * RPT + q] = __fmaf_rn(d0, sc.x, __fmul_rn(d1, sc.y));
    }
  }
}

// h = silu(gate) * up of the unit's row pair t (t < RL * RPT) of pick j, from
// the partials stashed by every compute thread; gs_*: the pick's global scales.
template <int RPT, bool WARP_RED>
__device__ __forceinline__ void gateup_epilogue(const float* red, int RL, int C, float gs_gate,
                                                float gs_up, int j, int rb, float xup,
                                                float* __restrict__ hbuf, int I, int t) {
  constexpr int V = 2 * RPT;
  const int gg = t / RPT, q = t - gg * RPT;
  const float gate = gs_gate * xup * sum_partial<V, WARP_RED>(red, gg, q, C);
  const float up = gs_up * xup * sum_partial<V, WARP_RED>(red, gg, RPT + q, C);
  hbuf[(size_t)j * I + rb * kGateUpRows + gg + q * RL] = gate / (1.0f + expf(-gate)) * up;
}

// Resident picks: slot bytes from HBM, units assigned round-robin over the
// persistent grid.  Warp-specialised: the C * RL compute threads wait only for
// their unit's bytes (the stage's "full" mbarrier), stash their partial sums
// and count their warp in on the stage's "stashed" mbarrier without waiting;
// one control warp (the CTA's last) waits on "stashed", refills the stage with
// a later unit's four segments by 1-D TMA bulk copies and forms h for the
// unit's rows.  No compute warp ever waits for another.  Every wait is
// bounded: a compute warp whose wait runs out sets the CTA's abort word and
// stops; the control warp, waiting on a stage no stopped warp will stash,
// sees the word, stops issuing, waits (bounded) for its copies in flight and
// returns.  A compute warp can never run more than the stage ring ahead of the
// control warp, since each of its units waits for a fill the control warp
// issues only after the stage's previous unit was stashed.
template <int RPT, bool WARP_RED>
__global__ void __launch_bounds__(kGateUpThreads + 32, 2)
gemv_gateup_kernel(const Plan* plan, const uint16_t* __restrict__ x,
                   float* __restrict__ hbuf, int H, int I, int RL, int NS, uint32_t* flags,
                   int subset, PickBounds bounds) {
  constexpr int V = 2 * RPT;
  constexpr int R = kGateUpRows;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float s_xmax[kGateUpThreads / 32 + 1];
  const int C = H / 32;
  const int NC = C * RL;  // compute threads; the control warp follows them
  const int tid = threadIdx.x, lane = tid & 31;
  const int g = tid / C, c = tid - g * C;
  const int cb = R * H / 2, sb = R * H / 16;
  const int stage_bytes = 2 * cb + 2 * sb;
  const int red_floats = WARP_RED ? RL * (C / 32) * V : NC * V;  // per stage
  uint8_t* base = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)NS * stage_bytes);
  uint64_t* stashed = full + NS;
  volatile int* abort_flag = reinterpret_cast<int*>(full + 2 * NS);
  float* red0 = reinterpret_cast<float*>(full + 2 * NS + 1);
  __shared__ int s_pcnt;
  // the launch's picks, once: no global round trip on the refill path
  __shared__ int s_j[MOE_MAX_TOPK];
  __shared__ const uint8_t* s_w[MOE_MAX_TOPK];
  __shared__ const uint8_t* s_s[MOE_MAX_TOPK];
  __shared__ float s_gs[MOE_MAX_TOPK][2];
  const int upp = I / R;  // units per pick
  // The down pass that follows (programmatic launch) takes an SM only once
  // this grid's CTAs there have left, and issues its first resident W2
  // copies while the last gate/up units finish.
  pdl_launch_dependents();

  auto issue = [&](int unit, int stage) {  // control warp, lane 0
    const int jl = unit / upp, rb = unit - jl * upp;
    const uint8_t* w = s_w[jl];
    const uint8_t* sc = s_s[jl];
    const size_t og = (size_t)rb * R, ou = (size_t)I + (size_t)rb * R;
    uint8_t* dst = base + (size_t)stage * stage_bytes;
    mbar_arrive_expect_tx(&full[stage], (uint32_t)stage_bytes);
    bulk_g2s(dst, w + og * (H / 2), cb, &full[stage]);
    bulk_g2s(dst + cb, w + ou * (H / 2), cb, &full[stage]);
    bulk_g2s(dst + 2 * cb, sc + og * (H / 16), sb, &full[stage]);
    bulk_g2s(dst + 2 * cb + sb, sc + ou * (H / 16), sb, &full[stage]);
  };
  int issued = 0;
  if (tid >= NC) {  // control warp: the plan, while x loads below
    pdl_wait();     // the plan comes from the kernel before this one
    // the subset's picks in one round of loads, checked before they address
    // memory: a bad plan skips the whole launch (MOE_FLAG_BAD_PLAN)
    const WarpPicks p = warp_picks(plan, subset, bounds, false, lane);
    plan_ok(p.ok || lane != 0, flags);
    if (lane < p.pcnt) {
      s_j[lane] = p.j;
      s_w[lane] = p.w;
      s_s[lane] = p.s;
      s_gs[lane][0] = p.gs0;
      s_gs[lane][1] = p.gs1;
    }
    if (lane == 0) {
      s_pcnt = p.pcnt;
      for (int s = 0; s < NS; ++s) {
        mbar_init(&full[s], 1);
        mbar_init(&stashed[s], (uint32_t)(NC / 32));  // one arrival per compute warp
      }
      fence_mbar_init();
      *abort_flag = 0;
    }
    __syncwarp();
  }
  // x: the step's input (one barrier, which also publishes the picks and the
  // mbarriers).  The first fills are issued after it, so the compute warps
  // never wait at the barrier for the copy issue.
  uint32_t xh[16];
  const float xup = load_x_f16(x, c < C ? c : 0, s_xmax, xh);
  const int pcnt = s_pcnt;
  const int nunits = pcnt * upp;
  const int my_units = units_of_block(nunits);

  if (tid >= NC) {  // ---- control warp
    if (lane == 0)
      for (; issued < NS && issued < my_units; ++issued)
        issue(blockIdx.x + issued * gridDim.x, issued);
    int s = 0, rbuf = 0;  // stage and partial-sum buffer of unit i (no runtime division)
    uint32_t sphase = 0;  // parity of stage s's current "stashed" phase
    bool stopped = false;
    for (int i = 0; i < my_units; ++i) {
      // every compute warp has stashed unit i, unless one stopped
      const bool got = mbar_wait_or_abort(&stashed[s], sphase, abort_flag, flags);
      if (!__all_sync(0xFFFFFFFFu, got)) {
        stopped = true;
        break;
      }
      const int unit = blockIdx.x + i * gridDim.x;
      if (lane == 0 && i + NS < my_units) {  // the stage's bytes are consumed
        issue(unit + NS * gridDim.x, s);
        ++issued;
      }
      // unit i's partials sit in buffer i % 2NS; the next unit to use that buffer
      // is i + 2NS, whose bytes are only requested after unit i + NS is stashed,
      // i.e. after this epilogue
      if (lane < RL * RPT) {
        const int jl = unit / upp;
        gateup_epilogue<RPT, WARP_RED>(red0 + rbuf * red_floats, RL, C, s_gs[jl][0],
                                       s_gs[jl][1], s_j[jl], unit - jl * upp, xup, hbuf, I, lane);
      }
      __syncwarp();
      if (++s == NS) {
        s = 0;
        sphase ^= 1u;
      }
      if (++rbuf == 2 * NS) rbuf = 0;
    }
    // after a stop: the last fill issued on each stage is the only one that may
    // still be in flight; let each land (bounded) before the CTA's memory goes
    if (stopped && lane == 0)
      for (int m = issued - NS > 0 ? issued - NS : 0; m < issued; ++m)
        if (!mbar_wait_bounded(&full[m % NS], (uint32_t)((m / NS) & 1), flags)) break;
    return;
  }
  // ---- compute threads (whole warps)
  int s = 0, rbuf = 0;
  uint32_t phase = 0;  // parity of stage s's current fill
  const uint64_t wait_ns = plan_wait_ns(plan);
  for (int i = 0; i < my_units; ++i) {
    const bool ok = mbar_wait_bounded(&full[s], phase, flags, wait_ns);
    if (__any_sync(0xFFFFFFFFu, !ok || *abort_flag)) {  // flagged: this warp stops
      if (lane == 0) *abort_flag = 1;
      break;
    }
    float a[V];
    gateup_partials<RPT>(base + (size_t)s * stage_bytes, H, RL, g, c, xh, a);
    stash_partials<V, WARP_RED>(a, red0 + rbuf * red_floats, g, c, C, lane);
    __syncwarp();  // the warp's partials are written before its arrival releases them
    if (lane == 0) mbar_arrive(&stashed[s]);
    if (++s == NS) {
      s = 0;
      phase ^= 1u;
    }
    if (++rbuf == 2 * NS) rbuf = 0;
  }
}

// ---------------------------------------------------------- read-through

// A read-through stage holds a gate/up unit (kGateUpRows row pairs of W13)
// or at least two whole W2 rows, whichever is larger.
__host__ __device__ inline int rt_stage_bytes(int H, int I) {
  const int gu = 2 * kGateUpRows * (H / 2) + 2 * kGateUpRows * (H / 16);
  const int w2 = 2 * (I / 2 + I / 16);
  return gu > w2 ? gu : w2;
}

// W2 rows in one read-through unit: the most whole rows (codes and scales)
// that fit a stage, an even number so the scale segment stays 16-byte sized.
__host__ __device__ inline int w2_unit_rows(int H, int I) {
  int r = rt_stage_bytes(H, I) / (I / 2 + I / 16);
  r &= ~1;
  return r < H ? r : H;
}

// The missed picks' host-link pass, one launch.  Its work list holds the
// gate/up units of every missed pick (rank order), then the W2 units of every
// missed pick: each missed expert's bytes are read once over the host link
// and written through to its victim slot.  A gate/up unit is computed on
// arrival with the functions above and counts itself for its pick once its h
// rows are written.  A W2 unit (whole rows, codes and scales) is reduced on
// arrival too, against gscale * w * h of its pick, once every gate/up unit of
// that pick has counted itself (a bounded wait; those units were all taken
// before any W2 unit, by CTAs that finish them without waiting on anything,
// so the wait always ends); its y' rows then count for their output blocks.
// Units are taken one at a time from a step counter, so CTAs that get more of
// the link take more.  The rows are reduced with the row routine of the down
// pass (h staged in shared memory instead of registers), so a missed pick's
// y' has the same bits as if it were resident.
// (Half the SMs, one CTA each; 96 registers a thread leave room on the SM for
// one CTA of the resident picks' gate/up beside it at the GLM shape.)
template <int RPT, bool WARP_RED>
__global__ void __maxnreg__(96)
gemv_readthrough_kernel(const Plan* plan, const uint16_t* __restrict__ x,
                        float* hbuf, float* ypart, float* __restrict__ out, int H, int I,
                        int RL, int NS, uint32_t* flags, uint32_t* ctr, PickBounds bounds) {
  constexpr int V = 2 * RPT;
  constexpr int R = kGateUpRows;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float s_xmax[kGateUpThreads / 32];
  __shared__ int s_unit[kMaxStages];  // link unit staged in each stage, -1: none
  __shared__ int s_next[2];           // by iteration parity: read after the writer moved on
  __shared__ int s_pick[MOE_MAX_TOPK];  // the missed picks, checked
  // their host and slot pointers and scales, read once: no plan round trip on
  // the fill path
  __shared__ const uint8_t* s_hw[MOE_MAX_TOPK];
  __shared__ const uint8_t* s_hsc[MOE_MAX_TOPK];
  __shared__ const uint8_t* s_dw[MOE_MAX_TOPK];
  __shared__ const uint8_t* s_ds[MOE_MAX_TOPK];
  __shared__ float s_pg[MOE_MAX_TOPK][3];  // gate, up global scales; down scale x router weight
  __shared__ int s_pcnt;
  __shared__ int s_hpick;   // missed pick whose f * h sits in hs (-1: none)
  __shared__ int s_hwait;   // the wait for a pick's h ended (1) or gave up (0)
  __shared__ int s_lastb[MOE_MAX_DIM / kOutBlockRows];
  __shared__ int s_nlast;
  __shared__ int s_u0;
  const int C = H / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int g = tid / C, c = tid - g * C;
  const int cb = R * H / 2, sb = R * H / 16;
  const int SB = rt_stage_bytes(H, I);  // stage bytes
  Stages S = carve(smem, NS, SB);
  const int red_floats = WARP_RED ? RL * (C / 32) * V : (int)blockDim.x * V;
  float* hs = reinterpret_cast<float*>(
      (reinterpret_cast<uintptr_t>(S.red + red_floats) + 15) & ~(uintptr_t)15);  // [I], transposed

  // The missed picks, each checked (index, slot and host pointers) before it
  // addresses memory: a bad plan skips the whole launch (MOE_FLAG_BAD_PLAN).
  if (tid < 32) {
    const WarpPicks p = warp_picks(plan, kPicksMiss, bounds, true, tid);
    plan_ok(p.ok || tid != 0, flags);
    if (tid < p.pcnt) {
      s_pick[tid] = p.j;
      s_hw[tid] = p.hw;
      s_hsc[tid] = p.hs;
      s_dw[tid] = p.w;
      s_ds[tid] = p.s;
      s_pg[tid][0] = p.gs0;
      s_pg[tid][1] = p.gs1;
      s_pg[tid][2] = __fmul_rn(p.gs2, p.wt);
    }
    if (tid == 0) {
      s_pcnt = p.pcnt;
      s_hpick = -1;
    }
  }
  // the stages and the CTA's first units, by the second warp while the first
  // reads the plan (a one-warp CTA: after it)
  if (tid == (nwarps > 1 ? 32 : 0)) {
    for (int s = 0; s < NS; ++s) mbar_init(&S.full[s], blockDim.x);
    fence_mbar_init();
    *S.abort_flag = 0;
    s_nlast = 0;
    s_u0 = (int)atomicAdd(&ctr[kWorkCtr], (uint32_t)NS);
  }
  __syncthreads();
  const int pcnt = s_pcnt;
  const int npicks = plan->npicks;
  auto pick_of = [&](int jl) { return s_pick[jl]; };
  const int upp = I / R;                   // gate/up units per pick
  const int R2 = w2_unit_rows(H, I);       // W2 rows per unit
  const int n2 = (H + R2 - 1) / R2;        // W2 units per pick
  const int NG = pcnt * upp;               // the gate/up units come first
  const int NL = NG + pcnt * n2;
  const uint64_t wait_ns = plan_wait_ns(plan);

  // link unit u: its byte segments in host memory and in the pick's slot
  auto segs = [&](int u, int& nseg) {
    Segs<4> sg;
    if (u < NG) {
      const int jl = u / upp, r = u - jl * upp;
      const uint8_t* hw = s_hw[jl];
      const uint8_t* hsc = s_hsc[jl];
      uint8_t* dw = const_cast<uint8_t*>(s_dw[jl]);
      uint8_t* ds = const_cast<uint8_t*>(s_ds[jl]);
      const size_t og = (size_t)r * R, ou = (size_t)I + (size_t)r * R;
      sg.src[0] = hw + og * (H / 2);
      sg.src[1] = hw + ou * (H / 2);
      sg.src[2] = hsc + og * (H / 16);
      sg.src[3] = hsc + ou * (H / 16);
      sg.dst[0] = dw + og * (H / 2);
      sg.dst[1] = dw + ou * (H / 2);
      sg.dst[2] = ds + og * (H / 16);
      sg.dst[3] = ds + ou * (H / 16);
      sg.n[0] = sg.n[1] = cb;
      sg.n[2] = sg.n[3] = sb;
      nseg = 4;
    } else {  // W2 rows r0 .. r0 + nr - 1: codes after the 2I W13 code rows, scales likewise
      const int v = u - NG, jl = v / n2, r0 = (v - jl * n2) * R2;
      const int nr = H - r0 < R2 ? H - r0 : R2;
      const size_t oc = (size_t)I * H + (size_t)r0 * (I / 2);
      const size_t os = (size_t)I * H / 8 + (size_t)r0 * (I / 16);
      sg.src[0] = s_hw[jl] + oc;
      sg.src[1] = s_hsc[jl] + os;
      sg.dst[0] = const_cast<uint8_t*>(s_dw[jl]) + oc;
      sg.dst[1] = const_cast<uint8_t*>(s_ds[jl]) + os;
      sg.n[0] = nr * (I / 2);
      sg.n[1] = nr * (I / 16);
      nseg = 2;
    }
    return sg;
  };
  auto fill = [&](int u, int stage) {  // every thread
    int n = 0;
    const Segs<4> sg = segs(u, n);
    stage_from_host(S.base + (size_t)stage * SB, sg, n, &S.full[stage]);
  };

  if (tid == 0) {
    const int u0 = s_u0;
    for (int s = 0; s < kMaxStages; ++s) s_unit[s] = (s < NS && u0 + s < NL) ? u0 + s : -1;
  }
  __syncthreads();
  for (int s = 0; s < NS; ++s)
    if (s_unit[s] >= 0) fill(s_unit[s], s);
  uint32_t xh[16];
  const float xup = load_x_f16(x, c, s_xmax, xh);

  int i_abort = -1;  // the iteration a timed-out wait stopped the loop at (uniform)
  for (int i = 0;; ++i) {
    const int stage = i % NS;
    const int unit = s_unit[stage];
    if (unit < 0) break;  // units are taken in order: none left for this CTA
    // the unit that refills this stage: taken now, used at the end
    const int taken = tid == 0 ? (int)atomicAdd(&ctr[kWorkCtr], 1u) : 0;
    if (!mbar_wait_bounded(&S.full[stage], (uint32_t)((i / NS) & 1), flags, wait_ns))
      *S.abort_flag = 1;
    if (tid == 0) s_nlast = 0;  // every thread read the last count before the previous barrier
    __syncthreads();
    if (*S.abort_flag) {  // flagged; the copies in flight are drained below
      i_abort = i;
      break;
    }
    const uint8_t* st = S.base + (size_t)stage * SB;
    int nseg = 0;
    const Segs<4> sg = segs(unit, nseg);
    const bool gu = unit < NG;  // uniform over the CTA
    int jl = 0, r = 0;
    if (gu) {
      jl = unit / upp;
      r = unit - jl * upp;
      float a[V];
      gateup_partials<RPT>(st, H, RL, g, c, xh, a);
      stash_partials<V, WARP_RED>(a, S.red, g, c, C, lane);
    } else {
      const int v = unit - NG;
      jl = v / n2;
      const int r0 = (v - jl * n2) * R2, nr = H - r0 < R2 ? H - r0 : R2;
      if (s_hpick != jl) {  // uniform: this pick's h into shared memory, once it is complete
        if (tid == 0)
          s_hwait = count_wait_bounded(&ctr[kHCtr + jl], (uint32_t)upp, flags, wait_ns) ? 1 : 0;
        __syncthreads();
        if (!s_hwait) {
          if (tid == 0) *S.abort_flag = 1;
          i_abort = i;
          break;  // uniform; the copies in flight are drained below
        }
        const int j = pick_of(jl);
        const float f = s_pg[jl][2];
        for (int e = tid; e < I; e += blockDim.x)  // transposed: lanes read distinct banks
          hs[(e & 31) * (I / 32) + (e >> 5)] = __fmul_rn(f, __ldcg(hbuf + (size_t)j * I + e));
        if (tid == 0) s_hpick = jl;
        __syncthreads();
      }
      const int j = pick_of(jl);
      for (int rr = warp; rr < nr; rr += nwarps) {  // a warp per row, as in the down pass
        const float y = w2_row_warp(st + rr * (I / 2), st + nr * (I / 2) + rr * (I / 16), hs, I,
                                    lane);
        if (lane == 0) ypart[(size_t)j * H + r0 + rr] = y;
      }
      if (lane == 0) __threadfence();  // this warp's y' rows before the counts below
      __syncthreads();
      {  // count the rows for their output blocks, a thread a block; combine what completes
        const int b = r0 / kOutBlockRows + tid;
        if (b * kOutBlockRows < r0 + nr) {
          const int lo = b * kOutBlockRows > r0 ? b * kOutBlockRows : r0;
          const int hi = (b + 1) * kOutBlockRows < r0 + nr ? (b + 1) * kOutBlockRows : r0 + nr;
          if (add_block_rows(ctr, b, (uint32_t)(hi - lo), npicks))
            s_lastb[atomicAdd(&s_nlast, 1)] = b;
        }
      }
      __syncthreads();
      combine_blocks(npicks, ypart, out, H, ctr, s_lastb, s_nlast);
    }
    if (tid == 0) {  // before the barrier: with one stage the next iteration reads it before any barrier
      const int nv = taken < NL ? taken : -1;
      s_next[i & 1] = nv;
      s_unit[stage] = nv;
    }
    __syncthreads();
    if (gu) {  // h rows of the unit, then the unit counts for its pick
      if (tid < RL * RPT) {
        gateup_epilogue<RPT, WARP_RED>(S.red, RL, C, s_pg[jl][0], s_pg[jl][1], pick_of(jl), r,
                                       xup, hbuf, I, tid);
        __threadfence();
      }
      __syncthreads();
      if (tid == 0) {
        __threadfence();
        atomicAdd(&ctr[kHCtr + jl], 1u);
      }
    }
    // the unit's bytes to its slot, after the signals above so that their
    // fences do not wait for these stores; nothing reads the slot this step
    write_through(st, sg, nseg);
    __syncthreads();  // every thread is done with the stage before its refill
    const int nxt = s_next[i & 1];
    if (nxt >= 0) fill(nxt, stage);
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  if (i_abort >= 0) {
    // Every thread's copies have landed; each fill's completion also arrives
    // on its stage's mbarrier, so wait (default limit) until the pending fills'
    // phases are complete: no arrival may reach this CTA's shared memory after
    // it exits.  Iteration it consumes phase it / NS of stage it % NS.
    __syncthreads();
    if (tid == 0)
      for (int d = 0; d < NS; ++d) {
        const int it = i_abort + d, stg = it % NS;
        if (s_unit[stg] >= 0 && !mbar_wait_bounded(&S.full[stg], (uint32_t)((it / NS) & 1), flags))
          break;
      }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- down

// Each CTA serves one pick (CTAs b, b + pcnt, ... share pick b % pcnt) and
// takes units of kDownUnitRows W2 rows (output blocks) of it.  Its warps work
// independently: warp w takes rows kDownItemRows * w .. of every unit of the
// CTA, through a ring of its own (stages of kDownItemRows code and scale rows,
// each filled by two 1-D TMA bulk copies on the stage's mbarrier), and
// reduces each row with w2_row_warp_g against gscale * w * h of the pick held
// in registers (or, for large I, in shared memory, transposed).  No barrier
// between warps until the CTA's exit, where its units are counted for the
// per-block combine.
template <int MB>  // h blocks a lane keeps in registers (0: read them from shared memory)
__global__ void __launch_bounds__(kDownThreads, 1)
gemv_down_kernel(const Plan* plan, const float* hbuf, float* ypart, int H, int I, int NSW,
                 uint32_t* flags, int subset, float* __restrict__ out, uint32_t* ctr,
                 PickBounds bounds) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_nlast;
  __shared__ int s_lastb[MOE_MAX_DIM / kDownUnitRows];
  constexpr int UR = kDownUnitRows, IR = kDownItemRows;
  // The plan was written by route/remap, which completed before the kernel
  // this one may overlap (programmatic launch) started: it is read at once.
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  int pbeg = 0, pcnt = 0;
  const bool range_ok = subset_range(plan, subset, pbeg, pcnt);
  if (!range_ok) {  // uniform: nothing is addressed through a bad plan
    if (tid == 0) plan_ok(false, flags);
    return;
  }
  // this CTA's pick and its share of the pick's units
  const int jl = pcnt > 0 ? (int)blockIdx.x % pcnt : 0;
  const int q = pcnt > 0 ? (int)blockIdx.x / pcnt : 0;
  const int nq = pcnt > 0 ? ((int)gridDim.x - jl + pcnt - 1) / pcnt : 0;
  const int units = H / UR;
  const int my_units = (pcnt > 0 && q < units) ? (units - 1 - q) / nq + 1 : 0;
  if (my_units == 0) return;  // uniform
  const int j = subset == kPicksAll ? jl : plan->order[pbeg + jl];
  if (!pick_ok(plan, j, plan->npicks, bounds, false)) {  // uniform
    if (tid == 0) plan_ok(false, flags);
    return;
  }
  const uint8_t* wsrc = plan->wptr[j] + (size_t)I * H;     // W2 codes
  const uint8_t* ssrc = plan->sptr[j] + (size_t)I * H / 8; // W2 scales

  // this warp's ring and its items: item n is rows row0(n) .. + IR
  const int item_b = IR * (I / 2 + I / 16);
  uint8_t* ring = smem + (size_t)warp * NSW * item_b;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)nwarps * NSW * item_b) + warp * NSW;
  float* hs = reinterpret_cast<float*>(smem + (size_t)nwarps * NSW * (item_b + 8));
  const int ipu = UR / IR;  // items per unit
  const int nitems = my_units * ipu;
  const int my_items = nitems > warp ? (nitems - 1 - warp) / nwarps + 1 : 0;
  auto row0 = [&](int n) {
    const int g = warp + n * nwarps;
    const int i = g / ipu;
    return (q + i * nq) * UR + (g - i * ipu) * IR;
  };
  auto issue = [&](int n, int s) {  // lane 0
    const int r0 = row0(n);
    uint8_t* dst = ring + (size_t)s * item_b;
    mbar_arrive_expect_tx(&bars[s], (uint32_t)item_b);
    bulk_g2s(dst, wsrc + (size_t)r0 * (I / 2), IR * (I / 2), &bars[s]);
    bulk_g2s(dst + IR * (I / 2), ssrc + (size_t)r0 * (I / 16), IR * (I / 16), &bars[s]);
  };
  const float f = __fmul_rn(plan->gs[j][2], plan->wts[j]);
  // The picks this kernel serves are resident (hit picks of a cached step, or
  // the caller's experts): their slot bytes were in place before the kernel
  // before this one started, so the first copies go out before the wait.
  if (lane == 0) {
    for (int s = 0; s < NSW; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
    for (int s = 0; s < NSW && s < my_items; ++s) issue(s, s);
  }
  pdl_wait();  // h comes from the kernel before this one
  for (int e = tid; e < I; e += blockDim.x)  // transposed: lanes read distinct banks
    hs[(e & 31) * (I / 32) + (e >> 5)] = __fmul_rn(f, __ldcg(hbuf + (size_t)j * I + e));
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
        hv[m][e] = c < C ? hs[e * C + c] : 0.f;
      }
  }
  int n = 0, s = 0;
  uint32_t phase = 0;  // parity of stage s's current fill
  const uint64_t wait_ns = plan_wait_ns(plan);
  for (; n < my_items; ++n) {
    const bool ok = mbar_wait_bounded(&bars[s], phase, flags, wait_ns);
    if (!__all_sync(0xFFFFFFFFu, ok)) break;  // flagged; this warp's rows stay unwritten
    const uint8_t* st = ring + (size_t)s * item_b;
    const int r0 = row0(n);
#pragma unroll
    for (int r = 0; r < IR; ++r) {
      const uint8_t* cw = st + r * (I / 2);
      const uint8_t* sc = st + IR * (I / 2) + r * (I / 16);
      float y;
      if constexpr (MB > 0)
        y = w2_row_warp_g(cw, sc, C, MB, lane, [&](int m, int e) { return hv[m][e]; });
      else
        y = w2_row_warp(cw, sc, hs, I, lane);
      if (lane == 0) ypart[(size_t)j * H + r0 + r] = y;
    }
    __syncwarp();  // every lane is done with the stage
    if (lane == 0 && n + NSW < my_items) issue(n + NSW, s);
    if (++s == NSW) {
      s = 0;
      phase ^= 1u;
    }
  }
  if (n < my_items && lane == 0)  // after a timeout: let the copies in flight land (bounded)
    for (int m = n; m < n + NSW && m < my_items; ++m)
      if (!mbar_wait_bounded(&bars[m % NSW], (uint32_t)((m / NSW) & 1), flags)) break;
  count_blocks(plan, ypart, out, H, ctr, q, nq, my_units, s_lastb, &s_nlast);
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
  s.C = H / 32;  // threads across a row, 32 columns each
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
  // stages, their two mbarriers, two sets of partial sums a stage, the abort word
  int ns = (per_cta - 16) / (stage + 16 + 2 * red_floats * 4);
  if (ns > 6) ns = 6;  // <= kMaxStages
  if (stages > 0 && stages < ns) ns = stages;
  s.NS = ns;
  s.smem = ns * stage + 16 * ns + 8 + 2 * ns * red_floats * 4;
  return s;
}

template <int RPT, bool WR>
cudaError_t run_gateup(cudaStream_t st, int grid, const GateUpShape& s, const Plan* plan,
                       const uint16_t* x, float* hbuf, int H, int I, uint32_t* flags,
                       int subset, bool pdl, const PickBounds& b) {
  auto kern = gemv_gateup_kernel<RPT, WR>;
  static int smem_set = 0;  // raise the opt-in limit once per size (not a stream operation)
  if (s.smem > smem_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, s.smem);
    if (e == cudaSuccess) e = prefer_max_shared(kern);
    if (e != cudaSuccess) return e;
    smem_set = s.smem;
  }
  if (pdl)
    return launch_pdl(kern, dim3(grid), dim3(s.NT + 32), s.smem, st, plan, x, hbuf, H, I, s.RL,
                      s.NS, flags, subset, b);
  kern<<<grid, s.NT + 32, s.smem, st>>>(plan, x, hbuf, H, I, s.RL, s.NS, flags, subset, b);
  return cudaGetLastError();
}

template <int RPT, bool WR>
cudaError_t run_readthrough(cudaStream_t st, int grid, const GateUpShape& s, const Plan* plan,
                            const uint16_t* x, const GemvWorkspace& ws, float* out, int H, int I,
                            uint32_t* flags, uint32_t* ctr, const PickBounds& b) {
  auto kern = gemv_readthrough_kernel<RPT, WR>;
  // stages, their mbarriers, the abort word, one set of partial sums, and the
  // W2 units' f * h (transposed, 16-byte aligned)
  const int V = 2 * s.RPT;
  const int red_floats = s.warp_red ? s.RL * (s.C / 32) * V : s.NT * V;
  const int smem = s.NS * rt_stage_bytes(H, I) + 8 * s.NS + 8 + red_floats * 4 + 16 + I * 4;
  static int smem_set = 0;
  if (smem > smem_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) e = prefer_max_shared(kern);
    if (e != cudaSuccess) return e;
    smem_set = smem;
  }
  kern<<<grid, s.NT, smem, st>>>(plan, x, ws.hbuf, ws.ypart, out, H, I, s.RL, s.NS, flags, ctr, b);
  return cudaGetLastError();
}

int gateup_grid(int I, int k, int num_sms, const GemvLaunch& how) {
  const int nunits = k * (I / kGateUpRows);
  const int grid = how.grid > 0 ? how.grid : 2 * num_sms;
  return grid < nunits ? grid : nunits;
}

struct DownShape {
  int NS, smem, stage;  // NS: stages per warp ring, stage: bytes of one
};

DownShape down_shape(int I, int stages) {
  DownShape d;
  const int nwarps = kDownThreads / 32;
  d.stage = kDownItemRows * (I / 2 + I / 16);
  // leave room on the SM for one CTA of the step's other kernels
  const int per_cta = 140 * 1024;
  int ns = (per_cta - I * 4) / (nwarps * (d.stage + 8));
  if (ns < 2) ns = (kSmemPerSm - 1024 - I * 4) / (nwarps * (d.stage + 8));  // large I
  if (ns > 8) ns = 8;
  if (stages > 0 && stages < ns) ns = stages;
  d.NS = ns;
  d.smem = nwarps * ns * (d.stage + 8) + I * 4;
  return d;
}

template <int MB>
cudaError_t run_down(cudaStream_t st, int grid, const DownShape& d, const Plan* plan,
                     const GemvWorkspace& ws, int H, int I, uint32_t* flags, int subset,
                     float* out, uint32_t* ctr, bool pdl, const PickBounds& b) {
  auto kern = gemv_down_kernel<MB>;
  static int smem_set = 0;
  if (d.smem > smem_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, d.smem);
    if (e == cudaSuccess) e = prefer_max_shared(kern);
    if (e != cudaSuccess) return e;
    smem_set = d.smem;
  }
  if (pdl)
    return launch_pdl(kern, dim3(grid), dim3(kDownThreads), d.smem, st, plan, ws.hbuf, ws.ypart,
                      H, I, d.NS, flags, subset, out, ctr, b);
  kern<<<grid, kDownThreads, d.smem, st>>>(plan, ws.hbuf, ws.ypart, H, I, d.NS, flags, subset,
                                           out, ctr, b);
  return cudaGetLastError();
}

}  // namespace

bool gemv_supported(int H, int I, int k) {
  const int C = I / 32;  // 32-element blocks of a W2 row: whole warps of them or part of one
  if (!(H % 128 == 0 && I % 128 == 0 && H <= MOE_MAX_DIM && I <= MOE_MAX_DIM && k >= 1 &&
        (C % 32 == 0 || 32 % C == 0) && H / 32 <= kGateUpThreads))
    return false;
  const GateUpShape s = gateup_shape(H, 0);
  return s.NT % 32 == 0 && s.NS >= 1 && down_shape(I, 0).NS >= 1;
}

#define GATEUP_DISPATCH(RUN, ...)                                  \
  switch (s.RPT * 2 + (s.warp_red ? 1 : 0)) {                      \
    case 2: return RUN<1, false>(__VA_ARGS__);                     \
    case 3: return RUN<1, true>(__VA_ARGS__);                      \
    case 4: return RUN<2, false>(__VA_ARGS__);                     \
    case 5: return RUN<2, true>(__VA_ARGS__);                      \
    case 8: return RUN<4, false>(__VA_ARGS__);                     \
    case 9: return RUN<4, true>(__VA_ARGS__);                      \
    default: return cudaErrorInvalidConfiguration;                 \
  }

cudaError_t launch_gemv_gateup(cudaStream_t st, const Plan* plan, const uint16_t* x, int H, int I,
                               int k, const GemvWorkspace& ws, uint32_t* flags, int num_sms,
                               const GemvLaunch& how) {
  const GateUpShape s = gateup_shape(H, how.stages);
  if (s.NS < 1 || s.NT > kGateUpThreads || how.from_host) return cudaErrorInvalidConfiguration;
  const int grid = gateup_grid(I, k, num_sms, how);
  GATEUP_DISPATCH(run_gateup, st, grid, s, plan, x, ws.hbuf, H, I, flags, how.subset, how.pdl,
                  how.bounds)
}

int gemv_readthrough_grid(int I, int k, int num_sms, const GemvLaunch& how) {
  return gateup_grid(I, k, num_sms, how);
}

cudaError_t launch_gemv_readthrough(cudaStream_t st, const Plan* plan, const uint16_t* x, int H,
                                    int I, int k, const GemvWorkspace& ws, uint32_t* flags,
                                    int num_sms, const GemvLaunch& how, float* out, uint32_t* ctr) {
  const GateUpShape s = gateup_shape(H, how.stages);
  if (s.NS < 1 || s.NT > kGateUpThreads || !how.from_host || how.subset != kPicksMiss)
    return cudaErrorInvalidConfiguration;
  const int grid = gemv_readthrough_grid(I, k, num_sms, how);
  GATEUP_DISPATCH(run_readthrough, st, grid, s, plan, x, ws, out, H, I, flags, ctr, how.bounds)
}
#undef GATEUP_DISPATCH

int gemv_down_grid(int H, int num_sms, const GemvLaunch& how) {
  (void)H;
  const int grid = how.grid > 0 ? how.grid : num_sms;
  return grid > MOE_MAX_TOPK ? grid : MOE_MAX_TOPK;  // at least one CTA per pick
}

cudaError_t launch_gemv_down(cudaStream_t st, const Plan* plan, int H, int I, int k,
                             const GemvWorkspace& ws, uint32_t* flags, int num_sms,
                             const GemvLaunch& how, float* out, uint32_t* ctr) {
  (void)k;
  const DownShape d = down_shape(I, how.stages);
  // resident slot bytes only: the kernel's first copies precede its wait on
  // the kernel before it
  if (d.NS < 1 || how.from_host || how.subset == kPicksMiss) return cudaErrorInvalidConfiguration;
  const int grid = gemv_down_grid(H, num_sms, how);
  const int C = I / 32;  // h blocks per W2 row: in registers up to two per lane
  if (C <= 32)
    return run_down<1>(st, grid, d, plan, ws, H, I, flags, how.subset, out, ctr, how.pdl, how.bounds);
  if (C == 64)
    return run_down<2>(st, grid, d, plan, ws, H, I, flags, how.subset, out, ctr, how.pdl, how.bounds);
  return run_down<0>(st, grid, d, plan, ws, H, I, flags, how.subset, out, ctr, how.pdl, how.bounds);
}

}  // namespace moe
