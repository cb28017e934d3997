// Activations -> residual multi-level NVFP4, the operand format of the
// block-scaled tensor-core MMA (E2M1 codes with one UE4M3 scale per 16
// elements; both MMA operands must be FP4 for kind::mxf4nvf4).
//
// One FP4 level carries ~3 bits, so a row is written as a sum of kLevels
// levels: level l quantises the residual r_l = v - sum_{l'<l} q_l' with its own
// fp32 level scale G_l = max|r_l| / (6 * 448), block scales s = the smallest
// UE4M3 >= max|r_l over the block| / (6 G_l) (rounded up, so no code saturates)
// and codes c = round-to-nearest-even E2M1 of r / (s G_l).  Each level shrinks
// the residual ~10x; 6 levels leave ~1e-6 of the row's RMS.  The MMA then
// computes one accumulator per level and the epilogue sums G_l * D_l.
//
// One CTA per row, one thread per 16-element block; the residual stays in
// registers across levels.
#include "internal.cuh"

namespace moe {
namespace {

__device__ __forceinline__ float block_reduce_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float m = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, red[w]);
  return m;
}

// Smallest E4M3 code whose value is >= v (v > 0, v <= 448).
__device__ __forceinline__ uint32_t e4m3_ceil(float v) {
  uint16_t two;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(two) : "f"(0.0f), "f"(v));
  uint32_t q = two & 0xFFu;
  const float back = e4m3x2_to_float2(q).x;
  if (back < v && q < 0x7Eu) q += 1;
  return q;
}

// Two floats -> one byte of E2M1 codes, round to nearest even, saturating;
// `lo` goes to the low nibble.
__device__ __forceinline__ uint32_t e2m1x2_rn(float lo, float hi) {
  uint16_t b;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
      : "=h"(b)
      : "f"(hi), "f"(lo));
  return b & 0xFFu;
}

template <bool BF16_IN>
__device__ void quantize_row(const void* __restrict__ src, int K, const QuantBuf& q, int row,
                             float* red) {
  const int t = threadIdx.x;
  const int nblk = K / 16;
  float r[16];
  if (t < nblk) {
    if constexpr (BF16_IN) {
      const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(src) +
                                                      (size_t)row * K + t * 16);
      const uint4 a = __ldg(p), b = __ldg(p + 1);
      const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        r[2 * i] = bf16_bits_to_float(w[i] & 0xFFFFu);
        r[2 * i + 1] = bf16_bits_to_float(w[i] >> 16);
      }
    } else {
      const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(src) +
                                                        (size_t)row * K + t * 16);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 v = __ldg(p + i);
        r[4 * i] = v.x;
        r[4 * i + 1] = v.y;
        r[4 * i + 2] = v.z;
        r[4 * i + 3] = v.w;
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = 0.f;
  }
  for (int l = 0; l < kLevels; ++l) {
    float bmax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) bmax = fmaxf(bmax, fabsf(r[i]));
    const float amax = block_reduce_max(bmax, red);
    const float G = amax / (6.0f * 448.0f);
    uint32_t sc = 0;
    uint32_t codes[2] = {0u, 0u};
    if (G > 0.f && bmax > 0.f) {
      float need = bmax / (6.0f * G);
      if (need > 448.f) need = 448.f;
      sc = e4m3_ceil(need);
      const float s = e4m3x2_to_float2(sc).x * G;
      if (s > 0.f) {
        const float inv = 1.0f / s;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t b = e2m1x2_rn(r[2 * i] * inv, r[2 * i + 1] * inv);
          codes[i >> 2] |= b << (8 * (i & 3));
          const float2 d = e2m1x2_to_float2(b);
          r[2 * i] -= d.x * s;
          r[2 * i + 1] -= d.y * s;
        }
      } else {
        sc = 0;
      }
    }
    if (t < nblk) {
      const size_t base = (size_t)row * kLevels + l;
      *reinterpret_cast<uint2*>(q.codes + base * (K / 2) + t * 8) = make_uint2(codes[0], codes[1]);
      q.scales[base * (K / 16) + t] = (uint8_t)sc;
      if (t == 0) q.gl[base] = G;
    }
  }
}

template <bool BF16_IN>
__global__ void __launch_bounds__(1024)
quantize_rows_kernel(const void* __restrict__ src, int K, QuantBuf q) {
  __shared__ float red[32];
  quantize_row<BF16_IN>(src, K, q, blockIdx.x, red);
}

// The rows named by the members of groups [g0, g1) (members are stored group
// after group, so they are one contiguous range; bounds as resolve_group takes them).
__global__ void __launch_bounds__(1024)
quantize_members_kernel(const float* __restrict__ src, int K, const GroupPlan* __restrict__ gp,
                        int g0, int g1, QuantBuf q) {
  __shared__ float red[32];
  const int ng = gp->n_groups;
  const int nh = min(max(gp->n_hit_groups, 0), ng);
  g0 = resolve_group(g0, nh, ng);
  g1 = resolve_group(g1, nh, ng);
  if (g0 >= ng || g1 <= g0) return;
  const int mbeg = gp->g_start[g0];
  const int mend = g1 < ng ? gp->g_start[g1] : gp->npicks;
  for (int i = mbeg + blockIdx.x; i < mend; i += gridDim.x) {
    quantize_row<false>(src, K, q, gp->members[i], red);
    __syncthreads();  // red is reused by the next row
  }
}

}  // namespace

cudaError_t launch_quantize_members(cudaStream_t st, const float* src, int K, const GroupPlan* gp,
                                    int g0, int g1, const QuantBuf& q, int grid) {
  const int nblk = K / 16;
  const int threads = ((nblk + 31) / 32) * 32;
  if (threads > 1024 || grid <= 0) return cudaErrorInvalidValue;
  quantize_members_kernel<<<grid, threads, 0, st>>>(src, K, gp, g0, g1, q);
  return cudaGetLastError();
}

cudaError_t launch_quantize_rows(cudaStream_t st, const void* src, bool bf16_in, int rows, int K,
                                 const QuantBuf& q) {
  if (rows <= 0) return cudaSuccess;
  const int nblk = K / 16;
  const int threads = ((nblk + 31) / 32) * 32;
  if (threads > 1024) return cudaErrorInvalidValue;
  if (bf16_in)
    quantize_rows_kernel<true><<<rows, threads, 0, st>>>(src, K, q);
  else
    quantize_rows_kernel<false><<<rows, threads, 0, st>>>(src, K, q);
  return cudaGetLastError();
}

}  // namespace moe
