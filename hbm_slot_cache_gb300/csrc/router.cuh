// Warp-level top-k router for one row of logits (shared by the cached-step and
// bypass routing kernels so both pick bit-identical ids and weights).
//
// "GLM 5.3 Testing: HBM Expert Allocation", "What the slot cache is": the
// router has chosen the top-8 expert ids before the expert kernel;
// "TensorFold GLM-5.3 explained": router ties break by a stable expert order.
// Ranking key: (logit descending, id ascending), -0 == +0, NaN below every
// number.  Weights: softmax over the k selected logits (NaN counts as -inf; a
// logit equal to the maximum contributes exactly 1), summed in rank order.
#pragma once
#include "internal.cuh"

namespace moe {

__device__ __forceinline__ uint32_t rank_key(float f) {
  if (isnan(f)) return 0u;                              // below -inf
  uint32_t u = __float_as_uint(f == 0.0f ? 0.0f : f);  // -0 ranks as +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) {
  return a > b ? a : b;
}
__device__ __forceinline__ unsigned long long umin64(unsigned long long a, unsigned long long b) {
  return a < b ? a : b;
}

// Softmax over the k selected logits; all 32 lanes call it, lane j < k holding
// the j-th selected logit, and lane j writes wts[j].
__device__ __forceinline__ void route_weights(float lsel, int k, int lane, float* wts) {
  const float l = (lane < k) ? (isnan(lsel) ? -INFINITY : lsel) : -INFINITY;
  float lmax = l;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xFFFFFFFFu, lmax, o));
  const float ej = (lane < k) ? ((l == lmax) ? 1.0f : expf(l - lmax)) : 0.0f;
  float sum = 0.f;
  for (int j = 0; j < k; ++j) sum += __shfl_sync(0xFFFFFFFFu, ej, j);
  if (lane < k) wts[lane] = ej / sum;
}

// The logit a ranking key was made from (rank_key inverted): -0 comes back as
// +0 and NaN as a NaN, which route_weights treats exactly like the originals.
__device__ __forceinline__ float key_logit(unsigned long long key) {
  const uint32_t kk = (uint32_t)(key >> 32);
  return __uint_as_float((kk & 0x80000000u) ? (kk & 0x7FFFFFFFu) : ~kk);
}

// Ranking key of logit f for expert e: larger key = earlier rank; never 0.
__device__ __forceinline__ unsigned long long route_key(float f, int e) {
  return ((unsigned long long)rank_key(f) << 32) | (0xFFFFFFFFu - (uint32_t)e);
}

// All 32 lanes call it.  ids[j] / wts[j] (j < k) are written by lanes 0 and j;
// returns true (on every lane) if any of the row's logits is NaN or infinite.
// KPL = keys per lane >= ceil(E / 32).  flags: the layer's error word.
template <int KPL>
__device__ __forceinline__ bool route_row(const float* __restrict__ lr, int E, int k, int lane,
                                          int32_t* ids, float* wts, uint32_t* flags) {
  unsigned long long key[KPL];
  bool bad = false;
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    const int e = lane + 32 * i;
    key[i] = 0ull;
    if (e < E) {
      const float f = lr[e];
      bad |= !isfinite(f);
      key[i] = route_key(f, e);
    }
  }
  unsigned long long best = 0ull;
#pragma unroll
  for (int i = 0; i < KPL; ++i) best = umax64(best, key[i]);
  float lsel = 0.f;  // lane j < k keeps the j-th selected logit
  for (int j = 0; j < k; ++j) {
    unsigned long long w = best;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) w = umax64(w, __shfl_xor_sync(0xFFFFFFFFu, w, o));
    const int e = (int)(0xFFFFFFFFu - (uint32_t)(w & 0xFFFFFFFFull));
    if ((e & 31) == lane) {  // the owning lane drops the winner and rescans
      best = 0ull;
#pragma unroll
      for (int i = 0; i < KPL; ++i) {
        if (lane + 32 * i == e) key[i] = 0ull;
        best = umax64(best, key[i]);
      }
    }
    if (lane == 0 && plan_ok(e >= 0 && e < E, flags)) ids[j] = e;
    if (lane == j && plan_ok(e >= 0 && e < E, flags)) lsel = lr[e];
  }
  route_weights(lsel, k, lane, wts);
  return __any_sync(0xFFFFFFFFu, bad) != 0;
}

}  // namespace moe
