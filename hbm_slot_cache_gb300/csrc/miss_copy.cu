// Miss copy: host backing -> HBM slot, byte for byte, by SM loads over the
// host link ("GLM 5.3 Testing: HBM Expert Allocation", "The build, measured
// ...": the miss handler copies the expert's weight row and scale row into the
// victim slot; an SM copy kernel ran at the NVLink-C2C ceiling).
//
// One launch covers all of a step's misses (the pages used four launches per
// layer: w13 rows, w2 rows and two scale tensors).  The grid is fixed, so the
// launch is graph-capturable; the miss count is read on the device and a step
// without misses exits at once.  Work is cut into 32 KB chunks (256 threads x
// 8 x 16 B); each thread keeps 8 independent 16-byte host loads in flight
// before storing them, so a grid of about a quarter of the SMs keeps ~1 MB in
// flight, enough to fill the host link, and leaves the other SMs to the
// resident experts' kernels that run beside it.
#include "internal.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 8;
constexpr long long kChunk = (long long)kThreads * kUnroll * 16;

__device__ __forceinline__ void copy_chunk(const uint8_t* __restrict__ src,
                                           uint8_t* __restrict__ dst, long long off,
                                           long long len) {
  uint4 buf[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const long long q = off + ((long long)u * kThreads + threadIdx.x) * 16;
    if (q < len) buf[u] = ld_stream16(src + q);
  }
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const long long q = off + ((long long)u * kThreads + threadIdx.x) * 16;
    if (q < len) *reinterpret_cast<uint4*>(dst + q) = buf[u];
  }
}

__global__ void __launch_bounds__(kThreads)
miss_copy_kernel(const Plan* __restrict__ plan, const uint8_t* __restrict__ host_w,
                 const uint8_t* __restrict__ host_s, uint8_t* __restrict__ slot_w,
                 uint8_t* __restrict__ slot_s, long long Bw, long long Bs, int part, int parts) {
  const int nall = plan->n_miss;
  const int m0 = nall * part / parts, m1 = nall * (part + 1) / parts;
  const int n = m1 - m0;
  if (n <= 0) return;
  const long long ncw = (Bw + kChunk - 1) / kChunk;
  const long long ncs = (Bs + kChunk - 1) / kChunk;
  const long long nc = ncw + ncs;
  for (long long c = blockIdx.x; c < (long long)n * nc; c += gridDim.x) {
    const int i = m0 + (int)(c / nc);
    const long long r = c - (long long)(i - m0) * nc;
    const long long e = plan->miss_e[i], v = plan->miss_v[i];
    if (r < ncw)
      copy_chunk(host_w + e * Bw, slot_w + v * Bw, r * kChunk, Bw);
    else
      copy_chunk(host_s + e * Bs, slot_s + v * Bs, (r - ncw) * kChunk, Bs);
  }
}

// Staged prefill ("GB300 GLM 5.3 Testing": stage a prefill's experts into HBM
// by DMA, up to 64 at a time, and run the grouped kernel from there): the
// experts of groups [q*C, q*C + C) go host -> staging half (q & 1), each read
// once over the host link, and those groups' pointers are set to the staged
// bytes for the grouped MMAs that follow.
__global__ void __launch_bounds__(kThreads)
stage_copy_kernel(GroupPlan* __restrict__ gp, int q, int C, LayerDev L, uint8_t* __restrict__ stage_w,
                  uint8_t* __restrict__ stage_s, long long Bw, long long Bs) {
  const int ng = gp->n_groups;
  const int g0 = q * C;
  if (g0 >= ng) return;
  const int n = min(C, ng - g0);
  const int half = (q & 1) * C;
  const long long ncw = (Bw + kChunk - 1) / kChunk;
  const long long ncs = (Bs + kChunk - 1) / kChunk;
  const long long nc = ncw + ncs;
  for (long long c = blockIdx.x; c < (long long)n * nc; c += gridDim.x) {
    const int i = (int)(c / nc);
    const long long r = c - (long long)i * nc;
    const long long e = gp->g_expert[g0 + i], b = half + i;
    if (r < ncw)
      copy_chunk(L.host_w + e * Bw, stage_w + b * Bw, r * kChunk, Bw);
    else
      copy_chunk(L.host_s + e * Bs, stage_s + b * Bs, (r - ncw) * kChunk, Bs);
  }
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      gp->g_wptr[g0 + i] = stage_w + (long long)(half + i) * Bw;
      gp->g_sptr[g0 + i] = stage_s + (long long)(half + i) * Bs;
    }
}

__global__ void __launch_bounds__(kThreads)
link_probe_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, long long bytes) {
  const long long nc = (bytes + kChunk - 1) / kChunk;
  for (long long c = blockIdx.x; c < nc; c += gridDim.x) copy_chunk(src, dst, c * kChunk, bytes);
}

}  // namespace

cudaError_t launch_miss_copy(cudaStream_t st, const Plan* plan, const uint8_t* host_w,
                             const uint8_t* host_s, uint8_t* slot_w, uint8_t* slot_s,
                             long long Bw, long long Bs, int grid, int part, int parts) {
  if (parts < 1 || part < 0 || part >= parts) return cudaErrorInvalidValue;
  static bool once = false;
  if (!once) {
    cudaError_t e = prefer_max_shared(miss_copy_kernel);
    if (e != cudaSuccess) return e;
    once = true;
  }
  miss_copy_kernel<<<grid, kThreads, 0, st>>>(plan, host_w, host_s, slot_w, slot_s, Bw, Bs, part,
                                               parts);
  return cudaGetLastError();
}

cudaError_t launch_stage_copy(cudaStream_t st, GroupPlan* gp, int q, int C, const LayerDev& L,
                              uint8_t* stage_w, uint8_t* stage_s, long long Bw, long long Bs,
                              int grid) {
  static bool once = false;
  if (!once) {
    cudaError_t e = prefer_max_shared(stage_copy_kernel);
    if (e != cudaSuccess) return e;
    once = true;
  }
  stage_copy_kernel<<<grid, kThreads, 0, st>>>(gp, q, C, L, stage_w, stage_s, Bw, Bs);
  return cudaGetLastError();
}

cudaError_t launch_link_probe(cudaStream_t st, const void* src, void* dst, size_t bytes,
                              int grid) {
  link_probe_kernel<<<grid, kThreads, 0, st>>>(static_cast<const uint8_t*>(src),
                                               static_cast<uint8_t*>(dst), (long long)bytes);
  return cudaGetLastError();
}

}  // namespace moe
