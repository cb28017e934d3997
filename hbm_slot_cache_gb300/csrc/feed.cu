// Step-input feeder: a device step cursor over device-resident input traces.
//
// A decode round is captured once as a CUDA graph over fixed input addresses
// ("GLM 5.3 Testing: HBM Expert Allocation", "What the slot cache is": fixed
// addresses and shapes make the round replayable as a graph).  To replay that
// one graph over many different steps, the graph's first node copies step t's
// router logits and activations from a trace held in device memory into the
// fixed buffers the step reads, t being a device-side cursor that the same
// launch advances.  Nothing on the host changes between replays.
//
// One launch copies one entry of each trace (16-byte words, all CTAs in a
// grid-stride loop) and then advances the cursor.  Every CTA reads the cursor
// before any CTA can change it: the CTA that finishes last (a done count in
// cursor[1], reset by that CTA) is the only writer, and it writes after every
// CTA has counted itself out, which each does after its copies used the value.
#include "internal.cuh"

namespace moe {
namespace {

constexpr int kFeedThreads = 512;

__global__ void __launch_bounds__(kFeedThreads)
feed_inputs_kernel(const uint4* __restrict__ a_src, uint4* __restrict__ a_dst, long long a_words,
                   const uint4* __restrict__ b_src, uint4* __restrict__ b_dst, long long b_words,
                   uint32_t steps, uint32_t* cursor) {
  __shared__ uint32_t s_c;
  if (threadIdx.x == 0) s_c = *reinterpret_cast<volatile uint32_t*>(cursor);
  __syncthreads();
  const uint32_t c = s_c;
  const long long t = (long long)(c % steps);
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long i0 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  for (long long i = i0; i < a_words; i += stride) a_dst[i] = __ldg(a_src + t * a_words + i);
  for (long long i = i0; i < b_words; i += stride) b_dst[i] = __ldg(b_src + t * b_words + i);
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&cursor[1], 1u) == gridDim.x - 1) {  // last CTA: every CTA has read c
      cursor[1] = 0u;
      cursor[0] = c + 1u;
      __threadfence();
    }
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_feed_inputs(const void* logits_trace, const void* x_trace,
                               size_t logits_bytes, size_t x_bytes, int steps, void* logits_dst,
                               void* x_dst, uint32_t* cursor, void* stream) {
  if (steps < 1 || !cursor || ((uintptr_t)cursor & 3) || (logits_bytes & 15) || (x_bytes & 15) ||
      (logits_bytes == 0 && x_bytes == 0))
    return MOE_ERR_ARG;
  if (logits_bytes && (!logits_trace || !logits_dst || ((uintptr_t)logits_trace & 15) ||
                       ((uintptr_t)logits_dst & 15)))
    return MOE_ERR_ARG;
  if (x_bytes && (!x_trace || !x_dst || ((uintptr_t)x_trace & 15) || ((uintptr_t)x_dst & 15)))
    return MOE_ERR_ARG;
  const long long aw = (long long)(logits_bytes / 16), bw = (long long)(x_bytes / 16);
  const long long words = aw > bw ? aw : bw;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  long long grid = (words + 4 * kFeedThreads - 1) / (4 * kFeedThreads);  // ~4 words a thread
  if (grid < 1) grid = 1;
  if (grid > sms) grid = sms;
  feed_inputs_kernel<<<(int)grid, kFeedThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(logits_trace), static_cast<uint4*>(logits_dst), aw,
      static_cast<const uint4*>(x_trace), static_cast<uint4*>(x_dst), bw, (uint32_t)steps,
      cursor);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
