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
  pdl_launch_dependents();  // a step's route/remap, launched programmatically, waits for this grid
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

// Host <-> device moves of a step's inputs and output by kernels that read or
// write page-locked host memory directly (its device-side address): every
// load of a launch is in flight at once, so a step's inputs cost a kernel
// launch and one host-link round trip instead of two copy-engine transfers,
// and its output one posted store per word.  Words of 16 bytes where both ends
// are 16-byte aligned, else 4 (logits, output) or 2 bytes (x).
constexpr int kIoThreads = 512;

__device__ __forceinline__ bool al16(const void* p) { return ((uintptr_t)p & 15) == 0; }

__global__ void __launch_bounds__(kIoThreads)
host_in_kernel(const float* lg_h, const uint16_t* x_h, float* lg_d, uint16_t* x_d, int nl,
               int nx) {
  pdl_launch_dependents();  // the step's route/remap waits for this grid
  const int stride = gridDim.x * blockDim.x, i0 = blockIdx.x * blockDim.x + threadIdx.x;
  if (al16(lg_h) && al16(lg_d) && (nl & 3) == 0) {
    for (int i = i0; i < nl / 4; i += stride)
      reinterpret_cast<uint4*>(lg_d)[i] = reinterpret_cast<const uint4*>(lg_h)[i];
  } else {
    for (int i = i0; i < nl; i += stride) lg_d[i] = lg_h[i];
  }
  if (al16(x_h) && al16(x_d) && (nx & 7) == 0) {
    for (int i = i0; i < nx / 8; i += stride)
      reinterpret_cast<uint4*>(x_d)[i] = reinterpret_cast<const uint4*>(x_h)[i];
  } else {
    for (int i = i0; i < nx; i += stride) x_d[i] = x_h[i];
  }
}

__global__ void __launch_bounds__(kIoThreads)
host_out_kernel(const float* out_d, float* out_h, int n) {
  const int stride = gridDim.x * blockDim.x, i0 = blockIdx.x * blockDim.x + threadIdx.x;
  if (al16(out_h) && al16(out_d) && (n & 3) == 0) {
    for (int i = i0; i < n / 4; i += stride)
      reinterpret_cast<uint4*>(out_h)[i] = reinterpret_cast<const uint4*>(out_d)[i];
  } else {
    for (int i = i0; i < n; i += stride) out_h[i] = out_d[i];
  }
}

int io_grid(int words) {
  const int g = (words + 4 * kIoThreads - 1) / (4 * kIoThreads);  // ~4 words a thread
  return g < 1 ? 1 : (g > 64 ? 64 : g);
}

}  // namespace

cudaError_t launch_host_in(cudaStream_t st, const float* lg_h, const uint16_t* x_h, float* lg_d,
                           uint16_t* x_d, int nl, int nx) {
  host_in_kernel<<<io_grid(nx / 8 > nl / 4 ? nx / 8 : nl / 4), kIoThreads, 0, st>>>(
      lg_h, x_h, lg_d, x_d, nl, nx);
  return cudaGetLastError();
}

cudaError_t launch_host_out(cudaStream_t st, const float* out_d, float* out_h, int n) {
  host_out_kernel<<<io_grid(n / 4), kIoThreads, 0, st>>>(out_d, out_h, n);
  return cudaGetLastError();
}

bool is_host_in_node(const void* func) { return func == reinterpret_cast<const void*>(host_in_kernel); }
bool is_host_out_node(const void* func) {
  return func == reinterpret_cast<const void*>(host_out_kernel);
}

cudaError_t set_host_in_node(cudaGraphExec_t ex, cudaGraphNode_t node, const float* lg_h,
                             const uint16_t* x_h, float* lg_d, uint16_t* x_d, int nl, int nx) {
  void* args[] = {&lg_h, &x_h, &lg_d, &x_d, &nl, &nx};
  cudaKernelNodeParams p{};
  p.func = reinterpret_cast<void*>(host_in_kernel);
  p.gridDim = dim3(io_grid(nx / 8 > nl / 4 ? nx / 8 : nl / 4));
  p.blockDim = dim3(kIoThreads);
  p.kernelParams = args;
  return cudaGraphExecKernelNodeSetParams(ex, node, &p);
}

cudaError_t set_host_out_node(cudaGraphExec_t ex, cudaGraphNode_t node, const float* out_d,
                              float* out_h, int n) {
  void* args[] = {&out_d, &out_h, &n};
  cudaKernelNodeParams p{};
  p.func = reinterpret_cast<void*>(host_out_kernel);
  p.gridDim = dim3(io_grid(n / 4));
  p.blockDim = dim3(kIoThreads);
  p.kernelParams = args;
  return cudaGraphExecKernelNodeSetParams(ex, node, &p);
}

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
