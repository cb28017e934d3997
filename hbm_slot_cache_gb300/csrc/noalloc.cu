// moe_expert_pass_noalloc: the one-row expert pass (gate/up -> SwiGLU -> down
// -> weighted combine) for callers that cannot allocate device memory.
//
// Some callers must not call cudaMalloc: a serving engine that has already
// reserved all free HBM for its own pools (KV cache, expert slot rings) and
// owns every further byte, or a latency-critical decode loop where an
// allocation's implicit device-wide synchronisation is not acceptable.  They
// bring their own inputs and outputs; the scratch the expert kernels need (the
// per-step plan, h, per-expert partial outputs and the tile tickets) lives in
// one file-scope __device__ array instead of a handle's workspace.
//
// The array is a fixed size (kScratchBytes, about 1.1 MB), held by every GPU
// that loads the library until the process exits.  Host code must not use the
// array's name as an address: the first call on each device, with that device
// current, resolves its device address with cudaGetSymbolAddress (so make that
// first call before any stream capture), and kernels get that address.
// All calls share the one array and it keeps the last call's contents: the
// tile tickets and the error-flags word are cleared on every call, and two
// calls whose work overlaps on the GPU (different streams without ordering)
// race on it.  A call's device-side error flags (a bounded wait that gave up,
// a plan check that failed) reach the caller through an optional device word.
// The array's address is looked up once per device for the life of the
// process: the pass must not be used on a device after cudaDeviceReset.
#include <mutex>

#include "internal.cuh"

namespace moe {
namespace {

constexpr int kMaxK = MOE_MAX_TOPK;
constexpr int kMaxDim = MOE_MAX_DIM;
constexpr size_t kPlanBytes = (sizeof(Plan) + 255) / 256 * 256;
constexpr size_t kHBytes = sizeof(float) * kMaxK * kMaxDim;     // h [k][inter]
constexpr size_t kYBytes = sizeof(float) * kMaxK * kMaxDim;     // y_j [k][hidden]
constexpr size_t kTileWords = kStepCounterWords;                 // step counters
constexpr size_t kTileBytes = (sizeof(uint32_t) * kTileWords + 255) / 256 * 256;
constexpr size_t kFlagBytes = 256;
constexpr size_t kScratchBytes = kPlanBytes + kHBytes + kYBytes + kTileBytes + kFlagBytes;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
struct DeviceScratch {
  unsigned char* base = nullptr;  // device address of g_noalloc_scratch
  int num_sms = 0;
};
DeviceScratch g_dev[kMaxDevices];
std::mutex g_setup_mu;

// Everything the plan needs, passed by value to the plan-builder kernel.
struct PlanArgs {
  const uint8_t* w[kMaxK];
  const uint8_t* s[kMaxK];
  float gs[kMaxK][3];
  float wts[kMaxK];
  int k;
};

// Writes the one-row plan into the scratch array and clears the tile tickets
// and the error flags.
__global__ void noalloc_plan_kernel(PlanArgs a, Plan* plan, uint32_t* tile_cnt, int ntiles,
                                    uint32_t* flags) {
  const int t = threadIdx.x;
  if (t < a.k) {
    plan->ids[t] = t;
    plan->wts[t] = a.wts[t];
    plan->wptr[t] = a.w[t];
    plan->sptr[t] = a.s[t];
    plan->gs[t][0] = a.gs[t][0];
    plan->gs[t][1] = a.gs[t][1];
    plan->gs[t][2] = a.gs[t][2];
    plan->gs[t][3] = 0.f;
  }
  if (t == 0) {
    plan->rows = 1;
    plan->npicks = a.k;
    plan->n_union = a.k;
    plan->n_miss = 0;
    plan->bypass = 0;
    plan->n_hit = 0;
    plan->wait_us = 0;  // the default wait limit
    *flags = 0u;
  }
  for (int i = t; i < ntiles; i += blockDim.x) tile_cnt[i] = 0;
}

// The call's error flags to the caller's word (after the expert kernels).
__global__ void noalloc_flags_kernel(const uint32_t* flags, uint32_t* flags_out) {
  *flags_out = *reinterpret_cast<const volatile uint32_t*>(flags);
}

// Once per device, with that device current: resolve the array's address.
int setup_device(int dev, DeviceScratch** out) {
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  DeviceScratch& d = g_dev[dev];
  if (!d.base) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    d.num_sms = sms;
    d.base = static_cast<unsigned char*>(p);
  }
  *out = &d;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_expert_pass_noalloc(int k, int hidden, int inter, const void* const* expert_w,
                                       const void* const* expert_s, const float* gscale,
                                       const float* weights, const uint16_t* x, float* out,
                                       uint32_t* flags_out, void* stream) {
  if (k < 1 || hidden < 1 || inter < 1 || !expert_w || !expert_s || !gscale || !weights || !x ||
      !out || ((uintptr_t)x & 15) || ((uintptr_t)out & 15) || ((uintptr_t)flags_out & 3))
    return MOE_ERR_ARG;
  if (k > kMaxK || hidden > kMaxDim || inter > kMaxDim || hidden % 128 || inter % 128 ||
      !gemv_supported(hidden, inter, k))
    return MOE_ERR_UNSUPPORTED;
  for (int j = 0; j < k; ++j)
    if (!expert_w[j] || !expert_s[j] || ((uintptr_t)expert_w[j] & 15) ||
        ((uintptr_t)expert_s[j] & 15))
      return MOE_ERR_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  DeviceScratch* d = nullptr;
  int rc = setup_device(dev, &d);
  if (rc != MOE_OK) return rc;

  Plan* plan = reinterpret_cast<Plan*>(d->base);
  GemvWorkspace ws;
  ws.hbuf = reinterpret_cast<float*>(d->base + kPlanBytes);
  ws.ypart = reinterpret_cast<float*>(d->base + kPlanBytes + kHBytes);
  ws.tile_cnt = reinterpret_cast<uint32_t*>(d->base + kPlanBytes + kHBytes + kYBytes);
  uint32_t* flags =
      reinterpret_cast<uint32_t*>(d->base + kPlanBytes + kHBytes + kYBytes + kTileBytes);
  ws.flags = flags;

  PlanArgs a;
  a.k = k;
  for (int j = 0; j < k; ++j) {
    a.w[j] = static_cast<const uint8_t*>(expert_w[j]);
    a.s[j] = static_cast<const uint8_t*>(expert_s[j]);
    a.gs[j][0] = gscale[3 * j + 0];
    a.gs[j][1] = gscale[3 * j + 1];
    a.gs[j][2] = gscale[3 * j + 2];
    a.wts[j] = weights[j];
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  noalloc_plan_kernel<<<1, 64, 0, st>>>(a, plan, ws.tile_cnt, (int)kTileWords, flags);
  cudaError_t e = cudaGetLastError();
  const GemvLaunch all{kPicksAll, false, 0, 0};  // the caller's experts: pointers unchecked
  if (e == cudaSuccess)
    e = launch_gemv_gateup(st, plan, x, hidden, inter, k, ws, flags, d->num_sms, all);
  if (e == cudaSuccess)
    e = launch_gemv_down(st, plan, hidden, inter, k, ws, flags, d->num_sms, all, out, ws.tile_cnt);
  if (e == cudaSuccess && flags_out) {
    noalloc_flags_kernel<<<1, 1, 0, st>>>(flags, flags_out);
    e = cudaGetLastError();
  }
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
