// Host side of the C ABI: handle lifetime, validation, per-step kernel
// sequence, counters and traces.  All device memory is allocated at create
// (fixed addresses; "GLM 5.3 Testing: HBM Expert Allocation", "What the slot
// cache is": fixed addresses and shapes keep the step CUDA-graph safe), and a
// step only enqueues kernels.
#include <climits>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <algorithm>
#include <array>
#include <vector>

#include "internal.cuh"

using namespace moe;

namespace {
constexpr int kDefaultPrefillChunk = 32;  // experts staged per prefill chunk (two chunks held)
// A cached multi-row step copies its misses in this many parts; the miss groups
// of a part run as soon as that part has landed, while the next one copies.
constexpr int kMissParts = 3;
}

struct moe_cache {
  int L, E, S, H, I, k;          // S: the largest ring of any layer
  std::vector<int> S_of;         // [L] ring size of each layer
  std::vector<size_t> slot_off;  // [L + 1] first slot of each layer in the slot arrays
  long long Bw, Bs;
  moe_cache_opts_t opts;
  int device, num_sms;
  // device state, per layer blocks
  uint8_t* slot_w = nullptr;   // [sum S_l][Bw], layer l from slot_off[l]
  uint8_t* slot_s = nullptr;   // [sum S_l][Bs]
  float* gscale = nullptr;     // [L][E][3]
  int32_t* map = nullptr;      // [L][E]
  int32_t* owner = nullptr;    // [sum S_l]
  uint32_t* stamp = nullptr;   // [sum S_l]
  uint32_t* clock = nullptr;   // [L]
  DevStats* stats = nullptr;   // [L]
  moe_step_record_t* trace = nullptr;  // [L][cap]
  uint32_t* trace_head = nullptr;      // [L]
  // per-step workspace
  Plan* plan = nullptr;
  GemvWorkspace gemv{};
  // multi-row / bypass workspace (sized for max_rows)
  int max_picks = 0;
  GroupPlan* gp = nullptr;  // device copy of the header; arrays below
  QuantBuf xq{}, hq{};      // residual NVFP4 activations: x by row, h by pick
  int32_t* ids_ws = nullptr;
  std::vector<void*> extra;  // further device allocations, freed with the handle
  // host backing (device-visible addresses)
  std::vector<const uint8_t*> host_w, host_s;
  // one-row steps fork the miss path onto a second stream
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  cudaEvent_t part_done[kMissParts] = {};  // multi-row steps: a part of the misses landed
  // staged prefill: two halves of `chunk` expert slots, events per chunk
  int chunk = 0, nchunks = 0;
  uint8_t* stage_w = nullptr;  // [2 * chunk][Bw]
  uint8_t* stage_s = nullptr;  // [2 * chunk][Bs]
  std::vector<cudaEvent_t> ev_staged, ev_used;  // [nchunks]
  // tensor maps of the slot arrays and of the staging halves (grouped MMA weight tiles)
  TmaSource tma_slots, tma_stage;
  // optional per-kernel timing events (caller-owned)
  cudaEvent_t ev[MOE_TIMING_EVENTS] = {};
  bool timing = false;
  // moe_cache_step_host: device staging for max_rows rows, one-row step graphs per layer
  float* st_logits = nullptr;   // [max_rows][E]
  uint16_t* st_x = nullptr;     // [max_rows][H]
  float* st_out = nullptr;      // [max_rows][H]
  cudaStream_t cap = nullptr;   // capture stream
  std::vector<cudaGraphExec_t> graph;  // [L], null until captured
  std::vector<cudaGraph_t> graph_src;  // [L] the captured graphs (their nodes address the copies)
  std::vector<std::array<cudaGraphNode_t, 2>> graph_cp;  // [L] input and output move nodes
  std::vector<char> graph_warm;        // [L]: one eager one-row step done
};

namespace {

int cuda_err(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

template <class T>
cudaError_t dalloc(T** p, size_t count) {
  return cudaMalloc(reinterpret_cast<void**>(p), count * sizeof(T) + (count == 0 ? 16 : 0));
}

void free_all(moe_cache* h) {
  cudaFree(h->slot_w);
  cudaFree(h->slot_s);
  cudaFree(h->gscale);
  cudaFree(h->map);
  cudaFree(h->owner);
  cudaFree(h->stamp);
  cudaFree(h->clock);
  cudaFree(h->stats);
  cudaFree(h->trace);
  cudaFree(h->trace_head);
  cudaFree(h->plan);
  cudaFree(h->gemv.hbuf);
  cudaFree(h->gemv.ypart);
  cudaFree(h->gemv.tile_cnt);
  for (void* p : h->extra) cudaFree(p);
  h->extra.clear();
  for (cudaEvent_t e : h->ev_staged) cudaEventDestroy(e);
  for (cudaEvent_t e : h->ev_used) cudaEventDestroy(e);
  h->ev_staged.clear();
  h->ev_used.clear();
  if (h->fork) cudaEventDestroy(h->fork);
  if (h->join) cudaEventDestroy(h->join);
  for (cudaEvent_t& ev : h->part_done) {
    if (ev) cudaEventDestroy(ev);
    ev = nullptr;
  }
  if (h->side) cudaStreamDestroy(h->side);
  h->fork = h->join = nullptr;
  h->side = nullptr;
  for (cudaGraphExec_t g : h->graph)
    if (g) cudaGraphExecDestroy(g);
  h->graph.clear();
  for (cudaGraph_t g : h->graph_src)
    if (g) cudaGraphDestroy(g);
  h->graph_src.clear();
  if (h->cap) cudaStreamDestroy(h->cap);
  h->cap = nullptr;
  cudaFree(h->st_logits);
  cudaFree(h->st_x);
  cudaFree(h->st_out);
  h->st_logits = nullptr;
  h->st_x = nullptr;
  h->st_out = nullptr;
}

// Group plan, quantised-activation buffers and bypass ids for steps of up to
// max_rows rows.
bool alloc_multirow(moe_cache* h) {
  const size_t P = (size_t)h->opts.max_rows * h->k;
  const size_t G = P < (size_t)h->E ? P : (size_t)h->E;
  const size_t J = P + G;
  const size_t R = (size_t)h->opts.max_rows;
  h->max_picks = (int)P;
  auto get = [&](size_t bytes) -> void* {
    void* p = nullptr;
    if (cudaMalloc(&p, bytes ? bytes : 16) != cudaSuccess) return nullptr;
    h->extra.push_back(p);
    return p;
  };
  GroupPlan g{};
  g.g_expert = static_cast<int32_t*>(get(4 * G));
  g.g_start = static_cast<int32_t*>(get(4 * G));
  g.g_count = static_cast<int32_t*>(get(4 * G));
  g.g_wptr = static_cast<const uint8_t**>(get(sizeof(void*) * G));
  g.g_sptr = static_cast<const uint8_t**>(get(sizeof(void*) * G));
  g.g_gs = static_cast<float*>(get(4 * 3 * G));
  g.members = static_cast<int32_t*>(get(4 * P));
  g.jobs = static_cast<int32_t*>(get(4 * J));
  g.wts = static_cast<float*>(get(4 * P));
  g.g_job = static_cast<int32_t*>(get(4 * (G + 1)));
  h->gp = static_cast<GroupPlan*>(get(sizeof(GroupPlan)));
  h->ids_ws = static_cast<int32_t*>(get(4 * P));
  h->xq.codes = static_cast<uint8_t*>(get(R * kLevels * (h->H / 2)));
  h->xq.scales = static_cast<uint8_t*>(get(R * kLevels * (h->H / 16)));
  h->xq.gl = static_cast<float*>(get(4 * R * kLevels));
  h->hq.codes = static_cast<uint8_t*>(get(P * kLevels * (h->I / 2)));
  h->hq.scales = static_cast<uint8_t*>(get(P * kLevels * (h->I / 16)));
  h->hq.gl = static_cast<float*>(get(4 * P * kLevels));
  for (void* p : h->extra)
    if (!p) return false;
  if (!g.g_expert || !g.g_start || !g.g_count || !g.g_wptr || !g.g_sptr || !g.g_gs ||
      !g.members || !g.jobs || !g.wts || !g.g_job || !h->gp || !h->ids_ws || !h->xq.codes || !h->xq.scales ||
      !h->xq.gl || !h->hq.codes || !h->hq.scales || !h->hq.gl)
    return false;
  return cudaMemcpy(h->gp, &g, sizeof g, cudaMemcpyHostToDevice) == cudaSuccess;
}

// Resolve a pinned host pointer to the address kernels use; -1 if not pinned.
int device_view(const void* p, const uint8_t** out) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_NOT_PINNED;
  }
  if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr) return MOE_ERR_NOT_PINNED;
  *out = static_cast<const uint8_t*>(a.devicePointer);
  return MOE_OK;
}

// True when every byte of the n-byte scale bank is a finite, non-negative E4M3
// code: sign bit clear and not the NaN code 0x7F.  The tensor-core path reads
// block scales as unsigned E4M3, so a sign bit would be read as a different
// value there than on the CUDA-core path; the check keeps both paths defined
// alike.  Word-wise (eight bytes at a time), then the tail.
bool scales_valid(const uint8_t* p, size_t n) {
  const uint64_t hi = 0x8080808080808080ull, lo = 0x0101010101010101ull;
  size_t i = 0;
  if (((uintptr_t)p & 7) == 0) {
    for (; i + 8 <= n; i += 8) {
      uint64_t v;
      std::memcpy(&v, p + i, 8);
      const uint64_t t = v ^ (0x7Full * lo);  // a zero byte where v has 0x7F
      if ((v & hi) || ((t - lo) & ~t & hi)) return false;
    }
  }
  for (; i < n; ++i)
    if ((p[i] & 0x80) || p[i] == 0x7F) return false;
  return true;
}

int init_state(moe_cache* h) {
  const size_t LE = (size_t)h->L * h->E, LS = h->slot_off[h->L];
  std::vector<int32_t> map(LE, -1), owner(LS, -1);
  if (h->opts.all_resident) {
    for (int l = 0; l < h->L; ++l)
      for (int e = 0; e < h->E; ++e) {
        map[(size_t)l * h->E + e] = e;
        owner[h->slot_off[l] + e] = e;
      }
  }
  cudaError_t e = cudaMemcpy(h->map, map.data(), LE * 4, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(h->owner, owner.data(), LS * 4, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemset(h->stamp, 0, LS * 4);
  if (e == cudaSuccess) e = cudaMemset(h->clock, 0, (size_t)h->L * 4);
  if (e == cudaSuccess) e = cudaMemset(h->stats, 0, (size_t)h->L * sizeof(DevStats));
  if (e == cudaSuccess) e = cudaMemset(h->trace_head, 0, (size_t)h->L * 4);
  if (e == cudaSuccess)
    e = cudaMemset(h->gemv.tile_cnt, 0, sizeof(uint32_t) * kStepCounterWords);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  return cuda_err(e);
}

LayerDev layer_dev(moe_cache* h, int l) {
  LayerDev d;
  d.map = h->map + (size_t)l * h->E;
  d.owner = h->owner + h->slot_off[l];
  d.stamp = h->stamp + h->slot_off[l];
  d.clock = h->clock + l;
  d.slot_w = h->slot_w + h->slot_off[l] * h->Bw;
  d.slot_s = h->slot_s + h->slot_off[l] * h->Bs;
  d.host_w = h->host_w[l];
  d.host_s = h->host_s[l];
  d.gscale = h->gscale + (size_t)l * h->E * 3;
  d.stats = h->stats + l;
  d.trace_cap = (uint32_t)h->opts.trace_capacity;
  d.trace = h->opts.trace_capacity ? h->trace + (size_t)l * h->opts.trace_capacity : nullptr;
  d.trace_head = h->trace_head + l;
  d.step_ctr = h->gemv.tile_cnt;
  return d;
}

}  // namespace

extern "C" {

int moe_expert_bytes(int hidden, int inter, uint64_t* Bw, uint64_t* Bs) {
  if (hidden <= 0 || inter <= 0 || !Bw || !Bs) return MOE_ERR_ARG;
  const uint64_t n = 3ull * (uint64_t)hidden * (uint64_t)inter;
  *Bw = n / 2;
  *Bs = n / 16;
  return MOE_OK;
}

int moe_cache_create(moe_cache_t** out, int layers, int experts, int slots, int hidden, int inter,
                     int top_k, const moe_host_layer_t* host_backing,
                     const moe_cache_opts_t* opts) {
  if (!out) return MOE_ERR_ARG;
  *out = nullptr;
  moe_cache_opts_t o{};
  o.copy_backend = MOE_COPY_SM;
  o.bypass_rows = MOE_MAX_CACHED_ROWS;
  o.max_rows = 0;
  if (opts) {
    o = *opts;
    if (o.bypass_rows <= 0) o.bypass_rows = MOE_MAX_CACHED_ROWS;
    if (o.prefill_chunk == 0) o.prefill_chunk = kDefaultPrefillChunk;
  } else {
    o.prefill_chunk = kDefaultPrefillChunk;
  }
  // Every cached step (up to bypass_rows rows) must fit the multi-row workspace,
  // so max_rows is at least bypass_rows; the default (0) is exactly that: a
  // decode-only handle with no bypass workspace and no prefill staging.
  if (o.max_rows < o.bypass_rows) o.max_rows = o.bypass_rows;
  if (o.prefill_chunk < -1 || o.batch_invariant < 0 || o.batch_invariant > 1) return MOE_ERR_ARG;
  if (o.batch_invariant && !mma_supported(hidden, inter)) return MOE_ERR_UNSUPPORTED;
  if (layers < 1 || experts < 1 || top_k < 1 || hidden < 1 || inter < 1 || !host_backing)
    return MOE_ERR_ARG;
  if (o.trace_capacity < 0 || o.copy_backend != MOE_COPY_SM) return MOE_ERR_ARG;
  if (experts > MOE_MAX_EXPERTS || top_k > MOE_MAX_TOPK || top_k > experts ||
      hidden % 128 || inter % 128 || hidden > MOE_MAX_DIM || inter > MOE_MAX_DIM ||
      o.bypass_rows > MOE_MAX_CACHED_ROWS || !gemv_supported(hidden, inter, top_k))
    return MOE_ERR_UNSUPPORTED;
  if (o.all_resident) slots = experts;
  std::vector<int> S_of(layers, slots);
  if (o.slots_per_layer && !o.all_resident)
    for (int l = 0; l < layers; ++l) S_of[l] = o.slots_per_layer[l];
  for (int l = 0; l < layers; ++l)
    if (S_of[l] < top_k || S_of[l] > experts) return MOE_ERR_ARG;
  o.slots_per_layer = nullptr;  // read here only

  moe_cache* h = new (std::nothrow) moe_cache();
  if (!h) return MOE_ERR_OOM;
  h->L = layers;
  h->E = experts;
  h->S_of = S_of;
  h->slot_off.assign(layers + 1, 0);
  for (int l = 0; l < layers; ++l) h->slot_off[l + 1] = h->slot_off[l] + S_of[l];
  h->S = *std::max_element(S_of.begin(), S_of.end());
  h->H = hidden;
  h->I = inter;
  h->k = top_k;
  h->opts = o;
  uint64_t bw, bs;
  moe_expert_bytes(hidden, inter, &bw, &bs);
  h->Bw = (long long)bw;
  h->Bs = (long long)bs;
  int rc = MOE_OK;
  cudaError_t e = cudaGetDevice(&h->device);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
  if (e != cudaSuccess) {
    delete h;
    return MOE_ERR_CUDA;
  }
  h->host_w.resize(layers);
  h->host_s.resize(layers);
  std::vector<float> gs((size_t)layers * experts * 3);
  for (int l = 0; l < layers; ++l) {
    const moe_host_layer_t& hl = host_backing[l];
    if (!hl.w || !hl.s || !hl.gscale || ((uintptr_t)hl.w & 15) || ((uintptr_t)hl.s & 15)) {
      delete h;
      return MOE_ERR_ARG;
    }
    if ((rc = device_view(hl.w, &h->host_w[l])) != MOE_OK ||
        (rc = device_view(hl.s, &h->host_s[l])) != MOE_OK) {
      delete h;
      return rc;
    }
    std::memcpy(gs.data() + (size_t)l * experts * 3, hl.gscale, sizeof(float) * experts * 3);
    bool seen = false;  // layers may share one bank: check each bank once
    for (int m = 0; m < l && !seen; ++m) seen = host_backing[m].s == hl.s;
    if (!seen && !scales_valid(static_cast<const uint8_t*>(hl.s), (size_t)experts * h->Bs)) {
      delete h;
      return MOE_ERR_ARG;
    }
  }
  const size_t LS = h->slot_off[layers], LE = (size_t)layers * experts;
  size_t max_picks = (size_t)o.max_rows * top_k;
  if (max_picks < (size_t)MOE_MAX_PICKS) max_picks = MOE_MAX_PICKS;
  const int cap = o.trace_capacity;
  bool ok = dalloc(&h->slot_w, LS * (size_t)h->Bw) == cudaSuccess &&
            dalloc(&h->slot_s, LS * (size_t)h->Bs) == cudaSuccess &&
            dalloc(&h->gscale, LE * 3) == cudaSuccess && dalloc(&h->map, LE) == cudaSuccess &&
            dalloc(&h->owner, LS) == cudaSuccess && dalloc(&h->stamp, LS) == cudaSuccess &&
            dalloc(&h->clock, (size_t)layers) == cudaSuccess &&
            dalloc(&h->stats, (size_t)layers) == cudaSuccess &&
            dalloc(&h->trace, (size_t)layers * (cap ? cap : 1)) == cudaSuccess &&
            dalloc(&h->trace_head, (size_t)layers) == cudaSuccess &&
            dalloc(&h->plan, 1) == cudaSuccess &&
            dalloc(&h->gemv.hbuf, (size_t)max_picks * inter) == cudaSuccess &&
            dalloc(&h->gemv.ypart, (size_t)max_picks * hidden) == cudaSuccess &&
            dalloc(&h->gemv.tile_cnt, (size_t)kStepCounterWords) == cudaSuccess;
  ok = ok && alloc_multirow(h);
  if (ok && o.max_rows > o.bypass_rows && o.prefill_chunk > 0) {
    // staged prefill: two halves of `chunk` expert slots, two events per chunk
    h->chunk = o.prefill_chunk < experts ? o.prefill_chunk : experts;
    h->nchunks = (experts + h->chunk - 1) / h->chunk;
    void* w = nullptr;
    void* sc = nullptr;
    ok = cudaMalloc(&w, (size_t)2 * h->chunk * h->Bw) == cudaSuccess;
    if (w) h->extra.push_back(w);
    ok = ok && cudaMalloc(&sc, (size_t)2 * h->chunk * h->Bs) == cudaSuccess;
    if (sc) h->extra.push_back(sc);
    h->stage_w = static_cast<uint8_t*>(w);
    h->stage_s = static_cast<uint8_t*>(sc);
    for (int q = 0; ok && q < h->nchunks; ++q) {
      cudaEvent_t a = nullptr, b = nullptr;
      ok = cudaEventCreateWithFlags(&a, cudaEventDisableTiming) == cudaSuccess;
      if (a) h->ev_staged.push_back(a);
      ok = ok && cudaEventCreateWithFlags(&b, cudaEventDisableTiming) == cudaSuccess;
      if (b) h->ev_used.push_back(b);
    }
  }
  // Multi-row steps read slot (and staged) weights as TMA tiles where the
  // shape allows; otherwise (and for host-memory experts) with cp.async.
  if (ok) {
    make_tma_source(h->slot_w, h->slot_s, LS, hidden, inter, h->Bw, h->Bs, h->num_sms,
                    &h->tma_slots);
    if (h->stage_w)
      make_tma_source(h->stage_w, h->stage_s, 2ull * h->chunk, hidden, inter, h->Bw, h->Bs,
                      h->num_sms, &h->tma_stage);
  }
  // The second stream carries the missed picks' read-through pass, the step's
  // critical path: highest priority, so its CTAs are placed before the
  // resident picks' persistent grids fill the SMs.
  int prio_least = 0, prio_greatest = 0;
  ok = ok && cudaDeviceGetStreamPriorityRange(&prio_least, &prio_greatest) == cudaSuccess;
  ok = ok &&
       cudaStreamCreateWithPriority(&h->side, cudaStreamNonBlocking, prio_greatest) ==
           cudaSuccess &&
       cudaEventCreateWithFlags(&h->fork, cudaEventDisableTiming) == cudaSuccess &&
       cudaEventCreateWithFlags(&h->join, cudaEventDisableTiming) == cudaSuccess;
  for (int q = 0; ok && q < kMissParts; ++q)
    ok = cudaEventCreateWithFlags(&h->part_done[q], cudaEventDisableTiming) == cudaSuccess;
  // host-buffer steps: staging for max_rows rows and a capture stream
  ok = ok && dalloc(&h->st_logits, (size_t)o.max_rows * experts) == cudaSuccess &&
       dalloc(&h->st_x, (size_t)o.max_rows * hidden) == cudaSuccess &&
       dalloc(&h->st_out, (size_t)o.max_rows * hidden) == cudaSuccess &&
       cudaStreamCreateWithFlags(&h->cap, cudaStreamNonBlocking) == cudaSuccess;
  if (ok) {
    h->graph.assign(layers, nullptr);
    h->graph_src.assign(layers, nullptr);
    h->graph_cp.assign(layers, {nullptr, nullptr});
    h->graph_warm.assign(layers, 0);
  }
  if (!ok) {
    cudaGetLastError();
    free_all(h);
    delete h;
    return MOE_ERR_OOM;
  }
  e = cudaMemcpy(h->gscale, gs.data(), gs.size() * sizeof(float), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemset(h->plan, 0, sizeof(Plan));  // wait_us 0: default limit
  if (e == cudaSuccess && o.all_resident) {
    for (int l = 0; l < layers && e == cudaSuccess; ++l) {
      e = cudaMemcpy(h->slot_w + h->slot_off[l] * h->Bw, host_backing[l].w,
                     (size_t)experts * h->Bw, cudaMemcpyHostToDevice);
      if (e == cudaSuccess)
        e = cudaMemcpy(h->slot_s + h->slot_off[l] * h->Bs, host_backing[l].s,
                       (size_t)experts * h->Bs, cudaMemcpyHostToDevice);
    }
  }
  if (e != cudaSuccess || (rc = init_state(h)) != MOE_OK) {
    free_all(h);
    delete h;
    return rc != MOE_OK ? rc : MOE_ERR_CUDA;
  }
  *out = h;
  return MOE_OK;
}

int moe_cache_step(moe_cache_t* h, int layer, int rows, const float* router_logits,
                   const uint16_t* x, float* out, void* stream) {
  if (!h || layer < 0 || layer >= h->L || rows < 1 || !router_logits || !x || !out)
    return MOE_ERR_ARG;
  if (((uintptr_t)x & 15) || ((uintptr_t)out & 15)) return MOE_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (rows > h->opts.bypass_rows && rows > h->opts.max_rows) return MOE_ERR_UNSUPPORTED;
  const bool one_row = rows == 1 && !h->opts.batch_invariant;
  if (!one_row && !mma_supported(h->H, h->I)) return MOE_ERR_UNSUPPORTED;
  const LayerDev L = layer_dev(h, layer);
  // inside a capture an event record must be an external node to be replayed
  auto mark = [&](int i, cudaStream_t s) -> cudaError_t {
    if (!h->timing) return cudaSuccess;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return e;
    return cudaEventRecordWithFlags(
        h->ev[i], s, cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : 0u);
  };
  uint32_t* flags = &(h->stats + layer)->flags;
  cudaError_t e = mark(0, st);
  if (one_row) {
    // One row.  After route/remap the missed picks take a second stream: one
    // read-through launch reads each missed expert once over the host link,
    // writes it through to the victim slot and computes its gate/up and then
    // its down rows on the way in.  Meanwhile the resident picks' gate/up and
    // down run on the caller's stream, so the hit experts' HBM reads overlap
    // the host-link transfer.  Each pick's weighted output y'_j is computed
    // with the same arithmetic whichever path it takes, and the CTA that
    // completes an output block's count over the step's picks (from either
    // launch) adds that block in rank order, so the result does not depend on
    // the hit/miss split.
    if (e == cudaSuccess)
      e = launch_route_remap(st, router_logits, rows, h->E, h->k, h->S_of[layer], h->Bw, h->Bs, L, h->plan,
                             h->opts.all_resident, nullptr);
    if (e == cudaSuccess) e = mark(1, st);
    if (e == cudaSuccess) e = cudaEventRecord(h->fork, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->side, h->fork, 0);
    // missed picks: a small grid keeps the host link saturated without taking
    // many SMs from the resident picks
    const int rt_grid = h->num_sms / 2 > 8 ? h->num_sms / 2 : 8;
    // the ring and bank every pointer of the plan must lie in (checked on the device)
    PickBounds pb;
    pb.slot_w = L.slot_w;
    pb.slot_s = L.slot_s;
    pb.slot_n = (unsigned long long)h->S_of[layer];
    pb.host_w = L.host_w;
    pb.host_s = L.host_s;
    pb.host_n = (unsigned long long)h->E;
    pb.Bw = h->Bw;
    pb.Bs = h->Bs;
    const GemvLaunch miss{kPicksMiss, true, rt_grid, 2, false, pb};
    // resident picks: slot bytes from HBM
    // Gate/up is launched normally, after route/remap, so the second stream's
    // higher priority places the read-through CTAs first (two gate/up CTAs
    // fill an SM's registers); the down pass starts as gate/up drains
    // (programmatic launch, not across timing events).
    const GemvLaunch hit_gu{kPicksHit, false, 0, 3, false, pb},
        hit_dn{kPicksHit, false, 0, 4, !h->timing, pb};
    if (e == cudaSuccess) e = mark(2, h->side);
    if (e == cudaSuccess)
      e = launch_gemv_readthrough(h->side, h->plan, x, h->H, h->I, h->k, h->gemv, flags,
                                  h->num_sms, miss, out, h->gemv.tile_cnt);
    if (e == cudaSuccess) e = mark(3, h->side);
    if (e == cudaSuccess) e = mark(4, h->side);
    if (e == cudaSuccess) e = cudaEventRecord(h->join, h->side);
    if (e == cudaSuccess)
      e = launch_gemv_gateup(st, h->plan, x, h->H, h->I, h->k, h->gemv, flags, h->num_sms,
                             hit_gu);
    if (e == cudaSuccess) e = mark(5, st);
    if (e == cudaSuccess)
      e = launch_gemv_down(st, h->plan, h->H, h->I, h->k, h->gemv, flags, h->num_sms, hit_dn,
                           out, h->gemv.tile_cnt);
    if (e == cudaSuccess) e = mark(6, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, h->join, 0);
    if (e == cudaSuccess) e = mark(7, st);
    return cuda_err(e);
  }
  // several rows: experts grouped, each read once for all its rows (tensor cores)
  const int npicks = rows * h->k;
  const bool cached_rows = rows <= h->opts.bypass_rows;
  if (cached_rows) {
    // The misses copy host -> slot on the second stream (a grid that keeps the
    // host link busy without taking the SMs) while the caller's stream runs
    // the hit groups below; the miss groups wait for the copy.
    if (e == cudaSuccess)
      e = launch_route_remap(st, router_logits, rows, h->E, h->k, h->S_of[layer], h->Bw, h->Bs, L, h->plan,
                             h->opts.all_resident, h->gp);
    if (e == cudaSuccess) e = mark(1, st);
    if (e == cudaSuccess) e = cudaEventRecord(h->fork, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->side, h->fork, 0);
    for (int q = 0; q < kMissParts && e == cudaSuccess; ++q) {
      if (!h->opts.all_resident)
        e = launch_miss_copy(h->side, h->plan, L.host_w, L.host_s, L.slot_w, L.slot_s, h->Bw,
                             h->Bs, std::max(8, h->num_sms / 2), q, kMissParts);
      if (e == cudaSuccess) e = cudaEventRecord(h->part_done[q], h->side);
    }
    if (e == cudaSuccess) e = cudaEventRecord(h->join, h->side);
  } else {
    // prefill bypass: experts read from host memory, cache untouched
    if (e == cudaSuccess)
      e = launch_route_rows(st, router_logits, rows, h->E, h->k, h->ids_ws, h->gp, L, h->Bw, h->Bs);
    if (e == cudaSuccess) e = mark(1, st);
  }
  if (e == cudaSuccess) e = mark(2, st);
  if (e == cudaSuccess) e = launch_quantize_rows(st, x, true, rows, h->H, h->xq);
  if (rows > h->opts.bypass_rows && h->chunk > 0) {
    // Staged prefill: chunk q's experts go host -> HBM staging on the second
    // stream while the caller's stream runs chunk q-1's grouped MMAs from the
    // staged bytes; a staging half is refilled only after the MMAs that read it.
    // Every chunk is launched (graph-safe); chunks past the step's groups exit.
    const int C = h->chunk;
    const int gx_gu = std::max(1, 2 * h->num_sms / (h->I / 64));
    const int gx_dn = std::max(1, 2 * h->num_sms / (h->H / 128));
    if (e == cudaSuccess) e = cudaEventRecord(h->fork, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->side, h->fork, 0);
    for (int q = 0; q < h->nchunks && e == cudaSuccess; ++q) {
      const int g0 = q * C, g1 = g0 + C;
      if (q >= 2) e = cudaStreamWaitEvent(h->side, h->ev_used[q - 2], 0);
      if (e == cudaSuccess)
        e = launch_stage_copy(h->side, h->gp, q, C, L, h->stage_w, h->stage_s, h->Bw, h->Bs,
                              std::max(8, h->num_sms / 2));
      if (e == cudaSuccess) e = cudaEventRecord(h->ev_staged[q], h->side);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(st, h->ev_staged[q], 0);
      if (e == cudaSuccess)
        e = launch_grouped_mma(st, h->gp, gx_gu, true, h->H, h->I, h->k, h->xq, h->gemv.hbuf,
                               flags, g0, g1, &h->tma_stage);
      if (e == cudaSuccess)
        e = launch_quantize_members(st, h->gemv.hbuf, h->I, h->gp, g0, g1, h->hq, h->num_sms);
      if (e == cudaSuccess)
        e = launch_grouped_mma(st, h->gp, gx_dn, false, h->H, h->I, h->k, h->hq, h->gemv.ypart,
                               flags, g0, g1, &h->tma_stage);
      if (e == cudaSuccess) e = cudaEventRecord(h->ev_used[q], st);
    }
    if (e == cudaSuccess) e = mark(3, st);
    if (e == cudaSuccess) e = mark(5, st);
    if (e == cudaSuccess) e = mark(4, st);
    if (e == cudaSuccess) e = mark(6, st);
  } else if (cached_rows) {
    // hit groups [0, n_hit) now, then each part of the miss groups once that
    // part's bytes are in the slots (the next part copies meanwhile): gate/up,
    // the members' h in residual NVFP4, down, each pass.  A union larger than
    // the ring (possible only when npicks > S) bypasses on the device and
    // reads host memory.
    int gr[kMissParts + 2] = {0, kHitGroups};
    for (int q = 1; q <= kMissParts; ++q) gr[q + 1] = miss_part(q, kMissParts);
    gr[kMissParts + 1] = INT_MAX;
    const bool may_bypass = npicks > h->S_of[layer];
    for (int pass = 0; pass <= kMissParts && e == cudaSuccess; ++pass) {
      if (pass >= 1) e = cudaStreamWaitEvent(st, h->part_done[pass - 1], 0);
      if (e == cudaSuccess)
        e = launch_grouped_mma(st, h->gp, npicks, true, h->H, h->I, h->k, h->xq, h->gemv.hbuf,
                               flags, gr[pass], gr[pass + 1], &h->tma_slots, may_bypass);
      if (e == cudaSuccess)
        e = launch_quantize_members(st, h->gemv.hbuf, h->I, h->gp, gr[pass], gr[pass + 1],
                                    h->hq, h->num_sms);
      if (e == cudaSuccess)
        e = launch_grouped_mma(st, h->gp, npicks, false, h->H, h->I, h->k, h->hq, h->gemv.ypart,
                               flags, gr[pass], gr[pass + 1], &h->tma_slots, may_bypass);
      if (e == cudaSuccess && pass == 0) e = mark(3, st);
      if (e == cudaSuccess && pass == 0) e = mark(5, st);
    }
    if (e == cudaSuccess) e = mark(4, st);
    if (e == cudaSuccess) e = mark(6, st);
  } else {
    if (e == cudaSuccess)
      e = launch_grouped_mma(st, h->gp, npicks, true, h->H, h->I, h->k, h->xq, h->gemv.hbuf,
                             flags);
    if (e == cudaSuccess) e = mark(3, st);
    if (e == cudaSuccess) e = mark(5, st);
    if (e == cudaSuccess) e = launch_quantize_rows(st, h->gemv.hbuf, false, npicks, h->I, h->hq);
    if (e == cudaSuccess)
      e = launch_grouped_mma(st, h->gp, npicks, false, h->H, h->I, h->k, h->hq, h->gemv.ypart,
                             flags);
    if (e == cudaSuccess) e = mark(4, st);
    if (e == cudaSuccess) e = mark(6, st);
  }
  if (e == cudaSuccess) e = launch_combine(st, h->gp, h->gemv.ypart, out, rows, h->H, h->k);
  if (e == cudaSuccess) e = mark(7, st);
  return cuda_err(e);
}

int moe_cache_stats(const moe_cache_t* h, int layer, moe_cache_stats_t* out) {
  if (!h || !out || layer < -1 || layer >= h->L) return MOE_ERR_ARG;
  std::vector<DevStats> ds(h->L);
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess)
    e = cudaMemcpy(ds.data(), h->stats, sizeof(DevStats) * h->L, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  std::memset(out, 0, sizeof *out);
  for (int l = 0; l < h->L; ++l) {
    if (layer >= 0 && l != layer) continue;
    out->steps += ds[l].steps;
    out->picks += ds[l].picks;
    out->hits += ds[l].hits;
    out->misses += ds[l].misses;
    out->evictions += ds[l].evictions;
    out->bytes_copied += ds[l].bytes_copied;
    out->bypass_calls += ds[l].bypass_calls;
    out->error_flags |= ds[l].flags;
  }
  return MOE_OK;
}

int moe_cache_slot_map(const moe_cache_t* h, int layer, int32_t* expert_of_slot) {
  if (!h || !expert_of_slot || layer < 0 || layer >= h->L) return MOE_ERR_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess)
    e = cudaMemcpy(expert_of_slot, h->owner + h->slot_off[layer],
                   sizeof(int32_t) * h->S_of[layer], cudaMemcpyDeviceToHost);
  return cuda_err(e);
}

int moe_cache_layer_slots(const moe_cache_t* h, int layer, int* slots) {
  if (!h || !slots || layer < 0 || layer >= h->L) return MOE_ERR_ARG;
  *slots = h->S_of[layer];
  return MOE_OK;
}

int moe_cache_slot_bytes(const moe_cache_t* h, int layer, int slot, void* w_dst, void* s_dst) {
  if (!h || layer < 0 || layer >= h->L || slot < 0 || slot >= h->S_of[layer]) return MOE_ERR_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  const size_t ls = h->slot_off[layer] + slot;
  if (e == cudaSuccess && w_dst)
    e = cudaMemcpy(w_dst, h->slot_w + ls * h->Bw, h->Bw, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && s_dst)
    e = cudaMemcpy(s_dst, h->slot_s + ls * h->Bs, h->Bs, cudaMemcpyDeviceToHost);
  return cuda_err(e);
}

int moe_cache_trace(const moe_cache_t* h, int layer, moe_step_record_t* recs, int max_recs,
                    int* n_recs) {
  if (!h || !recs || !n_recs || max_recs < 0 || layer < 0 || layer >= h->L) return MOE_ERR_ARG;
  const int cap = h->opts.trace_capacity;
  if (cap <= 0) return MOE_ERR_ARG;
  uint32_t head = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess)
    e = cudaMemcpy(&head, h->trace_head + layer, 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  uint32_t n = head < (uint32_t)cap ? head : (uint32_t)cap;
  if (n > (uint32_t)max_recs) n = (uint32_t)max_recs;
  const moe_step_record_t* base = h->trace + (size_t)layer * cap;
  for (uint32_t i = 0; i < n && e == cudaSuccess; ++i) {
    const uint32_t idx = (head - n + i) % (uint32_t)cap;
    e = cudaMemcpy(recs + i, base + idx, sizeof(moe_step_record_t), cudaMemcpyDeviceToHost);
  }
  *n_recs = (int)n;
  return cuda_err(e);
}

namespace {

// The device-side address of page-locked host memory (null for pageable or
// device memory).
void* mapped(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// The step's moves and kernels on stream s: logits and x host -> staging, the
// step over the staging buffers, out staging -> host.  Page-locked buffers are
// read and written by kernels through their device addresses; pageable ones
// go through copies (synchronous for the host).
int step_host_enqueue(moe_cache* h, int layer, int rows, const float* lg, const uint16_t* x,
                      float* out, cudaStream_t s) {
  const size_t nl = (size_t)rows * h->E, nx = (size_t)rows * h->H;
  const void* dlg = mapped(lg);
  const void* dx = mapped(x);
  void* dout = mapped(out);
  const bool direct = dlg && dx && dout;
  cudaError_t e =
      direct ? launch_host_in(s, static_cast<const float*>(dlg), static_cast<const uint16_t*>(dx),
                              h->st_logits, h->st_x, (int)nl, (int)nx)
             : cudaMemcpyAsync(h->st_logits, lg, nl * sizeof(float), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess && !direct)
    e = cudaMemcpyAsync(h->st_x, x, nx * sizeof(uint16_t), cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  const int rc = moe_cache_step(h, layer, rows, h->st_logits, h->st_x, h->st_out, s);
  if (rc != MOE_OK) return rc;
  return cuda_err(direct ? launch_host_out(s, h->st_out, static_cast<float*>(dout), (int)nx)
                         : cudaMemcpyAsync(out, h->st_out, nx * sizeof(float),
                                           cudaMemcpyDeviceToHost, s));
}

// Capture the layer's one-row step with its input and output moves (page-locked
// buffers); find the nodes of the two move kernels.
int capture_step_graph(moe_cache* h, int layer, const float* lg, const uint16_t* x, float* out) {
  cudaGraph_t g = nullptr;
  cudaError_t e = cudaStreamBeginCapture(h->cap, cudaStreamCaptureModeThreadLocal);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  const int rc = step_host_enqueue(h, layer, 1, lg, x, out, h->cap);
  e = cudaStreamEndCapture(h->cap, &g);
  if (rc != MOE_OK || e != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    cudaGetLastError();
    return rc != MOE_OK ? rc : MOE_ERR_CUDA;
  }
  size_t n = 0;
  e = cudaGraphGetNodes(g, nullptr, &n);
  std::vector<cudaGraphNode_t> nodes(n);
  if (e == cudaSuccess) e = cudaGraphGetNodes(g, nodes.data(), &n);
  std::array<cudaGraphNode_t, 2> cp = {nullptr, nullptr};
  for (size_t i = 0; i < n && e == cudaSuccess; ++i) {
    cudaGraphNodeType t;
    if ((e = cudaGraphNodeGetType(nodes[i], &t)) != cudaSuccess || t != cudaGraphNodeTypeKernel)
      continue;
    cudaKernelNodeParams kp{};
    if (cudaGraphKernelNodeGetParams(nodes[i], &kp) != cudaSuccess) {
      cudaGetLastError();
      continue;
    }
    if (is_host_in_node(kp.func)) cp[0] = nodes[i];
    else if (is_host_out_node(kp.func)) cp[1] = nodes[i];
  }
  cudaGraphExec_t ex = nullptr;
  if (e == cudaSuccess && cp[0] && cp[1]) e = cudaGraphInstantiate(&ex, g, 0);
  if (e != cudaSuccess || !ex) {
    cudaGraphDestroy(g);
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  h->graph[layer] = ex;
  h->graph_src[layer] = g;
  h->graph_cp[layer] = cp;
  return MOE_OK;
}

}  // namespace

int moe_cache_step_host(moe_cache_t* h, int layer, int rows, const float* router_logits,
                        const uint16_t* x, float* out, void* stream) {
  if (!h || layer < 0 || layer >= h->L || rows < 1 || rows > h->opts.max_rows || !router_logits ||
      !x || !out)
    return MOE_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // One-row steps with page-locked buffers replay a graph of the moves and the
  // step: the layer's first such step runs eagerly (its launches set every
  // kernel's attributes), the second captures the graph on the handle's own
  // stream, later ones point its move kernels at the call's buffers and launch it.
  const void* dlg = rows == 1 ? mapped(router_logits) : nullptr;
  const void* dx = rows == 1 ? mapped(x) : nullptr;
  void* dout = rows == 1 ? mapped(out) : nullptr;
  if (rows == 1 && !h->timing && h->graph_warm[layer] && dlg && dx && dout) {
    if (!h->graph[layer]) {
      const int rc = capture_step_graph(h, layer, router_logits, x, out);
      if (rc != MOE_OK) return rc;
    } else {
      const auto& cp = h->graph_cp[layer];
      cudaGraphExec_t ex = h->graph[layer];
      cudaError_t e = set_host_in_node(ex, cp[0], static_cast<const float*>(dlg),
                                       static_cast<const uint16_t*>(dx), h->st_logits, h->st_x,
                                       h->E, h->H);
      if (e == cudaSuccess)
        e = set_host_out_node(ex, cp[1], h->st_out, static_cast<float*>(dout), h->H);
      if (e != cudaSuccess) return MOE_ERR_CUDA;
    }
    return cuda_err(cudaGraphLaunch(h->graph[layer], st));
  }
  if (rows == 1 && !h->timing) h->graph_warm[layer] = 1;
  return step_host_enqueue(h, layer, rows, router_logits, x, out, st);
}

int moe_cache_reset(moe_cache_t* h) {
  if (!h) return MOE_ERR_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  return init_state(h);
}

int moe_cache_set_wait_timeout(moe_cache_t* h, int microseconds) {
  if (!h || microseconds < 0) return MOE_ERR_ARG;
  const uint32_t us = (uint32_t)microseconds;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(&h->plan->wait_us, &us, sizeof us, cudaMemcpyHostToDevice);
  return cuda_err(e);
}

int moe_cache_destroy(moe_cache_t* h) {
  if (!h) return MOE_OK;
  cudaDeviceSynchronize();
  free_all(h);
  delete h;
  return MOE_OK;
}

int moe_cache_set_timing_events(moe_cache_t* h, void* const* events) {
  if (!h) return MOE_ERR_ARG;
  if (!events) {
    h->timing = false;
    return MOE_OK;
  }
  for (int i = 0; i < MOE_TIMING_EVENTS; ++i) {
    if (!events[i]) return MOE_ERR_ARG;
    h->ev[i] = static_cast<cudaEvent_t>(events[i]);
  }
  h->timing = true;
  return MOE_OK;
}

const char* moe_cache_strerror(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_ARG: return "invalid argument";
    case MOE_ERR_NOT_PINNED: return "host backing is not pinned, device-mapped memory";
    case MOE_ERR_OOM: return "out of memory";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_UNSUPPORTED: return "shape or row count outside the supported limits";
    default: return "unknown error";
  }
}

int moe_host_alloc(void** out, size_t bytes) {
  if (!out || bytes == 0) return MOE_ERR_ARG;
  *out = nullptr;
  void* p = nullptr;
  if (cudaHostAlloc(&p, bytes, cudaHostAllocPortable | cudaHostAllocMapped) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_OOM;
  }
  void* dp = nullptr;
  if (cudaHostGetDevicePointer(&dp, p, 0) != cudaSuccess || dp != p) {
    cudaGetLastError();
    cudaFreeHost(p);
    return MOE_ERR_NOT_PINNED;
  }
  *out = p;
  return MOE_OK;
}

int moe_host_free(void* p) {
  if (!p) return MOE_OK;
  return cuda_err(cudaFreeHost(p));
}

int moe_probe_host_link(const void* host_src, void* dev_dst, size_t bytes, int method, int iters,
                        double* best_gbps) {
  if (!host_src || !dev_dst || !best_gbps || bytes == 0 || (bytes & 15) || iters < 1 ||
      ((uintptr_t)host_src & 15) || ((uintptr_t)dev_dst & 15) || (method != 0 && method != 1))
    return MOE_ERR_ARG;
  const uint8_t* src = nullptr;
  int rc = device_view(host_src, &src);
  if (rc != MOE_OK) return rc;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaStream_t st;
  cudaEvent_t a, b;
  if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) return MOE_ERR_CUDA;
  cudaEventCreate(&a);
  cudaEventCreate(&b);
  double best = 0.0;
  cudaError_t e = cudaSuccess;
  for (int it = 0; it < iters + 1 && e == cudaSuccess; ++it) {
    cudaEventRecord(a, st);
    if (method == 0)
      e = launch_link_probe(st, src, dev_dst, bytes, 2 * sms);
    else
      e = cudaMemcpyAsync(dev_dst, host_src, bytes, cudaMemcpyHostToDevice, st);
    cudaEventRecord(b, st);
    if (e == cudaSuccess) e = cudaEventSynchronize(b);
    float ms = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, a, b);
    if (e == cudaSuccess && it > 0 && ms > 0.f) {
      const double g = (double)bytes / (ms * 1e-3) / 1e9;
      if (g > best) best = g;
    }
  }
  cudaEventDestroy(a);
  cudaEventDestroy(b);
  cudaStreamDestroy(st);
  *best_gbps = best;
  return cuda_err(e);
}

}  // extern "C"
