// Offline slot-policy analysis over a routing trace (host code, no GPU).
//
// "GB300 GLM 5.3 Testing": the slot cache's LRU is compared with a hindsight
// static pin of the hottest experts and with hybrids that pin part of the
// ring and run LRU on the rest, on a recorded routing trace; the ring size S
// of each layer is then chosen from that layer's trace ("GLM 5.3 Testing: HBM
// Expert Allocation": per-layer S from traces).  This file evaluates those
// policies with the cache's exact rules and sizes per-layer rings for a total
// slot budget.
//
// The LRU rules are the device cache's: a step's picks are its rows' top-k
// ids; a pick hits if its expert was resident when the step began; each
// missing expert of the union is fetched once, in ascending expert id, into
// the unused-this-step slot with the smallest (last-use step, slot id); a
// union larger than the ring bypasses it (every expert of the union is read
// from host memory, the ring and its clock are untouched).
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <vector>

#include "../../include/moe_slot_cache.h"

namespace {

struct Ring {
  int S;
  std::vector<int32_t> slot_of;   // expert -> slot or -1
  std::vector<int32_t> owner;     // slot -> expert or -1
  std::vector<uint32_t> last;     // slot -> last-use step (0: never)
  uint32_t clock = 0;
  Ring(int experts, int slots) : S(slots), slot_of(experts, -1), owner(slots, -1), last(slots, 0) {}
};

// One step of the ring over the sorted union `u` (picks counted by the caller).
// Returns false (and changes nothing) if the union does not fit: a bypass.
bool ring_step(Ring& r, const std::vector<int32_t>& u, uint64_t* misses, uint64_t* evictions,
               std::vector<char>& used) {
  if ((int)u.size() > r.S) return false;
  const uint32_t t = ++r.clock;
  std::fill(used.begin(), used.begin() + r.S, 0);
  std::vector<int32_t> missing;
  for (int32_t e : u) {
    const int32_t v = r.slot_of[e];
    if (v >= 0) used[v] = 1;
    else missing.push_back(e);  // ascending: u is sorted
  }
  if (!missing.empty()) {
    std::vector<int32_t> free_slots;
    for (int v = 0; v < r.S; ++v)
      if (!used[v]) free_slots.push_back(v);
    const size_t n = missing.size();
    std::partial_sort(free_slots.begin(), free_slots.begin() + n, free_slots.end(),
                      [&](int32_t a, int32_t b) {
                        return r.last[a] != r.last[b] ? r.last[a] < r.last[b] : a < b;
                      });
    for (size_t i = 0; i < n; ++i) {
      const int32_t v = free_slots[i], e = missing[i];
      if (r.owner[v] >= 0) {
        r.slot_of[r.owner[v]] = -1;
        ++*evictions;
      }
      r.owner[v] = e;
      r.slot_of[e] = v;
      used[v] = 1;
    }
    *misses += n;
  }
  for (int v = 0; v < r.S; ++v)
    if (used[v]) r.last[v] = t;
  return true;
}

bool valid_trace(const int32_t* trace, int steps, int picks, int experts) {
  if (!trace || steps < 0 || picks < 1 || experts < 1 || experts > MOE_MAX_EXPERTS) return false;
  for (long long i = 0; i < (long long)steps * picks; ++i)
    if (trace[i] < 0 || trace[i] >= experts) return false;
  return true;
}

// Sorted union of one step's picks.
void step_union(const int32_t* p, int picks, std::vector<int32_t>& u) {
  u.assign(p, p + picks);
  std::sort(u.begin(), u.end());
  u.erase(std::unique(u.begin(), u.end()), u.end());
}

// Pin set of hindsight-static: the `n` most picked experts (ties: lower id).
std::vector<char> hottest(const int32_t* trace, int steps, int picks, int experts, int n) {
  std::vector<uint64_t> count(experts, 0);
  for (long long i = 0; i < (long long)steps * picks; ++i) ++count[trace[i]];
  std::vector<int32_t> ids(experts);
  for (int e = 0; e < experts; ++e) ids[e] = e;
  std::stable_sort(ids.begin(), ids.end(),
                   [&](int32_t a, int32_t b) { return count[a] > count[b]; });
  std::vector<char> pin(experts, 0);
  for (int i = 0; i < n && i < experts; ++i) pin[ids[i]] = 1;
  return pin;
}

// Pinned experts always resident; the rest through an LRU ring of `ring` slots.
void run_hybrid(const int32_t* trace, int steps, int picks, int experts, int pinned, int ring,
                moe_policy_result_t* out) {
  std::memset(out, 0, sizeof *out);
  const std::vector<char> pin = hottest(trace, steps, picks, experts, pinned);
  Ring r(experts, ring > 0 ? ring : 1);
  std::vector<char> used(r.S);
  std::vector<int32_t> u, rest;
  for (int s = 0; s < steps; ++s) {
    const int32_t* p = trace + (size_t)s * picks;
    step_union(p, picks, u);
    rest.clear();
    for (int32_t e : u)
      if (!pin[e]) rest.push_back(e);
    ++out->steps;
    if (ring <= 0) {  // pure static: every unpinned expert read from host memory
      for (int i = 0; i < picks; ++i) out->hits += pin[p[i]] ? 1 : 0;
      out->picks += picks;
      out->host_experts += rest.size();
      continue;
    }
    // hits: pinned picks + picks of ring-resident experts at step start
    uint64_t h = 0;
    for (int i = 0; i < picks; ++i) h += (pin[p[i]] || r.slot_of[p[i]] >= 0) ? 1 : 0;
    uint64_t m = 0, ev = 0;
    if (ring_step(r, rest, &m, &ev, used)) {
      out->picks += picks;
      out->hits += h;
      out->misses += m;
      out->evictions += ev;
      out->host_experts += m;
    } else {
      ++out->bypass_steps;
      out->host_experts += rest.size();
    }
  }
}

}  // namespace

extern "C" {

int moe_policy_lru(const int32_t* trace, int steps, int picks, int experts, int slots,
                   moe_policy_result_t* out) {
  if (!out || slots < 1 || slots > experts || !valid_trace(trace, steps, picks, experts))
    return MOE_ERR_ARG;
  run_hybrid(trace, steps, picks, experts, 0, slots, out);
  return MOE_OK;
}

int moe_policy_static(const int32_t* trace, int steps, int picks, int experts, int slots,
                      moe_policy_result_t* out) {
  if (!out || slots < 0 || slots > experts || !valid_trace(trace, steps, picks, experts))
    return MOE_ERR_ARG;
  run_hybrid(trace, steps, picks, experts, slots, 0, out);
  return MOE_OK;
}

int moe_policy_hybrid(const int32_t* trace, int steps, int picks, int experts, int slots,
                      int pinned, moe_policy_result_t* out) {
  if (!out || pinned < 0 || pinned > slots || slots > experts ||
      !valid_trace(trace, steps, picks, experts))
    return MOE_ERR_ARG;
  if (pinned == slots) {
    run_hybrid(trace, steps, picks, experts, pinned, 0, out);
  } else {
    run_hybrid(trace, steps, picks, experts, pinned, slots - pinned, out);
  }
  return MOE_OK;
}

int moe_policy_lru_curve(const int32_t* trace, int steps, int picks, int experts, int max_slots,
                         uint64_t* host_experts) {
  if (!host_experts || max_slots < 1 || max_slots > experts ||
      !valid_trace(trace, steps, picks, experts))
    return MOE_ERR_ARG;
  moe_policy_result_t r;
  for (int s = 1; s <= max_slots; ++s) {
    run_hybrid(trace, steps, picks, experts, 0, s, &r);
    host_experts[s - 1] = r.host_experts;
  }
  return MOE_OK;
}

int moe_policy_size_layers(const uint64_t* host_experts, int layers, int max_slots, int budget,
                           int min_slots, int32_t* slots_out) {
  if (!host_experts || !slots_out || layers < 1 || max_slots < 1 || min_slots < 1 ||
      min_slots > max_slots || budget < (long long)layers * min_slots)
    return MOE_ERR_ARG;
  // Exact: minimise the summed host-link experts over per-layer sizes in
  // [min_slots, max_slots] with sum <= budget (dynamic programme over layers).
  const int B = std::min<long long>(budget, (long long)layers * max_slots);
  const uint64_t INF = ~0ull;
  std::vector<uint64_t> cur(B + 1, INF), nxt(B + 1);
  std::vector<int32_t> pick((size_t)layers * (B + 1), -1);
  cur[0] = 0;
  for (int l = 0; l < layers; ++l) {
    std::fill(nxt.begin(), nxt.end(), INF);
    const uint64_t* c = host_experts + (size_t)l * max_slots;
    for (int b = 0; b <= B; ++b) {
      if (cur[b] == INF) continue;
      for (int s = min_slots; s <= max_slots && b + s <= B; ++s) {
        const uint64_t v = cur[b] + c[s - 1];
        if (v < nxt[b + s]) {
          nxt[b + s] = v;
          pick[(size_t)l * (B + 1) + b + s] = s;
        }
      }
    }
    cur.swap(nxt);
  }
  int best = -1;
  for (int b = 0; b <= B; ++b)
    if (cur[b] != INF && (best < 0 || cur[b] < cur[best])) best = b;
  if (best < 0) return MOE_ERR_ARG;
  for (int l = layers - 1, b = best; l >= 0; --l) {
    const int s = pick[(size_t)l * (B + 1) + b];
    slots_out[l] = s;
    b -= s;
  }
  return MOE_OK;
}

}  // extern "C"
