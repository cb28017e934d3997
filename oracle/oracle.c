/*
 * CPU oracle for the decode-time routed-MoE layer with an HBM expert slot cache.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the package smoke check and
 * the benchmark's CPU-baseline leg; never by the library.  Plain C, one
 * thread, double precision, no blocking or reordering beyond the definitions.
 * See oracle.h for the sources ([HEA], [GT], [TF], [SD], [OCP]) and the
 * readings taken where the pages are silent.
 *
 * Two independent halves:
 *   O-1  the layer's result: router -> NVFP4 dequant -> SwiGLU expert FFN ->
 *        weighted combine.  The slot cache changes only where bytes are read
 *        ([HEA] "What the slot cache is": the expert kernel reads the same
 *        bytes as the all-HBM case, only the index changes), so the result is
 *        the plain MoE layer.
 *   O-2  the cache trace: expert->slot map, hits, LRU victims, evictions.
 *        Two separate formulations (last-use stamps; an explicit recency list)
 *        that must agree.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- codecs */

/* E2M1 ([OCP] FP4): bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.
 * Exponent 0 is subnormal: value = 0.5 * mantissa.  [HEA] "What the slot
 * cache is" names the weights NVFP4; this is the element format NVFP4 uses. */
double orc_e2m1(unsigned code) {
  unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
  double mag;
  if (e == 0)
    mag = 0.5 * (double)m;
  else
    mag = ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
  return s ? -mag : mag;
}

/* E4M3 ([OCP] FP8, "FN" variant: no infinities, S.1111.111 is NaN):
 * bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0 mantissa; exponent 0 is
 * subnormal: 2^-6 * m/8.  The pages' FP8 block scales ([HEA] "What the slot
 * cache is": the scale row that travels with each expert's weight row). */
double orc_e4m3(unsigned code) {
  unsigned s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, -6);
  else
    mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
  return s ? -mag : mag;
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double orc_bf16(unsigned bits) {
  uint32_t u = (uint32_t)(bits & 0xFFFFu) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* ------------------------------------------------------------------ sizes */

/* One expert = three NVFP4 matrices (gate [I][H], up [I][H], down [H][I]):
 * 0.5 byte per weight plus one FP8 scale per 16 weights ([HEA] "What the slot
 * cache is": 18.874 MB of weights plus 2.359 MB of block scales at GLM shape;
 * "Five launches, four failures": scales are 12.5% of the weight bytes). */
void orc_expert_bytes(int64_t H, int64_t I, int64_t* Bw, int64_t* Bs) {
  int64_t weights = 3 * H * I;
  *Bw = weights / 2;
  *Bs = weights / 16;
}

/* ----------------------------------------------------------------- router */

/* Does expert a rank before expert b?  Larger logit first; NaN ranks below
 * every number; equal logits (including -0 == +0) rank the lower id first
 * ([TF]: router ties break by a stable expert order). */
static int orc_ranks_before(const float* l, int a, int b) {
  int na = isnan(l[a]) != 0, nb = isnan(l[b]) != 0;
  if (na || nb) {
    if (na && nb) return a < b;
    return nb;
  }
  if (l[a] > l[b]) return 1;
  if (l[a] < l[b]) return 0;
  return a < b;
}

/* Top-k router for one row ([HEA] "What the slot cache is": the router has
 * chosen top-8 expert ids; [SD]: the router weights by rank sum to one).
 * ids[0..k-1] in rank order; w[j] = exp(l_j - l_max) / sum over the k selected.
 * NaN counts as -inf for the weights; a logit equal to the maximum contributes
 * exactly 1 (so +inf and all -inf rows stay defined).  Returns
 * ORC_FLAG_NONFINITE_LOGIT if any of the row's E logits is NaN or infinite. */
unsigned orc_route(const float* logits, int E, int k, int32_t* ids, double* w) {
  unsigned flags = 0;
  char* taken = (char*)calloc((size_t)E, 1);
  for (int e = 0; e < E; ++e)
    if (!isfinite(logits[e])) flags |= ORC_FLAG_NONFINITE_LOGIT;
  for (int j = 0; j < k; ++j) {
    int best = -1;
    for (int e = 0; e < E; ++e) {
      if (taken[e]) continue;
      if (best < 0 || orc_ranks_before(logits, e, best)) best = e;
    }
    taken[best] = 1;
    ids[j] = best;
  }
  free(taken);
  double lmax = -INFINITY;
  for (int j = 0; j < k; ++j) {
    double l = isnan(logits[ids[j]]) ? -INFINITY : (double)logits[ids[j]];
    if (l > lmax) lmax = l;
  }
  double sum = 0.0;
  for (int j = 0; j < k; ++j) {
    double l = isnan(logits[ids[j]]) ? -INFINITY : (double)logits[ids[j]];
    w[j] = (l == lmax) ? 1.0 : exp(l - lmax);
    sum += w[j];
  }
  for (int j = 0; j < k; ++j) w[j] /= sum;
  return flags;
}

/* --------------------------------------------------------- NVFP4 matvec */

/* out[r] = sum_i W[r][i] * v[i] with W[r][i] = e2m1(code) * e4m3(scale) * gscale.
 * codes: [rows][K/2] bytes, element 2i in the low nibble of byte i;
 * scales: [rows][K/16] bytes, one per 16 consecutive elements of a row. */
void orc_nvfp4_matvec(const uint8_t* codes, const uint8_t* scales, double gscale,
                      int64_t rows, int64_t K, const double* v, double* out) {
  for (int64_t r = 0; r < rows; ++r) {
    const uint8_t* crow = codes + r * (K / 2);
    const uint8_t* srow = scales + r * (K / 16);
    double acc = 0.0;
    for (int64_t i = 0; i < K; ++i) {
      uint8_t byte = crow[i / 2];
      unsigned code = (i & 1) ? (byte >> 4) : (byte & 15u);
      double W = orc_e2m1(code) * orc_e4m3(srow[i / 16]) * gscale;
      acc += W * v[i];
    }
    out[r] = acc;
  }
}

/* ------------------------------------------------------------ expert FFN */

/* One routed expert: g = Wg x, u = Wu x, h = silu(g) * u, y = Wd h
 * ([HEA] "What the slot cache is": gate/up, SwiGLU and down over the expert's
 * weight row and scale row).  w_e/s_e point at the expert's bytes in the
 * layout of oracle.h; gs3 = (gate, up, down) fp32 global scales.
 * h_out (optional, [I]) receives h. */
void orc_expert_ffn(const uint8_t* w_e, const uint8_t* s_e, const float* gs3,
                    int64_t H, int64_t I, const double* x, double* y, double* h_out) {
  double* g = (double*)malloc(sizeof(double) * (size_t)I);
  double* u = (double*)malloc(sizeof(double) * (size_t)I);
  double* h = (double*)malloc(sizeof(double) * (size_t)I);
  orc_nvfp4_matvec(w_e, s_e, (double)gs3[0], I, H, x, g);
  orc_nvfp4_matvec(w_e + I * (H / 2), s_e + I * (H / 16), (double)gs3[1], I, H, x, u);
  for (int64_t r = 0; r < I; ++r) h[r] = g[r] / (1.0 + exp(-g[r])) * u[r];
  orc_nvfp4_matvec(w_e + 2 * I * (H / 2), s_e + 2 * I * (H / 16), (double)gs3[2], H, I, h, y);
  if (h_out) memcpy(h_out, h, sizeof(double) * (size_t)I);
  free(g);
  free(u);
  free(h);
}

/* ------------------------------------------------------------- MoE layer */

/* The layer's result for M rows (O-1).  w/s: E experts back to back
 * (Bw / Bs bytes each); gscale: [E][3]; logits fp32 [M][E]; x bf16 bits [M][H].
 * out[m][:] = sum_j wts[m][j] * y_{ids[m][j]}(x_m), j in rank order.
 * This is the same for a cached, an all-resident or a bypassed step. */
unsigned orc_moe_rows(const uint8_t* w, const uint8_t* s, const float* gscale,
                      int64_t E, int64_t H, int64_t I, int k, int M,
                      const float* logits, const uint16_t* x,
                      double* out, int32_t* ids, double* wts) {
  int64_t Bw, Bs;
  orc_expert_bytes(H, I, &Bw, &Bs);
  (void)E;
  unsigned flags = 0;
  double* xd = (double*)malloc(sizeof(double) * (size_t)H);
  double* y = (double*)malloc(sizeof(double) * (size_t)H);
  for (int m = 0; m < M; ++m) {
    flags |= orc_route(logits + (int64_t)m * E, (int)E, k, ids + m * k, wts + m * k);
    for (int64_t i = 0; i < H; ++i) xd[i] = orc_bf16(x[(int64_t)m * H + i]);
    double* o = out + (int64_t)m * H;
    for (int64_t i = 0; i < H; ++i) o[i] = 0.0;
    for (int j = 0; j < k; ++j) {
      int64_t e = ids[m * k + j];
      orc_expert_ffn(w + e * Bw, s + e * Bs, gscale + 3 * e, H, I, xd, y, NULL);
      for (int64_t i = 0; i < H; ++i) o[i] += wts[m * k + j] * y[i];
    }
  }
  free(xd);
  free(y);
  return flags;
}

/* -------------------------------------------------- cache trace (stamps) */

/* One layer-step of the slot cache (O-2), last-use-stamp formulation.
 * [HEA] "What the slot cache is": ids are mapped to slots on device; a miss
 * fills an LRU-victim slot and then updates the map.  [GT] "Correction,
 * September 14" counts misses per layer-step; [TF]: all rows of a round are
 * routed together and their union fetched once.
 *   map[E]: slot of each expert or -1; owner[S]: expert of each slot or -1;
 *   stamp[S]: step of last use (0 = never); t: this step, t >= 1.
 * Steps: U = union of the picks.  If |U| > S the step bypasses the cache:
 * state untouched, return -1.  Otherwise every resident id in U is a hit and
 * its slot is stamped t.  The missing ids, in ascending expert id, each take
 * the not-yet-used-this-step slot with the smallest (stamp, slot id); the
 * previous owner is evicted, then map/owner are set and the slot stamped t.
 * Outputs per pick: slot after the step, hit (resident at step start).
 * Per miss i: expert, slot, evicted expert (-1 if the slot was empty).
 * Returns the number of misses. */
int orc_lru_step(int E, int S, int32_t* map, int32_t* owner, uint32_t* stamp,
                 uint32_t t, int npicks, const int32_t* ids,
                 int32_t* slot_of_pick, int32_t* hit_of_pick,
                 int32_t* miss_e, int32_t* miss_v, int32_t* miss_evicted,
                 int32_t* n_union) {
  char* inU = (char*)calloc((size_t)E, 1);
  char* used = (char*)calloc((size_t)S, 1);
  int nU = 0;
  for (int p = 0; p < npicks; ++p) {
    if (!inU[ids[p]]) ++nU;
    inU[ids[p]] = 1;
  }
  *n_union = nU;
  for (int p = 0; p < npicks; ++p) hit_of_pick[p] = map[ids[p]] >= 0;
  if (nU > S) {
    for (int p = 0; p < npicks; ++p) slot_of_pick[p] = -1;
    free(inU);
    free(used);
    return -1;
  }
  for (int p = 0; p < npicks; ++p) {
    int v = map[ids[p]];
    if (v >= 0) {
      used[v] = 1;
      stamp[v] = t;
    }
  }
  int nmiss = 0;
  for (int e = 0; e < E; ++e) {
    if (!inU[e] || map[e] >= 0) continue;
    int best = -1;
    for (int v = 0; v < S; ++v) {
      if (used[v]) continue;
      if (best < 0 || stamp[v] < stamp[best]) best = v;
    }
    int ev = owner[best];
    if (ev >= 0) map[ev] = -1;
    map[e] = best;
    owner[best] = e;
    stamp[best] = t;
    used[best] = 1;
    miss_e[nmiss] = e;
    miss_v[nmiss] = best;
    miss_evicted[nmiss] = ev;
    ++nmiss;
  }
  for (int p = 0; p < npicks; ++p) slot_of_pick[p] = map[ids[p]];
  free(inU);
  free(used);
  return nmiss;
}

/* ---------------------------------------------- cache trace (recency list) */

/* The same step written as an explicit recency list: order[0] is the least
 * recently used slot, order[S-1] the most.  Initially order = 0, 1, ..., S-1.
 * A miss takes the first slot in the list not yet used this step.  At the end
 * of the step every slot used this step moves to the most-recent end, in
 * ascending slot id.  Same outputs and return value as orc_lru_step. */
int orc_lru_list_step(int E, int S, int32_t* map, int32_t* owner, int32_t* order,
                      int npicks, const int32_t* ids,
                      int32_t* slot_of_pick, int32_t* hit_of_pick,
                      int32_t* miss_e, int32_t* miss_v, int32_t* miss_evicted,
                      int32_t* n_union) {
  char* inU = (char*)calloc((size_t)E, 1);
  char* used = (char*)calloc((size_t)S, 1);
  int nU = 0;
  for (int p = 0; p < npicks; ++p) {
    if (!inU[ids[p]]) ++nU;
    inU[ids[p]] = 1;
  }
  *n_union = nU;
  for (int p = 0; p < npicks; ++p) hit_of_pick[p] = map[ids[p]] >= 0;
  if (nU > S) {
    for (int p = 0; p < npicks; ++p) slot_of_pick[p] = -1;
    free(inU);
    free(used);
    return -1;
  }
  for (int p = 0; p < npicks; ++p)
    if (map[ids[p]] >= 0) used[map[ids[p]]] = 1;
  int nmiss = 0;
  for (int e = 0; e < E; ++e) {
    if (!inU[e] || map[e] >= 0) continue;
    int victim = -1;
    for (int pos = 0; pos < S; ++pos) {
      if (!used[order[pos]]) {
        victim = order[pos];
        break;
      }
    }
    int ev = owner[victim];
    if (ev >= 0) map[ev] = -1;
    map[e] = victim;
    owner[victim] = e;
    used[victim] = 1;
    miss_e[nmiss] = e;
    miss_v[nmiss] = victim;
    miss_evicted[nmiss] = ev;
    ++nmiss;
  }
  int32_t* next = (int32_t*)malloc(sizeof(int32_t) * (size_t)S);
  int n = 0;
  for (int pos = 0; pos < S; ++pos)
    if (!used[order[pos]]) next[n++] = order[pos];
  for (int v = 0; v < S; ++v)
    if (used[v]) next[n++] = v;
  memcpy(order, next, sizeof(int32_t) * (size_t)S);
  free(next);
  for (int p = 0; p < npicks; ++p) slot_of_pick[p] = map[ids[p]];
  free(inU);
  free(used);
  return nmiss;
}
