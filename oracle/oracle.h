/*
 * CPU oracle for the decode-time routed-MoE layer with an HBM expert slot cache.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, single-threaded C
 * restatement of what the method computes, in double precision.  Only the
 * test suite, the package smoke check and the benchmark's CPU-baseline leg may
 * load it.  It shares no code, header, table or constant with the CUDA library
 * (hbm_slot_cache_gb300/csrc), and the library never calls it.
 *
 * Sources (web pages on the method; cited by page title and section):
 *   [HEA]  "GLM 5.3 Testing: HBM Expert Allocation", sections
 *          "What the slot cache is", "The build, measured on a synthetic
 *          GLM-shaped layer (M=1, graph-replayed)", "Five launches, four failures".
 *   [GT]   "GB300 GLM 5.3 Testing", sections "Correction, September 14" and
 *          "E1 v2: the first valid profile of this lane".
 *   [TF]   "TensorFold GLM-5.3 explained" (ring of slots, union fetch per round,
 *          exact-decoding rule: router ties break by a stable expert order).
 *   [SD]   "glm53 — GLM-5.3-Flash NVFP4" (servedeck), section on router weight
 *          by rank and "How it fits" (Flash expert shape).
 *   [OCP]  OCP Microscaling Formats (MX) v1.0 element encodings E2M1 and E4M3,
 *          the public definition the pages' "NVFP4" refers to.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - router: top-k by raw fp32 logit, descending; equal logits -> lower id
 *     first; NaN ranks below -inf.  Weights are the softmax of the k selected
 *     logits (renormalised over the k).
 *   - E2M1: element 2i of a row sits in the LOW nibble of byte i.
 *   - block scales: one E4M3 byte per 16 consecutive elements along K
 *     (the input dimension), row-major [rows][K/16].
 *   - expert byte layout: W13 [2I rows][H/2 bytes] (gate rows 0..I-1, up rows
 *     I..2I-1) then W2 [H rows][I/2 bytes]; scales in the same row order.
 *   - SwiGLU: h = silu(gate) * up, no clamp.
 *   - LRU: victims are the untouched-this-step slots with the smallest
 *     (last-use step, slot id); misses are filled in ascending expert id; empty
 *     slots have last use 0; a step whose id union exceeds S bypasses the cache
 *     and leaves it untouched.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORC_FLAG_NONFINITE_LOGIT 1u

double orc_e2m1(unsigned code);
double orc_e4m3(unsigned code);
double orc_bf16(unsigned bits);

void orc_expert_bytes(int64_t H, int64_t I, int64_t* Bw, int64_t* Bs);

unsigned orc_route(const float* logits, int E, int k, int32_t* ids, double* w);

void orc_nvfp4_matvec(const uint8_t* codes, const uint8_t* scales, double gscale,
                      int64_t rows, int64_t K, const double* v, double* out);

void orc_expert_ffn(const uint8_t* w_e, const uint8_t* s_e, const float* gs3,
                    int64_t H, int64_t I, const double* x, double* y, double* h_out);

unsigned orc_moe_rows(const uint8_t* w, const uint8_t* s, const float* gscale,
                      int64_t E, int64_t H, int64_t I, int k, int M,
                      const float* logits, const uint16_t* x,
                      double* out, int32_t* ids, double* wts);

int orc_lru_step(int E, int S, int32_t* map, int32_t* owner, uint32_t* stamp,
                 uint32_t t, int npicks, const int32_t* ids,
                 int32_t* slot_of_pick, int32_t* hit_of_pick,
                 int32_t* miss_e, int32_t* miss_v, int32_t* miss_evicted,
                 int32_t* n_union);

int orc_lru_list_step(int E, int S, int32_t* map, int32_t* owner, int32_t* order,
                      int npicks, const int32_t* ids,
                      int32_t* slot_of_pick, int32_t* hit_of_pick,
                      int32_t* miss_e, int32_t* miss_v, int32_t* miss_evicted,
                      int32_t* n_union);

#ifdef __cplusplus
}
#endif
#endif
