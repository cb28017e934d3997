// Grouped expert matmuls for multi-row steps on the 5th-generation tensor
// cores: tcgen05.mma kind::mxf4nvf4 with block scaling (E2M1 x E2M1, one UE4M3
// scale per 16 elements on both operands, fp32 accumulators in TMEM).
//
// Rows of a round are grouped by expert so each expert's bytes are read once
// for every row that chose it ("TensorFold GLM-5.3 explained": the round
// fetches the union of its rows' experts once and every row reads that copy).
// The weights are the MMA's A operand exactly as stored in the slot (or in
// host memory on a bypass): no decode on the CUDA cores.  The activations are
// the B operand in residual multi-level NVFP4 (quantize.cu): the N = 32
// columns of one MMA are 5 member rows x 6 levels, and the epilogue adds the
// levels with their fp32 level scales.
//
// One CTA (4 warps, one per TMEM lane quadrant) computes a 128-row weight tile
// for one job (5 members of one group) over the whole K:
//   gate/up: tile = 64 gate rows + the 64 matching up rows, so the epilogue
//            forms h = silu(gate) * up for those 64 rows directly;
//   down:    tile = 128 rows of W2, y_p = W2 h_p per member pick p.
// K is walked in chunks of up to 256 elements: A (128 x 128 B) and B
// (32 x 128 B) are copied with cp.async into the no-swizzle K-major core-matrix
// layout (8 rows x 16 B per core matrix; K-adjacent cores 128 B apart, 8-row
// groups 1 KB apart), and each row's scale words for the chunk land beside
// them.  Four stages: three chunks load while one computes.  Per chunk the
// scale factors go from shared memory to TMEM with tcgen05.st (two slots, by
// chunk parity), and one thread issues the chunk's MMAs and commits them to
// the mbarrier of that parity.
//
// Scale-factor placement: each 32-bit TMEM word holds the four UE4M3 scales of
// one row for one 64-element MMA step (byte b = elements 16b..16b+15).  Every
// warp writes its own lane quadrant, and each step's word is written to four
// adjacent columns, so the MMA finds the scales whichever of those columns its
// quadrant reads.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "internal.cuh"

namespace moe {
namespace {

constexpr int kThreads = 128;
constexpr int kTileM = 128;
constexpr int kTileN = 32;
constexpr int kMaxChunkBytes = 128;  // 256 FP4 elements per row per stage
constexpr int kABytes = kTileM * kMaxChunkBytes;
constexpr int kBBytes = kTileN * kMaxChunkBytes;
constexpr int kSfaBytes = kTileM * 16;  // the chunk's scale words, 16 B a row
constexpr int kSfbBytes = kTileN * 16;
constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;  // 22 KB
constexpr int kStages = 4;
constexpr int kTmemCols = 128;
constexpr int kColD = 0, kColSF = 32;  // SF stage s: A at 32 + 32 s, B at 48 + 32 s
constexpr int kSmemBytes = kStages * kStageBytes;  // 88 KB: two CTAs per SM

struct MmaArgs {
  const GroupPlan* gp;
  int K;        // inner dimension: H for gate/up, I for down
  int H, I, k;  // layer shape, top_k
  int gate_up;  // 1: gate/up + SwiGLU, 0: down
  QuantBuf act; // gate/up: by token row; down: by pick
  float* out;   // gate/up: h [P][I]; down: y [P][H]
  uint32_t* flags;
  int g0, g1;   // the launch's groups [g0, g1) (bounds as resolve_group takes them)
  // cp.async kernel only: a launch whose first group's expert lies in this
  // region (base, experts, bytes per expert; null: none) is left to the TMA
  // kernel launched beside it.  A step's groups are all in one place: the
  // slots, the staging halves, or host memory (a bypass).
  const uint8_t* skip_w;
  unsigned long long skip_n;
  long long skip_Bw;
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}

// 8-byte piece (scale words of a 128-element chunk)
__device__ __forceinline__ void cp_async8(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(smem_addr(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}

__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)(128u >> 4) << 16;   // K-adjacent core matrices: 128 B
  d |= (uint64_t)(1024u >> 4) << 32;  // 8-row groups: 1 KB
  d |= (uint64_t)1 << 46;             // sm_100-family descriptor version; no swizzle
  return d;
}

// kind::mxf4nvf4 instruction descriptor: A, B = E2M1, UE4M3 scales, K-major,
// M = 128, N = 32, dense.
__host__ __device__ constexpr uint32_t umma_idesc() {
  return (1u << 7) | (1u << 10) | ((uint32_t)(kTileN >> 3) << 17) | ((uint32_t)(kTileM >> 4) << 24);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&w)[4]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%1,%1,%1,%2,%2,%2,%2,%3,%3,%3,%3,%4,%4,%4,%4};" ::"r"(
          taddr),
      "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
      : "memory");
}

// Epilogue arithmetic shared by both grouped kernels, so a member gets the same
// bits from either: the levels of one accumulator row (columns
// s * kLevels + l) summed in level order with their level scales, and
// h = silu(gate) * up with the expert's global scales applied first.
__device__ __forceinline__ float level_sum(const float (&gl)[kLevels], const uint32_t* v) {
  float acc = 0.f;
#pragma unroll
  for (int l = 0; l < kLevels; ++l) acc = fmaf(gl[l], __uint_as_float(v[l]), acc);
  return acc;
}

__device__ __forceinline__ float swiglu_h(float gs_gate, float vg, float gs_up, float vu) {
  const float gate = gs_gate * vg;
  const float up = gs_up * vu;
  return gate / (1.0f + expf(-gate)) * up;
}

template <int P>  // 16-byte pieces per row per chunk (8: 256 elements, 4: 128)
__global__ void __launch_bounds__(kThreads)
grouped_mma_kernel(MmaArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) uint64_t s_bar[3];  // MMA commits of even / odd chunks; [2]: drain
  __shared__ uint32_t s_tmem;
  __shared__ int s_pick[kRowsPerJob], s_brow[kRowsPerJob];
  __shared__ float s_gl[kRowsPerJob][kLevels];
  __shared__ int s_fail;
  const GroupPlan* gp = a.gp;
  // this launch's jobs: those of groups [g0, g1)
  const int ng = gp->n_groups;
  const int nh = min(max(gp->n_hit_groups, 0), ng);
  const int g0 = resolve_group(a.g0, nh, ng);
  const int g1 = resolve_group(a.g1, nh, ng);
  const int jbeg = g0 < ng ? gp->g_job[g0] : gp->n_jobs;
  const int jend = gp->g_job[g1 < ng ? g1 : ng];
  if (jbeg + (int)blockIdx.x >= jend) return;  // uniform: before any TMEM or barrier use
  if (a.skip_w && expert_ptr_ok(gp->g_wptr[g0], a.skip_w, a.skip_n, a.skip_Bw)) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mt = blockIdx.y;
  const int K = a.K, H = a.H, I = a.I;
  constexpr int CB = P * 16;             // bytes per row per chunk
  constexpr int KSTEPS = CB / 32;        // 64-element MMA steps per chunk
  const int nchunks = K / (2 * CB);
  constexpr int AR = kTileM * P / kThreads;  // A rows per thread
  constexpr int BR = kTileN * P / kThreads;  // B rows per thread
  const int kc = tid % P;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&s_tmem)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    mbar_init(&s_bar[0], 1);
    mbar_init(&s_bar[1], 1);
    mbar_init(&s_bar[2], 1);
    fence_mbar_init();
    s_fail = 0;
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = s_tmem;
  const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
  int gc = 0;  // chunks this CTA has committed: barrier phases continue across jobs

  for (int job = jbeg + blockIdx.x; job < jend; job += gridDim.x) {
    // the job's plan entries are checked before they address memory (uniform
    // decision); a bad entry sets MOE_FLAG_BAD_PLAN and the job is skipped
    bool good = plan_ok(job >= 0 && job < gp->n_jobs, a.flags);
    const int jv = good ? gp->jobs[job] : 0;
    const int g = jv >> 8, tile = jv & 255;
    good = good && plan_ok(g >= 0 && g < ng, a.flags);
    const int gstart = good ? gp->g_start[g] : 0, gcount = good ? gp->g_count[g] : 1;
    good = good && plan_ok(gstart >= 0 && gcount >= 1 && gstart + gcount <= gp->npicks, a.flags);
    const int m0 = tile * kRowsPerJob;
    good = good && plan_ok(m0 < gcount, a.flags);
    good = __syncthreads_and(good);
    if (!good) continue;
    const int nmem = min(kRowsPerJob, gcount - m0);
    if (tid < kRowsPerJob) {
      int p = -1, br = 0;
      if (tid < nmem) {
        p = gp->members[gstart + m0 + tid];
        if (!plan_ok(p >= 0 && p < gp->npicks, a.flags)) p = 0;
        br = a.gate_up ? p / a.k : p;
      }
      s_pick[tid] = p;
      s_brow[tid] = br;
    }
    __syncthreads();
    if (tid < kRowsPerJob * kLevels) {
      const int s = tid / kLevels, l = tid - s * kLevels;
      s_gl[s][l] = (s < nmem) ? a.act.gl[(size_t)s_brow[s] * kLevels + l] : 0.f;
    }

    // weight rows of this tile
    const uint8_t* wbase = gp->g_wptr[g];
    const uint8_t* sbase = gp->g_sptr[g];
    size_t row_stride_w, row_stride_s;
    if (a.gate_up) {
      row_stride_w = H / 2;
      row_stride_s = H / 16;
    } else {
      wbase += (size_t)I * H;
      sbase += (size_t)I * H / 8;
      row_stride_w = I / 2;
      row_stride_s = I / 16;
    }
    auto src_row = [&](int r) -> size_t {  // tile row -> row index within the matrix block
      if (a.gate_up) return r < 64 ? (size_t)(64 * mt + r) : (size_t)(I + 64 * mt + r - 64);
      return (size_t)(kTileM * mt + r);
    };
    // this thread's cp.async pieces: A rows tid/P + (128/P) i, piece tid % P
    const uint8_t* a_src[AR];
#pragma unroll
    for (int i = 0; i < AR; ++i)
      a_src[i] = wbase + src_row(tid / P + (kThreads / P) * i) * row_stride_w + kc * 16;
    const uint8_t* b_src[BR];
    uint32_t b_ok[BR];
#pragma unroll
    for (int i = 0; i < BR; ++i) {
      const int n = tid / P + (kThreads / P) * i;
      const int s = n / kLevels, l = n - s * kLevels;
      const bool ok = n < kRowsPerJob * kLevels && s < nmem;
      b_ok[i] = ok ? 16u : 0u;
      b_src[i] = ok ? a.act.codes + ((size_t)s_brow[s] * kLevels + l) * (K / 2) + kc * 16 : a.act.codes;
    }
    // this thread's scale rows: A row 32*warp + lane, B row lane
    const uint8_t* sa_src = sbase + src_row(32 * warp + lane) * row_stride_s;
    const uint8_t* sb_src = nullptr;
    {
      const int s = lane / kLevels, l = lane - s * kLevels;
      if (lane < kRowsPerJob * kLevels && s < nmem)
        sb_src = a.act.scales + ((size_t)s_brow[s] * kLevels + l) * (K / 16);
    }

    // Chunk c goes to stage c % kStages: A and B codes in the core-matrix layout,
    // then each row's scale words (A: this thread's row; B: warp 0, row = lane).
    // Every thread commits one cp.async group per chunk (empty past the end), so
    // "chunk c landed" is a fixed wait_group count.
    auto load_chunk = [&](int c) {
      if (c < nchunks) {
        uint8_t* sA = smem + (c % kStages) * kStageBytes;
        uint8_t* sB = sA + kABytes;
        uint8_t* sSa = sB + kBBytes;
        uint8_t* sSb = sSa + kSfaBytes;
#pragma unroll
        for (int i = 0; i < AR; ++i) {
          const int r = tid / P + (kThreads / P) * i;
          cp_async16(sA + (r >> 3) * 1024 + kc * 128 + (r & 7) * 16, a_src[i] + (size_t)c * CB, 16u);
        }
#pragma unroll
        for (int i = 0; i < BR; ++i) {
          const int n = tid / P + (kThreads / P) * i;
          cp_async16(sB + (n >> 3) * 1024 + kc * 128 + (n & 7) * 16,
                     b_ok[i] ? b_src[i] + (size_t)c * CB : b_src[i], b_ok[i]);
        }
        constexpr int SW = CB / 8;  // scale bytes per row per chunk: 16 or 8
        if constexpr (SW == 16) {
          cp_async16(sSa + 16 * tid, sa_src + (size_t)c * SW, 16u);
          if (warp == 0)
            cp_async16(sSb + 16 * lane, sb_src ? sb_src + (size_t)c * SW : sa_src, sb_src ? 16u : 0u);
        } else {
          cp_async8(sSa + 16 * tid, sa_src + (size_t)c * SW, 8u);
          if (warp == 0)
            cp_async8(sSb + 16 * lane, sb_src ? sb_src + (size_t)c * SW : sa_src, sb_src ? 8u : 0u);
        }
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    };

#pragma unroll
    for (int c = 0; c < kStages - 1; ++c) load_chunk(c);
    bool ok = true;
    for (int c = 0; c < nchunks; ++c) {
      const int st = c % kStages, sf = (gc + c) & 1;
      asm volatile("cp.async.wait_group %0;" ::"n"(kStages - 2) : "memory");  // chunk c landed
      __syncthreads();
      // MMA(c-1) done => its stage may refill, and SF slot sf (last read by MMA(c-2)) is free
      if (c >= 1) {
        const int pc = gc + c - 1;
        if (!mbar_wait_bounded(&s_bar[pc & 1], (uint32_t)((pc >> 1) & 1), a.flags)) s_fail = 1;
      }
      load_chunk(c + kStages - 1);
      const uint8_t* sSa = smem + st * kStageBytes + kABytes + kBBytes;
      uint32_t w[4], wb[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        w[q] = q < KSTEPS ? reinterpret_cast<const uint32_t*>(sSa + 16 * tid)[q] : 0u;
        wb[q] = q < KSTEPS ? reinterpret_cast<const uint32_t*>(sSa + kSfaBytes + 16 * lane)[q] : 0u;
      }
      __syncwarp();  // tcgen05.st is .sync.aligned: the warp reconverges after the wait
      tmem_st16(tmem + lane_base + kColSF + 32 * sf, w);
      tmem_st16(tmem + lane_base + kColSF + 32 * sf + 16, wb);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncthreads();
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      if (s_fail) {
        ok = false;
        break;
      }
      if (tid == 0) {
        const uint32_t sA = smem_addr(smem + st * kStageBytes);
        const uint32_t sB = sA + kABytes;
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks) {
          const uint64_t da = umma_desc(sA + 256 * ks), db = umma_desc(sB + 256 * ks);
          const uint32_t sfa_t = tmem + kColSF + 32 * sf + 4 * ks;
          const uint32_t sfb_t = tmem + kColSF + 32 * sf + 16 + 4 * ks;
          const uint32_t acc = (c > 0 || ks > 0) ? 1u : 0u;
          asm volatile(
              "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
              "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
                  tmem + kColD),
              "l"(da), "l"(db), "r"(umma_idesc()), "r"(sfa_t), "r"(sfb_t), "r"(acc)
              : "memory");
        }
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                smem_addr(&s_bar[sf]))
            : "memory");
      }
    }
    if (ok) {
      const int pc = gc + nchunks - 1;
      if (!mbar_wait_bounded(&s_bar[pc & 1], (uint32_t)((pc >> 1) & 1), a.flags)) s_fail = 1;
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");  // nothing may land after exit
    __syncthreads();
    ok = s_fail == 0;  // uniform across the CTA
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (!ok) break;  // a timed-out wait leaves the barrier phases unknown: stop here
    gc += nchunks;

    uint32_t v[32];
    __syncwarp();
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
          "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
          "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(tmem + lane_base + kColD));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    const int row = 32 * warp + lane;  // tile row
    float val[kRowsPerJob];
#pragma unroll
    for (int s = 0; s < kRowsPerJob; ++s) val[s] = level_sum(s_gl[s], v + s * kLevels);
    const float* gsc = gp->g_gs + 3 * g;
    if (a.gate_up) {
      float* s_up = reinterpret_cast<float*>(smem);  // stages are idle now
      if (row >= 64)
#pragma unroll
        for (int s = 0; s < kRowsPerJob; ++s) s_up[(row - 64) * kRowsPerJob + s] = val[s];
      __syncthreads();
      if (row < 64) {
        for (int s = 0; s < nmem; ++s)
          a.out[(size_t)s_pick[s] * I + 64 * mt + row] =
              swiglu_h(gsc[0], val[s], gsc[1], s_up[row * kRowsPerJob + s]);
      }
    } else {
      for (int s = 0; s < nmem; ++s)
        a.out[(size_t)s_pick[s] * H + kTileM * mt + row] = gsc[2] * val[s];
    }
    // the next job rewrites s_pick / s_gl and the stages; TMEM reads are done
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (s_fail) {
    // A wait gave up, so MMAs this CTA committed may still be running: before
    // the TMEM is released, one more commit (it arrives once every earlier
    // tcgen05 operation of the issuing thread, thread 0, is complete) is waited
    // for under the default limit.
    if (tid == 0) {
      asm volatile(
          "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
              smem_addr(&s_bar[2]))
          : "memory");
      mbar_wait_bounded(&s_bar[2], 0u, a.flags);
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
  }
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols));
}

// ------------------------------------------------- TMA-staged grouped kernel
//
// The same jobs and arithmetic, the weight operand moved by the tensor memory
// accelerator.  Slot (or staging) bytes are viewed as 2-D row arrays (the
// TmaSource views), and each chunk's weight tile is two 128-row x 128-byte
// boxes (256 elements of K) in the 128-byte swizzle the MMA reads directly,
// plus the boxes of their scale words.  A work item is (job, tile): gate/up
// tiles pair 128 gate rows with the matching 128 up rows (one MMA each, so a
// TMEM lane holds both of its row's accumulators), down tiles are 256 W2
// rows.  One persistent CTA per SM takes items round robin, in five roles:
//   warp 10 (plan): reads each item's plan entries (checked) into a ring of
//     kTRing records in shared memory, ahead of the others, so no role waits
//     on a chain of global loads at an item boundary;
//   warp 4 (loads): keeps kTStages chunks in flight (TMA for the weight codes
//     and scales, 16-byte cp.async for the members' activation levels and
//     their scales) and runs on into the CTA's next item, so the HBM stream
//     does not stop at an item boundary;
//   warps 0-3 (scales, one TMEM lane quadrant each): move each chunk's scale
//     words into one of kTSfSlots TMEM slots and count in on the slot's
//     mbarrier;
//   warp 5, one thread (MMA): issues each chunk's MMAs into the item's
//     accumulator buffer (two, by item parity) once its scales are in, and
//     commits them to the stage's "empty" mbarrier (which also frees the
//     scale slot); after an item's last chunk it commits to the buffer's
//     "full" mbarrier;
//   warps 6-9 (epilogue, one lane quadrant each): read an item's accumulators,
//     release the buffer and the item's record, write h or y while the next
//     item's MMAs run.
// An item whose plan entries fail their checks (MOE_FLAG_BAD_PLAN) has no
// chunks; it still passes through the MMA thread and the epilogue so every
// role counts the same items.
// Every wait is bounded: one that runs out sets the CTA's abort word and
// everyone stops; copies and MMAs in flight are drained (bounded) before the
// TMEM is freed.

constexpr int kTThreads = 352;
constexpr int kTRows = 128;                     // rows of one MMA (M); two per item
constexpr int kTABytes = kTRows * 128;          // one weight box: 128 rows x 256 elements
constexpr int kTSfaBytes = kTRows * 16;         // its rows' scale words for the chunk
constexpr int kTOffSfa = 2 * kTABytes;
constexpr int kTOffB = kTOffSfa + 2 * kTSfaBytes;
constexpr int kTOffSfb = kTOffB + kBBytes;
constexpr int kTStageBytes = 41 * 1024;         // kTOffSfb + kSfbBytes, rounded up to 1 KB
constexpr int kTStages = 5;
constexpr int kTSmemBytes = kTStages * kTStageBytes + 1024;  // + room to align to 1 KB
constexpr int kTSfSlots = 4;                    // < kTStages (see the scale warps' wait)
constexpr int kTRing = 4;                       // item records decoded ahead
constexpr int kTTmemCols = 512;
// TMEM columns: accumulator buffer b at 64 b (half h at + 32 h); scale slot q
// at 128 + 48 q: SFA of half 0 at +0, half 1 at +16, SFB at +32, each K step's
// word written to four adjacent columns (the step's scale columns are 4-column
// aligned, as the MMA requires).
constexpr int kTColSF = 128;
static_assert(kTOffSfb + kSfbBytes <= kTStageBytes, "stage layout");
static_assert(kTStageBytes % 1024 == 0, "weight boxes must stay 1 KB aligned");
static_assert(kTSmemBytes <= 227 * 1024, "shared memory");
static_assert(kTColSF + 48 * kTSfSlots <= kTTmemCols && kTSfSlots < kTStages, "TMEM columns");

struct MmaTmaArgs {
  TmaMap map_w;  // codes view of the launch's matrix block
  TmaMap map_s;  // its scales view
  MmaArgs m;
  const uint8_t* base_w;
  const uint8_t* base_s;
  long long Bw, Bs;
  unsigned long long n;  // experts in the region
  int rps;               // view rows per expert: 3I (K = H) or 3H (K = I)
  int row0;              // first view row of the block within an expert: 0 (W13), 2H (W2)
};

// K-major operand in the 128-byte swizzle: 8-row groups 1 KB apart; a 64-element
// K step inside the 128-byte row advances the start address by 32 bytes.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1 << 16;              // leading byte offset: unused for this layout
  d |= (uint64_t)(1024u >> 4) << 32;   // 8-row groups: 1 KB
  d |= (uint64_t)1 << 46;              // sm_100-family descriptor version
  d |= (uint64_t)2 << 61;              // 128-byte swizzle
  return d;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const TmaMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// The mbarrier receives one arrival once this thread's earlier cp.async
// copies have landed (counted in its expected arrivals).
__device__ __forceinline__ void cp_async_bar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}

// One work item's plan entries, checked before they address memory (a bad
// entry sets MOE_FLAG_BAD_PLAN and the item is skipped by every warp alike:
// the plan does not change during the launch).
struct TItem {
  int g, gstart, m0, nmem, mt;
  int vw, vs;  // the group's expert in the region: codes, scales
};

__device__ __forceinline__ bool t_item(const MmaTmaArgs& a, int jbeg, int m_tiles, int it,
                                       TItem& t) {
  const GroupPlan* gp = a.m.gp;
  uint32_t* fl = a.m.flags;
  const int jo = it / m_tiles;
  const int job = jbeg + jo;
  t.mt = it - jo * m_tiles;
  if (!plan_ok(job >= 0 && job < gp->n_jobs, fl)) return false;
  const int jv = gp->jobs[job];
  t.g = jv >> 8;
  const int tile = jv & 255;
  if (!plan_ok(t.g >= 0 && t.g < gp->n_groups, fl)) return false;
  t.gstart = gp->g_start[t.g];
  const int gcount = gp->g_count[t.g];
  if (!plan_ok(t.gstart >= 0 && gcount >= 1 && t.gstart + gcount <= gp->npicks, fl)) return false;
  t.m0 = tile * kRowsPerJob;
  if (!plan_ok(t.m0 < gcount, fl)) return false;
  t.nmem = min(kRowsPerJob, gcount - t.m0);
  const uint8_t* w = gp->g_wptr[t.g];
  const uint8_t* s = gp->g_sptr[t.g];
  if (!plan_ok(expert_ptr_ok(w, a.base_w, a.n, a.Bw) && expert_ptr_ok(s, a.base_s, a.n, a.Bs), fl))
    return false;
  t.vw = (int)((w - a.base_w) / a.Bw);
  t.vs = (int)((s - a.base_s) / a.Bs);
  return true;
}

// Member s of the item's tile: its pick index, and the activation row its
// levels start at (gate/up: the token row, down: the pick).
__device__ __forceinline__ void t_member(const MmaTmaArgs& a, const TItem& t, int s, int& pick,
                                         int& brow) {
  pick = -1;
  brow = 0;
  if (s < t.nmem) {
    int p = a.m.gp->members[t.gstart + t.m0 + s];
    if (!plan_ok(p >= 0 && p < a.m.gp->npicks, a.m.flags)) p = 0;
    pick = p;
    brow = a.m.gate_up ? p / a.m.k : p;
  }
}

// One work item as the plan warp decoded it.
struct TRec {
  int good, mt, vw, vs;
  int pick[kRowsPerJob];  // -1: no member
  int brow[kRowsPerJob];  // the member's activation row
  float gl[kRowsPerJob][kLevels];
  float gs[3];
};

__global__ void __launch_bounds__(kTThreads, 1)
grouped_mma_tma_kernel(const __grid_constant__ MmaTmaArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t s_full[kTStages], s_empty[kTStages], s_sfready[kTSfSlots],
      s_accf[2], s_acce[2], s_rfull[kTRing], s_rfree[kTRing], s_drain;
  __shared__ TRec s_rec[kTRing];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  const MmaArgs& m = a.m;
  const GroupPlan* gp = m.gp;
  const int ng = gp->n_groups;
  const int nh = min(max(gp->n_hit_groups, 0), ng);
  const int g0 = resolve_group(m.g0, nh, ng);
  const int g1 = resolve_group(m.g1, nh, ng);
  const int jbeg = g0 < ng ? gp->g_job[g0] : gp->n_jobs;
  const int jend = gp->g_job[g1 < ng ? g1 : ng];
  const int m_tiles = m.gate_up ? m.I / kTRows : m.H / (2 * kTRows);
  const int n_items = max(jend - jbeg, 0) * m_tiles;
  const int mine =
      (int)blockIdx.x < n_items ? (n_items - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  if (mine == 0) return;  // uniform: before any TMEM or barrier use
  // experts outside the region (a bypass step's host memory): the cp.async kernel's
  if (!expert_ptr_ok(gp->g_wptr[g0], a.base_w, a.n, a.Bw)) return;
  const int nchunks = m.K / 256;
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_word = &s_abort;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&s_tmem)),
                 "r"(kTTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    for (int s = 0; s < kTStages; ++s) {
      mbar_init(&s_full[s], 33);  // the expect_tx arrival + one per loader lane (its cp.async)
      mbar_init(&s_empty[s], 1);  // the chunk's MMA commit
    }
    for (int q = 0; q < kTSfSlots; ++q) mbar_init(&s_sfready[q], 128);  // every scale thread
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_accf[b], 1);    // an item's last MMA commit
      mbar_init(&s_acce[b], 128);  // every epilogue thread has read the buffer
    }
    for (int q = 0; q < kTRing; ++q) {
      mbar_init(&s_rfull[q], 1);    // the plan warp wrote the record
      mbar_init(&s_rfree[q], 128);  // every epilogue thread is done with it (the last reader)
    }
    mbar_init(&s_drain, 1);
    fence_mbar_init();
    s_abort = 0;
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = s_tmem;

  if (warp == 10) {
    // ------------------------------------------------------------- plan
    for (int i = 0; i < mine; ++i) {
      const int slot = i % kTRing;
      if (i >= kTRing && !mbar_wait_or_abort(&s_rfree[slot], (uint32_t)((i / kTRing - 1) & 1),
                                             abort_word, m.flags)) {
        *abort_word = 1;
        break;
      }
      TItem t;
      const bool good = t_item(a, jbeg, m_tiles, (int)blockIdx.x + i * (int)gridDim.x, t);
      int pick = -1, brow = 0;
      if (good && lane < kRowsPerJob) t_member(a, t, lane, pick, brow);
      const int sm = lane / kLevels < kRowsPerJob ? lane / kLevels : 0;
      const int pick_s = __shfl_sync(0xFFFFFFFFu, pick, sm);
      const int brow_s = __shfl_sync(0xFFFFFFFFu, brow, sm);
      TRec& r = s_rec[slot];
      if (lane < kRowsPerJob * kLevels)
        r.gl[lane / kLevels][lane % kLevels] =
            (good && pick_s >= 0) ? m.act.gl[(size_t)brow_s * kLevels + lane % kLevels] : 0.f;
      if (lane < kRowsPerJob) {
        r.pick[lane] = pick;
        r.brow[lane] = brow;
      }
      if (lane < 3) r.gs[lane] = good ? gp->g_gs[3 * t.g + lane] : 0.f;
      if (lane == 0) {
        r.good = good ? 1 : 0;
        r.mt = good ? t.mt : 0;
        r.vw = good ? t.vw : 0;
        r.vs = good ? t.vs : 0;
      }
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        mbar_arrive(&s_rfull[slot]);
      }
    }
  } else if (warp == 4) {
    // ------------------------------------------------------------ loads
    int g = 0;  // chunks issued
    bool run = true;
    for (int i = 0; i < mine && run; ++i) {
      const int slot = i % kTRing;
      if (!mbar_wait_or_abort(&s_rfull[slot], (uint32_t)((i / kTRing) & 1), abort_word,
                              m.flags)) {
        *abort_word = 1;
        break;
      }
      const TRec& r = s_rec[slot];
      if (!r.good) continue;
      // this lane's activation pieces: rows n = lane / 8 + 4 q, piece lane % 8;
      // its scale row: n = lane.  Rows past the tile's members are zero-filled.
      const uint8_t* b_src[8];
      uint32_t b_n[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int n = (lane >> 3) + 4 * q;
        const int s = n / kLevels, l = n - s * kLevels;
        const bool ok = s < kRowsPerJob && r.pick[s < kRowsPerJob ? s : 0] >= 0;
        const int brow = ok ? r.brow[s] : 0;
        b_n[q] = ok ? 16u : 0u;
        b_src[q] = ok ? m.act.codes + ((size_t)brow * kLevels + l) * (m.K / 2) + (lane & 7) * 16
                      : m.act.codes;
      }
      const uint8_t* sfb_src;
      uint32_t sfb_n;
      {
        const int s = lane / kLevels, l = lane - s * kLevels;
        const bool ok = s < kRowsPerJob && r.pick[s < kRowsPerJob ? s : 0] >= 0;
        const int brow = ok ? r.brow[s] : 0;
        sfb_n = ok ? 16u : 0u;
        sfb_src = ok ? m.act.scales + ((size_t)brow * kLevels + l) * (m.K / 16) : m.act.scales;
      }
      int yw[2], ys[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int off = m.gate_up ? h * m.I + r.mt * kTRows : (2 * r.mt + h) * kTRows;
        yw[h] = r.vw * a.rps + a.row0 + off;
        ys[h] = r.vs * a.rps + a.row0 + off;
      }
      for (int c = 0; c < nchunks; ++c, ++g) {
        const int st = g % kTStages;
        if (g >= kTStages &&
            !mbar_wait_or_abort(&s_empty[st], (uint32_t)((g / kTStages - 1) & 1), abort_word,
                                m.flags)) {
          *abort_word = 1;
          run = false;
          break;
        }
        uint8_t* sg = smem + st * kTStageBytes;
        if (lane == 0) {
          mbar_arrive_expect_tx(&s_full[st], 2 * kTABytes + 2 * kTSfaBytes);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            tma_load_2d(sg + h * kTABytes, &a.map_w, c * 128, yw[h], &s_full[st]);
            tma_load_2d(sg + kTOffSfa + h * kTSfaBytes, &a.map_s, c * 16, ys[h], &s_full[st]);
          }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int n = (lane >> 3) + 4 * q;
          cp_async16(sg + kTOffB + (n >> 3) * 1024 + (lane & 7) * 128 + (n & 7) * 16,
                     b_n[q] ? b_src[q] + (size_t)c * 128 : b_src[q], b_n[q]);
        }
        cp_async16(sg + kTOffSfb + 16 * lane, sfb_n ? sfb_src + (size_t)c * 16 : sfb_src, sfb_n);
        cp_async_bar_arrive(&s_full[st]);
      }
    }
    // the last chunks issued have landed before the CTA may exit
    for (int d = g > kTStages ? g - kTStages : 0; d < g; ++d)
      mbar_wait_bounded(&s_full[d % kTStages], (uint32_t)((d / kTStages) & 1), m.flags);
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp < 4) {
    // ----------------------------------------------------------- scales
    // Chunk g's scales go to slot g % kTSfSlots once chunk g - kTSfSlots's
    // MMAs (the slot's last reader) are done.  That wait also keeps a thread
    // from arriving twice on a slot's mbarrier before the MMA thread saw the
    // first phase complete.
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    int g = 0;
    bool run = true;
    for (int i = 0; i < mine && run; ++i) {
      if (!mbar_wait_or_abort(&s_rfull[i % kTRing], (uint32_t)((i / kTRing) & 1), abort_word,
                              m.flags)) {
        *abort_word = 1;
        break;
      }
      if (!s_rec[i % kTRing].good) continue;
      for (int c = 0; c < nchunks; ++c, ++g) {
        const int st = g % kTStages, q = g % kTSfSlots;
        const int gp_ = g - kTSfSlots;
        if (!mbar_wait_or_abort(&s_full[st], (uint32_t)((g / kTStages) & 1), abort_word,
                                m.flags) ||
            (gp_ >= 0 && !mbar_wait_or_abort(&s_empty[gp_ % kTStages],
                                             (uint32_t)((gp_ / kTStages) & 1), abort_word,
                                             m.flags))) {
          *abort_word = 1;
          run = false;
          break;
        }
        const uint8_t* sg = smem + st * kTStageBytes;
        uint32_t w0[4], w1[4], wb[4];
        {
          const uint4 x0 = *reinterpret_cast<const uint4*>(sg + kTOffSfa + 16 * tid);
          const uint4 x1 = *reinterpret_cast<const uint4*>(sg + kTOffSfa + kTSfaBytes + 16 * tid);
          const uint4 xb = *reinterpret_cast<const uint4*>(sg + kTOffSfb + 16 * lane);
          w0[0] = x0.x; w0[1] = x0.y; w0[2] = x0.z; w0[3] = x0.w;
          w1[0] = x1.x; w1[1] = x1.y; w1[2] = x1.z; w1[3] = x1.w;
          wb[0] = xb.x; wb[1] = xb.y; wb[2] = xb.z; wb[3] = xb.w;
        }
        const uint32_t sft = kTColSF + 48 * q;
        __syncwarp();  // tcgen05.st is .sync.aligned: the warp reconverges after the waits
        tmem_st16(tmem + lane_base + sft, w0);
        tmem_st16(tmem + lane_base + sft + 16, w1);
        tmem_st16(tmem + lane_base + sft + 32, wb);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        mbar_arrive(&s_sfready[q]);
      }
    }
  } else if (warp == 5) {
    // -------------------------------------------------------------- MMAs
    if (lane == 0) {
      int g = 0, ni = 0;  // chunks consumed, items done
      bool run = true;
      for (int i = 0; i < mine && run; ++i) {
        if (!mbar_wait_or_abort(&s_rfull[i % kTRing], (uint32_t)((i / kTRing) & 1), abort_word,
                                m.flags)) {
          *abort_word = 1;
          break;
        }
        const bool good = s_rec[i % kTRing].good != 0;
        const int b = ni & 1;
        // the buffer's previous item (ni - 2) has been read by the epilogue
        if (ni >= 2 && !mbar_wait_or_abort(&s_acce[b], (uint32_t)(((ni >> 1) - 1) & 1),
                                           abort_word, m.flags)) {
          *abort_word = 1;
          break;
        }
        for (int c = 0; good && c < nchunks; ++c, ++g) {
          const int st = g % kTStages, q = g % kTSfSlots;
          // the chunk's scales are in TMEM (so its bytes have landed too)
          if (!mbar_wait_or_abort(&s_sfready[q], (uint32_t)((g / kTSfSlots) & 1), abort_word,
                                  m.flags)) {
            *abort_word = 1;
            run = false;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // cp.async bytes -> MMA
          const uint32_t sA = smem_addr(smem + st * kTStageBytes);
          const uint32_t sB = sA + kTOffB;
          const uint32_t sft = tmem + kTColSF + 48 * q;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t db = umma_desc(sB + 256 * ks);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint64_t da = umma_desc_sw128(sA + h * kTABytes + 32 * ks);
              const uint32_t acc = (c > 0 || ks > 0) ? 1u : 0u;
              asm volatile(
                  "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
                  "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
                      tmem + 64 * b + 32 * h),
                  "l"(da), "l"(db), "r"(umma_idesc()), "r"(sft + 16 * h + 4 * ks),
                  "r"(sft + 32 + 4 * ks), "r"(acc)
                  : "memory");
            }
          }
          asm volatile(
              "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                  smem_addr(&s_empty[st]))
              : "memory");
        }
        if (!run) break;
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                smem_addr(&s_accf[b]))
            : "memory");
        ++ni;
      }
    }
  } else {
    // --------------------------------------------------------- epilogue
    const int qd = warp & 3;  // warps 6, 7, 8, 9: lane quadrants 2, 3, 0, 1
    const int r = 32 * qd + lane;
    const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
    int ni = 0;
    for (int i = 0; i < mine; ++i) {
      const int slot = i % kTRing;
      if (!mbar_wait_or_abort(&s_rfull[slot], (uint32_t)((i / kTRing) & 1), abort_word,
                              m.flags)) {
        *abort_word = 1;
        break;
      }
      const TRec& rec = s_rec[slot];
      const bool good = rec.good != 0;
      const int mt = rec.mt;
      int pick[kRowsPerJob];
      float gl[kRowsPerJob][kLevels];
#pragma unroll
      for (int s = 0; s < kRowsPerJob; ++s) {
        pick[s] = rec.pick[s];
#pragma unroll
        for (int l = 0; l < kLevels; ++l) gl[s][l] = rec.gl[s][l];
      }
      const float gs0 = rec.gs[0], gs1 = rec.gs[1], gs2 = rec.gs[2];
      const int b = ni & 1;
      if (!mbar_wait_or_abort(&s_accf[b], (uint32_t)((ni >> 1) & 1), abort_word, m.flags)) {
        *abort_word = 1;
        break;
      }
      uint32_t v0[32], v1[32];
      if (good) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        __syncwarp();  // tcgen05.ld is .sync.aligned
        tmem_ld32(tmem + lane_base + 64 * b, v0);
        tmem_ld32(tmem + lane_base + 64 * b + 32, v1);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      }
      mbar_arrive(&s_acce[b]);
      mbar_arrive(&s_rfree[slot]);  // every other role is past this item's record
      ++ni;
      if (!good) continue;
      if (m.gate_up) {
        const int row = mt * kTRows + r;  // gate row = index into h
#pragma unroll
        for (int s = 0; s < kRowsPerJob; ++s)
          if (pick[s] >= 0)
            m.out[(size_t)pick[s] * m.I + row] =
                swiglu_h(gs0, level_sum(gl[s], v0 + s * kLevels), gs1,
                         level_sum(gl[s], v1 + s * kLevels));
      } else {
        const int row = 2 * mt * kTRows + r;
#pragma unroll
        for (int s = 0; s < kRowsPerJob; ++s)
          if (pick[s] >= 0) {
            m.out[(size_t)pick[s] * m.H + row] = gs2 * level_sum(gl[s], v0 + s * kLevels);
            m.out[(size_t)pick[s] * m.H + row + kTRows] = gs2 * level_sum(gl[s], v1 + s * kLevels);
          }
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (*abort_word) {  // uniform after the barrier
    // MMAs the MMA thread issued may still run: one more commit from it (it
    // arrives once all its earlier tcgen05 operations are complete) is waited
    // for under the default limit before the TMEM is released.
    if (tid == 5 * 32) {
      asm volatile(
          "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
              smem_addr(&s_drain))
          : "memory");
      mbar_wait_bounded(&s_drain, 0u, m.flags);
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
  }
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTTmemCols));
}

// out[m][o] = sum_j w[m*k + j] * y[m*k + j][o], j in rank order.
__global__ void combine_kernel(const GroupPlan* __restrict__ gp, const float* __restrict__ y,
                               float* __restrict__ out, int H, int k) {
  const int m = blockIdx.y;
  const int o = blockIdx.x * blockDim.x + threadIdx.x;
  if (o >= H) return;
  float acc = 0.f;
  for (int j = 0; j < k; ++j) {
    const int p = m * k + j;
    acc = fmaf(gp->wts[p], y[(size_t)p * H + o], acc);
  }
  out[(size_t)m * H + o] = acc;
}

cudaError_t run_mma_tma(cudaStream_t st, const MmaTmaArgs& a, int grid) {
  static bool set = false;
  if (!set) {
    cudaError_t e = cudaFuncSetAttribute(grouped_mma_tma_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kTSmemBytes);
    if (e == cudaSuccess) e = prefer_max_shared(grouped_mma_tma_kernel);
    if (e != cudaSuccess) return e;
    set = true;
  }
  grouped_mma_tma_kernel<<<grid, kTThreads, kTSmemBytes, st>>>(a);
  return cudaGetLastError();
}

template <int P>
cudaError_t run_mma(cudaStream_t st, const MmaArgs& a, int grid_x, int m_tiles) {
  auto kern = grouped_mma_kernel<P>;
  static bool set = false;
  if (!set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess) e = prefer_max_shared(kern);
    if (e != cudaSuccess) return e;
    set = true;
  }
  kern<<<dim3(grid_x, m_tiles), kThreads, kSmemBytes, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool make_tma_source(const uint8_t* w, const uint8_t* s, unsigned long long n, int H, int I,
                     long long Bw, long long Bs, int num_sms, TmaSource* out) {
  *out = TmaSource{};
  if (!w || !s || n == 0 || H % 256 != 0 || I % 256 != 0 || num_sms <= 0) return false;
  if (Bw != 3LL * H * I / 2 || Bs != 3LL * H * I / 16) return false;
  const unsigned long long rows13 = n * 3ull * (unsigned long long)I;
  const unsigned long long rows2 = n * 3ull * (unsigned long long)H;
  if (rows2 >= (1ull << 31) || rows13 >= (1ull << 31)) return false;  // TMA row coordinates
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return false;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  auto make = [&](TmaMap* dst, const uint8_t* base, unsigned long long row_bytes,
                  unsigned long long rows, unsigned box_x, bool swizzle) {
    CUtensorMap tm;
    cuuint64_t dims[2] = {row_bytes, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_x, (cuuint32_t)kTRows};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = encode(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base),
                              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    static_assert(sizeof(CUtensorMap) == sizeof(TmaMap), "tensor map size");
    if (r != CUDA_SUCCESS) return false;
    std::memcpy(dst->b, &tm, sizeof tm);
    return true;
  };
  const bool ok = make(&out->w13, w, H / 2, rows13, 128, true) &&
                  make(&out->w2, w, I / 2, rows2, 128, true) &&
                  make(&out->s13, s, H / 16, rows13, 16, false) &&
                  make(&out->s2, s, I / 16, rows2, 16, false);
  if (!ok) {
    *out = TmaSource{};
    return false;
  }
  out->base_w = w;
  out->base_s = s;
  out->n = n;
  out->grid = num_sms;
  out->ok = true;
  return true;
}

bool mma_supported(int H, int I) {
  auto ok = [](int K) { return K % 64 == 0 && (K <= 256 ? (K == 128 || K == 256) : K % 256 == 0); };
  return ok(H) && ok(I) && I % 64 == 0 && H % 128 == 0;
}

cudaError_t launch_grouped_mma(cudaStream_t st, const GroupPlan* gp, int grid_x, bool gate_up,
                               int H, int I, int k, const QuantBuf& act, float* out,
                               uint32_t* flags, int g0, int g1, const TmaSource* tma,
                               bool maybe_host) {
  if (grid_x <= 0) return cudaSuccess;
  MmaArgs a;
  a.gp = gp;
  a.K = gate_up ? H : I;
  a.H = H;
  a.I = I;
  a.k = k;
  a.gate_up = gate_up ? 1 : 0;
  a.act = act;
  a.out = out;
  a.flags = flags;
  a.g0 = g0;
  a.g1 = g1;
  a.skip_w = nullptr;
  a.skip_n = 0;
  a.skip_Bw = 0;
  if (tma && tma->ok) {
    MmaTmaArgs t;
    t.map_w = gate_up ? tma->w13 : tma->w2;
    t.map_s = gate_up ? tma->s13 : tma->s2;
    t.m = a;
    t.base_w = tma->base_w;
    t.base_s = tma->base_s;
    t.Bw = 3LL * H * I / 2;
    t.Bs = 3LL * H * I / 16;
    t.n = tma->n;
    t.rps = gate_up ? 3 * I : 3 * H;
    t.row0 = gate_up ? 0 : 2 * H;
    cudaError_t e = run_mma_tma(st, t, tma->grid);
    if (e != cudaSuccess || !maybe_host) return e;
    a.skip_w = tma->base_w;
    a.skip_n = tma->n;
    a.skip_Bw = t.Bw;
  }
  const int m_tiles = gate_up ? I / 64 : H / kTileM;
  if (a.K >= 256) return run_mma<8>(st, a, grid_x, m_tiles);
  return run_mma<4>(st, a, grid_x, m_tiles);
}

cudaError_t launch_combine(cudaStream_t st, const GroupPlan* gp, const float* y, float* out,
                           int rows, int H, int k) {
  dim3 grid((H + 255) / 256, rows);
  combine_kernel<<<grid, 256, 0, st>>>(gp, y, out, H, k);
  return cudaGetLastError();
}

}  // namespace moe
