// draft_tc.cu -- bf16 draft step on the 5th-generation tensor cores (sm_103a).
//
// Method: "DSpark: Confidence-Scheduled Speculative Decoding with
// Semi-Autoregressive Generation 요약 설명" §3.1 -- for draft position k the
// Markov head adds B_k = W1[x_{k-1}] W2 (rank r) to the backbone logits U_k,
// the result is normalised locally and x_k is sampled from it, left to right.
// One launch computes, for all R requests at once,
//     s = (U_k + A_k W2) / T        A_k = W1[x_{k-1}]  ([R x r], gathered)
// writes s to `scores`, and leaves per-(row, CTA) partials of the local
// normaliser and of the Philox-keyed Gumbel-max draw for the combine kernel.
//
// Structure (one CTA per SM, persistent):
//   * The grid is (number of 128-row tiles Mt) x (slots); CTA c owns row tile
//     c % Mt and the vocab tiles n = c / Mt, c / Mt + slots, ...  Its A tile
//     (128 x r bf16) stays in shared memory for the whole step; the Mt CTAs
//     that share a vocab tile stream the same W2 tile at about the same time,
//     so W2 comes from HBM about once per step.
//   * The A tile is gathered by the epilogue warps at the start: for step 1
//     from the anchors, for step k > 1 from step k-1's drawn tokens (each
//     row's packed best (key, group) that step's CTAs raised, then the token
//     inside that group).  Each CTA then writes step k-1's x, logp and lse for
//     its share of the row tile's rows, merging those rows' per-slot partials
//     for the lse.  So consecutive steps need no separate combine launch; one
//     combine follows the last step.
//   * warp 16 (producer): TMA of W2^T chunks [128 vocab rows x 64 K] into a
//     3-stage ring.  W2^T (K-major) is written once per draft call by
//     transpose_w2_kernel, so each vocab tile's B operand is one contiguous
//     128 x r block instead of r rows strided V apart.
//   * warp 17 (MMA): allocates 256 TMEM columns (two 128 x 128 fp32
//     accumulators) and issues tcgen05.mma (kind::f16, bf16 x bf16 -> fp32,
//     M = 128, N = 128, K = 16) from shared-memory descriptors: A and W2^T both
//     K-major, 128-byte swizzled.
//   * warp 18 (finalization, steps k > 1): writes step k-1's x, logp and lse
//     for its share of the row tile's rows, beside the pipeline.
//   * warps 0..15 (epilogue): warp w reads TMEM lanes 32 (w % 4) .. +31 (its
//     rows) and columns 32 (w / 4) .. +31 of the tile.  The four warps of a
//     row quarter share its U_k tile (32 rows x 128 columns, two TMA boxes with
//     128-byte rows, loaded by the quarter's column-group-0 warp once all four
//     have read the previous one; the first, and the next few into L2, before
//     the wait on the previous step).  Each warp computes s, stages it in
//     swizzled shared memory and stores it (coalesced st.global for several
//     row tiles, TMA for one), and updates per-row running statistics in
//     registers: max / sum-exp (online), and stage 1 of the two-level draw.
//   * Two-level draw: each warp's 32 columns of a row are one group; its key
//     L_j + G(DRAFT_GROUP, j) can beat the running best key b only if
//     -ln u < exp(L_j - b); since -ln u >= 1 - u, the cheap test
//     1 - u < exp(L_j - b) (with 0.1% slack) lets the two logarithms run only
//     for candidates.  Stage 2 (an id inside the drawn group) runs in the next
//     step's prologue, or in the combine after the last step.
//   * Every mbarrier wait is bounded (about 2 s of SM clocks); on expiry the
//     CTA flags DSPARK_DEV_TIMEOUT in the status word, stops issuing work,
//     drains what it issued, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace dspark {

namespace {

constexpr int kTileM = 128;
constexpr int kTileN = kDraftTileN;  // 128
constexpr int kChunkK = 64;          // 128 bytes of bf16: one swizzle atom row
constexpr int kStages = 3;
constexpr int kEpiWarps = 16;
constexpr int kThreads = (kEpiWarps + 3) * 32;
constexpr int kProducerWarp = kEpiWarps;
constexpr int kMmaWarp = kEpiWarps + 1;
constexpr int kFinWarp = kEpiWarps + 2;  // step k-1's x, logp, lse, beside the pipeline
constexpr int kMaxRank = 256;
// U tiles of the CTA's next units fetched into L2 before the step's wait (see
// the epilogue); more than a few competed with the previous step's last tiles.
constexpr int kUPrefetch = 4;
constexpr uint32_t kTmemCols = 256;

constexpr int kAChunkBytes = kTileM * kChunkK * 2;  // 16 KB
constexpr int kBChunkBytes = kChunkK * kTileN * 2;  // 16 KB (two 64-column boxes)
constexpr int kUBoxBytes = 32 * 64 * 2;             // 4 KB: 32 rows x 64 columns of U
constexpr int kUQuarterBytes = 2 * kUBoxBytes;      // 8 KB: a row quarter's 128 columns
constexpr int kSBoxBytes = 32 * 32 * 4;             // 4 KB per epilogue warp

// Shared memory layout (offsets from a 1024-aligned base).
constexpr int kOffA = 0;                                            // 4 x 16 KB
constexpr int kOffB = kOffA + (kMaxRank / kChunkK) * kAChunkBytes;  // 64 KB
constexpr int kOffU = kOffB + kStages * kBChunkBytes;               // 112 KB
constexpr int kOffS = kOffU + 4 * kUQuarterBytes;                   // 144 KB
constexpr int kOffMerge = kOffS + kEpiWarps * kSBoxBytes;           // 208 KB
constexpr int kMergeBytes = 5 * 4 * kTileM * 4;                     // 10 KB
constexpr int kOffRowBest = kOffMerge + kMergeBytes;                // [128 rows][4 groups] fp32
constexpr int kOffDrawn = kOffRowBest + kTileM * 4 * 4;  // [128] x_{k-1}, then [128] its score
constexpr int kOffBar = kOffDrawn + kTileM * 8;
constexpr int kNumBars = 1 + 2 * kStages + 2 + 2 + kEpiWarps + 1;
constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;  // + slack for 1024 alignment

// ------------------------------------------------------------------ PTX wrappers
// (mbarrier and bounded-wait wrappers shared with verify.cu are in ptx.cuh)
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// Fetch a U box into L2 only (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(map),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
      : "memory");
}

// L2 eviction priority for TMA loads whose lines should stay (evict_last).
__device__ __forceinline__ uint64_t l2_policy_keep() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, int x, int y,
                                                 uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y,
                                             int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          map),
      "r"(x), "r"(y), "r"(z), "r"(smem_addr(src))
      : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc], one instruction of M=128, N=128, K=16.
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i gets row (lane base + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for tcgen05.mma: start address, leading and
// stride byte offsets (16-byte units), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // version
  d |= (uint64_t)2 << 61;  // SWIZZLE_128B
  return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N) {
  return (1u << 4)                        // D format: F32
         | (1u << 7)                      // A format: BF16
         | (1u << 10)                     // B format: BF16
         | (0u << 15)                     // A K-major
         | (0u << 16)                     // B K-major
         | ((uint32_t)(N >> 3) << 17)     // N / 8
         | ((uint32_t)(M >> 4) << 24);    // M / 16
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction (the three-input form of max.f32).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// 1 + (w >> 9) 2^-23 as a float in [1, 2): the funnel shift of (0x7F : w) by 9
// places w's top 23 bits under the exponent field of 1.0f.
__device__ __forceinline__ float unit_float(uint32_t w) {
  return __uint_as_float(__funnelshift_r(w, 0x7Fu, 9));
}

__device__ __forceinline__ void named_barrier(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Arrive on a named barrier without waiting for it.
__device__ __forceinline__ void named_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}


struct Params {
  int R, gamma, V, r, k, Mt, slots, n_tiles, n_parts;
  float invT;
  uint64_t seed;
  const int32_t* x0;             // anchors (step 1)
  const __nv_bfloat16* W1;       // [V, r]
  const __nv_bfloat16* A_src;    // [R, r] precomputed A rows (RNN head), or nullptr
  const float4* prev_stats;      // step k-1 partials (k > 1)
  const int* prev_index;
  float4* pstats;                // this step's partials
  int* pindex;
  // [R] per row, the best (group key, group) any CTA of a step has reached,
  // packed as key_ord(key) << 32 | ~group (so that the u64 maximum takes the
  // larger key, then the smaller group): step k-1's (read by the prologue),
  // this step's (raised with atomicMax), and step k+1's (zeroed here).
  const unsigned long long* gbest_prev;
  unsigned long long* gbest_cur;
  unsigned long long* gbest_next;
  int32_t* x;                    // step k-1 outputs: each row by one CTA of its row tile
  float* logp;
  float* lse;
  int* status;
  float* scores;           // [R, gamma, V]: stored by the epilogue (kStg), read by stage 2
  long long wait_budget;  // SM clocks each bounded wait may take
  int withhold_w2;        // diagnostic: the producer issues no W2 loads, so the waits run out
  // W2^T kept in L2 across the steps (it fits); the last step hands its lines
  // back to the normal eviction order when done.
  int w2_keep;
  const __nv_bfloat16* w2t;
};

template <bool kStg>
__global__ void __launch_bounds__(kThreads, 1)
draft_step_tc_kernel(const __grid_constant__ CUtensorMap tmW2,
                     const __grid_constant__ CUtensorMap tmU,
                     const __grid_constant__ CUtensorMap tmS, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(smem + kOffBar);
  uint64_t* bar_a = bars;                         // A tile gathered (one arrive per epilogue warp)
  uint64_t* bar_full = bars + 1;                  // [kStages] W2 chunk loaded
  uint64_t* bar_empty = bars + 1 + kStages;       // [kStages] W2 chunk consumed
  uint64_t* bar_acc_full = bars + 1 + 2 * kStages;   // [2] accumulator ready
  uint64_t* bar_acc_empty = bar_acc_full + 2;        // [2] accumulator drained
  uint64_t* bar_u = bar_acc_empty + 2;               // [4] quarter's U tile loaded, [4..7] read
  uint64_t* bar_drain = bar_u + kEpiWarps;           // MMA drain at exit
  uint32_t* tmem_slot = (uint32_t*)(bars + kNumBars);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

  // The next step may be scheduled as soon as SMs free up: its CTAs set up and
  // prefetch W2 until their griddepcontrol.wait, which waits for this grid.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tile = blockIdx.x % p.Mt;
  const int slot = blockIdx.x / p.Mt;
  const int n_units = slot < p.n_tiles ? (p.n_tiles - 1 - slot) / p.slots + 1 : 0;
  const int n_chunks = p.r / kChunkK;

  if (threadIdx.x == 0) {
    mbar_init(bar_a, kEpiWarps);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_acc_full[b], 1);
      mbar_init(&bar_acc_empty[b], kEpiWarps);
    }
    for (int q = 0; q < 4; ++q) {
      mbar_init(&bar_u[q], 1);      // U tile of quarter q loaded
      mbar_init(&bar_u[4 + q], 4);  // read by the quarter's four warps
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  {
    float* rb = (float*)(smem + kOffRowBest);
    for (int i = threadIdx.x; i < kTileM * 4; i += blockDim.x) rb[i] = -INFINITY;
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_units > 0 && !p.withhold_w2) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      // W2^T is read again by the next step: where it fits in L2, its loads mark
      // it to be kept (evict_last) over the streamed U and scores.
      const uint64_t pol_w2 = l2_policy_keep();
      bool ok = true;
      for (int u = 0; u < n_units && ok; ++u) {
        const int n = slot + u * p.slots;
        for (int c = 0; c < n_chunks; ++c) {
          if (!mbar_wait(&bar_empty[stage], phase ^ 1u, abort_flag, p.wait_budget)) {
            ok = false;
            break;
          }
          uint8_t* dst = smem + kOffB + stage * kBChunkBytes;
          mbar_expect_tx(&bar_full[stage], kBChunkBytes);
          // W2^T rows n*128 .. +127, K columns c*64 .. +63 (one contiguous 64 KB block per tile)
          if (p.w2_keep)
            tma_load_2d_hint(dst, &tmW2, c * kChunkK, n * kTileN, &bar_full[stage], pol_w2);
          else
            tma_load_2d(dst, &tmW2, c * kChunkK, n * kTileN, &bar_full[stage]);
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Drain: wait (bounded) for the loads still in flight before leaving.
        int s = stage, ph = phase;
        for (int i = 0; i < kStages && i < issued; ++i) {
          s = (s + kStages - 1) % kStages;
          if (s == kStages - 1) ph ^= 1;
          mbar_drain(&bar_full[s], ph, p.wait_budget);
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_units > 0) {
      const uint32_t idesc = make_idesc(kTileM, kTileN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = mbar_wait(bar_a, 0, abort_flag, p.wait_budget);
      tc_fence_after();
      for (int u = 0; u < n_units && ok; ++u) {
        const int buf = u & 1;
        const uint32_t acc_phase = (u >> 1) & 1;
        if (!mbar_wait(&bar_acc_empty[buf], acc_phase ^ 1u, abort_flag, p.wait_budget)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * kTileN);
        for (int c = 0; c < n_chunks; ++c) {
          if (!mbar_wait(&bar_full[stage], phase, abort_flag, p.wait_budget)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_addr(smem + kOffA + c * kAChunkBytes);
          const uint32_t b_base = smem_addr(smem + kOffB + stage * kBChunkBytes);
#pragma unroll
          for (int kk = 0; kk < kChunkK / 16; ++kk) {
            // A: K-major, 128-byte rows, 8-row groups 1024 B apart; K advances 32 B.
            const uint64_t ad = smem_desc_sw128(a_base + kk * 32, 16, 1024);
            // W2^T: K-major like A (128 vocab rows of 128 bytes).
            const uint64_t bd = smem_desc_sw128(b_base + kk * 32, 16, 1024);
            tc_mma(d_tmem, ad, bd, idesc, (c | kk) != 0);
          }
          tc_commit(&bar_empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&bar_acc_full[buf]);
      }
      // All MMAs done before TMEM is freed.
      tc_commit(bar_drain);
      mbar_drain(bar_drain, 0, p.wait_budget);
    }
  } else if (warp == kFinWarp) {
    // ------------------------------------------------------------ finalization
    // x, logp and lse of step k-1 for the rows q = slot, slot + slots, ... of
    // this row tile (each row by one CTA), beside the pipeline: the row's
    // log-normaliser merged from its partials (lanes over the partials), its
    // drawn token and score from the epilogue warps' prologue (shared memory,
    // behind named barrier 2).
    if (p.k >= 2 && !p.A_src) {
      asm volatile("griddepcontrol.wait;" ::: "memory");
      named_barrier(2, (kEpiWarps + 1) * 32);
      const int m_row0 = m_tile * kTileM;
      for (int q = slot; q < kTileM; q += p.slots) {
        const int arow = m_row0 + q;
        if (arow >= p.R) break;
        float m = -INFINITY, S = 0.0f;
        for (int t = lane; t < p.n_parts; t += 32) {
          const float4 st = p.prev_stats[(size_t)arow * p.n_parts + t];
          lse_merge(m, S, st.x, st.y);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
          const float s2 = __shfl_xor_sync(0xffffffffu, S, o);
          lse_merge(m, S, m2, s2);
        }
        if (lane == 0) {
          const float l = m + logf(S);
          const size_t o = (size_t)arow * p.gamma + (p.k - 2);
          p.x[o] = ((const int*)(smem + kOffDrawn))[q];
          p.logp[o] = ((const float*)(smem + kOffDrawn))[kTileM + q] - l;
          p.lse[o] = l;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int cgrp = warp >> 2;
    const int row_local = quarter * 32 + lane;
    const int row = m_tile * kTileM + row_local;
    const bool row_ok = row < p.R;
    // The quarter's U tile: 32 rows x 128 columns as two 64-column boxes (128-byte rows,
    // 128-byte swizzle), loaded by the quarter's column-group-0 warp, read by all four.
    uint8_t* uq = smem + kOffU + quarter * kUQuarterBytes;
    uint8_t* sbox = smem + kOffS + warp * kSBoxBytes;
    const int row0 = m_tile * kTileM + quarter * 32;
    const int kpos = p.k - 1;
    const float L2E = 1.4426950408889634f;

    // Stage 1 of the two-level draw: one group key per (row, 32-column group).
    const PhiloxStream rng(p.seed, (uint32_t)row, (uint32_t)p.k, DSPARK_PURPOSE_DRAFT_GROUP);
    float run_m = -INFINITY, run_s = 0.0f, best = -INFINITY;
    int best_j = 0x7fffffff;
    // The first U tile, and the next few into L2: U is an input of the call
    // that no kernel of the draft writes, so it loads before the wait below,
    // while the previous step's last CTAs still run and HBM has room.
    if (cgrp == 0 && lane == 0 && n_units > 0) {
      mbar_expect_tx(&bar_u[quarter], kUQuarterBytes);
      tma_load_3d(uq, &tmU, slot * kTileN, kpos, row0, &bar_u[quarter]);
      tma_load_3d(uq + kUBoxBytes, &tmU, slot * kTileN + 64, kpos, row0, &bar_u[quarter]);
      for (int u = 1; u <= kUPrefetch && u < n_units; ++u) {
        const int n = slot + u * p.slots;
        tma_prefetch_3d(&tmU, n * kTileN, kpos, row0);
        tma_prefetch_3d(&tmU, n * kTileN + 64, kpos, row0);
      }
    }
    // Everything below reads or writes what the previous step (launched as this
    // grid's programmatic primary) wrote or reads: wait for its completion.
    // Its outputs are read with coherent loads (plain or ld.global.cg), never
    // the non-coherent path: this grid may have started while that step ran.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (slot == 0 && cgrp == 0 && row_ok) p.gbest_next[row] = 0ull;
    // U loads of this warp issued so far and those waited for (equal on exit
    // unless a wait failed: the one in flight must land before the CTA exits).
    int u_issued = n_units > 0 ? 1 : 0, u_landed = 0;
    // A tile: rows m_tile*128 + 8 warp .. +7 get W1[x_{k-1}], written straight into
    // the K-major 128-byte-swizzled layout the MMA reads (zero rows past R).
    // x_{k-1} is the anchor for k = 1, else step k-1's draw: its packed
    // per-row best gives the group, and lanes 4i .. 4i+3 (row i of the warp's
    // 8) draw the token inside it (stage 2).
    int xps[8];
    if (p.A_src) {  // the A rows come precomputed (RNN head); x_{k-1} is stored elsewhere
#pragma unroll
      for (int i = 0; i < 8; ++i) xps[i] = 0;
    } else if (p.k == 1) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int arow = m_tile * kTileM + warp * 8 + i;
        xps[i] = arow < p.R ? p.x0[arow] : 0;
      }
    } else {
      // The row's drawn group of step k-1: the packed best that step's CTAs
      // raised (the larger key, ties to the smaller group).
      const int sub = lane & 3;
      const int arow = m_tile * kTileM + warp * 8 + (lane >> 2);
      const bool ok_row = arow < p.R;
      const unsigned long long pb = ok_row ? __ldcg(p.gbest_prev + arow) : 0ull;
      const int gj = (pb >> 32) ? (int)~(uint32_t)pb : 0x7fffffff;
      // Stage 2: x_{k-1} inside group gj, from step k-1's stored scores.  The
      // row's four lanes take 8 ids each; each lane keys its largest score
      // exactly, filters the other seven against it (the draft epilogue's
      // test, on ids), and the four lanes' best keys are merged.
      int idx = 0x7fffffff;
      float sv = 0.0f;
      {
        const bool have_group = ok_row && gj >= 0 && gj < (p.V + kGroup - 1) / kGroup;
        const int v0 = (have_group ? gj : 0) * kGroup + 8 * sub;
        float bk = -INFINITY;
        if (have_group && v0 < p.V) {  // V % 8 == 0: the lane's 8 ids are all valid
          const float4* src =
              (const float4*)(p.scores + ((size_t)arow * p.gamma + (p.k - 2)) * p.V + v0);
          const float4 s0 = src[0], s1 = src[1];
          const float sc[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
          const uint4 w0 = rng_quad(p.seed, (uint32_t)arow, (uint32_t)(p.k - 1), DSPARK_PURPOSE_DRAFT,
                                    (uint32_t)v0 >> 2);
          const uint4 w1 = rng_quad(p.seed, (uint32_t)arow, (uint32_t)(p.k - 1), DSPARK_PURPOSE_DRAFT,
                                    ((uint32_t)v0 >> 2) + 1u);
          const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
          int im = 0;
          float sm = sc[0];
          uint32_t wm = w[0];
#pragma unroll
          for (int t = 1; t < 8; ++t)
            if (sc[t] > sm) {
              sm = sc[t];
              wm = w[t];
              im = t;
            }
          bk = __fadd_rn(sm, gumbel(wm));
          idx = v0 + im;
          sv = sm;
          const float L2E = 1.4426950408889634f;
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            if (t == im) continue;
            // element t can reach bk only if fl(f + 1.001 exp(s - bk)) >= 2
            const float d = unit_float(w[t]) + ex2_approx((sc[t] - bk) * L2E) * 1.001f;
            if (d >= 2.0f) {
              const float kt = __fadd_rn(sc[t], gumbel(w[t]));
              if (better(kt, v0 + t, bk, idx)) {
                bk = kt;
                idx = v0 + t;
                sv = sc[t];
              }
            }
          }
        }
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1) {
          const float k2 = __shfl_xor_sync(0xffffffffu, bk, o);
          const int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
          const float v2 = __shfl_xor_sync(0xffffffffu, sv, o);
          if (better(k2, i2, bk, idx)) {
            bk = k2;
            idx = i2;
            sv = v2;
          }
        }
      }
      if (ok_row && (idx < 0 || idx >= p.V)) {  // nothing drawn: every score of the row was NaN
        if (sub == 0) flag_status(p.status, DSPARK_DEV_BAD_INPUT);
        idx = 0;
      }
      if (sub == 0) {  // for the row's x, logp, lse of step k-1, written after the A tile
        const int q = warp * 8 + (lane >> 2);
        ((int*)(smem + kOffDrawn))[q] = idx;
        ((float*)(smem + kOffDrawn))[kTileM + q] = sv;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) xps[i] = __shfl_sync(0xffffffffu, idx, 4 * i);
    }
    uint4 gv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int arow = m_tile * kTileM + warp * 8 + i;
      int xp = xps[i];
      if (arow < p.R && (xp < 0 || xp >= p.V)) {
        if (lane == 0) flag_status(p.status, DSPARK_DEV_BAD_INPUT);
        xp = xp < 0 ? 0 : p.V - 1;
      }
      gv[i] = make_uint4(0u, 0u, 0u, 0u);
      if (arow < p.R && lane < p.r / 8)  // 16 bytes = 8 of the row's r bf16 per lane
        gv[i] = __ldg(reinterpret_cast<const uint4*>(
                          p.A_src ? p.A_src + (size_t)arow * p.r : p.W1 + (size_t)xp * p.r) +
                      lane);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int rl = warp * 8 + i;
      if (lane < p.r / 8) {
        const int c = lane >> 3, piece = lane & 7;
        *(uint4*)(smem + kOffA + c * kAChunkBytes + rl * 128 + ((piece ^ (rl & 7)) << 4)) = gv[i];
      }
    }
    fence_proxy_async();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_a);
    // The drawn rows are in shared memory: the finalization warp may go on.
    if (p.k >= 2 && !p.A_src) named_arrive(2, (kEpiWarps + 1) * 32);
    for (int u = 0; u < n_units; ++u) {
      const int n = slot + u * p.slots;
      const int buf = u & 1;
      const uint32_t acc_phase = (u >> 1) & 1;
      const int col0 = n * kTileN + cgrp * 32;
      // The row's best key over all CTAs of this step so far, read early (L2).
      const uint32_t gkey = row_ok ? (uint32_t)(__ldcg(p.gbest_cur + row) >> 32) : 0u;

      // U of this warp: row `lane`, its 32 columns of the quarter's tile.
      // Waits are decided warp-wide; on a failed one the warp leaves the loop
      // (every epilogue warp still reaches the merge barrier below).
      if (!__all_sync(0xffffffffu, mbar_wait(&bar_u[quarter], u & 1, abort_flag, p.wait_budget)))
        break;
      u_landed = u + 1;
      uint32_t upk[16];
      {
        // this warp's 32 columns: chunks 4 (cgrp & 1) .. +3 of box cgrp >> 1, row `lane`
        const uint8_t* rowp = uq + (cgrp >> 1) * kUBoxBytes + lane * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int pc = (4 * (cgrp & 1) + c) ^ (lane & 7);
          const uint4 q = *(const uint4*)(rowp + pc * 16);
          upk[4 * c + 0] = q.x;
          upk[4 * c + 1] = q.y;
          upk[4 * c + 2] = q.z;
          upk[4 * c + 3] = q.w;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_u[4 + quarter]);
      if (u + 1 < n_units && cgrp == 0) {
        // the next tile may overwrite the buffer once all four warps have read it
        const bool freed = __all_sync(0xffffffffu, mbar_wait(&bar_u[4 + quarter], u & 1, abort_flag,
                                                               p.wait_budget));
        if (!freed) break;
        if (lane == 0) {
          fence_proxy_async();
          mbar_expect_tx(&bar_u[quarter], kUQuarterBytes);
          tma_load_3d(uq, &tmU, (n + p.slots) * kTileN, kpos, row0, &bar_u[quarter]);
          tma_load_3d(uq + kUBoxBytes, &tmU, (n + p.slots) * kTileN + 64, kpos, row0,
                      &bar_u[quarter]);
        }
        u_issued = u + 2;
      }

      // Accumulator columns of this warp.
      if (!__all_sync(0xffffffffu, mbar_wait(&bar_acc_full[buf], acc_phase, abort_flag, p.wait_budget)))
        break;
      tc_fence_after();
      uint32_t acc[32];
      tmem_ld32(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * kTileN + cgrp * 32),
                acc);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_acc_empty[buf]);

      float s[32];
      {
        const float2 invT2 = make_float2(p.invT, p.invT);
#pragma unroll
        for (int i = 0; i < 16; ++i) {  // (u + acc) / T on float pairs
          const float2 u2 = make_float2(__uint_as_float(upk[i] << 16),
                                        __uint_as_float(upk[i] & 0xffff0000u));
          const float2 a2 = make_float2(__uint_as_float(acc[2 * i]), __uint_as_float(acc[2 * i + 1]));
          const float2 s2 = __fmul2_rn(__fadd2_rn(u2, a2), invT2);
          s[2 * i] = s2.x;
          s[2 * i + 1] = s2.y;
        }
      }

      // Stage s (128-byte rows, 128-byte swizzle) and store it: with TMA
      // (!kStg), or with coalesced 16-byte stores, lanes 8i .. 8i+7 writing one
      // row's 128 bytes (kStg: keeps the score stores off the TMA unit, which
      // also carries the U and W2 loads).
      if constexpr (!kStg) {
        if (lane == 0) bulk_wait_read0();
      }
      __syncwarp();
      {
        uint8_t* rowp = sbox + lane * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int pc = c ^ (lane & 7);
          *(float4*)(rowp + pc * 16) = make_float4(s[4 * c], s[4 * c + 1], s[4 * c + 2], s[4 * c + 3]);
        }
      }
      if constexpr (kStg) {
        __syncwarp();
        const int c = lane & 7;
        const int v = col0 + 4 * c;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int rr = 4 * i + (lane >> 3);
          const float4 val = *(const float4*)(sbox + rr * 128 + ((c ^ (rr & 7)) << 4));
          if (row0 + rr < p.R && v < p.V)
            __stcs((float4*)(p.scores + ((size_t)(row0 + rr) * p.gamma + kpos) * p.V + v), val);
        }
      } else {
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&tmS, sbox, col0, kpos, row0);
          bulk_commit();
        }
      }

      // Running statistics of this row over its 32 columns, which are one
      // group j of the two-level draw: the online (max, sum exp) of the row,
      // and stage 1 -- the group's log-mass L_j = mx + log st and its key
      // L_j + G(seed, row, k, DRAFT_GROUP, j).
      const int nvalid = row_ok ? min(32, p.V - col0) : 0;
      if (nvalid > 0) {
        if (nvalid < 32) {  // ragged last tile: columns past V take no part
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (i >= nvalid) s[i] = -INFINITY;
        }
        float mx = fmax3(s[0], s[1], s[2]);
#pragma unroll
        for (int i = 3; i < 31; i += 2) mx = fmax3(mx, s[i], s[i + 1]);
        mx = fmaxf(mx, s[31]);
        float st;
        {
          const float2 l2e = make_float2(L2E, L2E), nmx = make_float2(-mx * L2E, -mx * L2E);
          float2 sum = make_float2(0.0f, 0.0f);
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 a2 = __ffma2_rn(make_float2(s[i], s[i + 1]), l2e, nmx);
            sum = __fadd2_rn(sum, make_float2(ex2_approx(a2.x), ex2_approx(a2.y)));
          }
          st = sum.x + sum.y;
        }
        lse_merge(run_m, run_s, mx, st);
        const int gj = col0 >> 5;
        const float Lg = __fadd_rn(mx, logf(st));
        const uint4 w4 = rng.quad((uint32_t)col0 >> 7);  // groups 4n .. 4n+3 of vocab tile n
        const uint32_t wg = cgrp == 0 ? w4.x : cgrp == 1 ? w4.y : cgrp == 2 ? w4.z : w4.w;
        // Threshold: the best group key this row has reached so far in any of
        // the CTA's four column groups (shared memory) or in any CTA of this
        // step (global, raised with atomicMax).  Every published key is one a
        // group of the row reached, so a stale value is still a lower bound of
        // the row's maximum and no barrier is needed.
        volatile float* rowbest = (volatile float*)(smem + kOffRowBest) + row_local * 4;
        float thr = fmaxf(best, ord_key(gkey));
#pragma unroll
        for (int g2 = 0; g2 < 4; ++g2)
          if (g2 != cgrp) thr = fmaxf(thr, rowbest[g2]);
        // The group can reach thr only if 1 - u < exp(Lg - thr), tested as
        // fl(f + 1.001 exp(Lg - thr)) >= 2 (f = 1 + (w >> 9) 2^-23); with no
        // key yet the group is keyed exactly.
        const bool cand = thr == -INFINITY ||
                          unit_float(wg) + ex2_approx((Lg - thr) * L2E) * 1.001f >= 2.0f;
        bool raised = false;
        if (cand) {
          const float key = __fadd_rn(Lg, gumbel(wg));
          if (better(key, gj, best, best_j)) {
            best = key;
            best_j = gj;
            raised = true;
          }
        }
        // Publish for the row's other groups and CTAs.  A key equal to the
        // threshold is published too, so that the packed maximum ends on the
        // smaller of two groups with equal keys, as the partials' merge would.
        if (raised && best >= thr) {
          rowbest[cgrp] = best;
          if (best < INFINITY)
            atomicMax(p.gbest_cur + row,
                      ((unsigned long long)key_ord(best) << 32) | (unsigned long long)~(uint32_t)best_j);
        }
      }
    }

    // Merge the four column groups of each row, then write the row's partial.
    float* mg = (float*)(smem + kOffMerge);
    mg[(0 * 4 + cgrp) * kTileM + row_local] = run_m;
    mg[(1 * 4 + cgrp) * kTileM + row_local] = run_s;
    mg[(2 * 4 + cgrp) * kTileM + row_local] = best;
    ((int*)mg)[(4 * 4 + cgrp) * kTileM + row_local] = best_j;
    named_barrier(1, kEpiWarps * 32);
    if (cgrp == 0 && row_ok && n_units > 0) {
      float m = -INFINITY, S = 0.0f, bk = -INFINITY;
      int bi = 0x7fffffff;
      for (int g = 0; g < 4; ++g) {
        lse_merge(m, S, mg[(0 * 4 + g) * kTileM + row_local], mg[(1 * 4 + g) * kTileM + row_local]);
        const float k2 = mg[(2 * 4 + g) * kTileM + row_local];
        const int i2 = ((int*)mg)[(4 * 4 + g) * kTileM + row_local];
        if (better(k2, i2, bk, bi)) {
          bk = k2;
          bi = i2;
        }
      }
      const size_t o = (size_t)row * p.n_parts + slot;
      p.pstats[o] = make_float4(m, S, bk, 0.0f);
      p.pindex[o] = bi;
    }
    if (p.w2_keep && p.k == p.gamma) {
      // Last step: the W2^T rows of this CTA's vocab tiles (128-byte lines)
      // go back to the normal eviction order, so that what runs after the
      // draft gets the L2; the Mt CTAs that share the tiles split the lines.
      const int lines_per_row = p.r * 2 / 128;
      const int lines = n_units * kTileN * lines_per_row;
      for (int i = threadIdx.x + m_tile * kEpiWarps * 32; i < lines; i += p.Mt * kEpiWarps * 32) {
        const int u = i / (kTileN * lines_per_row), rest = i - u * (kTileN * lines_per_row);
        const size_t vrow = (size_t)(slot + u * p.slots) * kTileN + rest / lines_per_row;
        if (vrow < (size_t)p.V) {
          const char* a = (const char*)(p.w2t + vrow * p.r) + (rest % lines_per_row) * 128;
          asm volatile("applypriority.global.L2::evict_normal [%0], 128;" ::"l"(a) : "memory");
        }
      }
    }
    if (lane == 0) {
      if (cgrp == 0 && u_issued > u_landed)
        mbar_drain(&bar_u[quarter], (uint32_t)(u_issued - 1) & 1u, p.wait_budget);
      bulk_wait0();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) flag_status(p.status, DSPARK_DEV_TIMEOUT);
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// W2 [r, V] -> W2^T [V, r] (bf16), 64 x 64 tiles through shared memory, so the
// MMA's B operand of a vocab tile is one contiguous 128 x r block.  Both sides
// move 16-byte chunks (8 bf16): whole 128-byte rows in and out.  Needs
// V % 8 == 0 and r % 8 == 0 and a 16-byte aligned W2 (the tensor-core path
// checks all three).
__global__ void __launch_bounds__(256)
transpose_w2_kernel(const __nv_bfloat16* __restrict__ W2, int r, int V,
                    __nv_bfloat16* __restrict__ W2T) {
  __shared__ unsigned short tile[64][66];  // [k][v]; the padding spreads columns over banks
  const int k0 = blockIdx.y * 64, v0 = blockIdx.x * 64;
  const unsigned short* src = reinterpret_cast<const unsigned short*>(W2);
  unsigned short* dst = reinterpret_cast<unsigned short*>(W2T);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int c = threadIdx.x + 256 * h;  // 512 chunks: 64 k rows x 8 chunks of 8 vocab ids
    const int i = c >> 3, j = (c & 7) * 8;
    const int k = k0 + i, v = v0 + j;
    uint4 q = make_uint4(0u, 0u, 0u, 0u);
    if (k < r && v < V) q = __ldg(reinterpret_cast<const uint4*>(src + (size_t)k * V + v));
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      tile[i][j + 2 * e] = (unsigned short)(w[e] & 0xffffu);
      tile[i][j + 2 * e + 1] = (unsigned short)(w[e] >> 16);
    }
  }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int c = threadIdx.x + 256 * h;  // 64 vocab rows x 8 chunks of 8 k
    const int i = c >> 3, j = (c & 7) * 8;
    const int v = v0 + i, k = k0 + j;
    if (v < V && k < r) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        w[e] = (uint32_t)tile[j + 2 * e][i] | ((uint32_t)tile[j + 2 * e + 1][i] << 16);
      *reinterpret_cast<uint4*>(dst + (size_t)v * r + k) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)ptr;
  });
  return fn;
}

bool encode(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base,
            const cuuint64_t* dims, const cuuint64_t* strides_bytes, const cuuint32_t* box,
            CUtensorMapSwizzle sw) {
  auto fn = get_encode();
  if (!fn) return false;
  cuuint32_t estride[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(m, dt, (cuuint32_t)rank, const_cast<void*>(base), dims, strides_bytes, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// L2 size of the current device (bytes), once.
static size_t l2_bytes() {
  static size_t n = 0;
  if (n == 0) {
    int dev = 0, v = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev);
    n = v > 0 ? (size_t)v : 1;
  }
  return n;
}

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

}  // namespace

bool draft_tc_supported(int R, int V, int r) {
  (void)R;
  if (r % kChunkK != 0 || r > kMaxRank || V % 8 != 0) return false;
  return get_encode() != nullptr;
}

int draft_tc_parts(int R, int V) {
  const int Mt = (R + kTileM - 1) / kTileM;
  const int n_tiles = (V + kTileN - 1) / kTileN;
  int slots = sm_count() / Mt;
  if (slots < 1) slots = 1;
  if (slots > n_tiles) slots = n_tiles;
  return slots;
}

cudaError_t prepare_draft_tc(DraftTcPlan* plan, const void* U, const void* W2T, int R, int gamma,
                             int V, int r, float* scores) {
  static_assert(sizeof(CUtensorMap) == 128, "tensor map size");
  CUtensorMap* maps = reinterpret_cast<CUtensorMap*>(plan->maps);
  {
    // W2^T [V, r], K (r) innermost
    const cuuint64_t dims[2] = {(cuuint64_t)r, (cuuint64_t)V};
    const cuuint64_t strides[1] = {(cuuint64_t)r * 2};
    const cuuint32_t box[2] = {kChunkK, kTileN};
    if (!encode(&maps[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, W2T, dims, strides, box,
                CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)V, (cuuint64_t)gamma, (cuuint64_t)R};
    const cuuint64_t strides[2] = {(cuuint64_t)V * 2, (cuuint64_t)gamma * V * 2};
    const cuuint32_t box[3] = {64, 1, 32};
    if (!encode(&maps[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, U, dims, strides, box,
                CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)V, (cuuint64_t)gamma, (cuuint64_t)R};
    const cuuint64_t strides[2] = {(cuuint64_t)V * 4, (cuuint64_t)gamma * V * 4};
    const cuuint32_t box[3] = {32, 1, 32};
    if (!encode(&maps[2], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, scores, dims, strides, box,
                CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  // Once per process (thread-safe initialisation of a function-local static).
  static const cudaError_t attr_err = [] {
    cudaError_t e = cudaFuncSetAttribute(draft_step_tc_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(draft_step_tc_kernel<true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    return e;
  }();
  if (attr_err != cudaSuccess) return attr_err;
  plan->scores = scores;
  plan->w2t = W2T;
  plan->R = R;
  plan->gamma = gamma;
  plan->V = V;
  plan->r = r;
  return cudaSuccess;
}

cudaError_t launch_transpose_w2(const void* W2, int r, int V, void* W2T, cudaStream_t s) {
  dim3 grid((V + 63) / 64, (r + 63) / 64);
  transpose_w2_kernel<<<grid, 256, 0, s>>>((const __nv_bfloat16*)W2, r, V, (__nv_bfloat16*)W2T);
  return cudaGetLastError();
}

cudaError_t launch_draft_step_tc(const DraftTcPlan& plan, int k, float invT, uint64_t seed,
                                 const int32_t* x0, const void* W1, const DraftPartials& prev,
                                 const DraftPartials& cur, unsigned long long* gbest, int32_t* x,
                                 float* logp, float* lse, int* status, cudaStream_t s,
                                 const void* A_src, long long wait_budget, bool withhold_w2) {
  const int Mt = (plan.R + kTileM - 1) / kTileM;
  const int n_tiles = (plan.V + kTileN - 1) / kTileN;
  const int slots = draft_tc_parts(plan.R, plan.V);
  const CUtensorMap* maps = reinterpret_cast<const CUtensorMap*>(plan.maps);
  Params p;
  p.R = plan.R;
  p.gamma = plan.gamma;
  p.V = plan.V;
  p.r = plan.r;
  p.k = k;
  p.Mt = Mt;
  p.slots = slots;
  p.n_tiles = n_tiles;
  p.n_parts = slots;
  p.invT = invT;
  p.seed = seed;
  p.x0 = x0;
  p.W1 = (const __nv_bfloat16*)W1;
  p.A_src = (const __nv_bfloat16*)A_src;
  p.prev_stats = prev.stats;
  p.prev_index = prev.index;
  p.pstats = cur.stats;
  p.pindex = cur.index;
  p.gbest_prev = gbest + (size_t)((k + 2) % 3) * plan.R;  // step k-1's
  p.gbest_cur = gbest + (size_t)(k % 3) * plan.R;
  p.gbest_next = gbest + (size_t)((k + 1) % 3) * plan.R;
  p.x = x;
  p.logp = logp;
  p.lse = lse;
  p.status = status;
  p.scores = plan.scores;
  p.wait_budget = wait_budget > 0 ? wait_budget : kWaitBudget;
  p.withhold_w2 = withhold_w2 ? 1 : 0;
  p.w2t = (const __nv_bfloat16*)plan.w2t;
  // (rows of whole 128-byte lines, r % 64 == 0, so that each line the last
  // step hands back starts on a line boundary)
  p.w2_keep = plan.r % 64 == 0 && (size_t)plan.V * plan.r * 2 <= l2_bytes() / 4 * 3 ? 1 : 0;
  // Score stores: coalesced st.global when several row tiles share each W2
  // tile (the TMA unit then carries U and W2 for up to Mt CTAs' worth of
  // stores), TMA stores for a single row tile (R <= 128), where W2 dominates.
  auto kernel = Mt > 1 ? draft_step_tc_kernel<true> : draft_step_tc_kernel<false>;
  // Programmatic dependent launch on the previous kernel for k >= 2 (the
  // previous draft step) and for the RNN head (the state update of this step,
  // which itself follows the W2 transpose in stream order; see the kernel).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(Mt * slots);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (k >= 2 || A_src) ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, maps[0], maps[1], maps[2], p);
}

}  // namespace dspark
