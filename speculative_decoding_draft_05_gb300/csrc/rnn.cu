// rnn.cu -- the state update of the RNN draft head.
//
// "DSpark: Confidence-Scheduled Speculative Decoding with Semi-Autoregressive
// Generation 요약 설명", §3.1: the alternative sequential head keeps a state
// across the block and also takes the backbone's hidden state.  Read as an
// Elman recurrence in the Markov head's rank-r space,
//     h_0 = 0,  h_k = tanh(W1[x_{k-1}] + h_{k-1} Wh + Q_k),  B_k = bf16(h_k) W2,
// the bias contraction B_k is the Markov head's (draft_tc.cu, A taken from a
// buffer instead of gathered W1 rows).  This kernel runs before each draft
// step: it merges the previous step's per-CTA partials into the drawn group,
// draws x_{k-1} inside that group (stage 2 of the two-level draw, from the
// stored scores; it stores x, logp, lse of step k-1), then updates the state
// in fp32 and writes
// its bf16 rounding (nearest, ties to even) as the step's A rows.
//
// Grid: (row blocks of kRnnRows) x (column blocks of kRnnCols).  A CTA stages
// its column block of Wh (r x 64 bf16, 32 KB) and its rows' previous states
// (fp32) in shared memory; warp i merges row i's partials of step k-1, then
// lane l forms state columns c0 + 2l, c0 + 2l + 1 of row i.  The state is
// double-buffered (step k reads h_{k-1}, writes h_k) because the CTAs of one
// row read all of h_{k-1} while each writes only its own columns.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace dspark {

namespace {

constexpr int kRnnThreads = 256;
constexpr int kRnnRows = kRnnThreads / 32;  // one row per warp
constexpr int kRnnCols = 64;                // two columns per lane
constexpr int kRnnMaxR = 256;

__global__ void __launch_bounds__(kRnnThreads)
rnn_state_kernel(int k, const int32_t* __restrict__ x0, const __nv_bfloat16* __restrict__ W1,
                 const __nv_bfloat16* __restrict__ Wh, const float* __restrict__ Q,
                 const float4* __restrict__ prev_stats, const int* __restrict__ prev_index,
                 int n_parts, int R, int gamma, int V, int r, const float* __restrict__ h_prev,
                 float* __restrict__ h_next, __nv_bfloat16* __restrict__ A,
                 const float* __restrict__ scores, uint64_t seed, int32_t* __restrict__ x,
                 float* __restrict__ logp, float* __restrict__ lse, int* __restrict__ status) {
  __shared__ int s_x[kRnnRows];
  __shared__ float s_h[kRnnRows][kRnnMaxR];
  __shared__ __align__(16) __nv_bfloat162 s_w[kRnnMaxR][kRnnCols / 2];
  // The draft step that follows may be scheduled as SMs free up (it prefetches
  // W2 and waits for this grid before reading A).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = blockIdx.x * kRnnRows, c0 = blockIdx.y * kRnnCols;
  constexpr int kLoads = kRnnMaxR * 8 / kRnnThreads;  // 16-byte Wh vectors (and h values) per thread
  // Every global load of the prologue is issued before the first use, so the
  // CTA waits for one round of memory latency rather than one per load.  The
  // inputs (Wh, Q) are read first; when this kernel is launched as the
  // programmatic dependent of the previous draft step, the rest (the previous
  // state and partials, which that step's grid follows) only after its wait.
  uint4 wv[kLoads];
  float hv[kLoads];
#pragma unroll
  for (int u = 0; u < kLoads; ++u) {
    const int v = threadIdx.x + u * kRnnThreads;  // Wh[:, c0 : c0 + 64] as r rows of 8 vectors
    if (v < r * 8) wv[u] = __ldg((const uint4*)(Wh + (size_t)(v >> 3) * r + c0) + (v & 7));
  }
  const int row = row0 + warp;
  const int j = c0 + 2 * lane;
  float2 q = make_float2(0.0f, 0.0f);
  if (row < R) q = *(const float2*)(Q + ((size_t)row * gamma + (k - 1)) * r + j);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // What the previous draft step and state update wrote (state, partials,
  // scores) is read through L2 (ld.global.cg), never the non-coherent path:
  // this grid may have started while the previous step still ran.
#pragma unroll
  for (int u = 0; u < kLoads; ++u) {
    const int v = threadIdx.x + u * kRnnThreads;
    const int i = v / r, hrow = row0 + i;  // previous states of the CTA's rows
    hv[u] = (v < kRnnRows * r && k > 1 && hrow < R) ? __ldcg(h_prev + (size_t)hrow * r + (v - i * r)) : 0.0f;
  }
  // The previous step's partials of this warp's row (at most 2 per lane issued at once).
  float4 ps[2];
  int pi[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int t = lane + 32 * u;
    const bool use = k > 1 && row < R && t < n_parts;
    ps[u] = use ? __ldcg(prev_stats + (size_t)row * n_parts + t) : make_float4(-INFINITY, 0.0f, -INFINITY, 0.0f);
    pi[u] = use ? __ldcg(prev_index + (size_t)row * n_parts + t) : 0x7fffffff;
  }
#pragma unroll
  for (int u = 0; u < kLoads; ++u) {
    const int v = threadIdx.x + u * kRnnThreads;
    if (v < r * 8) *(uint4*)&s_w[v >> 3][(v & 7) * 4] = wv[u];
    if (v < kRnnRows * r) s_h[v / r][v % r] = hv[u];
  }
  {
    int xp = 0;
    if (row < R) {
      if (k == 1) {
        xp = x0[row];
      } else {
        // Merge step k-1's partials (lse and the drawn group), then draw x_{k-1}
        // inside that group from the stored scores (stage 2 of the two-level draw).
        float m = -INFINITY, S = 0.0f, key = -INFINITY, unused = 0.0f;
        int gj = 0x7fffffff;
        for (int t = lane; t < n_parts; t += 32) {
          const int u = (t - lane) >> 5;
          const float4 qs = u < 2 ? ps[u] : __ldcg(prev_stats + (size_t)row * n_parts + t);
          const int qi = u < 2 ? pi[u] : __ldcg(prev_index + (size_t)row * n_parts + t);
          lse_merge(m, S, qs.x, qs.y);
          if (better(qs.z, qi, key, gj)) {
            key = qs.z;
            gj = qi;
          }
        }
        warp_lse(m, S);
        warp_argmax3(key, gj, unused);
        if (gj < 0 || gj >= (V + kGroup - 1) / kGroup) gj = 0;  // NaN scores: flagged below
        const int v = gj * kGroup + lane;
        const bool valid = v < V;
        const float s_v = valid ? __ldcg(scores + ((size_t)row * gamma + (k - 2)) * V + v) : 0.0f;
        float k2, sv;
        int idx;
        group_draw_warp(s_v, valid, v, seed, (uint32_t)row, (uint32_t)(k - 1), DSPARK_PURPOSE_DRAFT, k2,
                        idx, sv);
        if (idx < 0 || idx >= V) {  // nothing drawn: every score of the row was NaN
          if (lane == 0) flag_status(status, DSPARK_DEV_BAD_INPUT);
          idx = 0;
        }
        xp = idx;
        if (lane == 0 && blockIdx.y == 0) {  // one CTA per row stores step k-1
          const float l = m + logf(S);
          const size_t o = (size_t)row * gamma + (k - 2);
          x[o] = idx;
          logp[o] = sv - l;
          lse[o] = l;
        }
      }
      if (xp < 0 || xp >= V) {
        if (lane == 0) flag_status(status, DSPARK_DEV_BAD_INPUT);
        xp = xp < 0 ? 0 : V - 1;
      }
    }
    if (lane == 0) s_x[warp] = xp;
  }
  __syncthreads();
  if (row >= R) return;
  const float2 w1 = __bfloat1622float2(*(const __nv_bfloat162*)(W1 + (size_t)s_x[warp] * r + j));
  float z0 = w1.x + q.x, z1 = w1.y + q.y;
  const float* hr = s_h[warp];
#pragma unroll 8
  for (int a = 0; a < r; ++a) {
    const float hv = hr[a];
    const float2 wv = __bfloat1622float2(s_w[a][lane]);
    z0 = fmaf(hv, wv.x, z0);
    z1 = fmaf(hv, wv.y, z1);
  }
  const float h0 = tanhf(z0), h1 = tanhf(z1);
  *(float2*)(h_next + (size_t)row * r + j) = make_float2(h0, h1);
  *(__nv_bfloat162*)(A + (size_t)row * r + j) = __floats2bfloat162_rn(h0, h1);
}

}  // namespace

cudaError_t launch_rnn_state(int k, const int32_t* x0, const void* W1, const void* Wh,
                             const float* Q, const DraftPartials& prev, int R, int gamma, int V,
                             int r, const float* h_prev, float* h_next, void* A,
                             const float* scores, uint64_t seed, int32_t* x, float* logp,
                             float* lse, int* status, cudaStream_t s) {
  if (r > kRnnMaxR || r % kRnnCols != 0) return cudaErrorInvalidValue;
  const dim3 grid((R + kRnnRows - 1) / kRnnRows, r / kRnnCols);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kRnnThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = k >= 2 ? 1 : 0;  // step 1 follows the W2 transpose: an ordinary launch
  return cudaLaunchKernelEx(&cfg, rnn_state_kernel, k, x0, (const __nv_bfloat16*)W1,
                            (const __nv_bfloat16*)Wh, Q, (const float4*)prev.stats,
                            (const int*)prev.index, prev.n_parts, R, gamma, V, r, h_prev, h_next,
                            (__nv_bfloat16*)A, scores, seed, x, logp, lse, status);
}

}  // namespace dspark
