// draft.cu -- semi-autoregressive draft step: anchor gather, CUDA-core
// contraction + fused epilogue (fp32 inputs, and bf16 where the tensor-core
// path does not apply), and the per-row combine that samples x_k.
//
// Method: "DSpark: Confidence-Scheduled Speculative Decoding with
// Semi-Autoregressive Generation 요약 설명" §3.1 (local normalisation, Markov
// head B = W1 W2 conditioned on the previous token, left-to-right sampling);
// "DSpark: Confidence-Scheduled Speculative Decoding with Semi-Autoregressive
// Generation" (notes), "DSpark 핵심 기술 1" (p_k = softmax(U_k + B_k)).
//
// One draft step k is two launches:
//   tile kernel  : B_k tile = A_k[rows] . W2[:, tile]  (A_k = W1[x_{k-1}])
//                  s = (U_k + B_k) / T -> scores; per (row, tile) partials
//                  (max, sum exp, and stage 1 of the two-level draw: the best
//                  group key L_j + G(DRAFT_GROUP, j) over the tile's four
//                  32-id groups, and that group's index)
//   combine      : per row, merge the tiles' partials -> lse_k and the drawn
//                  group; stage 2 draws x_k inside it from the stored scores
//                  (G(DRAFT, v)); logp_k; and gather A_{k+1} = W1[x_k].
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace dspark {

namespace {

template <typename T>
__global__ void gather_anchor_kernel(const T* __restrict__ W1, const int32_t* __restrict__ x0,
                                     int R, int V, int r, T* __restrict__ A,
                                     int* __restrict__ status) {
  const int row = blockIdx.x;
  if (row >= R) return;
  int t = x0[row];
  if (t < 0 || t >= V) {
    if (threadIdx.x == 0) flag_status(status, DSPARK_DEV_BAD_INPUT);
    t = t < 0 ? 0 : V - 1;
  }
  for (int i = threadIdx.x; i < r; i += blockDim.x) A[(size_t)row * r + i] = W1[(size_t)t * r + i];
}

constexpr int kSimtRows = 16;
constexpr int kSimtThreads = kDraftTileN;  // one thread per vocab column of the tile
constexpr int kMaxRank = 256;

template <typename T>
__global__ void __launch_bounds__(kSimtThreads)
draft_tile_simt_kernel(const T* __restrict__ U, const T* __restrict__ A, const T* __restrict__ W2,
                       int R, int gamma, int V, int r, int k, float invT, uint64_t seed,
                       float* __restrict__ scores, float4* __restrict__ pstats,
                       int* __restrict__ pindex, int n_tiles) {
  __shared__ float As[kSimtRows][kMaxRank];
  __shared__ float red_m[4][kSimtRows], red_s[4][kSimtRows], red_k[4][kSimtRows];
  __shared__ int red_i[4][kSimtRows];
  const int tile = blockIdx.x;
  const int row0 = blockIdx.y * kSimtRows;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int v = tile * kDraftTileN + tid;
  const bool valid = v < V;

  for (int i = tid; i < kSimtRows * r; i += kSimtThreads) {
    const int rr = i / r, c = i - rr * r;
    As[rr][c] = (row0 + rr < R) ? to_f32(A[(size_t)(row0 + rr) * r + c]) : 0.0f;
  }
  __syncthreads();

  float acc[kSimtRows];
#pragma unroll
  for (int rr = 0; rr < kSimtRows; ++rr) acc[rr] = 0.0f;
  if (valid) {
    for (int i = 0; i < r; ++i) {
      const float w = to_f32(W2[(size_t)i * V + v]);
#pragma unroll
      for (int rr = 0; rr < kSimtRows; ++rr) acc[rr] = fmaf(As[rr][i], w, acc[rr]);
    }
  }

#pragma unroll 1
  for (int rr = 0; rr < kSimtRows; ++rr) {
    const int row = row0 + rr;
    if (row >= R) break;  // uniform across the block
    float s = -INFINITY;
    if (valid) {
      const size_t o = ((size_t)row * gamma + (k - 1)) * V + v;
      s = (to_f32(U[o]) + acc[rr]) * invT;
      scores[o] = s;
    }
    // The warp's 32 columns are one group j of the two-level draw: its
    // log-mass L_j = m + log S and its stage-1 key L_j + G(DRAFT_GROUP, j).
    float m = valid ? s : -INFINITY, S = valid ? 1.0f : 0.0f;
    warp_lse(m, S);
    const int j = (tile * kDraftTileN + warp * 32) / kGroup;
    float key = -INFINITY;
    if (m != -INFINITY)
      key = __fadd_rn(__fadd_rn(m, logf(S)),
                      gumbel(rng_word(seed, (uint32_t)row, (uint32_t)k, DSPARK_PURPOSE_DRAFT_GROUP,
                                      (uint32_t)j)));
    if (lane == 0) {
      red_m[warp][rr] = m;
      red_s[warp][rr] = S;
      red_k[warp][rr] = key;
      red_i[warp][rr] = j;
    }
  }
  __syncthreads();
  if (tid < kSimtRows && row0 + tid < R) {
    const int rr = tid;
    float m = red_m[0][rr], S = red_s[0][rr], key = red_k[0][rr];
    int idx = red_i[0][rr];
    for (int w = 1; w < 4; ++w) {
      lse_merge(m, S, red_m[w][rr], red_s[w][rr]);
      if (better(red_k[w][rr], red_i[w][rr], key, idx)) {
        key = red_k[w][rr];
        idx = red_i[w][rr];
      }
    }
    const size_t po = (size_t)(row0 + rr) * n_tiles + tile;
    pstats[po] = make_float4(m, S, key, 0.0f);
    pindex[po] = idx;
  }
}

// One warp per row: merge the row's partials (lse_k and the drawn group),
// draw x_k inside that group from the stored scores (stage 2), gather W1[x_k].
template <typename T>
__global__ void draft_combine_kernel(const float4* __restrict__ pstats,
                                     const int* __restrict__ pindex, int n_tiles, int R, int gamma,
                                     int r, int k, const T* __restrict__ W1, T* __restrict__ A_next,
                                     const float* __restrict__ scores, uint64_t seed,
                                     int32_t* __restrict__ x, float* __restrict__ logp,
                                     float* __restrict__ lse, int V, int* __restrict__ status) {
  // Launched as a programmatic dependent of the draft step before it: wait for
  // that step, then read its partials and scores through L2 (ld.global.cg),
  // never the non-coherent path, since this grid may start while it runs.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= R) return;
  const float4* ps = pstats + (size_t)row * n_tiles;
  const int* pi = pindex + (size_t)row * n_tiles;
  float m = -INFINITY, S = 0.0f, key = -INFINITY, unused = 0.0f;
  int gj = 0x7fffffff;
  for (int t = lane; t < n_tiles; t += 32) {
    const float4 q = __ldcg(ps + t);
    lse_merge(m, S, q.x, q.y);
    const int qi = __ldcg(pi + t);
    if (better(q.z, qi, key, gj)) {
      key = q.z;
      gj = qi;
    }
  }
  warp_lse(m, S);
  warp_argmax3(key, gj, unused);
  const int n_groups = (V + kGroup - 1) / kGroup;
  if (gj < 0 || gj >= n_groups) {  // every score of the row was NaN
    if (lane == 0) flag_status(status, DSPARK_DEV_BAD_INPUT);
    gj = 0;
  }
  const int v = gj * kGroup + lane;
  const bool valid = v < V;
  const float sv = valid ? __ldcg(scores + ((size_t)row * gamma + (k - 1)) * V + v) : 0.0f;
  float k2, s_x;
  int idx;
  group_draw_warp(sv, valid, v, seed, (uint32_t)row, (uint32_t)k, DSPARK_PURPOSE_DRAFT, k2, idx, s_x);
  if (idx < 0 || idx >= V) {  // NaN scores inside the group
    if (lane == 0) flag_status(status, DSPARK_DEV_BAD_INPUT);
    idx = gj * kGroup;
  }
  const float l = m + logf(S);
  if (lane == 0) {
    const size_t o = (size_t)row * gamma + (k - 1);
    x[o] = idx;
    logp[o] = s_x - l;
    lse[o] = l;
  }
  if (A_next) {
    for (int i = lane; i < r; i += 32) A_next[(size_t)row * r + i] = W1[(size_t)idx * r + i];
  }
}

}  // namespace

cudaError_t launch_gather_anchor(const void* W1, const int32_t* x0, int R, int V, int r, int dtype,
                                 void* A, int* status, cudaStream_t s) {
  if (dtype == DSPARK_BF16)
    gather_anchor_kernel<__nv_bfloat16><<<R, 64, 0, s>>>((const __nv_bfloat16*)W1, x0, R, V, r,
                                                          (__nv_bfloat16*)A, status);
  else
    gather_anchor_kernel<float><<<R, 64, 0, s>>>((const float*)W1, x0, R, V, r, (float*)A, status);
  return cudaGetLastError();
}

cudaError_t launch_draft_tile_simt(const void* U, const void* A, const void* W2, int dtype, int R,
                                   int gamma, int V, int r, int k, float invT, uint64_t seed,
                                   float* scores, DraftPartials p, cudaStream_t s) {
  dim3 grid(p.n_parts, (R + kSimtRows - 1) / kSimtRows);
  if (dtype == DSPARK_BF16)
    draft_tile_simt_kernel<__nv_bfloat16><<<grid, kSimtThreads, 0, s>>>(
        (const __nv_bfloat16*)U, (const __nv_bfloat16*)A, (const __nv_bfloat16*)W2, R, gamma, V, r,
        k, invT, seed, scores, p.stats, p.index, p.n_parts);
  else
    draft_tile_simt_kernel<float><<<grid, kSimtThreads, 0, s>>>(
        (const float*)U, (const float*)A, (const float*)W2, R, gamma, V, r, k, invT, seed, scores,
        p.stats, p.index, p.n_parts);
  return cudaGetLastError();
}

cudaError_t launch_draft_combine(DraftPartials p, int R, int gamma, int V, int r, int k,
                                 const void* W1, int dtype, void* A_next, const float* scores,
                                 uint64_t seed, int32_t* x, float* logp, float* lse, int* status,
                                 cudaStream_t s) {
  const int warps = 8;
  // A programmatic dependent of the draft step before it (the kernel waits for
  // that step at entry), so that its launch overlaps the step's end.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((R + warps - 1) / warps);
  cfg.blockDim = dim3(warps * 32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (dtype == DSPARK_BF16)
    return cudaLaunchKernelEx(&cfg, draft_combine_kernel<__nv_bfloat16>, (const float4*)p.stats,
                              (const int*)p.index, p.n_parts, R, gamma, r, k,
                              (const __nv_bfloat16*)W1, (__nv_bfloat16*)A_next, (const float*)scores,
                              seed, x, logp, lse, V, status);
  return cudaLaunchKernelEx(&cfg, draft_combine_kernel<float>, (const float4*)p.stats,
                            (const int*)p.index, p.n_parts, R, gamma, r, k, (const float*)W1,
                            (float*)A_next, (const float*)scores, seed, x, logp, lse, V, status);
}

}  // namespace dspark
