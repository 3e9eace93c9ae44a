// rnn.cu -- the state update of the RNN draft head.
//
// "DSpark: Confidence-Scheduled Speculative Decoding with Semi-Autoregressive
// Generation 요약 설명", §3.1: the alternative sequential head keeps a state
// across the block and also takes the backbone's hidden state.  Read as an
// Elman recurrence in the Markov head's rank-r space,
//     h_0 = 0,  h_k = tanh(W1[x_{k-1}] + h_{k-1} Wh + Q_k),  B_k = bf16(h_k) W2,
// the bias contraction B_k is the Markov head's (draft_tc.cu, A taken from a
// buffer instead of gathered W1 rows).  This kernel runs before each draft
// step: it merges the previous step's per-CTA partials into x_{k-1} (and
// stores x, logp, lse of step k-1), then updates the state in fp32 and writes
// its bf16 rounding (nearest, ties to even) as the step's A rows.
//
// One CTA of kRnnThreads >= r threads takes kRnnRows rows: warp i merges row
// i, then thread j forms element j of every row's new state, streaming
// column j of Wh (coalesced across threads) once for all kRnnRows rows.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace dspark {

namespace {

constexpr int kRnnThreads = 256;  // >= r (r <= 256)
constexpr int kRnnRows = 4;

__global__ void __launch_bounds__(kRnnThreads)
rnn_state_kernel(int k, const int32_t* __restrict__ x0, const __nv_bfloat16* __restrict__ W1,
                 const __nv_bfloat16* __restrict__ Wh, const float* __restrict__ Q,
                 const float4* __restrict__ prev_stats, const int* __restrict__ prev_index,
                 int n_parts, int R, int gamma, int V, int r, float* __restrict__ h,
                 __nv_bfloat16* __restrict__ A, int32_t* __restrict__ x, float* __restrict__ logp,
                 float* __restrict__ lse, int* __restrict__ status) {
  __shared__ int s_x[kRnnRows];
  __shared__ float s_h[kRnnRows][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = blockIdx.x * kRnnRows;
  if (warp < kRnnRows) {
    const int row = row0 + warp;
    int xp = 0;
    if (row < R) {
      if (k == 1) {
        xp = x0[row];
      } else {
        float m = -INFINITY, S = 0.0f, key = -INFINITY, sv = 0.0f;
        int idx = 0x7fffffff;
        for (int t = lane; t < n_parts; t += 32) {
          const float4 q = prev_stats[(size_t)row * n_parts + t];
          const int qi = prev_index[(size_t)row * n_parts + t];
          lse_merge(m, S, q.x, q.y);
          if (better(q.z, qi, key, idx)) {
            key = q.z;
            idx = qi;
            sv = q.w;
          }
        }
        warp_lse(m, S);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float k2 = __shfl_xor_sync(0xffffffffu, key, o);
          const int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
          const float v2 = __shfl_xor_sync(0xffffffffu, sv, o);
          if (better(k2, i2, key, idx)) {
            key = k2;
            idx = i2;
            sv = v2;
          }
        }
        xp = idx;
        if (lane == 0) {
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
  for (int i = 0; i < kRnnRows; ++i) {
    const int row = row0 + i;
    if (threadIdx.x < r) s_h[i][threadIdx.x] = (row < R && k > 1) ? h[(size_t)row * r + threadIdx.x] : 0.0f;
  }
  __syncthreads();
  const int j = threadIdx.x;
  if (j >= r) return;
  float z[kRnnRows];
#pragma unroll
  for (int i = 0; i < kRnnRows; ++i) {
    const int row = row0 + i;
    z[i] = row < R ? __bfloat162float(W1[(size_t)s_x[i] * r + j]) +
                         Q[((size_t)row * gamma + (k - 1)) * r + j]
                   : 0.0f;
  }
  for (int a = 0; a < r; ++a) {
    const float w = __bfloat162float(Wh[(size_t)a * r + j]);
#pragma unroll
    for (int i = 0; i < kRnnRows; ++i) z[i] = fmaf(s_h[i][a], w, z[i]);
  }
#pragma unroll
  for (int i = 0; i < kRnnRows; ++i) {
    const int row = row0 + i;
    if (row < R) {
      const float hn = tanhf(z[i]);
      h[(size_t)row * r + j] = hn;
      A[(size_t)row * r + j] = __float2bfloat16_rn(hn);
    }
  }
}

}  // namespace

cudaError_t launch_rnn_state(int k, const int32_t* x0, const void* W1, const void* Wh,
                             const float* Q, const DraftPartials& prev, int R, int gamma, int V,
                             int r, float* h, void* A, int32_t* x, float* logp, float* lse,
                             int* status, cudaStream_t s) {
  if (r > kRnnThreads) return cudaErrorInvalidValue;
  rnn_state_kernel<<<(R + kRnnRows - 1) / kRnnRows, kRnnThreads, 0, s>>>(
      k, x0, (const __nv_bfloat16*)W1, (const __nv_bfloat16*)Wh, Q, prev.stats, prev.index,
      prev.n_parts, R, gamma, V, r, h, (__nv_bfloat16*)A, x, logp, lse, status);
  return cudaGetLastError();
}

}  // namespace dspark
