// schedule.cu -- hardware-aware prefix scheduler (Algorithm 1).
//
// "DSpark: Confidence-Scheduled Speculative Decoding with Semi-Autoregressive
// Generation 요약 설명", §3.2.2: prefix survival a_{r,j} = prod_{i<=j} c_{r,i};
// verify batch B = sum_r (1 + l_r); expected accepted tokens
// tau = sum_r (1 + sum_{j<=l_r} a_{r,j}); throughput Theta = tau * SPS(B) with
// SPS the engine's measured step-rate table.  Algorithm 1 extends prefixes in
// survival order and stops at the first candidate that does not improve Theta.
//
// One CTA does the whole problem (R * gamma <= 16384 candidates): survival
// products, a bitonic sort of 64-bit keys held 16 per thread in registers
// (strides below 16 inside a thread, up to 256 by warp shuffles, larger ones
// through shared memory), an exact int64 prefix sum of the fixed-point
// survivals, the Theta test of every prefix in parallel and a block-wide
// minimum to find the first non-improvement.
// Every step is exact or IEEE-rounded in a fixed order, so the result is
// bit-reproducible on any device.
#include "common.cuh"
#include "kernels.h"

namespace dspark {

namespace {

constexpr int kSchedThreads = 1024;
constexpr int kMaxCandidates = 16384;

__device__ __forceinline__ unsigned long long sort_key(float a, int j, int r) {
  // a >= 0: its bit pattern orders like the value.  Complementing it sorts by a
  // descending; the low word sorts ties by j, then r, ascending.
  return ((unsigned long long)(~__float_as_uint(a)) << 32) |
         ((unsigned long long)(unsigned)j << 16) | (unsigned long long)(unsigned)r;
}

__device__ __forceinline__ float key_survival(unsigned long long key) {
  return __uint_as_float(~(unsigned)(key >> 32));
}

constexpr int kPerThread = 16;  // keys held in registers by each sorting thread

__device__ __forceinline__ unsigned long long shfl_xor_u64(unsigned long long v, int d) {
  const unsigned lo = __shfl_xor_sync(0xffffffffu, (unsigned)v, d);
  const unsigned hi = __shfl_xor_sync(0xffffffffu, (unsigned)(v >> 32), d);
  return ((unsigned long long)hi << 32) | lo;
}

__device__ __forceinline__ long long fixed_survival(unsigned long long key) {
  return __float2ll_rn(__fmul_rn(key_survival(key), 281474976710656.0f));  // a * 2^48
}

template <int STRIDE>
__device__ __forceinline__ void reg_stage(unsigned long long (&k)[kPerThread], int base, int size) {
#pragma unroll
  for (int e = 0; e < kPerThread; ++e) {
    if (e & STRIDE) continue;
    const int e2 = e | STRIDE;
    const bool up = ((base + e) & size) == 0;
    if ((k[e] > k[e2]) == up) {
      const unsigned long long t = k[e];
      k[e] = k[e2];
      k[e2] = t;
    }
  }
}

// n_sort = max(512, next power of two >= R * gamma); threads t < n_sort / 16 sort.
__global__ void __launch_bounds__(kSchedThreads)
schedule_kernel(const float* __restrict__ conf, const double* __restrict__ sps, int R, int gamma,
                int n_sort, int32_t* __restrict__ ell, double* __restrict__ diag,
                int* __restrict__ status) {
  extern __shared__ unsigned long long keys[];  // [n_sort], staging for cross-warp stages
  __shared__ long long warp_tot[kSchedThreads / 32];
  __shared__ int stop_at;
  const int tid = threadIdx.x;
  const int n = R * gamma;
  const int sorters = n_sort / kPerThread;

  for (int r = tid; r < R; r += kSchedThreads) {
    ell[r] = 0;
    float a = 1.0f;
    for (int j = 0; j < gamma; ++j) {
      float c = conf[(size_t)r * gamma + j];
      if (!(c >= 0.0f) || c > 1.0f) {
        flag_status(status, DSPARK_DEV_BAD_INPUT);
        c = (c > 1.0f) ? 1.0f : 0.0f;  // NaN and negatives -> 0
      }
      a = (j == 0) ? c : __fmul_rn(a, c);
      const float av = (a == 0.0f) ? 0.0f : a;  // canonical +0
      keys[j * R + r] = sort_key(av, j, r);
    }
  }
  for (int i = n + tid; i < n_sort; i += kSchedThreads) keys[i] = ~0ull;
  if (tid == 0) stop_at = n + 1;
  __syncthreads();

  // Bitonic sort, ascending.  Thread t holds elements [16 t, 16 t + 16).
  unsigned long long k[kPerThread];
  const bool sorter = tid < sorters;
  const int base = tid * kPerThread;
  if (sorter) {
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) k[e] = keys[base + e];
  }
  for (int size = 2; size <= n_sort; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride >= 32 * kPerThread) {
        // partner in another warp: exchange through shared memory
        __syncthreads();
        if (sorter) {
#pragma unroll
          for (int e = 0; e < kPerThread; ++e) keys[base + e] = k[e];
        }
        __syncthreads();
        if (sorter) {
#pragma unroll
          for (int e = 0; e < kPerThread; ++e) {
            const int i = base + e;
            const unsigned long long v = keys[i ^ stride];
            const bool up = (i & size) == 0, lower = (i & stride) == 0;
            k[e] = (lower == up) ? (k[e] < v ? k[e] : v) : (k[e] > v ? k[e] : v);
          }
        }
      } else if (stride >= kPerThread) {
        // partner in another lane of the same warp
        if (sorter) {
          const int d = stride / kPerThread;
#pragma unroll
          for (int e = 0; e < kPerThread; ++e) {
            const int i = base + e;
            const unsigned long long v = shfl_xor_u64(k[e], d);
            const bool up = (i & size) == 0, lower = (i & stride) == 0;
            k[e] = (lower == up) ? (k[e] < v ? k[e] : v) : (k[e] > v ? k[e] : v);
          }
        }
      } else if (sorter) {
        // partner in this thread's registers (compile-time register indices)
        switch (stride) {
          case 8: reg_stage<8>(k, base, size); break;
          case 4: reg_stage<4>(k, base, size); break;
          case 2: reg_stage<2>(k, base, size); break;
          default: reg_stage<1>(k, base, size); break;
        }
      }
    }
  }

  // Exclusive prefix of the fixed-point survivals over the threads' chunks.
  long long local = 0;
  if (sorter) {
#pragma unroll
    for (int e = 0; e < kPerThread; ++e)
      if (base + e < n) local += fixed_survival(k[e]);
  }
  const int lane = tid & 31, warp = tid >> 5;
  long long incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    long long t = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    warp_tot[lane] = t;
  }
  __syncthreads();
  const long long run0 = (incl - local) + (warp > 0 ? warp_tot[warp - 1] : 0ll);

  // Theta test of every candidate (0-based index i, 1-based number i + 1):
  // before it B = R + i and tau = R + P_i; after it B = R + i + 1.
  const long long tau0 = (long long)R << 48;
  if (sorter) {
    long long run = run0;
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) {
      const int i = base + e;
      if (i < n) {
        const long long tau_prev = tau0 + run;
        run += fixed_survival(k[e]);
        const double th_prev = __dmul_rn(__ll2double_rn(tau_prev) * 0x1p-48, sps[R + i]);
        const double th_i = __dmul_rn(__ll2double_rn(tau0 + run) * 0x1p-48, sps[R + i + 1]);
        if (!(th_i > th_prev)) atomicMin(&stop_at, i + 1);
      }
    }
  }
  __syncthreads();
  const int taken = stop_at - 1;  // candidates 0..taken-1 were taken
  if (sorter) {
#pragma unroll
    for (int e = 0; e < kPerThread; ++e)
      if (base + e < taken) atomicAdd(&ell[(int)(k[e] & 0xffffu)], 1);
  }
  if (diag) {
    // tau after the taken candidates: the owner of index taken-1 finishes its chunk's sum.
    const bool owner = (taken == 0) ? (tid == 0)
                                    : (sorter && base <= taken - 1 && taken - 1 < base + kPerThread);
    if (owner) {
      long long tau = tau0 + (taken == 0 ? 0ll : run0);
#pragma unroll
      for (int e = 0; e < kPerThread; ++e)
        if (taken > 0 && base + e < taken) tau += fixed_survival(k[e]);
      diag[0] = (double)(R + taken);
      diag[1] = __ll2double_rn(tau) * 0x1p-48;
      diag[2] = __dmul_rn(__ll2double_rn(tau) * 0x1p-48, sps[R + taken]);
      diag[3] = (double)taken;
    }
  }
}

}  // namespace

cudaError_t launch_schedule(const float* conf, const double* sps, int R, int gamma, int32_t* ell,
                            double* diag, int* status, cudaStream_t s) {
  const int n = R * gamma;
  if (n > kMaxCandidates) return cudaErrorInvalidValue;
  int n_sort = 32 * kPerThread;
  while (n_sort < n) n_sort <<= 1;
  const size_t smem = (size_t)n_sort * sizeof(unsigned long long);
  cudaError_t e = cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  schedule_kernel<<<1, kSchedThreads, smem, s>>>(conf, sps, R, gamma, n_sort, ell, diag, status);
  return cudaGetLastError();
}

}  // namespace dspark
