// schedule.cu -- hardware-aware prefix scheduler (Algorithm 1).
//
// "DSpark: Confidence-Scheduled Speculative Decoding with Semi-Autoregressive
// Generation 요약 설명", §3.2.2: prefix survival a_{r,j} = prod_{i<=j} c_{r,i};
// verify batch B = sum_r (1 + l_r); expected accepted tokens
// tau = sum_r (1 + sum_{j<=l_r} a_{r,j}); throughput Theta = tau * SPS(B) with
// SPS the engine's measured step-rate table.  Algorithm 1 extends prefixes in
// survival order and stops at the first candidate that does not improve Theta.
//
// Two launches, every step exact or IEEE-rounded in a fixed order, so the
// result is bit-reproducible on any device:
//   schedule_rank  (up to one CTA per SM) each CTA builds the sort key of every
//                  candidate in shared memory.  Survival is non-increasing along
//                  a request, so every request's gamma keys are already sorted;
//                  a candidate's place in the global order is the sum over
//                  requests of how many of their keys are smaller (a binary
//                  search of <= 64 keys each), split across the CTA's warps.
//                  Keys are unique, so these ranks are a permutation: each
//                  candidate is written to its slot of the sorted array.
//   schedule_scan  (one CTA) exact int64 prefix sum of the fixed-point
//                  survivals in sorted order, the Theta test of every prefix in
//                  parallel (an exact integer comparison of the products
//                  tau * SPS, no floating point), a block-wide minimum for the
//                  first non-improvement, and the per-request counts l_r.
//
// Zero-overhead scheduling (same summary, §5.2): the capacity K comes from
// confidences two steps old without the early stop -- schedule_capacity is
// schedule_scan's exact Theta of every prefix followed by a block-wide
// argmax (first maximum) -- and the selection takes the top K of the current
// order (schedule_topk, one CTA).
#include "common.cuh"
#include "kernels.h"

namespace dspark {

namespace {

constexpr int kSchedThreads = 1024;
constexpr int kMaxCandidates = 16384;
constexpr int kPerThread = kMaxCandidates / kSchedThreads;  // 16

__device__ __forceinline__ unsigned long long sort_key(float a, int j, int r) {
  // a >= 0: its bit pattern orders like the value.  Complementing it sorts by a
  // descending; the low word sorts ties by j, then r, ascending.
  return ((unsigned long long)(~__float_as_uint(a)) << 32) |
         ((unsigned long long)(unsigned)j << 16) | (unsigned long long)(unsigned)r;
}

// a * 2^48 rounded to nearest, ties to even, for a in [0, 1], in integer
// arithmetic: a = m 2^(E - 150) with a 24-bit m (E = 0: m 2^-149).
__device__ __forceinline__ long long fixed_survival(unsigned long long key) {
  const unsigned bits = ~(unsigned)(key >> 32);
  const int E = (int)((bits >> 23) & 0xFF);
  const unsigned long long m = E ? ((bits & 0x7FFFFFu) | 0x800000u) : (bits & 0x7FFFFFu);
  const int sh = 102 - (E ? E : 1);  // a * 2^48 = m 2^-sh
  if (sh <= 0) return (long long)(m << (-sh));
  if (sh >= 25) return 0;  // below 1/2
  const unsigned long long q0 = m >> sh, rem = m & ((1ull << sh) - 1), half = 1ull << (sh - 1);
  return (long long)(q0 + ((rem > half || (rem == half && (q0 & 1))) ? 1 : 0));
}

// Exact test of t_a * s_a > t_b * s_b for fixed-point t > 0 and step rates
// s > 0 (finite doubles), in integer arithmetic only: s = m 2^e with an
// integer m < 2^53, so each product is a 117-bit integer times 2^e; compare the
// leading-bit positions, then the aligned 128-bit integers.  A step rate that
// is not positive and finite flags the status word and counts as no
// improvement.
struct U128 {
  unsigned long long hi, lo;
};

__device__ __forceinline__ bool split_rate(double s, unsigned long long& m, int& e) {
  const unsigned long long bits = (unsigned long long)__double_as_longlong(s);
  const int E = (int)((bits >> 52) & 0x7FF);
  const unsigned long long F = bits & ((1ull << 52) - 1);
  if ((bits >> 63) || E == 0x7FF || (E == 0 && F == 0)) return false;
  m = E ? (F | (1ull << 52)) : F;
  e = E ? E - 1075 : -1074;
  return true;
}

__device__ __forceinline__ int bitlen(const U128& x) {
  return x.hi ? 128 - __clzll((long long)x.hi) : 64 - __clzll((long long)x.lo);
}

__device__ __forceinline__ U128 shl(const U128& x, int d) {
  if (d == 0) return x;
  if (d >= 64) return U128{x.lo << (d - 64), 0ull};
  return U128{(x.hi << d) | (x.lo >> (64 - d)), x.lo << d};
}

__device__ __forceinline__ bool greater_split(long long ta, unsigned long long ma, int ea, long long tb,
                                              unsigned long long mb, int eb) {
  const U128 pa{__umul64hi((unsigned long long)ta, ma), (unsigned long long)ta * ma};
  const U128 pb{__umul64hi((unsigned long long)tb, mb), (unsigned long long)tb * mb};
  const int na = bitlen(pa), nb = bitlen(pb);
  if (na + ea != nb + eb) return na + ea > nb + eb;
  const U128 xa = na < nb ? shl(pa, nb - na) : pa;
  const U128 xb = nb < na ? shl(pb, na - nb) : pb;
  return xa.hi != xb.hi ? xa.hi > xb.hi : xa.lo > xb.lo;
}

// A step rate split once into one word: the 53-bit integer mantissa m in the
// low bits and e + 1075 (1 .. 2046) above them, s = m 2^e; 0 for a rate that
// is not positive and finite.
__device__ __forceinline__ unsigned long long pack_rate(double s) {
  unsigned long long m;
  int e;
  if (!split_rate(s, m, e)) return 0ull;
  return ((unsigned long long)(e + 1075) << 53) | m;
}

// The exact test on packed rates; a rate that is not positive and finite flags
// the status word and counts as no improvement.
__device__ __forceinline__ bool greater_packed(long long ta, unsigned long long ra, long long tb,
                                               unsigned long long rb, int* status) {
  if (!ra || !rb) {
    flag_status(status, DSPARK_DEV_BAD_INPUT);
    return false;
  }
  const unsigned long long kM = (1ull << 53) - 1;
  return greater_split(ta, ra & kM, (int)(ra >> 53) - 1075, tb, rb & kM, (int)(rb >> 53) - 1075);
}

__global__ void __launch_bounds__(kSchedThreads)
schedule_rank_kernel(const float* __restrict__ conf, int R, int gamma,
                     unsigned long long* __restrict__ sorted, int* __restrict__ status) {
  // The kernel after this one (scan, capacity or top-K) may be launched now; it
  // waits for this grid's completion before reading anything.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ unsigned long long keys[];  // [R][gamma], ascending along each request
  const int tid = threadIdx.x;
  const int n = R * gamma;
  // The confidences first, coalesced, into shared memory behind the keys (one
  // memory round trip), then each request's sequential products from there.
  float* cst = reinterpret_cast<float*>(keys + n);
#pragma unroll 4
  for (int i = tid; i < n; i += kSchedThreads) cst[i] = conf[i];
  __syncthreads();
  for (int r = tid; r < R; r += kSchedThreads) {
    float a = 1.0f;
    for (int j = 0; j < gamma; ++j) {
      float c = cst[r * gamma + j];
      if (!(c >= 0.0f) || c > 1.0f) {
        if (blockIdx.x == 0) flag_status(status, DSPARK_DEV_BAD_INPUT);
        c = (c > 1.0f) ? 1.0f : 0.0f;  // NaN and negatives -> 0
      }
      a = (j == 0) ? c : __fmul_rn(a, c);
      const float av = (a == 0.0f) ? 0.0f : a;  // canonical +0
      keys[r * gamma + j] = sort_key(av, j, r);
    }
  }
  __syncthreads();
  // Blocks of 32 candidates, one per lane; warp w counts, for every lane's
  // candidate, the keys below it in the lists of requests r = w, w + 32, ...
  // (all lanes probe the same list at once: no bank conflicts).  Each count is
  // a branch-free lower bound with the same number of steps for every lane
  // (ceil(log2 gamma)), four lists interleaved so that their probes overlap.
  __shared__ int part[kSchedThreads / 32][33];
  const int lane = tid & 31, warp = tid >> 5;
  const int blocks = (n + 31) / 32;
  constexpr int kW = kSchedThreads / 32;
  for (int blk = blockIdx.x; blk < blocks; blk += gridDim.x) {
    const int e = blk * 32 + lane;
    const unsigned long long key = e < n ? keys[e] : ~0ull;
    int below = 0;
    for (int r0 = warp; r0 < R; r0 += 4 * kW) {
      int pos[4];  // list start + running base, per list
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int r = r0 + q * kW;
        pos[q] = (r < R ? r : r0) * gamma;
      }
      for (int len = gamma; len > 1;) {  // the answer lies in [base, base + len]
        const int half = len >> 1;
#pragma unroll
        for (int q = 0; q < 4; ++q) pos[q] += keys[pos[q] + half] < key ? half : 0;
        len -= half;
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int r = r0 + q * kW;
        if (r < R) below += pos[q] - r * gamma + (keys[pos[q]] < key ? 1 : 0);
      }
    }
    part[warp][lane] = below;
    __syncthreads();
    if (warp == 0) {
      int rank = 0;
#pragma unroll 8
      for (int w = 0; w < kSchedThreads / 32; ++w) rank += part[w][lane];
      if (e < n) sorted[rank] = key;
    }
    __syncthreads();
  }
}

// Shared-memory slot of element i: one pad slot after every 16 elements, so
// that thread t reading its 16 consecutive 8-byte elements 16t + e hits banks
// 2(t + e) mod 32 -- at most two lanes of a warp per bank pair.
__device__ __forceinline__ int skew(int i) { return i + (i >> 4); }
constexpr int kStageSlots = kMaxCandidates + kMaxCandidates / 16 + 2;  // 8-byte slots

// Exclusive prefix of the fixed-point survivals of this thread's kPerThread
// sorted keys (staged coalesced in shared memory, then read into registers).
__device__ __forceinline__ long long stage_and_prefix(const unsigned long long* __restrict__ sorted,
                                                      int n, unsigned long long* stage,
                                                      long long* warp_tot,
                                                      unsigned long long (&k)[kPerThread]) {
  const int tid = threadIdx.x, base = tid * kPerThread;
#pragma unroll
  for (int i = tid; i < kMaxCandidates; i += kSchedThreads)
    stage[skew(i)] = i < n ? __ldcg(sorted + i) : ~0ull;  // L2 (see the scan kernel)
  __syncthreads();
  long long local = 0;
#pragma unroll
  for (int e = 0; e < kPerThread; ++e) {
    k[e] = stage[skew(base + e)];
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
  return (incl - local) + (warp > 0 ? warp_tot[warp - 1] : 0ll);
}

// The step rates sps[R + i], i = 0 .. n, packed (pack_rate) into the same
// shared memory, skewed like the keys, once every thread holds its keys in
// registers.
__device__ __forceinline__ void stage_rates(const double* __restrict__ sps, int R, int n,
                                            unsigned long long* st) {
  __syncthreads();
  for (int i = threadIdx.x; i <= n; i += kSchedThreads) st[skew(i)] = pack_rate(sps[R + i]);
  __syncthreads();
}

__global__ void __launch_bounds__(kSchedThreads)
schedule_scan_kernel(const unsigned long long* __restrict__ sorted, const double* __restrict__ sps,
                     int R, int gamma, int32_t* __restrict__ ell, double* __restrict__ diag,
                     int* __restrict__ status) {
  // Launched as the rank kernel's programmatic dependent: the sorted keys it
  // writes are read after this wait, through L2 (ld.global.cg), never the
  // non-coherent path, since this grid may start while the rank kernel runs.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ long long warp_tot[kSchedThreads / 32];
  __shared__ int stop_at;
  const int tid = threadIdx.x;
  const int n = R * gamma;
  const int base = tid * kPerThread;
  const int lane = tid & 31;
  for (int r = tid; r < R; r += kSchedThreads) ell[r] = 0;
  if (tid == 0) stop_at = n + 1;

  // Coalesced load of the sorted keys into shared memory, then 16 contiguous
  // keys per thread and their exclusive prefix; then the step rates.
  extern __shared__ unsigned long long stage[];  // [kStageSlots]
  unsigned long long k[kPerThread];
  const long long run0 = stage_and_prefix(sorted, n, stage, warp_tot, k);
  const unsigned long long* sv = stage;
  stage_rates(sps, R, n, stage);

  // Theta test of every candidate (0-based index i, 1-based number i + 1):
  // before it B = R + i and tau = R + P_i; after it B = R + i + 1.
  const long long tau0 = (long long)R << 48;
  long long run = run0;
  int first_fail = n + 1;  // this thread's first non-improving candidate (1-based)
#pragma unroll
  for (int e = 0; e < kPerThread; ++e) {
    const int i = base + e;
    if (i < n) {
      const long long tau_prev = tau0 + run;
      run += fixed_survival(k[e]);
      if (!greater_packed(tau0 + run, sv[skew(i + 1)], tau_prev, sv[skew(i)], status))
        first_fail = min(first_fail, i + 1);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) first_fail = min(first_fail, __shfl_xor_sync(0xffffffffu, first_fail, o));
  if (lane == 0 && first_fail <= n) atomicMin(&stop_at, first_fail);  // one per warp
  __syncthreads();
  const int taken = stop_at - 1;  // candidates 0..taken-1 were taken
#pragma unroll
  for (int e = 0; e < kPerThread; ++e)
    if (base + e < taken) atomicAdd(&ell[(int)(k[e] & 0xffffu)], 1);
  if (diag) {
    // tau after the taken candidates: the owner of index taken-1 finishes its chunk's sum.
    const bool owner =
        (taken == 0) ? (tid == 0) : (base <= taken - 1 && taken - 1 < base + kPerThread);
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

// The better of two (tau, number taken, packed step rate sps[R + k]) points by
// Theta = tau * sps[R + k], exactly; a tie goes to the smaller k (the first
// maximum).  k < 0: no point.
__device__ __forceinline__ void better_theta(long long& t, int& k, unsigned long long& sr, long long t2,
                                             int k2, unsigned long long sr2, int* status) {
  if (k2 < 0) return;
  if (k < 0 || greater_packed(t2, sr2, t, sr, status) ||
      (k2 < k && !greater_packed(t, sr, t2, sr2, status))) {
    t = t2;
    k = k2;
    sr = sr2;
  }
}

__global__ void __launch_bounds__(kSchedThreads)
schedule_capacity_kernel(const unsigned long long* __restrict__ sorted,
                         const double* __restrict__ sps, int R, int gamma,
                         int32_t* __restrict__ K_out, double* __restrict__ diag,
                         int* __restrict__ status) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // launched as the rank kernel's dependent
  __shared__ long long warp_tot[kSchedThreads / 32];
  __shared__ long long red_t[kSchedThreads / 32];
  __shared__ int red_k[kSchedThreads / 32];
  __shared__ unsigned long long red_s[kSchedThreads / 32];
  extern __shared__ unsigned long long stage[];  // [kMaxCandidates]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = R * gamma, base = tid * kPerThread;
  unsigned long long k[kPerThread];
  long long run = stage_and_prefix(sorted, n, stage, warp_tot, k);
  const long long tau0 = (long long)R << 48;
  const unsigned long long* sv = stage;
  stage_rates(sps, R, n, stage);
  // this thread's best prefix; thread 0 also holds the empty one (k = 0)
  long long bt = tau0;
  int bk = tid == 0 ? 0 : -1;
  unsigned long long bs = sv[skew(0)];  // sps[R], thread 0's empty prefix
#pragma unroll
  for (int e = 0; e < kPerThread; ++e) {
    const int i = base + e;
    if (i < n) {
      run += fixed_survival(k[e]);
      better_theta(bt, bk, bs, tau0 + run, i + 1, sv[skew(i + 1)], status);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const long long t2 = __shfl_xor_sync(0xffffffffu, bt, o);
    const int k2 = __shfl_xor_sync(0xffffffffu, bk, o);
    const unsigned long long s2 = __shfl_xor_sync(0xffffffffu, bs, o);
    better_theta(bt, bk, bs, t2, k2, s2, status);
  }
  if (lane == 0) {
    red_t[warp] = bt;
    red_k[warp] = bk;
    red_s[warp] = bs;
  }
  __syncthreads();
  if (warp == 0) {
    bt = red_t[lane];
    bk = red_k[lane];
    bs = red_s[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const long long t2 = __shfl_xor_sync(0xffffffffu, bt, o);
      const int k2 = __shfl_xor_sync(0xffffffffu, bk, o);
      const unsigned long long s2 = __shfl_xor_sync(0xffffffffu, bs, o);
      better_theta(bt, bk, bs, t2, k2, s2, status);
    }
    if (lane == 0) {
      K_out[0] = bk;
      if (diag) {
        diag[0] = (double)(R + bk);
        diag[1] = __ll2double_rn(bt) * 0x1p-48;
        diag[2] = __dmul_rn(__ll2double_rn(bt) * 0x1p-48, sps[R + bk]);
        diag[3] = (double)bk;
      }
    }
  }
}

__global__ void __launch_bounds__(kSchedThreads)
schedule_topk_kernel(const unsigned long long* __restrict__ sorted, const int32_t* __restrict__ K,
                     int R, int gamma, int32_t* __restrict__ ell, int* __restrict__ status) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // launched as the rank kernel's dependent
  const int n = R * gamma;
  for (int r = threadIdx.x; r < R; r += kSchedThreads) ell[r] = 0;
  __syncthreads();
  int k = *K;
  if (k < 0) {
    if (threadIdx.x == 0) flag_status(status, DSPARK_DEV_BAD_INPUT);
    k = 0;
  }
  if (k > n) k = n;
  for (int i = threadIdx.x; i < k; i += kSchedThreads)
    atomicAdd(&ell[(int)(__ldcg(sorted + i) & 0xffffu)], 1);
}

int sm_count_sched() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

// Launch as a programmatic dependent of the kernel before it on the stream
// (the rank kernel), so that its launch overlaps that kernel's end.
template <typename... Params, typename... Args>
cudaError_t launch_after_rank(void (*kernel)(Params...), size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(kSchedThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}

}  // namespace

size_t schedule_sorted_bytes(int R, int gamma) {
  return (size_t)R * gamma * sizeof(unsigned long long);
}

cudaError_t launch_schedule_rank(const float* conf, int R, int gamma, unsigned long long* sorted,
                                 int* status, cudaStream_t s) {
  const int n = R * gamma;
  if (n > kMaxCandidates) return cudaErrorInvalidValue;
  const size_t smem = (size_t)n * (sizeof(unsigned long long) + sizeof(float));  // keys + conf
  // Once per process (thread-safe initialisation of a function-local static).
  static const cudaError_t attr_err =
      cudaFuncSetAttribute(schedule_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)(kMaxCandidates * (sizeof(unsigned long long) + sizeof(float))));
  if (attr_err != cudaSuccess) return attr_err;
  int blocks = (n + 31) / 32;  // 32 candidates per CTA pass
  const int sms = sm_count_sched();
  if (blocks > sms) blocks = sms;
  if (blocks < 1) blocks = 1;
  schedule_rank_kernel<<<blocks, kSchedThreads, smem, s>>>(conf, R, gamma, sorted, status);
  return cudaGetLastError();
}

cudaError_t launch_schedule_scan(const unsigned long long* sorted, const double* sps, int R,
                                 int gamma, int32_t* ell, double* diag, int* status,
                                 cudaStream_t s) {
  if (R * gamma > kMaxCandidates) return cudaErrorInvalidValue;
  const size_t smem = kStageSlots * sizeof(unsigned long long);
  // Once per process (thread-safe initialisation of a function-local static).
  static const cudaError_t attr_err =
      cudaFuncSetAttribute(schedule_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (attr_err != cudaSuccess) return attr_err;
  return launch_after_rank(schedule_scan_kernel, smem, s, sorted, sps, R, gamma, ell, diag, status);
}

cudaError_t launch_schedule_capacity(const unsigned long long* sorted, const double* sps, int R,
                                     int gamma, int32_t* K, double* diag, int* status,
                                     cudaStream_t s) {
  if (R * gamma > kMaxCandidates) return cudaErrorInvalidValue;
  const size_t smem = kStageSlots * sizeof(unsigned long long);
  // Once per process (thread-safe initialisation of a function-local static).
  static const cudaError_t attr_err =
      cudaFuncSetAttribute(schedule_capacity_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (attr_err != cudaSuccess) return attr_err;
  return launch_after_rank(schedule_capacity_kernel, smem, s, sorted, sps, R, gamma, K, diag, status);
}

cudaError_t launch_schedule_topk(const unsigned long long* sorted, const int32_t* K, int R,
                                 int gamma, int32_t* ell, int* status, cudaStream_t s) {
  if (R * gamma > kMaxCandidates) return cudaErrorInvalidValue;
  return launch_after_rank(schedule_topk_kernel, 0, s, sorted, K, R, gamma, ell, status);
}

}  // namespace dspark
