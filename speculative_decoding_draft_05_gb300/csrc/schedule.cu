// schedule.cu -- hardware-aware prefix scheduler (Algorithm 1).
//
// "DSpark: Confidence-Scheduled Speculative Decoding with Semi-Autoregressive
// Generation 요약 설명", §3.2.2: prefix survival a_{r,j} = prod_{i<=j} c_{r,i};
// verify batch B = sum_r (1 + l_r); expected accepted tokens
// tau = sum_r (1 + sum_{j<=l_r} a_{r,j}); throughput Theta = tau * SPS(B) with
// SPS the engine's measured step-rate table.  Algorithm 1 extends prefixes in
// survival order and stops at the first candidate that does not improve Theta.
//
// Every step is exact or IEEE-rounded in a fixed order, so the result is
// bit-reproducible on any device.  Each kernel runs in CTAs of 128 threads with
// at most 56 registers and no dynamic shared memory: one fits on an SM beside
// a tensor-core draft step's CTA, so a schedule issued on a side stream next
// to the draft takes no SM from it (CTAs of 1024 threads with the keys staged
// in shared memory had waited for SMs between draft steps and delayed them).
//   schedule_keys  one thread per request: the sequential products and the
//                  sort key of each of its gamma candidates, to global memory.
//   schedule_rank  one thread per candidate.  Survival is non-increasing along
//                  a request, so every request's gamma keys are already sorted;
//                  a candidate's place in the global order is the sum over
//                  requests of how many of their keys are smaller (a binary
//                  search of <= 64 keys each, the lists streamed through a
//                  3 KB shared-memory window).  Keys are unique, so these ranks
//                  are a permutation: each candidate is written to its slot of
//                  the sorted array.
//   schedule_scan  (one CTA) exact int64 prefix sum of the fixed-point
//                  survivals in sorted order, the Theta test of every prefix
//                  (an exact integer comparison of the products tau * SPS, no
//                  floating point), a block-wide minimum for the first
//                  non-improvement, and the per-request counts l_r.
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

constexpr int kSchedThreads = 128;
constexpr int kMaxCandidates = 16384;
constexpr int kChunkKeys = 384;  // schedule_rank's shared-memory window: 3 KB of keys
// (128 threads, at least 9 CTAs' worth of registers per SM: <= 56 registers)
#define SCHED_BOUNDS __launch_bounds__(kSchedThreads, 9)

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

__global__ void SCHED_BOUNDS
schedule_keys_kernel(const float* __restrict__ conf, int R, int gamma,
                     unsigned long long* __restrict__ keys, int* __restrict__ status) {
  // The rank kernel may be launched now; it waits for this grid before reading.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int r = blockIdx.x * kSchedThreads + threadIdx.x;
  if (r >= R) return;
  float a = 1.0f;
  for (int j = 0; j < gamma; ++j) {
    float c = conf[(size_t)r * gamma + j];
    if (!(c >= 0.0f) || c > 1.0f) {
      flag_status(status, DSPARK_DEV_BAD_INPUT);
      c = (c > 1.0f) ? 1.0f : 0.0f;  // NaN and negatives -> 0
    }
    a = (j == 0) ? c : __fmul_rn(a, c);
    const float av = (a == 0.0f) ? 0.0f : a;  // canonical +0
    keys[(size_t)r * gamma + j] = sort_key(av, j, r);
  }
}

__global__ void SCHED_BOUNDS
schedule_rank_kernel(const unsigned long long* __restrict__ keys, int R, int gamma,
                     unsigned long long* __restrict__ sorted) {
  // The kernel after this one (scan, capacity or top-K) may be launched now; it
  // waits for this grid's completion before reading anything.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // The keys come from the kernel before (this grid's programmatic primary):
  // read after its completion, through L2 (ld.global.cg), never the
  // non-coherent path, since this grid may start while that kernel runs.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ unsigned long long chunk[kChunkKeys];
  const int n = R * gamma;
  const int e = blockIdx.x * kSchedThreads + threadIdx.x;  // this thread's candidate
  const bool valid = e < n;
  const unsigned long long key = valid ? __ldcg(keys + e) : 0ull;
  // The requests' lists pass through shared memory a few at a time (each key
  // is read from L2 once per CTA); every thread counts the keys below its own
  // in each list, a branch-free lower bound with the same number of steps
  // (ceil(log2 gamma)) for all lanes, four lists interleaved.  All lanes probe
  // the same list at once (at gamma <= 16 its keys span the banks at most once).
  const int per = kChunkKeys / gamma;  // whole lists per chunk (gamma <= 64)
  int below = 0;
  for (int r0 = 0; r0 < R; r0 += per) {
    const int nl = min(per, R - r0);
    __syncthreads();
    for (int i = threadIdx.x; i < nl * gamma; i += kSchedThreads)
      chunk[i] = __ldcg(keys + (size_t)r0 * gamma + i);
    __syncthreads();
    if (!valid) continue;
    int l = 0;
    for (; l + 4 <= nl; l += 4) {
      int pos[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) pos[q] = (l + q) * gamma;
      for (int len = gamma; len > 1;) {  // the answer lies in [base, base + len]
        const int half = len >> 1;
#pragma unroll
        for (int q = 0; q < 4; ++q) pos[q] += chunk[pos[q] + half] < key ? half : 0;
        len -= half;
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) below += pos[q] - (l + q) * gamma + (chunk[pos[q]] < key ? 1 : 0);
    }
    for (; l < nl; ++l) {
      int pos = l * gamma;
      for (int len = gamma; len > 1;) {
        const int half = len >> 1;
        pos += chunk[pos + half] < key ? half : 0;
        len -= half;
      }
      below += pos - l * gamma + (chunk[pos] < key ? 1 : 0);
    }
  }
  if (valid) sorted[below] = key;
}

// Exclusive prefix over the block of one int64 per thread (kSchedThreads).
__device__ __forceinline__ long long block_exclusive_sum(long long v, long long* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  long long before = 0;
  for (int w = 0; w < warp; ++w) before += warp_tot[w];
  return before + incl - v;
}

// This thread's contiguous share [b0, b1) of the n sorted candidates, and the
// exact exclusive prefix of their fixed-point survivals.  The sorted keys are
// the rank kernel's output: read through L2 (see the scan kernel).
__device__ __forceinline__ long long share_prefix(const unsigned long long* __restrict__ sorted,
                                                  int n, int& b0, int& b1, long long* warp_tot) {
  const int per = (n + kSchedThreads - 1) / kSchedThreads;
  b0 = min(n, (int)threadIdx.x * per);
  b1 = min(n, b0 + per);
  long long local = 0;
#pragma unroll 8
  for (int i = b0; i < b1; ++i) local += fixed_survival(__ldcg(sorted + i));
  return block_exclusive_sum(local, warp_tot);
}

__global__ void SCHED_BOUNDS
schedule_scan_kernel(const unsigned long long* __restrict__ sorted, const double* __restrict__ sps,
                     int R, int gamma, int32_t* __restrict__ ell, double* __restrict__ diag,
                     int* __restrict__ status) {
  // Launched as the rank kernel's programmatic dependent: the sorted keys it
  // writes are read after this wait, through L2 (ld.global.cg), never the
  // non-coherent path, since this grid may start while the rank kernel runs.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ long long warp_tot[kSchedThreads / 32];
  __shared__ int stop_at;
  const int tid = threadIdx.x, lane = tid & 31;
  const int n = R * gamma;
  for (int r = tid; r < R; r += kSchedThreads) ell[r] = 0;
  if (tid == 0) stop_at = n + 1;
  int b0, b1;
  const long long run0 = share_prefix(sorted, n, b0, b1, warp_tot);

  // Theta test of every candidate (0-based index i, 1-based number i + 1):
  // before it B = R + i and tau = R + P_i; after it B = R + i + 1.
  const long long tau0 = (long long)R << 48;
  long long run = run0;
  int first_fail = n + 1;  // this thread's first non-improving candidate (1-based)
  unsigned long long rate_before = b0 < b1 ? pack_rate(sps[R + b0]) : 0ull;
#pragma unroll 4
  for (int i = b0; i < b1; ++i) {
    const long long tau_prev = tau0 + run;
    run += fixed_survival(__ldcg(sorted + i));
    const unsigned long long rate_after = pack_rate(sps[R + i + 1]);
    if (!greater_packed(tau0 + run, rate_after, tau_prev, rate_before, status))
      first_fail = min(first_fail, i + 1);
    rate_before = rate_after;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) first_fail = min(first_fail, __shfl_xor_sync(0xffffffffu, first_fail, o));
  if (lane == 0 && first_fail <= n) atomicMin(&stop_at, first_fail);  // one per warp
  __syncthreads();
  const int taken = stop_at - 1;  // candidates 0..taken-1 were taken
  for (int i = b0; i < min(b1, taken); ++i) atomicAdd(&ell[(int)(__ldcg(sorted + i) & 0xffffu)], 1);
  if (diag) {
    // tau after the taken candidates: the owner of index taken-1 finishes its share's sum.
    const bool owner = (taken == 0) ? (tid == 0) : (b0 <= taken - 1 && taken - 1 < b1);
    if (owner) {
      long long tau = tau0 + (taken == 0 ? 0ll : run0);
      for (int i = b0; i < taken; ++i) tau += fixed_survival(__ldcg(sorted + i));
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

__global__ void SCHED_BOUNDS
schedule_capacity_kernel(const unsigned long long* __restrict__ sorted,
                         const double* __restrict__ sps, int R, int gamma,
                         int32_t* __restrict__ K_out, double* __restrict__ diag,
                         int* __restrict__ status) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // launched as the rank kernel's dependent
  __shared__ long long warp_tot[kSchedThreads / 32];
  __shared__ long long red_t[kSchedThreads / 32];
  __shared__ int red_k[kSchedThreads / 32];
  __shared__ unsigned long long red_s[kSchedThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = R * gamma;
  int b0, b1;
  long long run = share_prefix(sorted, n, b0, b1, warp_tot);
  const long long tau0 = (long long)R << 48;
  // this thread's best prefix; thread 0 also holds the empty one (k = 0)
  long long bt = tau0;
  int bk = tid == 0 ? 0 : -1;
  unsigned long long bs = pack_rate(sps[R]);  // thread 0's empty prefix
#pragma unroll 4
  for (int i = b0; i < b1; ++i) {
    run += fixed_survival(__ldcg(sorted + i));
    better_theta(bt, bk, bs, tau0 + run, i + 1, pack_rate(sps[R + i + 1]), status);
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
  if (tid == 0) {
    for (int w = 1; w < kSchedThreads / 32; ++w) better_theta(bt, bk, bs, red_t[w], red_k[w], red_s[w], status);
    K_out[0] = bk;
    if (diag) {
      diag[0] = (double)(R + bk);
      diag[1] = __ll2double_rn(bt) * 0x1p-48;
      diag[2] = __dmul_rn(__ll2double_rn(bt) * 0x1p-48, sps[R + bk]);
      diag[3] = (double)bk;
    }
  }
}

__global__ void SCHED_BOUNDS
schedule_topk_kernel(const unsigned long long* __restrict__ sorted, const int32_t* __restrict__ K,
                     int R, int gamma, int32_t* __restrict__ ell, int* __restrict__ status) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // launched as the rank kernel's dependent
  const int n = R * gamma;
  for (int r = threadIdx.x; r < R; r += kSchedThreads) ell[r] = 0;
  __syncthreads();
  int k = __ldcg(K);
  if (k < 0) {
    if (threadIdx.x == 0) flag_status(status, DSPARK_DEV_BAD_INPUT);
    k = 0;
  }
  if (k > n) k = n;
  for (int i = threadIdx.x; i < k; i += kSchedThreads)
    atomicAdd(&ell[(int)(__ldcg(sorted + i) & 0xffffu)], 1);
}

// Launch as a programmatic dependent of the kernel before it on the stream,
// so that its launch overlaps that kernel's end.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), int grid, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kSchedThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}

// The scheduler's kernels ask for the largest shared-memory carveout, the one
// the draft steps run with, so that an SM can hold a CTA of each at once (an
// SM changes its carveout only when idle).  Once per process.
cudaError_t set_carveouts() {
  static const cudaError_t err = [] {
    const int kMax = (int)cudaSharedmemCarveoutMaxShared;
    cudaError_t e = cudaFuncSetAttribute(schedule_keys_kernel,
                                         cudaFuncAttributePreferredSharedMemoryCarveout, kMax);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(schedule_rank_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, kMax);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(schedule_scan_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, kMax);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(schedule_capacity_kernel,
                               cudaFuncAttributePreferredSharedMemoryCarveout, kMax);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(schedule_topk_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, kMax);
    return e;
  }();
  return err;
}

}  // namespace

// The sorted keys, then the keys in candidate order.
size_t schedule_sorted_bytes(int R, int gamma) {
  return 2 * (size_t)R * gamma * sizeof(unsigned long long);
}

cudaError_t launch_schedule_rank(const float* conf, int R, int gamma, unsigned long long* sorted,
                                 int* status, cudaStream_t s) {
  const int n = R * gamma;
  if (n > kMaxCandidates) return cudaErrorInvalidValue;
  unsigned long long* keys = sorted + n;
  cudaError_t e = set_carveouts();
  if (e != cudaSuccess) return e;
  schedule_keys_kernel<<<(R + kSchedThreads - 1) / kSchedThreads, kSchedThreads, 0, s>>>(
      conf, R, gamma, keys, status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int grid = (n + kSchedThreads - 1) / kSchedThreads;
  return launch_dependent(schedule_rank_kernel, grid, s, (const unsigned long long*)keys, R, gamma,
                          sorted);
}

cudaError_t launch_schedule_scan(const unsigned long long* sorted, const double* sps, int R,
                                 int gamma, int32_t* ell, double* diag, int* status,
                                 cudaStream_t s) {
  if (R * gamma > kMaxCandidates) return cudaErrorInvalidValue;
  return launch_dependent(schedule_scan_kernel, 1, s, sorted, sps, R, gamma, ell, diag, status);
}

cudaError_t launch_schedule_capacity(const unsigned long long* sorted, const double* sps, int R,
                                     int gamma, int32_t* K, double* diag, int* status,
                                     cudaStream_t s) {
  if (R * gamma > kMaxCandidates) return cudaErrorInvalidValue;
  return launch_dependent(schedule_capacity_kernel, 1, s, sorted, sps, R, gamma, K, diag, status);
}

cudaError_t launch_schedule_topk(const unsigned long long* sorted, const int32_t* K, int R,
                                 int gamma, int32_t* ell, int* status, cudaStream_t s) {
  if (R * gamma > kMaxCandidates) return cudaErrorInvalidValue;
  return launch_dependent(schedule_topk_kernel, 1, s, sorted, K, R, gamma, ell, status);
}

}  // namespace dspark
