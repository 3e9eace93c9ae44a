// verify.cu -- standard rejection sampling over the scheduled prefixes, the
// soft acceptance label, and the residual / bonus draw.
//
// "DSpark: Confidence-Scheduled Speculative Decoding with Semi-Autoregressive
// Generation 요약 설명": opening bullets (the target verifies the drafted block
// by rejection sampling, which preserves the target distribution), §3 (the
// accepted length counts the target's bonus token), §3.2.1 (soft label
// c*_k = 1 - 1/2 |p^d_k - p^t_k|_1).  "DSpark: ... Semi-Autoregressive
// Generation" (notes), "배경": accept the longest prefix.
//
// Launches:
//   verify_index  one CTA: the scheduled rows (r, j), j <= l_r, as a flat list.
//   verify_rows   a CTA per listed row at a time: LSE of Z_j / T,
//                 c*_j = sum_v min(p^d_j, p^t_j), and the accept test of x_j;
//                 Z_j is streamed twice (the second pass hits L2) and the
//                 score row once, with several 16-byte loads in flight.
//   verify_draw   (vocab chunks x requests) CTAs: first rejection n, then
//                 stage 1 of the two-level Gumbel-max draw from
//                 norm(max(0, p^t - p^d)) at row n + 1 or from p^t at the bonus
//                 row l + 1: the best 32-id group key per chunk;
//   verify_emit   one CTA per request: merges the chunks into the drawn group,
//                 draws the token inside it (stage 2), writes tokens, n_acc,
//                 n_emit and the NaN padding of c* / LSE^t beyond l.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"
#include "kernels.h"

namespace dspark {

namespace {

constexpr int kVerifyThreads = 512;

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr int kWarps = kVerifyThreads / 32;

// Eight consecutive elements starting at 8g (row is 16-byte aligned, V % 8 == 0).
__device__ __forceinline__ void load8(const float* __restrict__ row, int g, float (&o)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(row) + 2 * g);
  const float4 b = __ldg(reinterpret_cast<const float4*>(row) + 2 * g + 1);
  o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
  o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}

__device__ __forceinline__ void load8(const __nv_bfloat16* __restrict__ row, int g, float (&o)[8]) {
  const uint4 a = __ldg(reinterpret_cast<const uint4*>(row) + g);
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o[2 * i] = __uint_as_float(w[i] << 16);
    o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

template <int NWARPS = kWarps>
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum(v);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.0f;
  if (threadIdx.x < 32) {
    t = lane < NWARPS ? red[lane] : 0.0f;
    t = warp_sum(t);
    if (lane == 0) red[0] = t;
  }
  __syncthreads();
  t = red[0];
  __syncthreads();
  return t;
}

// Block-wide argmax over NWARPS warps (rk, ri hold NWARPS entries).
template <int NWARPS>
__device__ __forceinline__ void block_argmax(float& key, int& idx, float* rk, int* ri) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  warp_argmax(key, idx);
  if (lane == 0) {
    rk[warp] = key;
    ri[warp] = idx;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    float k2 = lane < NWARPS ? rk[lane] : -INFINITY;
    int i2 = lane < NWARPS ? ri[lane] : 0x7fffffff;
    warp_argmax(k2, i2);
    if (lane == 0) {
      rk[0] = k2;
      ri[0] = i2;
    }
  }
  __syncthreads();
  key = rk[0];
  idx = ri[0];
  __syncthreads();
}

__device__ __forceinline__ int clamp_ell(const int32_t* ell, int r, int gamma, int* status,
                                         bool report) {
  int L = ell[r];
  if (L < 0 || L > gamma) {
    if (report) flag_status(status, DSPARK_DEV_BAD_INPUT);
    L = L < 0 ? 0 : gamma;
  }
  return L;
}

// ---------------------------------------------------------------------------
// Scheduled rows as a flat list: entry i = r * gamma + (j - 1) for the rows
// (r, j), 1 <= j <= l_r, in request order; *count = their number.  One CTA,
// a block-wide exclusive scan of l over tiles of 1024 requests.
constexpr int kIndexThreads = 1024;

__global__ void __launch_bounds__(kIndexThreads)
verify_index_kernel(const int32_t* __restrict__ ell, int R, int gamma, uint32_t* __restrict__ list,
                    int* __restrict__ count, int* __restrict__ status, ZRows zr) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // the row kernel may launch
  __shared__ int warp_tot[kIndexThreads / 32];
  __shared__ int carry;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < R; base += kIndexThreads) {
    const int r = base + threadIdx.x;
    const int L = r < R ? clamp_ell(ell, r, gamma, status, true) : 0;
    if (zr.off && r < R) {  // a packed Z must hold rows 1 .. l_r + 1 of every request
      const long long a = zr.off[r], b = zr.off[r + 1];
      if (a < 0 || b - a < 1 + L || b > zr.n_rows) flag_status(status, DSPARK_DEV_BAD_INPUT);
    }
    int v = L;  // inclusive scan within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += t;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
      int w = warp_tot[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += t;
      }
      warp_tot[lane] = w;  // inclusive totals of warps 0..lane
    }
    __syncthreads();
    const int excl = carry + (warp ? warp_tot[warp - 1] : 0) + v - L;
    for (int j = 0; j < L; ++j) list[excl + j] = (uint32_t)(r * gamma + j);
    __syncthreads();
    if (threadIdx.x == kIndexThreads - 1) carry = excl + L;
    __syncthreads();
  }
  if (threadIdx.x == 0) *count = carry;
}

// Block-wide (max, sum exp(x - max)) of the per-thread pairs over NWARPS warps;
// every thread gets the result.
template <int NWARPS>
__device__ __forceinline__ void block_ms(float& m, float& s, float* rm, float* rs) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  warp_lse(m, s);
  if (lane == 0) {
    rm[warp] = m;
    rs[warp] = s;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    float mm = lane < NWARPS ? rm[lane] : -INFINITY;
    float ss = lane < NWARPS ? rs[lane] : 0.0f;
    warp_lse(mm, ss);
    if (lane == 0) {
      rm[0] = mm;
      rs[0] = ss;
    }
  }
  __syncthreads();
  m = rm[0];
  s = rs[0];
  __syncthreads();
}

// Eight consecutive elements of a row held raw (as loaded) until they are used,
// so that several 16-byte loads per thread are in flight at once.
template <typename T> struct Raw8;
template <> struct Raw8<__nv_bfloat16> {
  uint4 a;
  __device__ __forceinline__ void load(const __nv_bfloat16* row, int g) {
    a = __ldg(reinterpret_cast<const uint4*>(row) + g);
  }
  __device__ __forceinline__ void unpack(float (&o)[8]) const {
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = __uint_as_float(w[i] << 16);
      o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
};
template <> struct Raw8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* row, int g) {
    a = __ldg(reinterpret_cast<const float4*>(row) + 2 * g);
    b = __ldg(reinterpret_cast<const float4*>(row) + 2 * g + 1);
  }
  __device__ __forceinline__ void unpack(float (&o)[8]) const {
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
    o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
  }
};

// LSE^t_j, c*_j and the accept test of x_j for every listed row (r, j), one
// CTA per row at a time (rows i = CTA, CTA + grid, ...), two CTAs of 512
// threads per SM.  Pass 1 streams Z_j from HBM (64 bytes of Z in flight per
// thread) into an online (max, sum exp) of Z_j / T; pass 2 streams
// Z_j again -- from L2, which holds the rows in flight (2 per SM, 92 MB at
// V = 151,936) -- with the draft scores (streaming loads, read once) into
// sum_v min(p^d, p^t).  So HBM sees Z and the scores about once.  The row's list
// entry is loaded a row ahead and its scalars (x_j, the draft LSE, logp_j,
// then the logit Z_j[x_j]) one pass ahead of their use.
constexpr int kRowThreads = 512;
constexpr int kRowWarps = kRowThreads / 32;
// 16-byte loads of Z per thread in flight: pass 1 (Z alone) and pass 2 (Z and
// the scores).  Larger values spill at the 64 registers two CTAs per SM allow.
template <typename T> constexpr int row_unroll() { return sizeof(T) == 2 ? 4 : 2; }
template <typename T> constexpr int row_unroll2() { return sizeof(T) == 2 ? 2 : 1; }

template <typename T>
__global__ void __launch_bounds__(kRowThreads, 2)
verify_rows_stream_kernel(const int32_t* __restrict__ x, const float* __restrict__ logp,
                          const float* __restrict__ lse, const float* __restrict__ scores,
                          const T* __restrict__ Z, const uint32_t* __restrict__ list,
                          const int* __restrict__ count, int gamma, int V, float invT,
                          uint64_t seed, float* __restrict__ cstar, float* __restrict__ lse_t_ws,
                          int* __restrict__ acc_ws, int* __restrict__ status, ZRows zr) {
  // Launched as a programmatic dependent of the previous kernel: wait for it
  // before anything else, then let the next kernel's launch begin.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ float rm[kRowWarps], rs[kRowWarps];
  __shared__ float s_ld;
  constexpr int kRowUnroll = row_unroll<T>();  // 64 bytes of Z per thread in flight
  // What the kernels before this one in the chain wrote (the row list and its
  // count here; LSE^t, the accept flags and the draw partials further on) is
  // read through L2 (ld.global.cg), never through the non-coherent path: a
  // programmatic dependent may start while the kernel before it still runs.
  const int n_rows = __ldcg(count);
  const int groups = V >> 3;
  // Equal waves: with w = ceil(rows / grid) rows per CTA, only the first
  // ceil(rows / w) CTAs take rows, so every working CTA takes w or w - 1 and no
  // last wave runs part-empty (1088 rows on 304 CTAs: 272 CTAs x 4 rows).
  const int waves = n_rows > 0 ? (n_rows + (int)gridDim.x - 1) / (int)gridDim.x : 1;
  const int stride = (n_rows + waves - 1) / waves;
  uint32_t item = (int)blockIdx.x < n_rows ? __ldcg(list + blockIdx.x) : 0u;
  for (int i = blockIdx.x; i < n_rows && (int)blockIdx.x < stride; i += stride) {
    const uint32_t item_next = i + stride < n_rows ? __ldcg(list + i + stride) : 0u;
    const int r = (int)(item / (uint32_t)gamma), j = (int)(item - (uint32_t)r * gamma) + 1;
    const size_t rj = (size_t)r * gamma + (j - 1);
    const T* z = Z + zr.row(r, j) * V;
    const float* srow = scores + rj * V;
    int xj = 0;
    float ld0 = 0.0f, lp = 0.0f;
    if (threadIdx.x == 0) {
      xj = x[rj];
      ld0 = lse[rj];
      lp = logp[rj];
    }

    // Pass 1: (max, sum exp) of Z_j / T.
    float m = -INFINITY, S = 0.0f;
    for (int g0 = threadIdx.x; g0 < groups; g0 += kRowThreads * kRowUnroll) {
      Raw8<T> raw[kRowUnroll];
#pragma unroll
      for (int u = 0; u < kRowUnroll; ++u) {
        const int g = g0 + u * kRowThreads;
        if (g < groups) raw[u].load(z, g);
      }
#pragma unroll
      for (int u = 0; u < kRowUnroll; ++u) {
        if (g0 + u * kRowThreads >= groups) break;
        float e[8];
        raw[u].unpack(e);
        float mx = -INFINITY;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          e[t] *= invT;
          mx = fmaxf(mx, e[t]);
        }
        if (mx > m) {
          S = (m == -INFINITY) ? 0.0f : S * __expf(m - mx);
          m = mx;
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) S += __expf(e[t] - m);
      }
    }
    block_ms<kRowWarps>(m, S, rm, rs);
    const float Lt = m + logf(S);
    T zraw = T();
    if (threadIdx.x == 0) {
      s_ld = ld0;
      if (xj < 0 || xj >= V) {
        flag_status(status, DSPARK_DEV_BAD_INPUT);
        xj = xj < 0 ? 0 : V - 1;
      }
      zraw = z[xj];  // first used after pass 2
    }
    __syncthreads();
    const float ld = s_ld;

    // Pass 2: sum over the row of min(p^d, p^t) = exp(min(s - lse^d, z / T - LSE^t)).
    float acc = 0.0f;
    constexpr int kRowUnroll2 = row_unroll2<T>();
    for (int g0 = threadIdx.x; g0 < groups; g0 += kRowThreads * kRowUnroll2) {
      Raw8<T> raw[kRowUnroll2];
      float4 sa[kRowUnroll2], sb[kRowUnroll2];
#pragma unroll
      for (int u = 0; u < kRowUnroll2; ++u) {
        const int g = g0 + u * kRowThreads;
        if (g < groups) {
          raw[u].load(z, g);
          sa[u] = __ldcs(reinterpret_cast<const float4*>(srow) + 2 * g);
          sb[u] = __ldcs(reinterpret_cast<const float4*>(srow) + 2 * g + 1);
        }
      }
#pragma unroll
      for (int u = 0; u < kRowUnroll2; ++u) {
        if (g0 + u * kRowThreads >= groups) break;
        float e[8];
        raw[u].unpack(e);
        const float sv[8] = {sa[u].x, sa[u].y, sa[u].z, sa[u].w, sb[u].x, sb[u].y, sb[u].z, sb[u].w};
#pragma unroll
        for (int t = 0; t < 8; ++t) acc += __expf(fminf(sv[t] - ld, e[t] * invT - Lt));
      }
    }
    const float csum = block_sum<kRowWarps>(acc, rs);
    if (threadIdx.x == 0) {
      const float u = uniform01(rng_word(seed, (uint32_t)r, (uint32_t)j, DSPARK_PURPOSE_ACCEPT, 0u));
      const float rhs = (to_f32(zraw) * invT - Lt) - lp;
      acc_ws[rj] = logf(u) < rhs ? 1 : 0;
      cstar[rj] = csum;
      lse_t_ws[(size_t)r * (gamma + 1) + (j - 1)] = Lt;
    }
    item = item_next;
  }
}

// Leading accepts of request r (the first rejection is at row n + 1), by one
// warp: lanes read 32 accept flags at a time and the first zero among them
// ends the run (one L2 round trip for gamma <= 32).
__device__ __forceinline__ int leading_accepts_warp(const int* __restrict__ acc_ws, int r, int gamma,
                                                    int L) {
  const int lane = threadIdx.x & 31;
  for (int base = 0; base < L; base += 32) {
    const int a = base + lane < L ? __ldcg(acc_ws + (size_t)r * gamma + base + lane) : 1;
    const unsigned zero = __ballot_sync(0xffffffffu, a == 0);
    if (zero) return base + __ffs((int)zero) - 1;
  }
  return L;
}

// Philox4x32-10 round keys of one seed, passed by value as a kernel parameter:
// the rounds read them as constant-bank operands rather than holding 20
// registers.
struct PhiloxKeys {
  uint32_t k0[10], k1[10];
};
PhiloxKeys philox_keys(uint64_t seed) {
  PhiloxKeys K;
  uint32_t k0 = (uint32_t)(seed & 0xffffffffu), k1 = (uint32_t)(seed >> 32);
  for (int i = 0; i < 10; ++i) {
    K.k0[i] = k0;
    K.k1[i] = k1;
    k0 += kPhiloxW0;
    k1 += kPhiloxW1;
  }
  return K;
}

// The same words as PhiloxStream (one (request, position, purpose), varying first
// counter word q), with the round keys taken from a PhiloxKeys parameter.
struct KeyedPhilox {
  uint32_t a1, b_hi, b_lo, pk1;
  __device__ __forceinline__ KeyedPhilox(const PhiloxKeys& K, uint32_t request, uint32_t position,
                                         uint32_t purpose) {
    const unsigned long long p1 = (unsigned long long)kPhiloxM1 * request;
    const uint32_t a0 = (uint32_t)(p1 >> 32) ^ position ^ K.k0[0];
    a1 = (uint32_t)p1;
    const unsigned long long pb = (unsigned long long)kPhiloxM0 * a0;
    b_hi = (uint32_t)(pb >> 32);
    b_lo = (uint32_t)pb;
    pk1 = purpose ^ K.k1[0];
  }
  __device__ __forceinline__ uint4 quad(const PhiloxKeys& K, uint32_t q) const {
    const unsigned long long p0 = (unsigned long long)kPhiloxM0 * q;
    const uint32_t c2 = (uint32_t)(p0 >> 32) ^ pk1;
    const uint32_t c3 = (uint32_t)p0;
    const unsigned long long p1 = (unsigned long long)kPhiloxM1 * c2;
    uint4 c = make_uint4((uint32_t)(p1 >> 32) ^ a1 ^ K.k0[1], (uint32_t)p1, b_hi ^ c3 ^ K.k1[1], b_lo);
#pragma unroll
    for (int i = 2; i < 10; ++i) {
      const unsigned long long m0 = (unsigned long long)kPhiloxM0 * c.x;
      const unsigned long long m1 = (unsigned long long)kPhiloxM1 * c.z;
      c = make_uint4((uint32_t)(m1 >> 32) ^ c.y ^ K.k0[i], (uint32_t)m1,
                     (uint32_t)(m0 >> 32) ^ c.w ^ K.k1[i], (uint32_t)m0);
    }
    return c;
  }
};

constexpr int kDrawThreads = 256;

// The residual row of the rejection draw, element by element.  With
// a = z/T - LSE^t = ln p^t(v) and delta = ln p^t(v) - ln p^d(v) written as
//   delta = (z/T - s) - (LSE^t - lse^d),
// both differences in parentheses are single roundings of small numbers when
// the two distributions nearly agree, so delta keeps its relative precision
// where p^t - p^d cancels.  The residual is max(0, p^t - p^d) =
// p^t (1 - e^-delta) for delta > 0 and zero otherwise, and its log-weight
// a + ln(1 - e^-delta) is evaluated without the cancelling subtraction.
// Explicitly rounded operations: every evaluation sees the same a and delta.
__device__ __forceinline__ void residual_terms(float z, float s, float invT, float Lt, float dL,
                                               float& a, float& delta) {
  a = __fmaf_rn(z, invT, -Lt);
  delta = __fsub_rn(__fmaf_rn(z, invT, -s), dL);
}

__device__ __forceinline__ float residual_lw(float a, float delta) {
  return __fadd_rn(a, logf(-expm1f(-delta)));
}

// One contiguous global -> shared copy by the bulk-copy engine, completing on
// `bar` (16-byte aligned addresses, bytes a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Bounded wait on a warp's own copy barrier: false after `budget` SM clocks.
__device__ __forceinline__ bool bar_wait_bounded(uint64_t* bar, uint32_t parity, long long budget) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > budget) return false;
  return true;
}

constexpr int kDrawWarpBytes = 32 * 4 * 32 * 2;  // a warp's four groups per lane of bf16 Z: 8 KB
constexpr int kDrawSmemBytes = (kDrawThreads / 32) * kDrawWarpBytes + (kDrawThreads / 32) * 8;

// max of two packed bf16 pairs, lane by lane (exact: a comparison).
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// The raw loads of one 32-id group of a target row (the last group of a row may
// hold fewer ids: nv, a multiple of 8; the missing ones read as -inf), and its
// log-mass log sum_v e^{z_v / T}: the maximum first -- on packed bf16 pairs,
// before any unpacking -- then the sum of exp on float pairs, one unpack per id.
template <typename T> struct GroupZ;
template <> struct GroupZ<__nv_bfloat16> {
  static constexpr uint32_t kNegInf2 = 0xff80ff80u;  // two bf16 -inf
  uint4 q[4];
  __device__ __forceinline__ void load(const __nv_bfloat16* __restrict__ z, int g0, int nv) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
      q[c] = 8 * c < nv ? __ldg(reinterpret_cast<const uint4*>(z) + g0 + c)
                        : make_uint4(kNegInf2, kNegInf2, kNegInf2, kNegInf2);
  }
  // From a shared-memory copy of the group: piece pc is read at step c = pc - rot
  // (mod 4), so that lanes spread over the banks; pieces past nv read as -inf.
  __device__ __forceinline__ void load_shared(const uint8_t* g, int nv, int rot) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int pc = (c + rot) & 3;
      q[c] = 8 * pc < nv ? *(const uint4*)(g + pc * 16)
                         : make_uint4(kNegInf2, kNegInf2, kNegInf2, kNegInf2);
    }
  }
  __device__ __forceinline__ float log_mass(float invT) const {
    const float L2E = 1.4426950408889634f;
    uint32_t m4[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) m4[c] = bmax2(bmax2(q[c].x, q[c].y), bmax2(q[c].z, q[c].w));
    const uint32_t m2 = bmax2(bmax2(m4[0], m4[1]), bmax2(m4[2], m4[3]));
    const float mz = fmaxf(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xffff0000u));
    if (mz == -INFINITY) return -INFINITY;
    const float m = mz * invT;  // T > 0: the largest z/T is the largest z, scaled
    const float2 k2 = make_float2(invT * L2E, invT * L2E), n2 = make_float2(-m * L2E, -m * L2E);
    float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t w[4] = {q[c].x, q[c].y, q[c].z, q[c].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 e2 = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
        const float2 a2 = __ffma2_rn(e2, k2, n2);
        acc = __fadd2_rn(acc, make_float2(ex2_approx(a2.x), ex2_approx(a2.y)));
      }
    }
    return __fadd_rn(m, logf(acc.x + acc.y));
  }
};
template <> struct GroupZ<float> {
  float4 q[8];
  __device__ __forceinline__ void load_shared(const uint8_t*, int, int) {}  // bf16 rows only
  __device__ __forceinline__ void load(const float* __restrict__ z, int g0, int nv) {
#pragma unroll
    for (int c = 0; c < 8; ++c)
      q[c] = 4 * c < nv ? __ldg(reinterpret_cast<const float4*>(z) + 2 * g0 + c)
                        : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  }
  __device__ __forceinline__ float log_mass(float invT) const {
    const float L2E = 1.4426950408889634f;
    float mz = fmax3(q[0].x, q[0].y, q[0].z);
    mz = fmax3(mz, q[0].w, q[1].x);
    mz = fmax3(mz, q[1].y, q[1].z);
    mz = fmaxf(mz, q[1].w);
#pragma unroll
    for (int c = 2; c < 8; ++c) mz = fmax3(fmax3(mz, q[c].x, q[c].y), q[c].z, q[c].w);
    if (mz == -INFINITY) return -INFINITY;
    const float m = mz * invT;
    const float2 k2 = make_float2(invT * L2E, invT * L2E), n2 = make_float2(-m * L2E, -m * L2E);
    float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float2 lo = __ffma2_rn(make_float2(q[c].x, q[c].y), k2, n2);
      const float2 hi = __ffma2_rn(make_float2(q[c].z, q[c].w), k2, n2);
      acc = __fadd2_rn(acc, make_float2(ex2_approx(lo.x), ex2_approx(lo.y)));
      acc = __fadd2_rn(acc, make_float2(ex2_approx(hi.x), ex2_approx(hi.y)));
    }
    return __fadd_rn(m, logf(acc.x + acc.y));
  }
};

// Log-mass of one 32-id group of the rejected row's residual: log sum_v of
// e^a (1 - e^-delta) over the ids with delta > 0 (see residual_terms), -inf
// when there is none.  Two halves of 16 ids, each scaled by its largest e^a
// and merged online; the raw loads of a half are unpacked twice (the maximum,
// then the sum), so the group needs no array of its values.
template <typename T>
__device__ __forceinline__ float residual_group_log_mass(const T* __restrict__ z,
                                                         const float* __restrict__ srow, int v0,
                                                         int nv, float invT, float Lt, float dL) {
  const float L2E = 1.4426950408889634f;
  const int g0 = v0 >> 3;  // first 8-id chunk
  float m = -INFINITY, S = 0.0f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (16 * h >= nv) break;
    Raw8<T> rz[2];
    float4 sa[2], sb[2];
#pragma unroll
    for (int c = 0; c < 2; ++c)
      if (16 * h + 8 * c < nv) {
        rz[c].load(z, g0 + 2 * h + c);
        sa[c] = __ldg(reinterpret_cast<const float4*>(srow) + 2 * (g0 + 2 * h + c));
        sb[c] = __ldg(reinterpret_cast<const float4*>(srow) + 2 * (g0 + 2 * h + c) + 1);
      }
    float mh = -INFINITY;
#pragma unroll
    for (int c = 0; c < 2; ++c)
      if (16 * h + 8 * c < nv) {
        float e[8];
        rz[c].unpack(e);
        const float sv[8] = {sa[c].x, sa[c].y, sa[c].z, sa[c].w, sb[c].x, sb[c].y, sb[c].z, sb[c].w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float av, dt;
          residual_terms(e[i], sv[i], invT, Lt, dL, av, dt);
          if (dt > 0.0f) mh = fmaxf(mh, av);
        }
      }
    if (mh == -INFINITY) continue;
    float Sh = 0.0f;
    const float nm = -mh * L2E;
#pragma unroll
    for (int c = 0; c < 2; ++c)
      if (16 * h + 8 * c < nv) {
        float e[8];
        rz[c].unpack(e);
        const float sv[8] = {sa[c].x, sa[c].y, sa[c].z, sa[c].w, sb[c].x, sb[c].y, sb[c].z, sb[c].w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float av, dt;
          residual_terms(e[i], sv[i], invT, Lt, dL, av, dt);
          if (dt > 0.0f) Sh += ex2_approx(__fmaf_rn(av, L2E, nm)) * -expm1f(-dt);
        }
      }
    lse_merge(m, S, mh, Sh);
  }
  return (m == -INFINITY || !(S > 0.0f)) ? -INFINITY : __fadd_rn(m, logf(S));
}

// Stage 1 of the two-level draw over one chunk of 256 gpt groups of the drawn
// row (the rejected row's residual, or the bonus row's p^t): each thread takes
// gpt consecutive groups (4: they share one Philox quad, word j & 3 keying
// group j; 1 when there are too few requests to fill the GPU otherwise), one
// after another.  For a bf16 bonus row at gpt = 4 each warp first brings its
// 8 KB of Z into shared memory with one bulk copy (dynamic shared memory of
// kDrawSmemBytes), so that the loads are whole-line requests rather than 32
// scattered 16-byte pieces per instruction.  A group's key is
// L_j + G(seed, r, row, RESAMPLE_GROUP, j); it can beat the running best key
// b only if 1 - u_j < exp(L_j - b), tested as fl(f + 1.001 exp(L_j - b)) >= 2
// (f = 1 + (w >> 9) 2^-23), so the two logarithms run only for candidates.  b
// is the best key any thread of the CTA has reached so far (shared memory,
// raised with atomicMax in key_ord form; a stale value is still a lower bound
// of the chunk's maximum).  Writes the chunk's (best group key, group index)
// partial; the emit kernel merges the chunks and draws the token inside the
// winning group.
template <typename T>
__global__ void __launch_bounds__(kDrawThreads, 4)
verify_draw_kernel(const float* __restrict__ lse, const float* __restrict__ scores,
                   const T* __restrict__ Z, const int32_t* __restrict__ ell, int gamma, int V,
                   float invT, const PhiloxKeys keys, const float* __restrict__ lse_t_ws,
                   const int* __restrict__ acc_ws, float2* __restrict__ partials, int n_chunks,
                   int gpt, int* __restrict__ status, ZRows zr) {
  // Launched as a programmatic dependent of the previous kernel: wait for it
  // before anything else, then let the next kernel's launch begin.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ float rk[kDrawThreads / 32];
  __shared__ int ri[kDrawThreads / 32];
  __shared__ int s_n;
  __shared__ uint32_t s_best;  // key_ord of the CTA's best key so far (0: none)
  const int r = blockIdx.y, chunk = blockIdx.x;
  const int L = clamp_ell(ell, r, gamma, nullptr, false);
  if (threadIdx.x < 32) {
    const int n0 = leading_accepts_warp(acc_ws, r, gamma, L);
    if (threadIdx.x == 0) {
      s_n = n0;
      s_best = 0u;
    }
  }
  __syncthreads();
  volatile uint32_t* cta_best = &s_best;
  const int n = s_n;
  const bool residual = n < L;
  const int row = n + 1;  // 1-based position of the drawn token
  const T* z = Z + zr.row(r, row) * V;
  const float* srow = scores + ((size_t)r * gamma + (residual ? row - 1 : 0)) * V;
  float Lt = 0.0f, dL = 0.0f;
  if (residual) {
    Lt = __ldcg(lse_t_ws + (size_t)r * (gamma + 1) + (row - 1));
    dL = __fsub_rn(Lt, lse[(size_t)r * gamma + (row - 1)]);
  }
  const int n_groups = (V + kGroup - 1) / kGroup;
  const float L2E = 1.4426950408889634f;
  float best = -INFINITY;
  int bj = 0x7fffffff;
  auto consider = [&](float Lg, int j, uint32_t w) {
    if (Lg == -INFINITY) return;
    const float thr = ord_key(*cta_best);
    const bool cand = thr == -INFINITY ||
                      __uint_as_float(__funnelshift_r(w, 0x7Fu, 9)) +
                              ex2_approx((Lg - thr) * L2E) * 1.001f >= 2.0f;
    if (cand) {
      const float key = __fadd_rn(Lg, gumbel(w));
      if (better(key, j, best, bj)) {
        best = key;
        bj = j;
      }
      if (best > thr && best < INFINITY) atomicMax(&s_best, key_ord(best));
    }
  };
  const int j0 = (chunk * kDrawThreads + threadIdx.x) * gpt;  // gpt = 1 or 4: 4 | j0
  // bf16 bonus rows at four groups per thread: the warp's 8 KB of Z (four
  // groups per lane) come by one bulk copy into shared memory, issued by lane 0
  // for the whole warp (the warp's ids from s0 up to the row's end).
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long s0 = (long long)(j0 - gpt * lane) * kGroup;  // the warp's first id
  const bool staged = sizeof(T) == 2 && !residual && gpt == 4;
  extern __shared__ __align__(128) uint8_t draw_smem[];
  uint8_t* wbuf = draw_smem + warp * kDrawWarpBytes;
  if (staged && s0 < V) {
    uint64_t* wbar = (uint64_t*)(draw_smem + (kDrawThreads / 32) * kDrawWarpBytes) + warp;
    if (lane == 0) {
      mbar_init(wbar, 1);
      fence_barrier_init();
      const uint32_t bytes = (uint32_t)min((long long)kDrawWarpBytes, (V - s0) * 2);
      mbar_expect_tx(wbar, bytes);
      bulk_load(wbuf, z + s0, bytes, wbar);
    }
    __syncwarp();
    if (!bar_wait_bounded(wbar, 0, kWaitBudget)) {
      if (lane == 0) flag_status(status, DSPARK_DEV_TIMEOUT);
      mbar_drain(wbar, 0, kWaitBudget);
    }
  }
  if (j0 < n_groups) {
    const KeyedPhilox rng(keys, (uint32_t)r, (uint32_t)row, DSPARK_PURPOSE_RESAMPLE_GROUP);
    const uint4 q = rng.quad(keys, (uint32_t)j0 >> 2);
    auto word = [&](int g) {
      const int t = (j0 + g) & 3;
      return t == 0 ? q.x : t == 1 ? q.y : t == 2 ? q.z : q.w;
    };
    const int ng = min(gpt, n_groups - j0);
    if (staged) {
      // Lane l takes its groups in the order (g + l / 4) % 4 and each group's
      // pieces from l % 4 on: the pieces a step reads fall in eight distinct
      // 16-byte bank groups across the warp.
      const uint8_t* tbuf = wbuf + lane * (4 * kGroup * 2);
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const int G = (g + (lane >> 2)) & 3;
        if (G >= ng) continue;
        const int j = j0 + G;
        GroupZ<T> gz;
        gz.load_shared(tbuf + G * kGroup * 2, min(kGroup, V - j * kGroup), lane);
        consider(gz.log_mass(invT), j, word(G));
      }
    } else if (!residual) {  // loads straight from global memory
#pragma unroll 1
      for (int g = 0; g < ng; ++g) {
        const int j = j0 + g;
        GroupZ<T> cur;
        cur.load(z, j * (kGroup / 8), min(kGroup, V - j * kGroup));
        consider(cur.log_mass(invT), j, word(g));
      }
    } else {
#pragma unroll 1
      for (int g = 0; g < ng; ++g) {
        const int j = j0 + g;
        consider(residual_group_log_mass(z, srow, j * kGroup, min(kGroup, V - j * kGroup), invT, Lt,
                                         dL),
                 j, word(g));
      }
    }
  }
  block_argmax<kDrawThreads / 32>(best, bj, rk, ri);
  if (threadIdx.x == 0)
    partials[(size_t)r * n_chunks + chunk] = make_float2(best, __int_as_float(bj));
}

// Per request: merge the chunks' partials into the drawn group (for a residual
// that is zero everywhere, draw the group from p^t over the whole row
// instead), draw the token inside it (stage 2, warp 0: lane t keys id
// 32 j + t with G(seed, r, row, RESAMPLE, v)), then write tokens, n_acc,
// n_emit and the NaN padding of c* / LSE^t beyond l.
template <typename T>
__global__ void __launch_bounds__(kVerifyThreads)
verify_emit_kernel(const int32_t* __restrict__ x, const float* __restrict__ lse,
                   const float* __restrict__ scores, const T* __restrict__ Z,
                   const int32_t* __restrict__ ell, int gamma, int V, float invT, uint64_t seed,
                   const float* __restrict__ lse_t_ws, const int* __restrict__ acc_ws,
                   const float2* __restrict__ partials, int n_chunks, int32_t* __restrict__ n_acc,
                   int32_t* __restrict__ tokens, int32_t* __restrict__ n_emit,
                   float* __restrict__ cstar, float* __restrict__ lse_t_out, ZRows zr) {
  // Launched as a programmatic dependent of the previous kernel: wait for it
  // before anything else, then let the next kernel's launch begin.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ float rk[kWarps];
  __shared__ int ri[kWarps];
  __shared__ int s_n, s_tok;
  const int r = blockIdx.x;
  const int L = clamp_ell(ell, r, gamma, nullptr, false);
  if (threadIdx.x < 32) {
    const int n0 = leading_accepts_warp(acc_ws, r, gamma, L);
    if (threadIdx.x == 0) s_n = n0;
  }
  __syncthreads();
  const int n = s_n;
  const int row = n + 1;
  bool residual = n < L;
  const T* z = Z + zr.row(r, row) * V;
  float best = -INFINITY;
  int gj = 0x7fffffff;
  for (int c = threadIdx.x; c < n_chunks; c += kVerifyThreads) {
    const float2 p = __ldcg(partials + (size_t)r * n_chunks + c);
    const int pi = __float_as_int(p.y);
    if (better(p.x, pi, best, gj)) {
      best = p.x;
      gj = pi;
    }
  }
  block_argmax<kWarps>(best, gj, rk, ri);
  const int n_groups = (V + kGroup - 1) / kGroup;
  if (best == -INFINITY) {
    // Residual zero everywhere (p^t = p^d numerically): draw from p^t, stage 1
    // over every group of the row here.
    residual = false;
    const PhiloxStream rng(seed, (uint32_t)r, (uint32_t)row, DSPARK_PURPOSE_RESAMPLE_GROUP);
    gj = 0x7fffffff;
    for (int j = threadIdx.x; j < n_groups; j += kVerifyThreads) {
      const int v0 = j * kGroup;
      GroupZ<T> gz;
      gz.load(z, v0 >> 3, min(kGroup, V - v0));
      const float Lg = gz.log_mass(invT);
      const float key = __fadd_rn(Lg, gumbel(rng.word((uint32_t)j)));
      if (better(key, j, best, gj)) {
        best = key;
        gj = j;
      }
    }
    block_argmax<kWarps>(best, gj, rk, ri);
  }
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    if (gj < 0 || gj >= n_groups) gj = 0;  // NaN logits only
    const int v = gj * kGroup + lane;
    bool valid = v < V;
    float lw = 0.0f;
    if (valid) {
      const float zv = to_f32(z[v]);
      if (residual) {
        const float Lt = __ldcg(lse_t_ws + (size_t)r * (gamma + 1) + (row - 1));
        const float dL = __fsub_rn(Lt, lse[(size_t)r * gamma + (row - 1)]);
        float a, dt;
        residual_terms(zv, scores[((size_t)r * gamma + (row - 1)) * V + v], invT, Lt, dL, a, dt);
        valid = dt > 0.0f;
        if (valid) lw = residual_lw(a, dt);
      } else {
        lw = zv * invT;
      }
    }
    float key, lwb;
    int tok;
    group_draw_warp(lw, valid, v, seed, (uint32_t)r, (uint32_t)row, DSPARK_PURPOSE_RESAMPLE, key, tok,
                    lwb);
    if (lane == 0) s_tok = tok < V ? tok : gj * kGroup;
  }
  __syncthreads();
  const int idx = s_tok;
  int32_t* trow = tokens + (size_t)r * (gamma + 1);
  for (int t = threadIdx.x; t < gamma + 1; t += kVerifyThreads) {
    int32_t out = -1;
    if (t < n) out = x[(size_t)r * gamma + t];
    else if (t == n) out = idx;
    trow[t] = out;
    if (t < gamma && t >= L) cstar[(size_t)r * gamma + t] = __int_as_float(0x7fc00000);
    if (lse_t_out)
      lse_t_out[(size_t)r * (gamma + 1) + t] =
          t < L ? __ldcg(lse_t_ws + (size_t)r * (gamma + 1) + t) : __int_as_float(0x7fc00000);
  }
  if (threadIdx.x == 0) {
    n_acc[r] = n;
    n_emit[r] = n + 1;
  }
}

}  // namespace

int verify_sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

// Launch `kernel` as a programmatic dependent of the stream's previous kernel
// (the kernel waits for it with griddepcontrol.wait at entry).
template <typename... Params, typename... Args>
cudaError_t launch_chained_smem(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                                cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}

template <typename... Params, typename... Args>
cudaError_t launch_chained(void (*kernel)(Params...), dim3 grid, dim3 block, cudaStream_t s,
                           Args... args) {
  return launch_chained_smem(kernel, grid, block, 0, s, args...);
}

cudaError_t launch_verify_rows(const int32_t* x, const float* logp, const float* lse,
                               const float* scores, const void* Z, int dtype, const int32_t* ell,
                               int R, int gamma, int V, float invT, uint64_t seed, float* cstar,
                               float* lse_t_ws, int* acc_ws, uint32_t* row_list, int* row_count,
                               int* status, ZRows zr, cudaStream_t s) {
  verify_index_kernel<<<1, kIndexThreads, 0, s>>>(ell, R, gamma, row_list, row_count, status, zr);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long rows_max = (long long)R * gamma;
  const int cap = 2 * verify_sm_count();  // two CTAs of 512 threads per SM
  const int grid = (int)(rows_max < cap ? rows_max : cap);
  if (dtype == DSPARK_BF16)
    return launch_chained(verify_rows_stream_kernel<__nv_bfloat16>, dim3(grid), dim3(kRowThreads), s,
                          x, logp, lse, scores, (const __nv_bfloat16*)Z, (const uint32_t*)row_list,
                          (const int*)row_count, gamma, V, invT, seed, cstar, lse_t_ws, acc_ws,
                          status, zr);
  return launch_chained(verify_rows_stream_kernel<float>, dim3(grid), dim3(kRowThreads), s, x, logp,
                        lse, scores, (const float*)Z, (const uint32_t*)row_list,
                        (const int*)row_count, gamma, V, invT, seed, cstar, lse_t_ws, acc_ws, status,
                        zr);
}

// Groups per thread of the draw: 4 when four-group chunks still give at least
// two waves of draw CTAs (four per SM), else 1.
static int draw_gpt(int R, int V) {
  const long long n_groups = (V + kGroup - 1) / kGroup;
  const long long chunks4 = (n_groups + 4 * kDrawThreads - 1) / (4 * kDrawThreads);
  return (long long)R * chunks4 >= 2LL * 4 * verify_sm_count() ? 4 : 1;
}

static int draw_chunks(int V, int gpt) {
  const int n_groups = (V + kGroup - 1) / kGroup;
  return (n_groups + gpt * kDrawThreads - 1) / (gpt * kDrawThreads);
}

// Partials per request the workspace holds: the larger count (one group per thread).
int verify_draw_chunks(int V) { return draw_chunks(V, 1); }

// Draw CTAs per request of this launch (both launches below must agree).
int verify_draw_launch_chunks(int R, int V) { return draw_chunks(V, draw_gpt(R, V)); }

cudaError_t launch_verify_draw(const float* lse, const float* scores, const void* Z, int dtype,
                               const int32_t* ell, int R, int gamma, int V, float invT,
                               uint64_t seed, const float* lse_t_ws, const int* acc_ws,
                               float2* partials, int* status, ZRows zr, cudaStream_t s) {
  const int gpt = draw_gpt(R, V);
  const int chunks = draw_chunks(V, gpt);
  dim3 grid(chunks, R);
  if (dtype == DSPARK_BF16) {
    static bool smem_set = false;  // the staged bonus draw's shared memory (> 48 KB: opt in)
    if (!smem_set) {
      const cudaError_t e = cudaFuncSetAttribute(
          verify_draw_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
          kDrawSmemBytes);
      if (e != cudaSuccess) return e;
      smem_set = true;
    }
    return launch_chained_smem(verify_draw_kernel<__nv_bfloat16>, grid, dim3(kDrawThreads),
                               gpt == 4 ? (size_t)kDrawSmemBytes : 0, s, lse, scores,
                               (const __nv_bfloat16*)Z, ell, gamma, V, invT, philox_keys(seed),
                               lse_t_ws, acc_ws, partials, chunks, gpt, status, zr);
  }
  return launch_chained(verify_draw_kernel<float>, grid, dim3(kDrawThreads), s, lse, scores,
                        (const float*)Z, ell, gamma, V, invT, philox_keys(seed), lse_t_ws, acc_ws,
                        partials, chunks, gpt, status, zr);
}

cudaError_t launch_verify_emit(const int32_t* x, const float* lse, const float* scores,
                               const void* Z, int dtype, const int32_t* ell, int R, int gamma, int V,
                               float invT, uint64_t seed, const float* lse_t_ws, const int* acc_ws,
                               const float2* partials, int32_t* n_acc, int32_t* tokens,
                               int32_t* n_emit, float* cstar, float* lse_t, ZRows zr,
                               cudaStream_t s) {
  const int chunks = verify_draw_launch_chunks(R, V);
  if (dtype == DSPARK_BF16)
    return launch_chained(verify_emit_kernel<__nv_bfloat16>, dim3(R), dim3(kVerifyThreads), s, x,
                          lse, scores, (const __nv_bfloat16*)Z, ell, gamma, V, invT, seed, lse_t_ws,
                          acc_ws, partials, chunks, n_acc, tokens, n_emit, cstar, lse_t, zr);
  return launch_chained(verify_emit_kernel<float>, dim3(R), dim3(kVerifyThreads), s, x, lse, scores,
                        (const float*)Z, ell, gamma, V, invT, seed, lse_t_ws, acc_ws, partials,
                        chunks, n_acc, tokens, n_emit, cstar, lse_t, zr);
}

}  // namespace dspark
