// common.cuh -- device helpers shared by the DSpark kernels.
//
// Philox4x32-10 follows Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers:
// As Easy as 1, 2, 3" (SC'11).  The counter layout, uniform map and Gumbel map
// are the library's convention, stated in include/dspark.h.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dspark.h"

namespace dspark {

constexpr uint32_t kPhiloxM0 = 0xD2511F53u;
constexpr uint32_t kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u;
constexpr uint32_t kPhiloxW1 = 0xBB67AE85u;

// Ten rounds; the key advances by the Weyl constants between rounds.
__device__ __forceinline__ uint4 philox10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const unsigned long long p0 = (unsigned long long)kPhiloxM0 * c.x;
    const unsigned long long p1 = (unsigned long long)kPhiloxM1 * c.z;
    c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ k0, (uint32_t)p1, (uint32_t)(p0 >> 32) ^ c.w ^ k1,
                   (uint32_t)p0);
    k0 += kPhiloxW0;
    k1 += kPhiloxW1;
  }
  return c;
}

// Philox4x32-10 words for one fixed (seed, request, position, purpose) and a
// varying first counter word q.  The same ten rounds as philox10(); the parts
// that do not depend on q -- the round keys, round 1's product of the request
// word, round 2's product of that round's first output -- are computed once.
struct PhiloxStream {
  uint32_t rk0[10], rk1[10];
  uint32_t a0, a1;      // round-1 outputs 0 and 1 (independent of q)
  uint32_t b_hi, b_lo;  // round-2 product M0 * a0
  uint32_t pk1;         // purpose ^ round-1 key word 1

  __device__ __forceinline__ PhiloxStream(uint64_t seed, uint32_t request, uint32_t position,
                                          uint32_t purpose) {
    uint32_t k0 = (uint32_t)(seed & 0xffffffffu), k1 = (uint32_t)(seed >> 32);
#pragma unroll
    for (int i = 0; i < 10; ++i) {
      rk0[i] = k0;
      rk1[i] = k1;
      k0 += kPhiloxW0;
      k1 += kPhiloxW1;
    }
    const unsigned long long p1 = (unsigned long long)kPhiloxM1 * request;
    a0 = (uint32_t)(p1 >> 32) ^ position ^ rk0[0];
    a1 = (uint32_t)p1;
    const unsigned long long pb = (unsigned long long)kPhiloxM0 * a0;
    b_hi = (uint32_t)(pb >> 32);
    b_lo = (uint32_t)pb;
    pk1 = purpose ^ rk1[0];
  }

  __device__ __forceinline__ uint4 quad(uint32_t q) const {
    // round 1: (q, position, request, purpose) -> (a0, a1, c2, c3)
    const unsigned long long p0 = (unsigned long long)kPhiloxM0 * q;
    const uint32_t c2 = (uint32_t)(p0 >> 32) ^ pk1;
    const uint32_t c3 = (uint32_t)p0;
    // round 2: M0 * a0 is fixed
    const unsigned long long p1 = (unsigned long long)kPhiloxM1 * c2;
    uint4 c = make_uint4((uint32_t)(p1 >> 32) ^ a1 ^ rk0[1], (uint32_t)p1, b_hi ^ c3 ^ rk1[1], b_lo);
#pragma unroll
    for (int i = 2; i < 10; ++i) {
      const unsigned long long m0 = (unsigned long long)kPhiloxM0 * c.x;
      const unsigned long long m1 = (unsigned long long)kPhiloxM1 * c.z;
      c = make_uint4((uint32_t)(m1 >> 32) ^ c.y ^ rk0[i], (uint32_t)m1,
                     (uint32_t)(m0 >> 32) ^ c.w ^ rk1[i], (uint32_t)m0);
    }
    return c;
  }

  __device__ __forceinline__ uint32_t word(uint32_t v) const {
    const uint4 w = quad(v >> 2);
    const uint32_t s = v & 3u;
    return s == 0 ? w.x : s == 1 ? w.y : s == 2 ? w.z : w.w;
  }
};

__device__ __forceinline__ uint32_t seed_lo(uint64_t s) { return (uint32_t)(s & 0xffffffffu); }
__device__ __forceinline__ uint32_t seed_hi(uint64_t s) { return (uint32_t)(s >> 32); }

// The four words for vocab ids 4q..4q+3 at (request, position, purpose).
__device__ __forceinline__ uint4 rng_quad(uint64_t seed, uint32_t request, uint32_t position,
                                          uint32_t purpose, uint32_t q) {
  return philox10(make_uint4(q, position, request, purpose), seed_lo(seed), seed_hi(seed));
}

__device__ __forceinline__ uint32_t rng_word(uint64_t seed, uint32_t request, uint32_t position,
                                             uint32_t purpose, uint32_t v) {
  const uint4 w = rng_quad(seed, request, position, purpose, v >> 2);
  const uint32_t s = v & 3u;
  return s == 0 ? w.x : s == 1 ? w.y : s == 2 ? w.z : w.w;
}

// u = (2 (w >> 9) + 1) 2^-24, exact in fp32.
__device__ __forceinline__ float uniform01(uint32_t w) {
  return __fmul_rn((float)(((w >> 9) << 1) | 1u), 5.9604644775390625e-8f);
}

// G = -ln(-ln u) with the accurate logf (never the approximate intrinsic:
// ln u near 1 needs full relative accuracy).
__device__ __forceinline__ float gumbel(uint32_t w) { return -logf(-logf(uniform01(w))); }

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// (value, index) order used by every argmax: larger value wins, ties go to the
// lower index.  NaN keys never win.
__device__ __forceinline__ bool better(float a, int ia, float b, int ib) {
  return a > b || (a == b && ia < ib);
}

__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (better(ov, oi, v, i)) {
      v = ov;
      i = oi;
    }
  }
}

// Warp-level argmax carrying a value at the argmax (ties to the lower index).
__device__ __forceinline__ void warp_argmax3(float& key, int& idx, float& val) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ok = __shfl_xor_sync(0xffffffffu, key, o);
    const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
    const float ov = __shfl_xor_sync(0xffffffffu, val, o);
    if (better(ok, oi, key, idx)) {
      key = ok;
      idx = oi;
      val = ov;
    }
  }
}

// Ids per group of the two-level Gumbel-max draw: stage 1 draws a group of
// kGroup consecutive ids by Gumbel-max over the groups' log-masses, stage 2
// draws an id of that group by Gumbel-max over its log-weights.
constexpr int kGroup = DSPARK_GROUP;

// Stage 2 by one warp over group j: lane t holds id v = kGroup j + t with
// log-weight lw (`valid`: v < V and the weight is non-zero) and keys it
// lw + G(seed, request, position, purpose, v).  Every lane returns the best
// key, its id and its log-weight (ties to the lower id).
__device__ __forceinline__ void group_draw_warp(float lw, bool valid, int v, uint64_t seed,
                                                uint32_t request, uint32_t position,
                                                uint32_t purpose, float& key, int& idx,
                                                float& lw_best) {
  key = valid ? __fadd_rn(lw, gumbel(rng_word(seed, request, position, purpose, (uint32_t)v)))
              : -INFINITY;
  idx = valid ? v : 0x7fffffff;
  lw_best = lw;
  warp_argmax3(key, idx, lw_best);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Merge a (max, sum of exp(x - max)) pair into another.
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
    return;
  }
  if (m2 > m) {
    s = s * __expf(m - m2) + s2;
    m = m2;
  } else {
    s = s + s2 * __expf(m2 - m);
  }
}

__device__ __forceinline__ void warp_lse(float& m, float& s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    lse_merge(m, s, m2, s2);
  }
}

// Order-preserving map of a float key onto uint32: unsigned order equals float
// order for every non-NaN value, and 0 lies below all of them (it stands for
// "no key yet", so a zero-filled array starts every row at -inf).
__device__ __forceinline__ uint32_t key_ord(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float ord_key(uint32_t o) {
  if (o == 0u) return -INFINITY;
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

// Device status word: OR bits in with an atomic.
__device__ __forceinline__ void flag_status(int* status, int bits) {
  if (status) atomicOr(status, bits);
}

}  // namespace dspark
