// sts.cu -- Sequential Temperature Scaling of the confidence head and the
// static-threshold scheduler.
//
// "DSpark: Confidence-Scheduled Speculative Decoding with Semi-Autoregressive
// Generation 요약 설명", §3.2.1: on held-out data the cumulative prefix survival
// is calibrated by a left-to-right 1-D grid search that minimises each
// position's Expected Calibration Error with the earlier positions'
// calibration held fixed.  §4.3.3: a static threshold on the survival prunes
// the verify length.
//
// Per position k (three launches):
//   sts_ece     (grid temperatures x sample chunks) CTAs: for every sample,
//               ahat = ahat_prev * temper(c_k; T_g) (the map in fp32, the
//               product in fp64), its bin b = min(floor(ahat M), M - 1), and
//               (ahat - Y_k) added to bin b in 2^-40 fixed point (int64), so
//               each ECE is exact for the given ahat and independent of the
//               summation order;
//   sts_pick    one CTA: ECE(g) = sum_b |S_b| 2^-40 / N, the first grid entry
//               with the smallest ECE becomes T_k; the bins are cleared;
//   sts_update  ahat_prev *= temper(c_k; T_k), Y &= y_k.
#include "common.cuh"
#include "kernels.h"

namespace dspark {

namespace {

constexpr int kStsThreads = 256;
constexpr int kStsChunk = 16384;  // samples per sts_ece CTA
constexpr double kFix = 1099511627776.0;  // 2^40

// sigmoid(logit(c) / T); 0 and 1 stay, T = 1 returns c.  NaN counts as 0.
__device__ __forceinline__ float temper(float c, float T) {
  if (!(c > 0.0f)) return 0.0f;
  if (!(c < 1.0f)) return 1.0f;
  if (T == 1.0f) return c;
  const float z = (logf(c) - log1pf(-c)) / T;
  return 1.0f / (1.0f + expf(-z));
}

__global__ void __launch_bounds__(kStsThreads)
sts_ece_kernel(const float* __restrict__ conf, const uint8_t* __restrict__ accept, int N, int gamma,
               int k, const double* __restrict__ grid, int M, const double* __restrict__ ahat,
               const uint8_t* __restrict__ Y, long long* __restrict__ bins) {
  extern __shared__ long long sb[];  // [M]
  for (int b = threadIdx.x; b < M; b += kStsThreads) sb[b] = 0;
  __syncthreads();
  const int g = blockIdx.x;
  const float T = (float)grid[g];
  const int s0 = blockIdx.y * kStsChunk, s1 = min(N, s0 + kStsChunk);
  for (int s = s0 + threadIdx.x; s < s1; s += kStsThreads) {
    const double a = ahat[s] * (double)temper(conf[(size_t)s * gamma + k], T);
    const int yk = Y[s] && accept[(size_t)s * gamma + k];
    int b = (int)floor(a * M);
    b = b > M - 1 ? M - 1 : (b < 0 ? 0 : b);
    atomicAdd((unsigned long long*)&sb[b], (unsigned long long)llrint((a - (double)yk) * kFix));
  }
  __syncthreads();
  for (int b = threadIdx.x; b < M; b += kStsThreads)
    if (sb[b]) atomicAdd((unsigned long long*)&bins[(size_t)g * M + b], (unsigned long long)sb[b]);
}

__global__ void __launch_bounds__(kStsThreads)
sts_pick_kernel(long long* __restrict__ bins, const double* __restrict__ grid, int G, int M, int N,
                int k, double* __restrict__ temps, double* __restrict__ ece,
                int* __restrict__ choice) {
  __shared__ double be[kStsThreads];
  __shared__ int bg[kStsThreads];
  double best = INFINITY;
  int arg = 0x7fffffff;
  for (int g = threadIdx.x; g < G; g += kStsThreads) {
    unsigned long long tot = 0;  // sum of |S_b| in 2^-40 units (exact)
    for (int b = 0; b < M; ++b) {
      const long long v = bins[(size_t)g * M + b];
      tot += (unsigned long long)(v < 0 ? -v : v);
    }
    const double e = (double)tot / kFix / (double)N;
    if (e < best || (e == best && g < arg)) {
      best = e;
      arg = g;
    }
  }
  be[threadIdx.x] = best;
  bg[threadIdx.x] = arg;
  __syncthreads();
  for (int o = kStsThreads / 2; o > 0; o >>= 1) {
    if (threadIdx.x < o) {
      const double e2 = be[threadIdx.x + o];
      const int g2 = bg[threadIdx.x + o];
      if (e2 < be[threadIdx.x] || (e2 == be[threadIdx.x] && g2 < bg[threadIdx.x])) {
        be[threadIdx.x] = e2;
        bg[threadIdx.x] = g2;
      }
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    *choice = bg[0];
    temps[k] = grid[bg[0]];
    if (ece) ece[k] = be[0];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < G * M; i += kStsThreads) bins[i] = 0;
}

__global__ void __launch_bounds__(kStsThreads)
sts_update_kernel(const float* __restrict__ conf, const uint8_t* __restrict__ accept, int N,
                  int gamma, int k, const double* __restrict__ grid,
                  const int* __restrict__ choice, double* __restrict__ ahat,
                  uint8_t* __restrict__ Y) {
  const int s = blockIdx.x * kStsThreads + threadIdx.x;
  if (s >= N) return;
  const float T = (float)grid[*choice];
  ahat[s] *= (double)temper(conf[(size_t)s * gamma + k], T);
  Y[s] = Y[s] && accept[(size_t)s * gamma + k];
}

__global__ void sts_init_kernel(int N, double* __restrict__ ahat, uint8_t* __restrict__ Y) {
  const int s = blockIdx.x * kStsThreads + threadIdx.x;
  if (s < N) {
    ahat[s] = 1.0;
    Y[s] = 1;
  }
}

// l_r = number of leading positions whose survival prod temper(c; T_j) (or
// prod c without temperatures) is at least theta.  One thread per request.
__global__ void __launch_bounds__(kStsThreads)
schedule_threshold_kernel(const float* __restrict__ conf, const double* __restrict__ temps,
                          double theta, int R, int gamma, int32_t* __restrict__ ell) {
  const int r = blockIdx.x * kStsThreads + threadIdx.x;
  if (r >= R) return;
  double a = 1.0;
  int l = 0;
  for (int j = 0; j < gamma; ++j) {
    const float c = conf[(size_t)r * gamma + j];
    a *= (double)temper(c, temps ? (float)temps[j] : 1.0f);
    if (!(a >= theta)) break;
    l = j + 1;
  }
  ell[r] = l;
}

}  // namespace

StsWorkspace sts_workspace_layout(int N, int G, int M) {
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  StsWorkspace w;
  w.choice = 0;
  w.bins = 256;
  w.ahat = al(w.bins + (size_t)G * M * sizeof(long long));
  w.Y = al(w.ahat + (size_t)N * sizeof(double));
  w.total = al(w.Y + (size_t)N);
  return w;
}

cudaError_t launch_sts_calibrate(const float* conf, const uint8_t* accept, int N, int gamma,
                                 const double* grid, int G, int M, double* temps, double* ece,
                                 void* workspace, cudaStream_t s) {
  const StsWorkspace L = sts_workspace_layout(N, G, M);
  char* ws = (char*)workspace;
  int* choice = (int*)(ws + L.choice);
  long long* bins = (long long*)(ws + L.bins);
  double* ahat = (double*)(ws + L.ahat);
  uint8_t* Y = (uint8_t*)(ws + L.Y);
  cudaError_t e = cudaMemsetAsync(bins, 0, (size_t)G * M * sizeof(long long), s);
  if (e != cudaSuccess) return e;
  const int nb = (N + kStsThreads - 1) / kStsThreads;
  sts_init_kernel<<<nb, kStsThreads, 0, s>>>(N, ahat, Y);
  const dim3 egrid(G, (N + kStsChunk - 1) / kStsChunk);
  for (int k = 0; k < gamma; ++k) {
    sts_ece_kernel<<<egrid, kStsThreads, M * sizeof(long long), s>>>(conf, accept, N, gamma, k, grid,
                                                                     M, ahat, Y, bins);
    sts_pick_kernel<<<1, kStsThreads, 0, s>>>(bins, grid, G, M, N, k, temps, ece, choice);
    sts_update_kernel<<<nb, kStsThreads, 0, s>>>(conf, accept, N, gamma, k, grid, choice, ahat, Y);
  }
  return cudaGetLastError();
}

cudaError_t launch_schedule_threshold(const float* conf, const double* temps, double theta, int R,
                                      int gamma, int32_t* ell, cudaStream_t s) {
  schedule_threshold_kernel<<<(R + kStsThreads - 1) / kStsThreads, kStsThreads, 0, s>>>(
      conf, temps, theta, R, gamma, ell);
  return cudaGetLastError();
}

}  // namespace dspark
