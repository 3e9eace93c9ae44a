// api.cu -- the C-ABI of libdspark.so (declared in include/dspark.h): argument
// checks, workspace layout, and the launch sequence of each call.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "../../include/dspark.h"
#include "kernels.h"

namespace dspark {

static thread_local char g_last_error[256] = "";

static int cuda_fail(cudaError_t e, const char* where) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s", where, cudaGetErrorString(e));
  return DSPARK_ERR_CUDA;
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

DraftWorkspace draft_workspace_layout(int R, int gamma, int V, int r, int dtype) {
  (void)gamma;
  DraftWorkspace w;
  const size_t esize = dtype == DSPARK_BF16 ? 2 : 4;
  const size_t tiles = (size_t)((V + kDraftTileN - 1) / kDraftTileN);
  const size_t rows = ((size_t)R + 127) / 128 * 128;  // A padded to whole 128-row tiles
  w.status = 0;
  w.a_rows = align256(w.status + 4);
  w.stats = align256(w.a_rows + rows * (size_t)r * esize);
  w.index = align256(w.stats + (size_t)R * tiles * sizeof(float4));
  w.stats2 = align256(w.index + (size_t)R * tiles * sizeof(int));
  w.index2 = align256(w.stats2 + (size_t)R * tiles * sizeof(float4));
  w.gbest = align256(w.index2 + (size_t)R * tiles * sizeof(int));  // uint64 [3, R]
  w.w2t = align256(w.gbest + 3 * (size_t)R * sizeof(unsigned long long));  // bf16 W2^T [V, r]
  w.total = align256(w.w2t + (dtype == DSPARK_BF16 ? (size_t)V * r * 2 : 0));
  return w;
}

// Scratch layout of verify (byte offsets, 256-aligned): status word and the
// scheduled-row count (the first 256 bytes), LSE^t [R, gamma+1], accept flags
// [R, gamma], the scheduled-row list [R * gamma] (u32), draw partials
// [R, chunks] (float2).
struct VerifyScratch {
  size_t count, lse_t, acc, list, partials, total;
};
static VerifyScratch verify_scratch_layout(int R, int gamma, int V) {
  VerifyScratch v;
  v.count = 4;
  v.lse_t = 256;
  v.acc = align256(v.lse_t + (size_t)R * (gamma + 1) * sizeof(float));
  v.list = align256(v.acc + (size_t)R * gamma * sizeof(int));
  v.partials = align256(v.list + (size_t)R * gamma * sizeof(uint32_t));
  v.total = align256(v.partials + (size_t)R * verify_draw_chunks(V) * sizeof(float2));
  return v;
}

static int check_common(int R, int gamma, int V, float T, int dtype) {
  if (R <= 0 || gamma <= 0 || V <= 0) return DSPARK_ERR_INVALID_ARG;
  if (!(T > 0.0f) || !isfinite(T)) return DSPARK_ERR_INVALID_ARG;
  if (dtype != DSPARK_F32 && dtype != DSPARK_BF16) return DSPARK_ERR_INVALID_ARG;
  if (gamma > 64 || R > 65535 || V % 8 != 0 || V < 8) return DSPARK_ERR_UNSUPPORTED;
  return DSPARK_OK;
}

// Optional event timing: while enabled, every kernel launch of the library is
// bracketed by two CUDA events recorded on the launch's stream.  Host-side
// state only (events, no device memory); not thread-safe.
struct Profiler {
  static constexpr int kMax = 8192;
  bool on = false;
  bool created = false;
  int n = 0;
  int launches[kKindCount] = {};
  int kind[kMax];
  cudaEvent_t ev[2 * kMax];
};
static Profiler g_prof;

static void prof_begin(int kind, cudaStream_t s) {
  if (!g_prof.on) return;
  g_prof.launches[kind] += 1;
  if (g_prof.n < Profiler::kMax) {
    g_prof.kind[g_prof.n] = kind;
    cudaEventRecord(g_prof.ev[2 * g_prof.n], s);
  }
}

static void prof_end(cudaStream_t s) {
  if (!g_prof.on || g_prof.n >= Profiler::kMax) return;
  cudaEventRecord(g_prof.ev[2 * g_prof.n + 1], s);
  g_prof.n += 1;
}

}  // namespace dspark

using namespace dspark;

extern "C" {

const char* dspark_status_string(int status) {
  switch (status) {
    case DSPARK_OK: return "ok";
    case DSPARK_ERR_INVALID_ARG: return "invalid argument";
    case DSPARK_ERR_UNSUPPORTED: return "unsupported size or dtype";
    case DSPARK_ERR_WORKSPACE: return "workspace missing or too small";
    case DSPARK_ERR_CUDA: return "CUDA error";
    case DSPARK_ERR_DEVICE_INPUT: return "device input out of range";
    case DSPARK_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

const char* dspark_last_error(void) { return g_last_error; }

int dspark_version(void) { return 10000; }

size_t dspark_draft_workspace_bytes(int R, int gamma, int V, int r, int dtype) {
  if (R <= 0 || gamma <= 0 || V <= 0 || r <= 0) return 0;
  return draft_workspace_layout(R, gamma, V, r, dtype).total;
}

int dspark_transpose_w2(const void* W2, int r, int V, void* W2T, void* stream) {
  if (!W2 || !W2T || r <= 0 || V <= 0) return DSPARK_ERR_INVALID_ARG;
  if (r > 256 || r % 64 != 0 || V % 8 != 0) return DSPARK_ERR_UNSUPPORTED;
  if (!aligned16(W2) || !aligned16(W2T)) return DSPARK_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  prof_begin(kKindPrepare, s);
  const cudaError_t e = launch_transpose_w2(W2, r, V, W2T, s);
  prof_end(s);
  if (e != cudaSuccess) return cuda_fail(e, "transpose_w2");
  return DSPARK_OK;
}

// The Markov-head draft; W2 is [r, V] as stored, or (w2t) the K-major W2^T
// [V, r] that dspark_transpose_w2 wrote, which the tensor-core steps read.
static int draft_markov(const void* U, const void* W1, const void* W2, bool w2t,
                        const int32_t* x0, int dtype, int R, int gamma, int V, int r,
                        float temperature, uint64_t seed, int32_t* x, float* logp, float* lse,
                        float* scores, void* workspace, size_t workspace_bytes, void* stream) {
  if (!U || !W1 || !W2 || !x0 || !x || !logp || !lse || !scores) return DSPARK_ERR_INVALID_ARG;
  if (r <= 0) return DSPARK_ERR_INVALID_ARG;
  int st = check_common(R, gamma, V, temperature, dtype);
  if (st != DSPARK_OK) return st;
  if (r > 256 || r % 16 != 0 || (dtype == DSPARK_BF16 && r % 64 != 0)) return DSPARK_ERR_UNSUPPORTED;
  if (!aligned16(U) || !aligned16(W1) || !aligned16(W2) || !aligned16(scores))
    return DSPARK_ERR_INVALID_ARG;
  const DraftWorkspace L = draft_workspace_layout(R, gamma, V, r, dtype);
  if (!workspace || workspace_bytes < L.total || ((uintptr_t)workspace & 255u))
    return DSPARK_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  char* ws = (char*)workspace;
  int* status = (int*)(ws + L.status);
  void* A = ws + L.a_rows;
  const bool tc = dtype == DSPARK_BF16 && draft_tc_supported(R, V, r);
  if (w2t && !tc) return DSPARK_ERR_UNSUPPORTED;  // W2^T feeds the tensor-core steps only
  const int n_parts = tc ? draft_tc_parts(R, V) : (V + kDraftTileN - 1) / kDraftTileN;
  DraftPartials p{(float4*)(ws + L.stats), (int*)(ws + L.index), n_parts};
  DraftPartials p2{(float4*)(ws + L.stats2), (int*)(ws + L.index2), n_parts};
  const float invT = 1.0f / temperature;
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int), s);
  if (e != cudaSuccess) return cuda_fail(e, "draft status reset");
  const size_t esize = dtype == DSPARK_BF16 ? 2 : 4;
  const size_t pad_rows = ((size_t)R + 127) / 128 * 128 - (size_t)R;
  if (pad_rows) {
    e = cudaMemsetAsync((char*)A + (size_t)R * r * esize, 0, pad_rows * r * esize, s);
    if (e != cudaSuccess) return cuda_fail(e, "draft pad reset");
  }
  if (tc) {
    // Tensor-core path: each step gathers its A tile itself; partials alternate
    // between two buffers; one combine after the last step.
    const void* W2T = W2;
    if (!w2t) {
      W2T = ws + L.w2t;
      prof_begin(kKindPrepare, s);
      e = launch_transpose_w2(W2, r, V, ws + L.w2t, s);
      prof_end(s);
      if (e != cudaSuccess) return cuda_fail(e, "transpose_w2");
    }
    DraftTcPlan plan;
    e = prepare_draft_tc(&plan, U, W2T, R, gamma, V, r, scores);
    if (e != cudaSuccess) return cuda_fail(e, "draft tensor maps");
    unsigned long long* gbest = (unsigned long long*)(ws + L.gbest);
    e = cudaMemsetAsync(gbest, 0, 3 * (size_t)R * sizeof(unsigned long long), s);
    if (e != cudaSuccess) return cuda_fail(e, "draft key reset");
    const DraftPartials buf[2] = {p, p2};
    for (int k = 1; k <= gamma; ++k) {
      prof_begin(kKindDraftTile, s);
      e = launch_draft_step_tc(plan, k, invT, seed, x0, W1, buf[(k + 1) & 1], buf[k & 1], gbest, x,
                               logp, lse, status, s);
      prof_end(s);
      if (e != cudaSuccess) return cuda_fail(e, "draft_step");
    }
    prof_begin(kKindDraftCombine, s);
    e = launch_draft_combine(buf[gamma & 1], R, gamma, V, r, gamma, W1, dtype, nullptr, scores, seed,
                             x, logp, lse, status, s);
    prof_end(s);
    if (e != cudaSuccess) return cuda_fail(e, "draft_combine");
    return DSPARK_OK;
  }
  prof_begin(kKindPrepare, s);
  e = launch_gather_anchor(W1, x0, R, V, r, dtype, A, status, s);
  prof_end(s);
  if (e != cudaSuccess) return cuda_fail(e, "gather_anchor");
  for (int k = 1; k <= gamma; ++k) {
    prof_begin(kKindDraftTile, s);
    e = launch_draft_tile_simt(U, A, W2, dtype, R, gamma, V, r, k, invT, seed, scores, p, s);
    prof_end(s);
    if (e != cudaSuccess) return cuda_fail(e, "draft_tile");
    prof_begin(kKindDraftCombine, s);
    e = launch_draft_combine(p, R, gamma, V, r, k, W1, dtype, k < gamma ? A : nullptr, scores, seed,
                             x, logp, lse, status, s);
    prof_end(s);
    if (e != cudaSuccess) return cuda_fail(e, "draft_combine");
  }
  return DSPARK_OK;
}

int dspark_draft_sample(const void* U, const void* W1, const void* W2, const int32_t* x0,
                        int dtype, int R, int gamma, int V, int r, float temperature,
                        uint64_t seed, int32_t* x, float* logp, float* lse, float* scores,
                        void* workspace, size_t workspace_bytes, void* stream) {
  return draft_markov(U, W1, W2, false, x0, dtype, R, gamma, V, r, temperature, seed, x, logp,
                      lse, scores, workspace, workspace_bytes, stream);
}

int dspark_draft_sample_w2t(const void* U, const void* W1, const void* W2T, const int32_t* x0,
                            int R, int gamma, int V, int r, float temperature, uint64_t seed,
                            int32_t* x, float* logp, float* lse, float* scores, void* workspace,
                            size_t workspace_bytes, void* stream) {
  return draft_markov(U, W1, W2T, true, x0, DSPARK_BF16, R, gamma, V, r, temperature, seed, x,
                      logp, lse, scores, workspace, workspace_bytes, stream);
}

// The RNN head's extra scratch after the draft workspace: the state h [2][R, r]
// fp32 (double-buffered across steps) and the A rows [R padded to 128, r] bf16.
struct RnnWorkspace {
  size_t h, A, total;
};
static RnnWorkspace rnn_workspace_layout(int R, int gamma, int V, int r) {
  RnnWorkspace w;
  w.h = align256(draft_workspace_layout(R, gamma, V, r, DSPARK_BF16).total);
  w.A = align256(w.h + 2 * (size_t)R * r * sizeof(float));
  w.total = align256(w.A + ((size_t)R + 127) / 128 * 128 * r * 2);
  return w;
}

size_t dspark_draft_rnn_workspace_bytes(int R, int gamma, int V, int r) {
  if (R <= 0 || gamma <= 0 || V <= 0 || r <= 0) return 0;
  return rnn_workspace_layout(R, gamma, V, r).total;
}

static int draft_rnn(const void* U, const void* W1, const void* W2, bool w2t, const void* Wh,
                     const float* Q, const int32_t* x0, int dtype, int R, int gamma, int V, int r,
                     float temperature, uint64_t seed, int32_t* x, float* logp, float* lse,
                     float* scores, void* workspace, size_t workspace_bytes, void* stream) {
  if (!U || !W1 || !W2 || !Wh || !Q || !x0 || !x || !logp || !lse || !scores)
    return DSPARK_ERR_INVALID_ARG;
  if (r <= 0) return DSPARK_ERR_INVALID_ARG;
  int st = check_common(R, gamma, V, temperature, dtype);
  if (st != DSPARK_OK) return st;
  if (dtype != DSPARK_BF16 || r > 256 || r % 64 != 0 || V % 8 != 0) return DSPARK_ERR_UNSUPPORTED;
  if (!aligned16(U) || !aligned16(W1) || !aligned16(W2) || !aligned16(scores) || !aligned16(Wh) ||
      !aligned16(Q))
    return DSPARK_ERR_INVALID_ARG;
  const DraftWorkspace L = draft_workspace_layout(R, gamma, V, r, dtype);
  const RnnWorkspace LR = rnn_workspace_layout(R, gamma, V, r);
  if (!workspace || workspace_bytes < LR.total || ((uintptr_t)workspace & 255u))
    return DSPARK_ERR_WORKSPACE;
  if (!draft_tc_supported(R, V, r)) return DSPARK_ERR_UNSUPPORTED;  // needs the driver's TMA encoder
  cudaStream_t s = (cudaStream_t)stream;
  char* ws = (char*)workspace;
  int* status = (int*)(ws + L.status);
  float* h = (float*)(ws + LR.h);
  void* A = ws + LR.A;
  const int n_parts = draft_tc_parts(R, V);
  DraftPartials p{(float4*)(ws + L.stats), (int*)(ws + L.index), n_parts};
  DraftPartials p2{(float4*)(ws + L.stats2), (int*)(ws + L.index2), n_parts};
  const float invT = 1.0f / temperature;
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int), s);
  if (e == cudaSuccess)  // A's rows past R stay zero: the contraction reads whole 128-row tiles
    e = cudaMemsetAsync(A, 0, ((size_t)R + 127) / 128 * 128 * r * 2, s);
  if (e != cudaSuccess) return cuda_fail(e, "draft_rnn reset");
  const void* W2T = W2;
  if (!w2t) {
    W2T = ws + L.w2t;
    prof_begin(kKindPrepare, s);
    e = launch_transpose_w2(W2, r, V, ws + L.w2t, s);
    prof_end(s);
    if (e != cudaSuccess) return cuda_fail(e, "transpose_w2");
  }
  DraftTcPlan plan;
  e = prepare_draft_tc(&plan, U, W2T, R, gamma, V, r, scores);
  if (e != cudaSuccess) return cuda_fail(e, "draft tensor maps");
  unsigned long long* gbest = (unsigned long long*)(ws + L.gbest);
  e = cudaMemsetAsync(gbest, 0, 3 * (size_t)R * sizeof(unsigned long long), s);
  if (e != cudaSuccess) return cuda_fail(e, "draft key reset");
  const DraftPartials buf[2] = {p, p2};
  for (int k = 1; k <= gamma; ++k) {
    prof_begin(kKindRnnState, s);
    e = launch_rnn_state(k, x0, W1, Wh, Q, buf[(k + 1) & 1], R, gamma, V, r,
                         h + (size_t)((k + 1) & 1) * R * r, h + (size_t)(k & 1) * R * r, A, scores,
                         seed, x, logp, lse, status, s);
    prof_end(s);
    if (e != cudaSuccess) return cuda_fail(e, "rnn_state");
    prof_begin(kKindDraftTile, s);
    e = launch_draft_step_tc(plan, k, invT, seed, x0, W1, buf[(k + 1) & 1], buf[k & 1], gbest, x,
                             logp, lse, status, s, A);
    prof_end(s);
    if (e != cudaSuccess) return cuda_fail(e, "draft_step");
  }
  prof_begin(kKindDraftCombine, s);
  e = launch_draft_combine(buf[gamma & 1], R, gamma, V, r, gamma, W1, dtype, nullptr, scores, seed, x,
                           logp, lse, status, s);
  prof_end(s);
  if (e != cudaSuccess) return cuda_fail(e, "draft_combine");
  return DSPARK_OK;
}

int dspark_draft_sample_rnn(const void* U, const void* W1, const void* W2, const void* Wh,
                            const float* Q, const int32_t* x0, int dtype, int R, int gamma, int V,
                            int r, float temperature, uint64_t seed, int32_t* x, float* logp,
                            float* lse, float* scores, void* workspace, size_t workspace_bytes,
                            void* stream) {
  return draft_rnn(U, W1, W2, false, Wh, Q, x0, dtype, R, gamma, V, r, temperature, seed, x, logp,
                   lse, scores, workspace, workspace_bytes, stream);
}

int dspark_draft_sample_rnn_w2t(const void* U, const void* W1, const void* W2T, const void* Wh,
                                const float* Q, const int32_t* x0, int R, int gamma, int V, int r,
                                float temperature, uint64_t seed, int32_t* x, float* logp,
                                float* lse, float* scores, void* workspace,
                                size_t workspace_bytes, void* stream) {
  return draft_rnn(U, W1, W2T, true, Wh, Q, x0, DSPARK_BF16, R, gamma, V, r, temperature, seed, x,
                   logp, lse, scores, workspace, workspace_bytes, stream);
}

size_t dspark_schedule_workspace_bytes(int R, int gamma) {
  if (R <= 0 || gamma <= 0) return 0;
  return 256 + align256(schedule_sorted_bytes(R, gamma));
}

int dspark_schedule(const float* conf, const double* sps, int sps_len, int R, int gamma,
                    int32_t* ell, double* diag, void* workspace, size_t workspace_bytes,
                    void* stream) {
  if (!conf || !sps || !ell) return DSPARK_ERR_INVALID_ARG;
  if (R <= 0 || gamma <= 0) return DSPARK_ERR_INVALID_ARG;
  if (gamma > 64 || (long long)R * gamma > 16384) return DSPARK_ERR_UNSUPPORTED;
  if ((long long)sps_len < (long long)R * (1 + gamma) + 1) return DSPARK_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < dspark_schedule_workspace_bytes(R, gamma) ||
      ((uintptr_t)workspace & 255u))
    return DSPARK_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  int* status = (int*)workspace;
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int), s);
  if (e != cudaSuccess) return cuda_fail(e, "schedule status reset");
  unsigned long long* sorted = (unsigned long long*)((char*)workspace + 256);
  prof_begin(kKindSchedule, s);
  e = launch_schedule_rank(conf, R, gamma, sorted, status, s);
  prof_end(s);
  if (e != cudaSuccess) return cuda_fail(e, "schedule_rank");
  prof_begin(kKindSchedule, s);
  e = launch_schedule_scan(sorted, sps, R, gamma, ell, diag, status, s);
  prof_end(s);
  if (e != cudaSuccess) return cuda_fail(e, "schedule_scan");
  return DSPARK_OK;
}

static int schedule_args(const float* conf, int R, int gamma, void* workspace,
                         size_t workspace_bytes) {
  if (!conf) return DSPARK_ERR_INVALID_ARG;
  if (R <= 0 || gamma <= 0) return DSPARK_ERR_INVALID_ARG;
  if (gamma > 64 || (long long)R * gamma > 16384) return DSPARK_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < dspark_schedule_workspace_bytes(R, gamma) ||
      ((uintptr_t)workspace & 255u))
    return DSPARK_ERR_WORKSPACE;
  return DSPARK_OK;
}

int dspark_schedule_capacity(const float* conf_old, const double* sps, int sps_len, int R,
                             int gamma, int32_t* K, double* diag, void* workspace,
                             size_t workspace_bytes, void* stream) {
  if (!sps || !K) return DSPARK_ERR_INVALID_ARG;
  if (R > 0 && gamma > 0 && (long long)sps_len < (long long)R * (1 + gamma) + 1)
    return DSPARK_ERR_INVALID_ARG;
  int st = schedule_args(conf_old, R, gamma, workspace, workspace_bytes);
  if (st != DSPARK_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  int* status = (int*)workspace;
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int), s);
  if (e != cudaSuccess) return cuda_fail(e, "schedule_capacity status reset");
  unsigned long long* sorted = (unsigned long long*)((char*)workspace + 256);
  prof_begin(kKindSchedule, s);
  e = launch_schedule_rank(conf_old, R, gamma, sorted, status, s);
  prof_end(s);
  if (e != cudaSuccess) return cuda_fail(e, "schedule_rank");
  prof_begin(kKindSchedule, s);
  e = launch_schedule_capacity(sorted, sps, R, gamma, K, diag, status, s);
  prof_end(s);
  if (e != cudaSuccess) return cuda_fail(e, "schedule_capacity");
  return DSPARK_OK;
}

int dspark_schedule_topk(const float* conf, const int32_t* K, int R, int gamma, int32_t* ell,
                         void* workspace, size_t workspace_bytes, void* stream) {
  if (!K || !ell) return DSPARK_ERR_INVALID_ARG;
  int st = schedule_args(conf, R, gamma, workspace, workspace_bytes);
  if (st != DSPARK_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  int* status = (int*)workspace;
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int), s);
  if (e != cudaSuccess) return cuda_fail(e, "schedule_topk status reset");
  unsigned long long* sorted = (unsigned long long*)((char*)workspace + 256);
  prof_begin(kKindSchedule, s);
  e = launch_schedule_rank(conf, R, gamma, sorted, status, s);
  prof_end(s);
  if (e != cudaSuccess) return cuda_fail(e, "schedule_rank");
  prof_begin(kKindSchedule, s);
  e = launch_schedule_topk(sorted, K, R, gamma, ell, status, s);
  prof_end(s);
  if (e != cudaSuccess) return cuda_fail(e, "schedule_topk");
  return DSPARK_OK;
}

size_t dspark_sts_workspace_bytes(int N, int G, int M) {
  if (N <= 0 || G <= 0 || M <= 0) return 0;
  return sts_workspace_layout(N, G, M).total;
}

int dspark_sts_calibrate(const float* conf, const uint8_t* accept, int N, int gamma,
                         const double* grid, int G, int M, double* temps, double* ece,
                         void* workspace, size_t workspace_bytes, void* stream) {
  if (!conf || !accept || !grid || !temps) return DSPARK_ERR_INVALID_ARG;
  if (N <= 0 || gamma <= 0 || G <= 0 || M <= 0) return DSPARK_ERR_INVALID_ARG;
  if (N > (1 << 22) || M > 1024 || gamma > 64) return DSPARK_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < dspark_sts_workspace_bytes(N, G, M) ||
      ((uintptr_t)workspace & 255u))
    return DSPARK_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = launch_sts_calibrate(conf, accept, N, gamma, grid, G, M, temps, ece, workspace, s);
  if (e != cudaSuccess) return cuda_fail(e, "sts_calibrate");
  return DSPARK_OK;
}

int dspark_schedule_threshold(const float* conf, const double* temps, double theta, int R,
                              int gamma, int32_t* ell, void* stream) {
  if (!conf || !ell) return DSPARK_ERR_INVALID_ARG;
  if (R <= 0 || gamma <= 0 || !(theta == theta)) return DSPARK_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  prof_begin(kKindSchedule, s);
  cudaError_t e = launch_schedule_threshold(conf, temps, theta, R, gamma, ell, s);
  prof_end(s);
  if (e != cudaSuccess) return cuda_fail(e, "schedule_threshold");
  return DSPARK_OK;
}

size_t dspark_verify_workspace_bytes(int R, int gamma, int V) {
  if (R <= 0 || gamma <= 0 || V <= 0) return 0;
  return verify_scratch_layout(R, gamma, V).total;
}

}  // extern "C"

// The verify launches on `workspace` (already validated); zr addresses Z.
static int verify_enqueue(const int32_t* x, const float* logp, const float* lse,
                          const float* scores, const void* Z, int dtype, const int32_t* ell, int R,
                          int gamma, int V, float temperature, uint64_t seed, int32_t* n_acc,
                          int32_t* tokens, int32_t* n_emit, float* cstar, float* lse_t,
                          void* workspace, ZRows zr, cudaStream_t s, const char* what) {
  char* ws = (char*)workspace;
  int* status = (int*)ws;
  const VerifyScratch lay = verify_scratch_layout(R, gamma, V);
  float* lse_t_ws = (float*)(ws + lay.lse_t);
  int* acc_ws = (int*)(ws + lay.acc);
  float2* partials = (float2*)(ws + lay.partials);
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int), s);
  if (e != cudaSuccess) return cuda_fail(e, what);
  const float invT = 1.0f / temperature;
  prof_begin(kKindVerifyRows, s);
  e = launch_verify_rows(x, logp, lse, scores, Z, dtype, ell, R, gamma, V, invT, seed, cstar,
                         lse_t_ws, acc_ws, (uint32_t*)(ws + lay.list), (int*)(ws + lay.count),
                         status, zr, s);
  prof_end(s);
  if (e != cudaSuccess) return cuda_fail(e, what);
  prof_begin(kKindVerifyDraw, s);
  e = launch_verify_draw(lse, scores, Z, dtype, ell, R, gamma, V, invT, seed, lse_t_ws, acc_ws,
                         partials, status, zr, s);
  prof_end(s);
  if (e != cudaSuccess) return cuda_fail(e, what);
  prof_begin(kKindVerifyEmit, s);
  e = launch_verify_emit(x, lse, scores, Z, dtype, ell, R, gamma, V, invT, seed, lse_t_ws, acc_ws,
                         partials, n_acc, tokens, n_emit, cstar, lse_t, zr, s);
  prof_end(s);
  if (e != cudaSuccess) return cuda_fail(e, what);
  return DSPARK_OK;
}

static int verify_args(const int32_t* x, const float* logp, const float* lse, const float* scores,
                       const void* Z, int dtype, const int32_t* ell, int R, int gamma, int V,
                       float temperature, const int32_t* n_acc, const int32_t* tokens,
                       const int32_t* n_emit, const float* cstar) {
  if (!x || !logp || !lse || !scores || !Z || !ell || !n_acc || !tokens || !n_emit || !cstar)
    return DSPARK_ERR_INVALID_ARG;
  int st = check_common(R, gamma, V, temperature, dtype);
  if (st != DSPARK_OK) return st;
  if (!aligned16(Z) || !aligned16(scores)) return DSPARK_ERR_INVALID_ARG;
  return DSPARK_OK;
}

extern "C" {

int dspark_verify(const int32_t* x, const float* logp, const float* lse, const float* scores,
                  const void* Z, int dtype, const int32_t* ell, int R, int gamma, int V,
                  float temperature, uint64_t seed, int32_t* n_acc, int32_t* tokens,
                  int32_t* n_emit, float* cstar, float* lse_t, void* workspace,
                  size_t workspace_bytes, void* stream) {
  int st = verify_args(x, logp, lse, scores, Z, dtype, ell, R, gamma, V, temperature, n_acc, tokens,
                       n_emit, cstar);
  if (st != DSPARK_OK) return st;
  if (!workspace || workspace_bytes < dspark_verify_workspace_bytes(R, gamma, V) ||
      ((uintptr_t)workspace & 255u))
    return DSPARK_ERR_WORKSPACE;
  return verify_enqueue(x, logp, lse, scores, Z, dtype, ell, R, gamma, V, temperature, seed, n_acc,
                        tokens, n_emit, cstar, lse_t, workspace, ZRows{nullptr, gamma, 0},
                        (cudaStream_t)stream, "verify");
}

int dspark_verify_packed(const int32_t* x, const float* logp, const float* lse,
                         const float* scores, const void* Zp, int dtype, const int32_t* row_offsets,
                         int n_rows, const int32_t* ell, int R, int gamma, int V,
                         float temperature, uint64_t seed, int32_t* n_acc, int32_t* tokens,
                         int32_t* n_emit, float* cstar, float* lse_t, void* workspace,
                         size_t workspace_bytes, void* stream) {
  int st = verify_args(x, logp, lse, scores, Zp, dtype, ell, R, gamma, V, temperature, n_acc, tokens,
                       n_emit, cstar);
  if (st != DSPARK_OK) return st;
  if (!row_offsets || n_rows < R) return DSPARK_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < dspark_verify_workspace_bytes(R, gamma, V) ||
      ((uintptr_t)workspace & 255u))
    return DSPARK_ERR_WORKSPACE;
  return verify_enqueue(x, logp, lse, scores, Zp, dtype, ell, R, gamma, V, temperature, seed, n_acc,
                        tokens, n_emit, cstar, lse_t, workspace, ZRows{row_offsets, gamma, n_rows},
                        (cudaStream_t)stream, "verify_packed");
}

int dspark_read_device_status(const void* workspace, void* stream, int32_t* out) {
  if (!workspace || !out) return DSPARK_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(out, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "read_device_status");
  return DSPARK_OK;
}

}  // extern "C"

// Scratch of dspark_verify_noalloc: a file-scope device array.  In host code
// its name is only a stand-in; the kernels get the device address that
// cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) unsigned char g_verify_noalloc_scratch[DSPARK_VERIFY_NOALLOC_SCRATCH_BYTES];
static std::mutex g_noalloc_mu;
// Per device: the address and the id of the context it was looked up in.  A
// cudaDeviceReset ends the primary context; the next one loads the module
// again, possibly elsewhere, so the address is looked up again when the
// current context's id differs.
static void* g_noalloc_addr[64] = {};
static unsigned long long g_noalloc_ctx[64] = {};

typedef CUresult (*PFN_ctx_get_current)(CUcontext*);
typedef CUresult (*PFN_ctx_get_id)(CUcontext, unsigned long long*);

// Id of the current context (0 if the driver cannot tell): two driver calls,
// no synchronisation, allowed during stream capture.
static unsigned long long current_ctx_id() {
  static PFN_ctx_get_current get_current = nullptr;
  static PFN_ctx_get_id get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = (PFN_ctx_get_current)f;
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = (PFN_ctx_get_id)f;
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

static int noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "verify_noalloc current device");
  if (dev < 0 || dev >= 64) {
    snprintf(g_last_error, sizeof(g_last_error), "dspark_verify_noalloc: device %d not supported", dev);
    return DSPARK_ERR_UNSUPPORTED;
  }
  // Before the device's first runtime call there is no current context (id
  // 0): the lookup creates it, and its id is recorded afterwards.
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  const unsigned long long ctx = current_ctx_id();
  if (!g_noalloc_addr[dev] || ctx == 0 || ctx != g_noalloc_ctx[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_verify_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "verify_noalloc scratch address");
    g_noalloc_addr[dev] = p;
    g_noalloc_ctx[dev] = ctx != 0 ? ctx : current_ctx_id();
  }
  *out = g_noalloc_addr[dev];
  return DSPARK_OK;
}

extern "C" {

int dspark_verify_noalloc(const int32_t* x, const float* logp, const float* lse,
                          const float* scores, const void* Z, int dtype, const int32_t* ell, int R,
                          int gamma, int V, float temperature, uint64_t seed, int32_t* n_acc,
                          int32_t* tokens, int32_t* n_emit, float* cstar, float* lse_t,
                          void* stream) {
  if (!x || !logp || !lse || !scores || !Z || !ell || !n_acc || !tokens || !n_emit || !cstar)
    return DSPARK_ERR_INVALID_ARG;
  int st = check_common(R, gamma, V, temperature, dtype);
  if (st != DSPARK_OK) return st;
  if (!aligned16(Z) || !aligned16(scores)) return DSPARK_ERR_INVALID_ARG;
  const VerifyScratch lay = verify_scratch_layout(R, gamma, V);
  const size_t need = lay.total;
  if (need > DSPARK_VERIFY_NOALLOC_SCRATCH_BYTES) {
    snprintf(g_last_error, sizeof(g_last_error),
             "dspark_verify_noalloc: R=%d, gamma=%d needs %zu bytes of scratch, the static array "
             "holds %u",
             R, gamma, need, (unsigned)DSPARK_VERIFY_NOALLOC_SCRATCH_BYTES);
    return DSPARK_ERR_UNSUPPORTED;
  }
  void* scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != DSPARK_OK) return st;
  return verify_enqueue(x, logp, lse, scores, Z, dtype, ell, R, gamma, V, temperature, seed, n_acc,
                        tokens, n_emit, cstar, lse_t, scratch, ZRows{nullptr, gamma, 0},
                        (cudaStream_t)stream, "verify_noalloc");
}

int dspark_selftest_draft_timeout(const void* U, const void* W1, const void* W2,
                                  const int32_t* x0, int R, int gamma, int V, int r,
                                  long long wait_cycles, int32_t* x, float* logp, float* lse,
                                  float* scores, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  if (!U || !W1 || !W2 || !x0 || !x || !logp || !lse || !scores) return DSPARK_ERR_INVALID_ARG;
  if (wait_cycles < 1000 || wait_cycles > 4000000000ll) return DSPARK_ERR_INVALID_ARG;
  int st = check_common(R, gamma, V, 1.0f, DSPARK_BF16);
  if (st != DSPARK_OK) return st;
  if (!aligned16(U) || !aligned16(W1) || !aligned16(W2) || !aligned16(scores))
    return DSPARK_ERR_INVALID_ARG;
  if (!draft_tc_supported(R, V, r)) return DSPARK_ERR_UNSUPPORTED;
  const DraftWorkspace L = draft_workspace_layout(R, gamma, V, r, DSPARK_BF16);
  if (!workspace || workspace_bytes < L.total || ((uintptr_t)workspace & 255u))
    return DSPARK_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  char* ws = (char*)workspace;
  int* status = (int*)(ws + L.status);
  const int n_parts = draft_tc_parts(R, V);
  DraftPartials p{(float4*)(ws + L.stats), (int*)(ws + L.index), n_parts};
  DraftPartials p2{(float4*)(ws + L.stats2), (int*)(ws + L.index2), n_parts};
  unsigned long long* gbest = (unsigned long long*)(ws + L.gbest);
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int), s);
  if (e == cudaSuccess) e = cudaMemsetAsync(gbest, 0, 3 * (size_t)R * sizeof(unsigned long long), s);
  if (e != cudaSuccess) return cuda_fail(e, "selftest reset");
  DraftTcPlan plan;
  e = prepare_draft_tc(&plan, U, ws + L.w2t, R, gamma, V, r, scores);
  if (e != cudaSuccess) return cuda_fail(e, "selftest tensor maps");
  e = launch_draft_step_tc(plan, 1, 1.0f, 0, x0, W1, p2, p, gbest, x, logp, lse, status, s, nullptr,
                           wait_cycles, true);
  if (e != cudaSuccess) return cuda_fail(e, "selftest draft_step");
  return DSPARK_OK;
}

int dspark_profile_start(void) {
  if (!g_prof.created) {
    for (int i = 0; i < 2 * Profiler::kMax; ++i) {
      cudaError_t e = cudaEventCreate(&g_prof.ev[i]);
      if (e != cudaSuccess) return cuda_fail(e, "profile event create");
    }
    g_prof.created = true;
  }
  g_prof.n = 0;
  for (int k = 0; k < kKindCount; ++k) g_prof.launches[k] = 0;
  g_prof.on = true;
  return DSPARK_OK;
}

int dspark_stream_probe(const void* in, float* out, size_t n, void* stream) {
  if (!in || !out || n == 0 || n % 8 != 0 || !aligned16(in) || !aligned16(out))
    return DSPARK_ERR_INVALID_ARG;
  cudaError_t e = launch_stream_probe(in, out, n, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "stream_probe");
  return DSPARK_OK;
}

int dspark_profile_stop(double* ms_by_kind, int* launches_by_kind, int* timed_launches) {
  if (!g_prof.on) return DSPARK_ERR_INVALID_ARG;
  g_prof.on = false;
  for (int k = 0; k < kKindCount; ++k) {
    if (ms_by_kind) ms_by_kind[k] = 0.0;
    if (launches_by_kind) launches_by_kind[k] = g_prof.launches[k];
  }
  if (timed_launches) *timed_launches = g_prof.n;
  if (g_prof.n == 0) return DSPARK_OK;
  cudaError_t e = cudaEventSynchronize(g_prof.ev[2 * g_prof.n - 1]);
  if (e != cudaSuccess) return cuda_fail(e, "profile sync");
  for (int i = 0; i < g_prof.n; ++i) {
    float ms = 0.0f;
    e = cudaEventElapsedTime(&ms, g_prof.ev[2 * i], g_prof.ev[2 * i + 1]);
    if (e != cudaSuccess) return cuda_fail(e, "profile elapsed");
    if (ms_by_kind) ms_by_kind[g_prof.kind[i]] += ms;
  }
  return DSPARK_OK;
}

}  // extern "C"
