// kernels.h -- host-side launchers of the DSpark kernels (internal to libdspark.so).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace dspark {

// Per-row draft partials over a subset of the vocabulary: max m, sum exp(s - m),
// and stage 1 of the two-level draw: the best group key L_j + G(DRAFT_GROUP, j)
// of the subset's 32-id groups, with that group's index j.  The CUDA-core path
// writes one part per 128-column tile, the tensor-core path one part per CTA
// slot.
struct DraftPartials {
  float4* stats;  // [R, n_parts] (m, S, best group key, unused)
  int* index;     // [R, n_parts] best group index
  int n_parts;
};

constexpr int kDraftTileN = 128;  // vocab columns per tile (both contraction paths)

// Workspace layout of dspark_draft_sample (byte offsets, 256-aligned).
struct DraftWorkspace {
  // two partial buffers; gbest: [3][R] per-row packed best (key, group) of a step's CTAs
  size_t status, a_rows, stats, index, stats2, index2, gbest, w2t, total;
};
DraftWorkspace draft_workspace_layout(int R, int gamma, int V, int r, int dtype);

cudaError_t launch_gather_anchor(const void* W1, const int32_t* x0, int R, int V, int r, int dtype,
                                 void* A, int* status, cudaStream_t s);

// fp32 / bf16 CUDA-core contraction + fused epilogue for draft step k (1-based).
cudaError_t launch_draft_tile_simt(const void* U, const void* A, const void* W2, int dtype, int R,
                                   int gamma, int V, int r, int k, float invT, uint64_t seed,
                                   float* scores, DraftPartials p, cudaStream_t s);

// bf16 tcgen05 contraction (TMA-fed, TMEM accumulators) + fused epilogue.
// Tensor maps of one draft call (W2, U, scores), encoded once on the host.
struct DraftTcPlan {
  alignas(64) unsigned char maps[3][128];
  float* scores;
  const void* w2t;  // W2^T [V, r] bf16, read by every step
  int R, gamma, V, r;
};
cudaError_t prepare_draft_tc(DraftTcPlan* plan, const void* U, const void* W2T, int R, int gamma,
                             int V, int r, float* scores);
cudaError_t launch_transpose_w2(const void* W2, int r, int V, void* W2T, cudaStream_t s);
// Step k (1-based): gathers A from x0 (k = 1) or from step k-1's drawn
// tokens (its packed per-row best, then the token inside that group; the
// partials `prev` give step k-1's lse, which it stores with x and logp),
// writes `cur`.  gbest is the [3][R] array of per-row packed bests
// (key_ord(key) << 32 | ~group): step k reads row (k - 1) % 3, raises row
// k % 3 and zeroes row (k + 1) % 3 for the next step; rows 1 and 2 must be
// zero before step 1.
cudaError_t launch_draft_step_tc(const DraftTcPlan& plan, int k, float invT, uint64_t seed,
                                 const int32_t* x0, const void* W1, const DraftPartials& prev,
                                 const DraftPartials& cur, unsigned long long* gbest, int32_t* x,
                                 float* logp, float* lse, int* status, cudaStream_t s,
                                 const void* A_src = nullptr, long long wait_budget = 0,
                                 bool withhold_w2 = false);
// RNN head, step k: x_{k-1} (anchor for k = 1, else the merge of `prev`, whose
// x/logp/lse it also stores), h_k = tanh(W1[x_{k-1}] + h_{k-1} Wh + Q_k) from
// h_prev into h_next ([R, r] fp32 each; h_prev unread for k = 1), and
// A [R, r] = bf16(h_k) for the contraction.  r a multiple of 64, at most 256;
// Wh 16-byte aligned.
cudaError_t launch_rnn_state(int k, const int32_t* x0, const void* W1, const void* Wh,
                             const float* Q, const DraftPartials& prev, int R, int gamma, int V,
                             int r, const float* h_prev, float* h_next, void* A,
                             const float* scores, uint64_t seed, int32_t* x, float* logp,
                             float* lse, int* status, cudaStream_t s);
bool draft_tc_supported(int R, int V, int r);
int draft_tc_parts(int R, int V);  // partials per row written by the tensor-core path

cudaError_t launch_draft_combine(DraftPartials p, int R, int gamma, int V, int r, int k,
                                 const void* W1, int dtype, void* A_next, const float* scores,
                                 uint64_t seed, int32_t* x, float* logp, float* lse, int* status,
                                 cudaStream_t s);

// Scheduler: rank-and-scatter sort into `sorted` (R * gamma keys), then the scan.
size_t schedule_sorted_bytes(int R, int gamma);
cudaError_t launch_schedule_rank(const float* conf, int R, int gamma, unsigned long long* sorted,
                                 int* status, cudaStream_t s);
cudaError_t launch_schedule_scan(const unsigned long long* sorted, const double* sps, int R,
                                 int gamma, int32_t* ell, double* diag, int* status,
                                 cudaStream_t s);
// Zero-overhead scheduling: capacity K (first global Theta maximum along the
// sorted order, written to device memory), then the top K of a sorted order.
cudaError_t launch_schedule_capacity(const unsigned long long* sorted, const double* sps, int R,
                                     int gamma, int32_t* K, double* diag, int* status,
                                     cudaStream_t s);
cudaError_t launch_schedule_topk(const unsigned long long* sorted, const int32_t* K, int R,
                                 int gamma, int32_t* ell, int* status, cudaStream_t s);

// Where the target row of request r at (1-based) position j starts, in rows
// of V elements: the padded [R, gamma+1, V] layout (off == nullptr) or a packed
// [n_rows, V] buffer whose request r occupies rows off[r] .. off[r] + l_r
// (positions 1 .. l_r + 1), the index clamped into the buffer.
struct ZRows {
  const int32_t* off;  // [R + 1] row offsets, or nullptr for the padded layout
  int gamma, n_rows;
#ifdef __CUDACC__
  __device__ __forceinline__ size_t row(int r, int j) const {
    if (!off) return (size_t)r * (gamma + 1) + (j - 1);
    long long q = (long long)off[r] + (j - 1);
    q = q < 0 ? 0 : (q >= n_rows ? n_rows - 1 : q);
    return (size_t)q;
  }
#endif
};

// LSE^t, c* and the accept flag of every scheduled row (r, j <= l_r).
// row_list ([R * gamma] u32) and *row_count are scratch: the list of those rows
// that verify_index builds first and the row kernel then takes from.
cudaError_t launch_verify_rows(const int32_t* x, const float* logp, const float* lse,
                               const float* scores, const void* Z, int dtype, const int32_t* ell,
                               int R, int gamma, int V, float invT, uint64_t seed, float* cstar,
                               float* lse_t_ws, int* acc_ws, uint32_t* row_list, int* row_count,
                               int* status, ZRows zr, cudaStream_t s);

// The drawn token: verify_draw over vocab chunks, then verify_emit per request.
int verify_draw_chunks(int V);
cudaError_t launch_verify_draw(const float* lse, const float* scores, const void* Z, int dtype,
                               const int32_t* ell, int R, int gamma, int V, float invT,
                               uint64_t seed, const float* lse_t_ws, const int* acc_ws,
                               float2* partials, int* status, ZRows zr, cudaStream_t s);
cudaError_t launch_verify_emit(const int32_t* x, const float* lse, const float* scores,
                               const void* Z, int dtype, const int32_t* ell, int R, int gamma, int V,
                               float invT, uint64_t seed, const float* lse_t_ws, const int* acc_ws,
                               const float2* partials, int32_t* n_acc, int32_t* tokens,
                               int32_t* n_emit, float* cstar, float* lse_t, ZRows zr,
                               cudaStream_t s);

// Sequential temperature scaling: workspace (byte offsets, 256-aligned) of the
// chosen grid index, the [G, M] fixed-point bins, the running survival [N]
// (fp64) and the running outcome [N] (u8).
struct StsWorkspace {
  size_t choice, bins, ahat, Y, total;
};
StsWorkspace sts_workspace_layout(int N, int G, int M);
cudaError_t launch_sts_calibrate(const float* conf, const uint8_t* accept, int N, int gamma,
                                 const double* grid, int G, int M, double* temps, double* ece,
                                 void* workspace, cudaStream_t s);
cudaError_t launch_schedule_threshold(const float* conf, const double* temps, double theta, int R,
                                      int gamma, int32_t* ell, cudaStream_t s);

// Contiguous bf16 -> fp32 stream of n values (n % 8 == 0): a bandwidth probe.
cudaError_t launch_stream_probe(const void* in, float* out, size_t n, cudaStream_t s);

// Kernel kinds for the optional event timing (dspark_profile_*).
enum KernelKind {
  kKindPrepare = 0,  // W2 transpose (bf16) or anchor gather (fp32)
  kKindDraftTile = 1,
  kKindDraftCombine = 2,
  kKindSchedule = 3,  // both scheduler launches
  kKindVerifyRows = 4,
  kKindVerifyDraw = 5,  // stage 1 of the residual / bonus draw
  kKindRnnState = 6,    // RNN head: state update before each draft step
  kKindVerifyEmit = 7,  // stage 2 of the draw and the emitted tokens
  kKindCount = 8
};

}  // namespace dspark
