/*
 * dspark.h -- C-ABI of the DSpark per-round sampling library (libdspark.so).
 *
 * Three calls make one speculative-decoding round on one GPU, in stream order:
 *
 *   dspark_draft_sample -> dspark_schedule -> dspark_verify
 *
 * Sources (page title, section):
 *   "DSpark: Confidence-Scheduled Speculative Decoding with Semi-Autoregressive
 *    Generation 요약 설명" (greeksharifa.github.io) -- cited below as [summary]:
 *    opening bullets (draft proposes a block, the target verifies the accepted
 *    prefix by rejection sampling, which keeps the target distribution),
 *    §3 (tau counts the bonus token), §3.1 (semi-autoregressive draft, Markov
 *    head B = W1 W2), §3.2.1 (soft label c*), §3.2.2 (prefix scheduler,
 *    Algorithm 1).
 *   "DSpark: Confidence-Scheduled Speculative Decoding with Semi-Autoregressive
 *    Generation" (notes-ybman-uk.pages.dev) -- cited as [notes]: "DSpark 핵심
 *    기술 1" (p_k = softmax(U_k + B_k)), "배경" (accept the longest prefix).
 *
 * Conventions shared by all calls
 * -------------------------------
 * - Every pointer except `stream`, `diag`-less NULLs and the host-side
 *   `out` of dspark_read_device_status is a DEVICE pointer on the current
 *   device.  The caller allocates and owns every buffer (inputs, outputs,
 *   workspace).  The library never allocates or frees memory and keeps no
 *   state between calls.  Inputs are read-only, outputs write-only; no
 *   output may alias an input or another output.
 * - Arrays are dense, row-major, with the layouts stated per argument.
 *   Request r, draft position k (1-based) lives at index [r][k-1].
 * - `stream` is a cudaStream_t (NULL = legacy default stream).  All calls only
 *   enqueue work and return; none synchronises.  Results are ready when the
 *   stream reaches them.
 * - Randomness is Philox4x32-10 (Salmon et al., SC'11), keyed by the 64-bit
 *   `seed` (key = (seed & 0xffffffff, seed >> 32)).  The draw for
 *   (request r, position p, purpose q, index v) uses counter
 *   (v >> 2, p, r, q) and output word (v & 3).  Purposes: DRAFT = 0 (draft
 *   Gumbel noise of vocab id v, p = k), ACCEPT = 1 (accept uniform, p = j,
 *   v = 0), RESAMPLE = 2 (residual or bonus Gumbel noise of vocab id v,
 *   p = row), DRAFT_GROUP = 3 and RESAMPLE_GROUP = 4 (the same for group
 *   index v).  A word w maps to u = (2 (w >> 9) + 1) 2^-24 in (0,1); Gumbel
 *   noise is G = -ln(-ln u).
 * - Every token draw is a two-level Gumbel-max over log-weights lw(v): the
 *   vocabulary is cut into groups of 32 consecutive ids (group j = ids
 *   32j .. 32j+31, the last one shorter when V % 32 != 0); the group is
 *   j* = argmax_j L_j + G(.., *_GROUP, j) with L_j = log sum_{v in j} e^{lw(v)},
 *   then the token is argmax_{v in j*} lw(v) + G(.., v).  This samples
 *   p(v) = e^{lw(v)} / sum_u e^{lw(u)} exactly, like one Gumbel-max over all
 *   ids, with one random word per group plus 32 for the chosen group.  Keys
 *   are compared in fp32; ties go to the lowest group and the lowest id.
 * - Return value: a dspark_status.  Host-side argument errors are returned
 *   before anything is enqueued.  Errors found on the device (bad token ids,
 *   l_r outside [0, gamma], confidence outside [0,1]) set bits in a status
 *   word at the start of the call's workspace; the kernels clamp the bad value
 *   and finish.  dspark_read_device_status() reads that word.
 *
 * Limits: 1 <= R, 1 <= gamma <= 64, 8 <= V < 2^31 with V % 8 == 0,
 *   R * gamma <= 16384 for dspark_schedule, 16 <= r <= 256 with r % 16 == 0
 *   (r % 64 == 0 for BF16), 0 < temperature < inf.  Beyond these:
 *   DSPARK_ERR_UNSUPPORTED.
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DSPARK_OK = 0,
  DSPARK_ERR_INVALID_ARG = 1,  /* NULL pointer, non-positive size, bad temperature, bad dtype */
  DSPARK_ERR_UNSUPPORTED = 2,  /* outside the limits above */
  DSPARK_ERR_WORKSPACE = 3,    /* workspace NULL or smaller than the *_workspace_bytes query */
  DSPARK_ERR_CUDA = 4,         /* a CUDA launch or runtime call failed: dspark_last_error() */
  DSPARK_ERR_DEVICE_INPUT = 5, /* (device status) an input value was out of range */
  DSPARK_ERR_TIMEOUT = 6       /* (device status) a bounded device-side wait gave up */
} dspark_status;

typedef enum { DSPARK_F32 = 0, DSPARK_BF16 = 1 } dspark_dtype;

enum {
  DSPARK_PURPOSE_DRAFT = 0,
  DSPARK_PURPOSE_ACCEPT = 1,
  DSPARK_PURPOSE_RESAMPLE = 2,
  DSPARK_PURPOSE_DRAFT_GROUP = 3,
  DSPARK_PURPOSE_RESAMPLE_GROUP = 4
};
/* Ids per group of the two-level Gumbel-max draw. */
enum { DSPARK_GROUP = 32 };

/* Device status word bits (OR-ed together).  DSPARK_DEV_TIMEOUT: a bounded
 * device-side wait gave up (the tensor-core draft's pipeline barriers; the
 * verify draw's wait for its bulk copy of a target row); the outputs of that
 * call are then not valid, and the context stays usable. */
enum { DSPARK_DEV_BAD_INPUT = 1, DSPARK_DEV_TIMEOUT = 2 };

/* Text of a status code; static storage. */
const char* dspark_status_string(int status);
/* Text of the last CUDA error seen by this thread's calls (empty if none). */
const char* dspark_last_error(void);
/* 10000 * major + 100 * minor + patch. */
int dspark_version(void);

/* ------------------------------------------------------------------------
 * dspark_draft_sample -- semi-autoregressive draft ([summary] §3.1; [notes]
 * "DSpark 핵심 기술 1").  For k = 1..gamma, left to right, for every request r:
 *   B_k     = W1[x_{k-1}] W2               (x_0 = x0[r]; one [R x r] x [r x V]
 *                                           contraction per k, fp32 accumulate)
 *   s_k(v)  = (U_k(v) + B_k(v)) / T         -> scores[r][k-1][v]
 *   lse_k   = log sum_v exp(s_k(v))         -> lse[r][k-1]
 *   x_k     = two-level Gumbel-max over lw = s_k, stream (seed, r, k, DRAFT_GROUP
 *             / DRAFT)                       -> x[r][k-1]
 *   logp_k  = s_k(x_k) - lse_k              -> logp[r][k-1]
 * so p^d_k(v) = exp(scores - lse) is the locally normalised draft
 * distribution that verification needs.
 *
 * U       [R, gamma, V]  dtype      backbone logits
 * W1      [V, r]         dtype      Markov head, first factor
 * W2      [r, V]         dtype      Markov head, second factor
 * x0      [R]            int32      anchor token per request, in [0, V)
 * dtype   DSPARK_F32 (fp32 CUDA-core contraction) or DSPARK_BF16 (tensor cores)
 * x       [R, gamma]     int32      out
 * logp    [R, gamma]     float      out
 * lse     [R, gamma]     float      out
 * scores  [R, gamma, V]  float      out
 * workspace: >= dspark_draft_workspace_bytes(R, gamma, V, r, dtype) bytes,
 *   256-byte aligned.  Contents need no initialisation and are scratch.
 * U, W1, W2 and scores must be 16-byte aligned.
 * ---------------------------------------------------------------------- */
size_t dspark_draft_workspace_bytes(int R, int gamma, int V, int r, int dtype);
int dspark_draft_sample(const void* U, const void* W1, const void* W2, const int32_t* x0,
                        int dtype, int R, int gamma, int V, int r, float temperature,
                        uint64_t seed, int32_t* x, float* logp, float* lse, float* scores,
                        void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * dspark_transpose_w2 -- the Markov head's second factor in the layout the
 * tensor-core draft reads: W2T[v][a] = W2[a][v], so that each block of 128
 * vocabulary ids is one contiguous 128 x r block (K-major operand).  The bf16
 * dspark_draft_sample does this itself on every call (a read and a write of
 * r V bf16); a caller whose head weights stay fixed across rounds does it once
 * and passes W2T to dspark_draft_sample_w2t / dspark_draft_sample_rnn_w2t.
 *
 * W2   [r, V]  bf16   in;  W2T  [V, r]  bf16   out (caller-allocated)
 * r a multiple of 64, at most 256; V a multiple of 8 (else
 * DSPARK_ERR_UNSUPPORTED); W2 and W2T 16-byte aligned (else
 * DSPARK_ERR_INVALID_ARG).  Enqueued on `stream`; no host synchronisation.
 * ---------------------------------------------------------------------- */
int dspark_transpose_w2(const void* W2, int r, int V, void* W2T, void* stream);

/* dspark_draft_sample_w2t -- dspark_draft_sample, bf16, with the second factor
 * given as dspark_transpose_w2's W2T [V, r] instead of W2 [r, V]; the same
 * computation and outputs (bit for bit), without the per-call transpose.
 * Shapes the tensor-core draft does not take return DSPARK_ERR_UNSUPPORTED.
 * workspace: >= dspark_draft_workspace_bytes(R, gamma, V, r, DSPARK_BF16). */
int dspark_draft_sample_w2t(const void* U, const void* W1, const void* W2T, const int32_t* x0,
                            int R, int gamma, int V, int r, float temperature, uint64_t seed,
                            int32_t* x, float* logp, float* lse, float* scores, void* workspace,
                            size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * dspark_draft_sample_rnn -- the draft with the RNN head instead of the Markov
 * head ([summary] §3.1: the alternative sequential head keeps a state across
 * the block and also takes the backbone's hidden state).  Read as an Elman
 * recurrence in the Markov head's rank-r space:
 *   h_0 = 0,  h_k = tanh(W1[x_{k-1}] + h_{k-1} Wh + Q_k)   (fp32 state),
 *   B_k = bf16(h_k) W2                                       (bf16 contraction),
 * then s_k, lse_k, x_k, logp_k exactly as dspark_draft_sample.  With Wh = 0
 * and Q = 0 it is dspark_draft_sample with W1 replaced by bf16(tanh(W1)).
 *
 * Wh [r, r] bf16 (row a, column j: h_{k-1}[a]'s weight on h_k[j]);
 * Q  [R, gamma, r] float: the backbone hidden state of each position,
 *    projected into the head's space;
 * other arguments and outputs as dspark_draft_sample (bf16 only; r a multiple
 * of 64, at most 256; Wh and Q 16-byte aligned, else DSPARK_ERR_INVALID_ARG).
 * workspace: >= dspark_draft_rnn_workspace_bytes(R, gamma, V, r) bytes,
 *   256-byte aligned.
 * ---------------------------------------------------------------------- */
size_t dspark_draft_rnn_workspace_bytes(int R, int gamma, int V, int r);
int dspark_draft_sample_rnn(const void* U, const void* W1, const void* W2, const void* Wh,
                            const float* Q, const int32_t* x0, int dtype, int R, int gamma, int V,
                            int r, float temperature, uint64_t seed, int32_t* x, float* logp,
                            float* lse, float* scores, void* workspace, size_t workspace_bytes,
                            void* stream);
/* dspark_draft_sample_rnn_w2t -- dspark_draft_sample_rnn with W2 given as
 * dspark_transpose_w2's W2T [V, r] (bf16); same outputs, no per-call transpose.
 * workspace: >= dspark_draft_rnn_workspace_bytes(R, gamma, V, r). */
int dspark_draft_sample_rnn_w2t(const void* U, const void* W1, const void* W2T, const void* Wh,
                                const float* Q, const int32_t* x0, int R, int gamma, int V, int r,
                                float temperature, uint64_t seed, int32_t* x, float* logp,
                                float* lse, float* scores, void* workspace,
                                size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * dspark_schedule -- hardware-aware prefix scheduler, Algorithm 1
 * ([summary] §3.2.2).
 *   a_{r,j} = prod_{i<=j} c_{r,i}   (sequential fp32 product; c clamped to [0,1])
 *   Candidates (r, j) are sorted by a descending, ties by smaller j, then
 *   smaller r.  Start with l = 0, B = R, tau = R, Theta_0 = tau * sps[B].
 *   Taking candidate i: B += 1, tau += a_i, Theta_i = tau * sps[B]; stop at the
 *   first i with Theta_i <= Theta_{i-1}.  l_r = number of taken candidates of r.
 *   tau is kept exactly in 2^-48 fixed point (each a rounded to nearest, ties
 *   to even); the test Theta_i > Theta_{i-1} compares the exact products
 *   tau * sps[B] (no rounding).  diag's Theta* is ((double)tau * 2^-48) * sps[B*].
 *   Step rates must be positive and finite: others flag DSPARK_DEV_BAD_INPUT
 *   and count as no improvement.
 *
 * conf    [R, gamma]   float   predicted conditional acceptance c_{r,j}
 * sps     [sps_len]    double  measured step rate (steps/s) indexed by verify
 *                              batch size B; sps_len >= R * (1 + gamma) + 1
 * ell     [R]          int32   out: scheduled verify length l_r in [0, gamma]
 * diag    [4] double or NULL   out: B*, tau*, Theta*, number of taken candidates
 * workspace: >= dspark_schedule_workspace_bytes(R, gamma) bytes, 256-byte aligned
 *   (holds the R * gamma sorted candidates).
 * ---------------------------------------------------------------------- */
size_t dspark_schedule_workspace_bytes(int R, int gamma);
int dspark_schedule(const float* conf, const double* sps, int sps_len, int R, int gamma,
                    int32_t* ell, double* diag, void* workspace, size_t workspace_bytes,
                    void* stream);

/* ------------------------------------------------------------------------
 * Zero-overhead scheduling ([summary] §5.2).  The serving scheduler sets the
 * next capacity K from confidences two steps old and takes, among the current
 * candidates, the top K by current survival, so it never waits on this step's
 * scheduling; when K is predicted from the past, Algorithm 1's early stop is
 * left out, so that a throughput cliff of an irregular SPS curve does not trap
 * it at a local optimum.  Two calls:
 *
 * dspark_schedule_capacity -- K from conf_old: the candidates in Algorithm
 *   1's order (survival a descending, ties by smaller j, then smaller r),
 *   Theta_i = tau_i * sps[R + i] for i = 0 .. R gamma taken candidates (tau_i
 *   exact in 2^-48 fixed point, Theta compared exactly, as in
 *   dspark_schedule); K = the smallest i at which Theta_i is the maximum.
 *   K >= dspark_schedule's count, with equality when Theta is unimodal along
 *   the path.
 *   conf_old [R, gamma] float; sps as for dspark_schedule;
 *   K    [1] int32 (device)       out: the capacity
 *   diag [4] double or NULL       out: R + K, tau*, Theta*, K
 * dspark_schedule_topk -- l_r = number of candidates of request r among the
 *   first min(K, R gamma) of conf's order (K read from device memory, so it
 *   can come straight from dspark_schedule_capacity).  K < 0 flags
 *   DSPARK_DEV_BAD_INPUT and counts as 0.
 *   conf [R, gamma] float; K [1] int32 (device); ell [R] int32 out.
 * Both take a workspace of dspark_schedule_workspace_bytes(R, gamma) bytes
 * (256-byte aligned) and the limits of dspark_schedule.
 * ---------------------------------------------------------------------- */
int dspark_schedule_capacity(const float* conf_old, const double* sps, int sps_len, int R,
                             int gamma, int32_t* K, double* diag, void* workspace,
                             size_t workspace_bytes, void* stream);
int dspark_schedule_topk(const float* conf, const int32_t* K, int R, int gamma, int32_t* ell,
                         void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Sequential Temperature Scaling ([summary] §3.2.1) and the static-threshold
 * scheduler ([summary] §4.3.3).
 *
 * temper(c; T) = sigmoid(logit(c) / T) (0 and 1 stay, T = 1 returns c), in
 * fp32; calibrated survival ahat_{s,k} = prod_{i<=k} temper(c_{s,i}; T_i)
 * (fp64 product).
 *
 * dspark_sts_calibrate -- on held-out samples s = 0..N-1 with raw confidences
 *   conf [N, gamma] float and outcomes accept [N, gamma] uint8 (1 = position k
 *   accepted given its prefix accepted; the survival label is
 *   Y_{s,k} = prod_{i<=k} accept_{s,i}), a left-to-right 1-D grid search:
 *   for k = 1..gamma, with T_1..T_{k-1} fixed, T_k = the first entry of grid
 *   [G] (device, fp64, positive) with the smallest
 *     ECE_k = (1/N) sum_b | sum_{s in bin b} (ahat_{s,k} - Y_{s,k}) |,
 *   M equal-width bins on [0, 1], b = min(floor(ahat M), M - 1).  The bin
 *   sums are exact in 2^-40 fixed point, so each ECE is independent of the
 *   summation order.
 *   temps [gamma] double (device) out; ece [gamma] double (device) or NULL out.
 *   workspace: >= dspark_sts_workspace_bytes(N, G, M) bytes, 256-byte aligned.
 *   Limits: N <= 2^22, M <= 1024, gamma <= 64 (else DSPARK_ERR_UNSUPPORTED).
 * dspark_schedule_threshold -- l_r = the number of leading positions of
 *   request r whose survival prod_{i<=j} temper(c_{r,i}; T_i) is at least
 *   theta (temps [gamma] device, or NULL for the raw product of c).  The
 *   survival does not increase along a request, so the result is a prefix.
 *   conf [R, gamma] float; ell [R] int32 out.
 * ---------------------------------------------------------------------- */
size_t dspark_sts_workspace_bytes(int N, int G, int M);
int dspark_sts_calibrate(const float* conf, const uint8_t* accept, int N, int gamma,
                         const double* grid, int G, int M, double* temps, double* ece,
                         void* workspace, size_t workspace_bytes, void* stream);
int dspark_schedule_threshold(const float* conf, const double* temps, double theta, int R,
                              int gamma, int32_t* ell, void* stream);

/* ------------------------------------------------------------------------
 * dspark_verify -- standard rejection sampling over the scheduled prefixes
 * ([summary] opening bullets, §3; [notes] "배경") and the soft label
 * ([summary] §3.2.1).  With p^t_j = softmax(Z_j / T) and
 * p^d_j = exp(scores_j - lse_j), for every request r with l = ell[r]:
 *   c*_j = sum_v min(p^d_j(v), p^t_j(v))  (= 1 - 1/2 |p^d_j - p^t_j|_1), j <= l
 *   accept x_j (j = 1..l, in order) iff
 *     ln u_j < (Z_j[x_j]/T - LSE^t_j) - logp_j,  u_j = U01(seed, r, j, ACCEPT, 0)
 *   n = number of leading accepts.
 *   n < l : token drawn from norm(max(0, p^t_{n+1} - p^d_{n+1})): two-level
 *           Gumbel-max over lw = ln max(0, p^t - p^d) (-inf where zero), stream
 *           (seed, r, n+1, RESAMPLE_GROUP / RESAMPLE); if that residual is zero
 *           everywhere, over lw = Z_{n+1}/T instead
 *   n = l : bonus token: two-level Gumbel-max over lw = Z_{l+1}/T, stream
 *           (seed, r, l+1, RESAMPLE_GROUP / RESAMPLE)
 *   Emitted tokens: x_1..x_n, token; n_emit = n + 1.
 *
 * x, logp, lse, scores   the draft's outputs (layouts as in dspark_draft_sample)
 * Z       [R, gamma+1, V]  dtype  target logits at positions 1..gamma+1
 * ell     [R]              int32  verify lengths (dspark_schedule's output)
 * n_acc   [R]              int32  out: accepted draft tokens n
 * tokens  [R, gamma+1]     int32  out: emitted tokens, -1 after the n_emit-th
 * n_emit  [R]              int32  out: n + 1
 * cstar   [R, gamma]       float  out: c*_j for j <= l, NaN for j > l
 * lse_t   [R, gamma+1] float or NULL  out: LSE^t_j for j <= l, NaN otherwise
 * workspace: >= dspark_verify_workspace_bytes(R, gamma, V) bytes.
 * Z and scores must be 16-byte aligned.
 * ---------------------------------------------------------------------- */
size_t dspark_verify_workspace_bytes(int R, int gamma, int V);
int dspark_verify(const int32_t* x, const float* logp, const float* lse, const float* scores,
                  const void* Z, int dtype, const int32_t* ell, int R, int gamma, int V,
                  float temperature, uint64_t seed, int32_t* n_acc, int32_t* tokens,
                  int32_t* n_emit, float* cstar, float* lse_t, void* workspace,
                  size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * dspark_verify_packed -- dspark_verify over a packed target-logit buffer.
 * A serving engine that lets each request verify a different length runs its
 * target on the concatenated rows of all requests ([summary] §5.3: tokens of
 * the requests are laid out flat, with sequence boundaries passed alongside,
 * to avoid padding), so its target logits come packed: request r occupies
 * rows row_offsets[r] .. row_offsets[r] + l_r of Zp (positions 1 .. l_r + 1;
 * rows beyond l_r + 1 up to row_offsets[r + 1] may exist and are not read).
 * Same arithmetic, outputs and workspace as dspark_verify; only the target
 * rows are addressed through the offsets.
 *
 * Zp          [n_rows, V] bf16 or fp32, 16-byte aligned
 * row_offsets [R + 1]     int32 (device), non-decreasing,
 *                         row_offsets[r + 1] - row_offsets[r] >= 1 + l_r,
 *                         row_offsets[R] <= n_rows
 * n_rows      rows of Zp (>= R).  Offsets that break these rules flag
 *             DSPARK_DEV_BAD_INPUT; every row index is clamped into Zp.
 * ---------------------------------------------------------------------- */
int dspark_verify_packed(const int32_t* x, const float* logp, const float* lse,
                         const float* scores, const void* Zp, int dtype, const int32_t* row_offsets,
                         int n_rows, const int32_t* ell, int R, int gamma, int V,
                         float temperature, uint64_t seed, int32_t* n_acc, int32_t* tokens,
                         int32_t* n_emit, float* cstar, float* lse_t, void* workspace,
                         size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * dspark_verify_noalloc -- dspark_verify for callers that cannot allocate
 * device memory.  The paper has no counterpart; this is a deployment aid.
 *
 * Some callers have no way to obtain a device buffer at the point where they
 * verify: an engine that carves all of its device memory into fixed pools at
 * start-up and has none left to hand out, or code running where a cudaMalloc
 * would synchronise the device in the middle of a serving round.  This entry
 * point takes the same inputs and outputs as dspark_verify (caller-owned,
 * same layouts and meaning) but no workspace: its scratch (the status word,
 * LSE^t of every row, the accept flags and the per-chunk partials of the
 * drawn token, the list of scheduled rows) lives in a file-scope device array
 * of DSPARK_VERIFY_NOALLOC_SCRATCH_BYTES bytes that every GPU which loads the
 * library holds until the process exits.
 *
 * - Size limit: dspark_verify_workspace_bytes(R, gamma, V) =
 *   256 + align256(4 R (gamma+1)) + 2 align256(4 R gamma)
 *   + align256(8 R ceil(V / 16384)) bytes must fit in the array (with
 *   gamma = 16 and V = 151,936 that is R <= 15,194); larger
 *   problems return DSPARK_ERR_UNSUPPORTED, with the reason in
 *   dspark_last_error(), before anything is enqueued.
 * - The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current) and caches it together
 *   with the id of the current context; make that first call before any
 *   stream capture.  After cudaDeviceReset (a new primary context, where the
 *   module may load elsewhere) the next call sees a new context id and looks
 *   the address up again: make that call outside stream capture too.
 * - It allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 * - Every call shares the one array, which keeps the previous call's
 *   contents; the call clears the status word itself.  Calls whose work
 *   overlaps on the GPU (other streams, or the same array from other host
 *   threads) race on the array: serialise them.
 * - Device-side input errors are clamped as in dspark_verify; their status
 *   word is internal to the array and not reported.
 * ---------------------------------------------------------------------- */
#define DSPARK_VERIFY_NOALLOC_SCRATCH_BYTES (4u << 20)
int dspark_verify_noalloc(const int32_t* x, const float* logp, const float* lse,
                          const float* scores, const void* Z, int dtype, const int32_t* ell, int R,
                          int gamma, int V, float temperature, uint64_t seed, int32_t* n_acc,
                          int32_t* tokens, int32_t* n_emit, float* cstar, float* lse_t,
                          void* stream);

/* Copies the device status word of `workspace` (as written by the last call
 * that used it) to *out after synchronising `stream`.  *out is a HOST pointer.
 * Returns DSPARK_OK, or DSPARK_ERR_CUDA if the copy failed. */
int dspark_read_device_status(const void* workspace, void* stream, int32_t* out);

/* ========================================================================
 * Diagnostics and measurement aids.  Not part of the method and outside the
 * draft -> schedule -> verify contract: a caller of the path needs none of
 * them.  They exist for benchmarks and for testing the library's own error
 * paths, and make the same ownership promises (no allocation, caller buffers).
 * ======================================================================== */

/* ------------------------------------------------------------------------
 * Optional per-kernel timing (for benchmarks; not thread-safe).
 * dspark_profile_start() makes every later kernel launch of this library be
 * bracketed by two CUDA events recorded on the launch's own stream (the first
 * call creates 16384 events; no device memory).  dspark_profile_stop()
 * synchronises on the last event and returns, per kernel kind, the summed
 * event-timed milliseconds and the launch count (each may be NULL), plus how
 * many launches were timed (at most 8192 per start/stop window; the launch
 * counts keep counting beyond that).
 * ---------------------------------------------------------------------- */
enum {
  DSPARK_KERNEL_PREPARE = 0,        /* draft set-up: W2 transpose (bf16) or anchor gather (fp32) */
  DSPARK_KERNEL_DRAFT_TILE = 1,     /* draft contraction + fused epilogue (gamma launches) */
  DSPARK_KERNEL_DRAFT_COMBINE = 2,  /* per-row combine + next gather (gamma launches) */
  DSPARK_KERNEL_SCHEDULE = 3,
  DSPARK_KERNEL_VERIFY_ROWS = 4,
  DSPARK_KERNEL_VERIFY_DRAW = 5,    /* stage 1 of the residual / bonus draw */
  DSPARK_KERNEL_RNN_STATE = 6,      /* RNN head: state update (gamma launches) */
  DSPARK_KERNEL_VERIFY_EMIT = 7,    /* stage 2 of the draw, emitted tokens */
  DSPARK_KERNEL_KINDS = 8
};
int dspark_profile_start(void);
int dspark_profile_stop(double* ms_by_kind, int* launches_by_kind, int* timed_launches);

/* ------------------------------------------------------------------------
 * dspark_stream_probe -- a bandwidth probe: out[i] = (float)in[i] for n bf16
 * values, streamed contiguously in 16-byte pieces.  It moves the draft step's
 * traffic mix (2 bytes read, 4 written per element) without the draft's
 * access pattern, so its bandwidth is a ceiling for that mix on this GPU.
 * in (bf16) and out (float) are device pointers, 16-byte aligned, not
 * overlapping; n % 8 == 0 (else DSPARK_ERR_INVALID_ARG).
 * ---------------------------------------------------------------------- */
int dspark_stream_probe(const void* in, float* out, size_t n, void* stream);

/* ------------------------------------------------------------------------
 * dspark_selftest_draft_timeout -- exercises the tensor-core draft's bounded
 * device waits.  It enqueues draft step k = 1 of dspark_draft_sample (bf16,
 * temperature 1, seed 0) with the W2 operand loads withheld, so that the
 * contraction's wait for its first operand chunk can never complete, and with
 * every device wait limited to wait_cycles SM clocks (1000 .. 4e9; the
 * library's own limit is 4e9, about 2 s).  The kernel then gives up: the role
 * that timed out raises the CTA's abort flag, the others see it, every copy
 * already issued is waited for (also bounded), tensor memory is freed, and
 * DSPARK_DEV_TIMEOUT is set in the status word of `workspace`.  The context
 * stays usable.  Arguments, layouts and workspace as dspark_draft_sample
 * (dtype bf16, r a multiple of 64); x, logp, lse and scores receive
 * unspecified values.
 * ---------------------------------------------------------------------- */
int dspark_selftest_draft_timeout(const void* U, const void* W1, const void* W2,
                                  const int32_t* x0, int R, int gamma, int V, int r,
                                  long long wait_cycles, int32_t* x, float* logp, float* lse,
                                  float* scores, void* workspace, size_t workspace_bytes,
                                  void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H */
