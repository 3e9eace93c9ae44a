/*
 * dspark_oracle.c -- plain, slow CPU oracle for the DSpark per-round sampling path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * loads this file.  It is used by tests/, by __graft_entry__.smoke() and by
 * the cpu_baseline / reference leg of bench.py.  It shares no code, header,
 * table or helper with the CUDA path under speculative_decoding_draft_05_gb300/csrc.
 *
 * Everything is written as plain loops in double precision, in the order the
 * pages state the method.  The few places where a floating-point value decides
 * an integer (a Gumbel argmax, the accept test, the scheduler's stop test)
 * take that decision in the kernel's precision (fp32 keys, fixed-point tau,
 * fp64 theta), as the comments say at each place.
 *
 * Sources (page title, section):
 *   [P1] "DSpark: Confidence-Scheduled Speculative Decoding with Semi-Autoregressive
 *        Generation 요약 설명" (greeksharifa.github.io): summary bullets (standard
 *        rejection sampling preserves the target distribution), §3 (latency
 *        L = (T_draft + T_verify)/tau, tau includes the bonus token), §3.1 (local
 *        normalisation, Markov head B = W1 W2 conditioned on the previous token,
 *        left-to-right sampling), §3.2.1 (soft label c* = 1 - 1/2 |p^d - p^t|_1),
 *        §3.2.2 (prefix survival, B, tau, Theta, Algorithm 1), Appendix A.
 *   [P2] "DSpark: Confidence-Scheduled Speculative Decoding with Semi-Autoregressive
 *        Generation" (notes-ybman-uk.pages.dev): "DSpark 핵심 기술 1" -- the draft
 *        distribution p_k(v | x0, x<k) = softmax(U_k(v) + B_k(x0, x<k, v));
 *        "배경" -- accept the longest prefix by rejection sampling.
 *   Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy
 *        as 1, 2, 3", SC'11.
 *   Rejection rule (the textbook form the pages call "standard rejection
 *        sampling"): Leviathan, Kalman, Matias, "Fast Inference from Transformers
 *        via Speculative Decoding", ICML 2023; Chen et al., "Accelerating Large
 *        Language Model Decoding with Speculative Sampling", 2023.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_PURPOSE_DRAFT 0u
#define ORACLE_PURPOSE_ACCEPT 1u
#define ORACLE_PURPOSE_RESAMPLE 2u
#define ORACLE_PURPOSE_DRAFT_GROUP 3u
#define ORACLE_PURPOSE_RESAMPLE_GROUP 4u
#define ORACLE_GROUP 32

/* ------------------------------------------------------------------------- */
/* Philox4x32-10 (SC'11).  One round maps (c0,c1,c2,c3) with key (k0,k1) to   */
/* (hi(M1*c2)^c1^k0, lo(M1*c2), hi(M0*c0)^c3^k1, lo(M0*c0)); the key is       */
/* bumped by the Weyl constants (W0,W1) before every round after the first.  */
/* ------------------------------------------------------------------------- */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += W0;
      k1 += W1;
    }
    uint64_t p0 = (uint64_t)M0 * (uint64_t)c0;
    uint64_t p1 = (uint64_t)M1 * (uint64_t)c2;
    uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
    uint32_t n1 = (uint32_t)p1;
    uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
    uint32_t n3 = (uint32_t)p0;
    c0 = n0;
    c1 = n1;
    c2 = n2;
    c3 = n3;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

/* The random word for (seed, request, position, purpose, vocab id):
 * counter = (v >> 2, position, request, purpose), key = (seed lo, seed hi),
 * and the word is output number (v & 3). */
uint32_t oracle_rng_word(uint64_t seed, uint32_t request, uint32_t position, uint32_t purpose,
                         uint32_t v) {
  uint32_t ctr[4] = {v >> 2, position, request, purpose};
  uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
  uint32_t out[4];
  oracle_philox4x32_10(ctr, key, out);
  return out[v & 3u];
}

/* Uniform on the open interval (0,1): u = (2*(w >> 9) + 1) * 2^-24.  Never 0
 * or 1, and exactly representable in fp32 as well as fp64. */
double oracle_uniform(uint32_t w) { return ((double)(w >> 9) * 2.0 + 1.0) * 0x1p-24; }

/* Standard Gumbel variate G = -ln(-ln u). */
double oracle_gumbel(uint32_t w) { return -log(-log(oracle_uniform(w))); }

/* ------------------------------------------------------------------------- */
/* Markov head bias, [P1] §3.1: B = W1 W2 of rank r, conditioned on the       */
/* immediately previous token: B(v) = sum_i W1[prev, i] * W2[i, v].           */
/* ------------------------------------------------------------------------- */
void oracle_markov_bias(const double* W1, const double* W2, int V, int r, int32_t prev,
                        double* out /* [V] */) {
  for (int v = 0; v < V; ++v) out[v] = 0.0;
  const double* w1row = W1 + (size_t)prev * r;
  for (int i = 0; i < r; ++i) {
    const double a = w1row[i];
    const double* w2row = W2 + (size_t)i * V;
    for (int v = 0; v < V; ++v) out[v] += a * w2row[v];
  }
}

void oracle_markov_bias_rows(const double* W1, const double* W2, int V, int r, const int32_t* prev,
                             int n, double* out /* [n, V] */) {
  for (int i = 0; i < n; ++i) oracle_markov_bias(W1, W2, V, r, prev[i], out + (size_t)i * V);
}

/* log(sum_v exp(x_v)) with the maximum taken out first. */
static double logsumexp(const double* x, int n) {
  double m = -INFINITY;
  for (int i = 0; i < n; ++i)
    if (x[i] > m) m = x[i];
  double s = 0.0;
  for (int i = 0; i < n; ++i) s += exp(x[i] - m);
  return m + log(s);
}

/* argmax of fp32-rounded keys, lowest index on ties; also the fp64 gap between
 * the chosen key and the best other key (the decision's margin). */
static int argmax_fp32(const double* key, int n, double* margin) {
  int best = -1;
  float bf = -INFINITY;
  for (int v = 0; v < n; ++v) {
    if (isnan(key[v])) continue;
    float f = (float)key[v];
    if (best < 0 || f > bf) {
      bf = f;
      best = v;
    }
  }
  if (margin) {
    double other = -INFINITY;
    for (int v = 0; v < n; ++v)
      if (v != best && !isnan(key[v]) && key[v] > other) other = key[v];
    *margin = (best >= 0) ? key[best] - other : 0.0;
  }
  return best;
}

/* ------------------------------------------------------------------------- */
/* Draft step, [P1] §3.1 and [P2] "DSpark 핵심 기술 1":                         */
/*   for k = 1..gamma (left to right):                                        */
/*     s_k(v)  = (U_k(v) + B_k(v)) / T,   B_k = W1[x_{k-1}] W2, x_0 = anchor   */
/*     lse_k   = log sum_v exp(s_k(v))    (local normalisation)                */
/*     x_k     = argmax_v s_k(v) + G(seed, request, k, DRAFT, v)  (Gumbel-max) */
/*     logp_k  = s_k(x_k) - lse_k                                             */
/* The argmax compares fp32-rounded keys (the kernel's precision).            */
/* ------------------------------------------------------------------------- */
typedef struct {
  int n_req, gamma, V, r;
  double T;
  uint64_t seed;
  const int32_t* req_ids;
  const double *U, *W1, *W2;
  const int32_t* x0;
  int32_t* x;
  double *logp, *lse, *scores, *margin;
} draft_job;

/* One draft position k of request i, shared by both heads: s holds the bias */
/* B_k on entry and the scores s_k = (U_k + B_k) / T on return; the token is  */
/* the Gumbel argmax of s_k, its log-probability s_k[x] - lse(s_k).           */
/* ------------------------------------------------------------------------- */
/* Two-level Gumbel-max: draw v with probability proportional to e^{lw[v]}    */
/* (lw[v] = -inf for weight zero).  The ids are cut into groups of 32         */
/* consecutive ids (the last one possibly shorter).  Stage 1 draws a group j  */
/* by Gumbel-max over the groups' log-masses                                  */
/*   L_j = log sum_{v in j} e^{lw[v]},  key_j = L_j + G(seed, req, pos, pg, j); */
/* stage 2 draws v inside that group by Gumbel-max over                       */
/*   lw[v] + G(seed, req, pos, pe, v).                                        */
/* P(v) = P(group of v) P(v | group) = (e^{L_j} / sum_i e^{L_i}) (e^{lw[v]} /  */
/* e^{L_j}) = e^{lw[v]} / sum_u e^{lw[u]}: the same law as one Gumbel-max over */
/* all ids.  Both argmaxes decide on fp32-rounded keys, ties to the lowest id. */
/* margin = the smaller of the two stages' top-1 minus top-2 key gaps.        */
/* gkey holds ceil(V/32) doubles.  Returns -1 if every weight is zero.        */
/* ------------------------------------------------------------------------- */
static int two_level_argmax(const double* lw, int V, uint64_t seed, uint32_t req, uint32_t pos,
                            uint32_t pg, uint32_t pe, double* gkey, double* margin) {
  const int ng = (V + ORACLE_GROUP - 1) / ORACLE_GROUP;
  for (int j = 0; j < ng; ++j) {
    const int a = j * ORACLE_GROUP, b = (a + ORACLE_GROUP < V) ? a + ORACLE_GROUP : V;
    double m = -INFINITY;
    for (int v = a; v < b; ++v)
      if (lw[v] > m) m = lw[v];
    if (m == -INFINITY) {
      gkey[j] = NAN; /* no weight in this group: it cannot be drawn */
      continue;
    }
    double t = 0.0;
    for (int v = a; v < b; ++v) t += exp(lw[v] - m);
    gkey[j] = (m + log(t)) + oracle_gumbel(oracle_rng_word(seed, req, pos, pg, (uint32_t)j));
  }
  double m1 = 0.0, m2 = 0.0;
  const int j = argmax_fp32(gkey, ng, &m1);
  if (j < 0) {
    if (margin) *margin = 0.0;
    return -1;
  }
  const int a = j * ORACLE_GROUP, n = ((a + ORACLE_GROUP < V) ? a + ORACLE_GROUP : V) - a;
  double ekey[ORACLE_GROUP];
  for (int t = 0; t < n; ++t)
    ekey[t] = (lw[a + t] == -INFINITY)
                  ? NAN
                  : lw[a + t] + oracle_gumbel(oracle_rng_word(seed, req, pos, pe, (uint32_t)(a + t)));
  const int t = argmax_fp32(ekey, n, &m2);
  if (margin) *margin = m1 < m2 ? m1 : m2;
  return a + t;
}

static int32_t draft_sample(const draft_job* J, int i, int k, double* s, double* key) {
  const int g = J->gamma, V = J->V;
  const uint32_t req = (uint32_t)J->req_ids[i];
  const double* Uk = J->U + ((size_t)i * g + (k - 1)) * V;
  for (int v = 0; v < V; ++v) s[v] = (Uk[v] + s[v]) / J->T;
  const double lse = logsumexp(s, V);
  /* x_k ~ softmax(s): two-level Gumbel-max over the scores */
  double margin = 0.0;
  const int xk = two_level_argmax(s, V, J->seed, req, (uint32_t)k, ORACLE_PURPOSE_DRAFT_GROUP,
                                  ORACLE_PURPOSE_DRAFT, key, &margin);
  const size_t o = (size_t)i * g + (k - 1);
  J->x[o] = xk;
  J->logp[o] = s[xk] - lse;
  J->lse[o] = lse;
  if (J->margin) J->margin[o] = margin;
  if (J->scores) memcpy(J->scores + o * V, s, sizeof(double) * (size_t)V);
  return xk;
}

static void draft_one(const draft_job* J, int i, double* s, double* key) {
  int32_t prev = J->x0[i];
  for (int k = 1; k <= J->gamma; ++k) {
    oracle_markov_bias(J->W1, J->W2, J->V, J->r, prev, s);
    prev = draft_sample(J, i, k, s, key);
  }
}

/* ------------------------------------------------------------------------- */
/* RNN head, [P1] §3.1: the alternative sequential head keeps a state across */
/* the block and also takes the backbone's hidden state.  Reading: an Elman  */
/* recurrence in the Markov head's rank-r space,                              */
/*   h_0 = 0,  h_k = tanh(W1[x_{k-1}] + h_{k-1} Wh + Q_k),  B_k = h_k W2,     */
/* with Q_k [r] the backbone hidden state of position k projected into the   */
/* head (an input) and Wh [r, r].  The state is exact (fp64 here); the       */
/* contraction takes it rounded to bf16 (nearest, ties to even), like every  */
/* operand of the bf16 contraction.  Everything else is the Markov draft.    */
/* ------------------------------------------------------------------------- */
double oracle_round_bf16(double v) {
  if (!isfinite(v) || v == 0.0) return v;
  int e;
  const double f = frexp(v, &e);            /* v = f 2^e, |f| in [0.5, 1) */
  const double q = nearbyint(ldexp(f, 8));  /* 8 significant bits: |q| in [128, 256] */
  return ldexp(q, e - 8);
}

static void draft_rnn_one(const draft_job* J, const double* Wh, const double* Q, double* hstate,
                          int i, double* s, double* key) {
  const int g = J->gamma, V = J->V, r = J->r;
  int32_t prev = J->x0[i];
  double* h = (double*)calloc((size_t)r, sizeof(double));
  double* hn = (double*)malloc(sizeof(double) * (size_t)r);
  double* A = (double*)malloc(sizeof(double) * (size_t)r);
  for (int k = 1; k <= g; ++k) {
    const double* Qk = Q + ((size_t)i * g + (k - 1)) * r;
    for (int j = 0; j < r; ++j) {
      double z = J->W1[(size_t)prev * r + j] + Qk[j];
      for (int a = 0; a < r; ++a) z += h[a] * Wh[(size_t)a * r + j];
      hn[j] = tanh(z);
    }
    for (int j = 0; j < r; ++j) {
      h[j] = hn[j];
      A[j] = oracle_round_bf16(hn[j]);
    }
    if (hstate) memcpy(hstate + ((size_t)i * g + (k - 1)) * r, h, sizeof(double) * (size_t)r);
    for (int v = 0; v < V; ++v) s[v] = 0.0;
    for (int a = 0; a < r; ++a) {
      const double* w2row = J->W2 + (size_t)a * V;
      for (int v = 0; v < V; ++v) s[v] += A[a] * w2row[v];
    }
    prev = draft_sample(J, i, k, s, key);
  }
  free(h);
  free(hn);
  free(A);
}

typedef struct {
  draft_job base;
  const double *Wh, *Q;
  double* hstate;  // optional [n_req, gamma, r]: the state h_k of every step
} draft_rnn_job;

typedef struct {
  const void* job;
  int n, nthreads, tid;
  void (*fn)(const void*, int, double*, double*);
  size_t scratch;
} worker_arg;

static void* worker(void* p) {
  worker_arg* w = (worker_arg*)p;
  double* a = (double*)malloc(sizeof(double) * w->scratch);
  double* b = (double*)malloc(sizeof(double) * w->scratch);
  for (int i = w->tid; i < w->n; i += w->nthreads) w->fn(w->job, i, a, b);
  free(a);
  free(b);
  return NULL;
}

static void run_parallel(const void* job, int n, int nthreads, size_t scratch,
                         void (*fn)(const void*, int, double*, double*)) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > n) nthreads = n > 0 ? n : 1;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * nthreads);
  worker_arg* args = (worker_arg*)malloc(sizeof(worker_arg) * nthreads);
  for (int t = 0; t < nthreads; ++t) {
    args[t].job = job;
    args[t].n = n;
    args[t].nthreads = nthreads;
    args[t].tid = t;
    args[t].fn = fn;
    args[t].scratch = scratch;
    pthread_create(&th[t], NULL, worker, &args[t]);
  }
  for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
  free(th);
  free(args);
}

static void draft_fn(const void* job, int i, double* a, double* b) {
  draft_one((const draft_job*)job, i, a, b);
}

static void draft_rnn_fn(const void* job, int i, double* a, double* b) {
  const draft_rnn_job* J = (const draft_rnn_job*)job;
  draft_rnn_one(&J->base, J->Wh, J->Q, J->hstate, i, a, b);
}

int oracle_draft_rnn(int n_req, const int32_t* req_ids, int gamma, int V, int r, double T,
                     uint64_t seed, const double* U, const double* W1, const double* W2,
                     const double* Wh, const double* Q, const int32_t* x0, int32_t* x, double* logp,
                     double* lse, double* scores, double* margin, double* hstate, int nthreads) {
  if (n_req < 0 || gamma < 1 || V < 1 || r < 1 || !(T > 0.0)) return 1;
  for (int i = 0; i < n_req; ++i)
    if (x0[i] < 0 || x0[i] >= V) return 2;
  draft_rnn_job J = {{n_req, gamma, V, r, T, seed, req_ids, U, W1, W2, x0, x, logp, lse, scores,
                      margin},
                     Wh, Q, hstate};
  run_parallel(&J, n_req, nthreads, (size_t)V, draft_rnn_fn);
  return 0;
}

int oracle_draft(int n_req, const int32_t* req_ids, int gamma, int V, int r, double T,
                 uint64_t seed, const double* U, const double* W1, const double* W2,
                 const int32_t* x0, int32_t* x, double* logp, double* lse, double* scores,
                 double* margin, int nthreads) {
  if (n_req < 0 || gamma < 1 || V < 1 || r < 1 || !(T > 0.0)) return 1;
  for (int i = 0; i < n_req; ++i)
    if (x0[i] < 0 || x0[i] >= V) return 2;
  draft_job J = {n_req, gamma, V, r, T, seed, req_ids, U, W1, W2, x0, x, logp, lse, scores, margin};
  run_parallel(&J, n_req, nthreads, (size_t)V, draft_fn);
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Hardware-aware prefix scheduler, [P1] §3.2.2 (Algorithm 1):                */
/*   a_{r,j} = prod_{i<=j} c_{r,i}; candidates sorted by survival (ties:      */
/*   smaller j, then smaller r); start with l = 0 for all, B = R, tau = R,    */
/*   Theta_0 = tau * SPS(B); take candidates in order, B += 1, tau += a,      */
/*   Theta = tau * SPS(B); stop at the first candidate whose Theta does not   */
/*   strictly improve; l_r = number of taken candidates of request r.         */
/* Precision (the kernel's, since these values decide integers): a is the    */
/* sequential fp32 product; tau is held exactly in 2^-48 fixed point, each a */
/* rounded to nearest (ties to even); the stop test compares the exact       */
/* products tau_i * SPS[B_i] and tau_{i-1} * SPS[B_{i-1}] (no rounding), the */
/* plain reading of "Theta does not improve".  The reported Theta* is the    */
/* fp64 value ((double)tau_fixed * 2^-48) * SPS[B].                          */
/* ------------------------------------------------------------------------- */
typedef struct {
  float a;
  int j, r;
} cand;

/* Exact comparison of t_a * s_a > t_b * s_b for t > 0 (integers) and s > 0
 * (finite doubles): s = m 2^e with an integer m < 2^53, so each product is a
 * 117-bit integer times a power of two; compare leading-bit positions, then
 * the aligned integers. */
static int bitlen128(unsigned __int128 x) {
  int n = 0;
  while (x) {
    ++n;
    x >>= 1;
  }
  return n;
}

static int exact_greater(int64_t ta, double sa, int64_t tb, double sb) {
  int ea, eb;
  const double fa = frexp(sa, &ea), fb = frexp(sb, &eb); /* s = f 2^e, f in [0.5, 1) */
  const unsigned __int128 pa = (unsigned __int128)(uint64_t)ta * (uint64_t)ldexp(fa, 53);
  const unsigned __int128 pb = (unsigned __int128)(uint64_t)tb * (uint64_t)ldexp(fb, 53);
  const int la = bitlen128(pa) + ea, lb = bitlen128(pb) + eb;
  if (la != lb) return la > lb;
  const int da = bitlen128(pa), db = bitlen128(pb);
  const unsigned __int128 xa = da < db ? pa << (db - da) : pa;
  const unsigned __int128 xb = db < da ? pb << (da - db) : pb;
  return xa > xb;
}

static int cand_cmp(const void* pa, const void* pb) {
  const cand* x = (const cand*)pa;
  const cand* y = (const cand*)pb;
  if (x->a > y->a) return -1;
  if (x->a < y->a) return 1;
  if (x->j != y->j) return x->j < y->j ? -1 : 1;
  if (x->r != y->r) return x->r < y->r ? -1 : 1;
  return 0;
}

/* The candidates (r, j) with their survivals, sorted (a descending, ties by
 * smaller j, then smaller r); a_out (may be NULL) receives a. */
static cand* sorted_candidates(int R, int gamma, const float* c, float* a_out) {
  const int n = R * gamma;
  cand* cs = (cand*)malloc(sizeof(cand) * (size_t)n);
  for (int r = 0; r < R; ++r) {
    float a = 1.0f;
    for (int j = 0; j < gamma; ++j) {
      float cj = c[(size_t)r * gamma + j];
      if (!(cj >= 0.0f)) cj = 0.0f; /* NaN or negative: no survival */
      if (cj > 1.0f) cj = 1.0f;
      a = (j == 0) ? cj : a * cj;
      float av = a;
      if (av == 0.0f) av = 0.0f; /* canonical +0 */
      cs[(size_t)r * gamma + j].a = av;
      cs[(size_t)r * gamma + j].j = j;
      cs[(size_t)r * gamma + j].r = r;
      if (a_out) a_out[(size_t)r * gamma + j] = av;
    }
  }
  qsort(cs, (size_t)n, sizeof(cand), cand_cmp);
  return cs;
}

static int rates_ok(int R, int gamma, const double* sps) {
  for (int b = R; b <= R * (1 + gamma); ++b)
    if (!(sps[b] > 0.0) || !isfinite(sps[b])) return 0; /* step rates must be positive */
  return 1;
}

int oracle_schedule(int R, int gamma, const float* c, const double* sps, int sps_len, int32_t* ell,
                    double* diag /* [4]: B*, tau*, Theta*, n* (may be NULL) */,
                    float* a_out /* [R, gamma] (may be NULL) */) {
  if (R < 1 || gamma < 1) return 1;
  if (sps_len < R * (1 + gamma) + 1) return 1;
  const int n = R * gamma;
  cand* cs = sorted_candidates(R, gamma, c, a_out);
  for (int r = 0; r < R; ++r) ell[r] = 0;
  if (!rates_ok(R, gamma, sps)) {
    free(cs);
    return 3;
  }
  int64_t tau = (int64_t)R << 48;
  int B = R;
  int taken = 0;
  for (int i = 0; i < n; ++i) {
    const int64_t q = (int64_t)nearbyint((double)cs[i].a * 0x1p48);
    const int64_t tau_i = tau + q;
    if (!exact_greater(tau_i, sps[B + 1], tau, sps[B])) break;
    tau = tau_i;
    B += 1;
    ell[cs[i].r] += 1;
    taken += 1;
  }
  if (diag) {
    diag[0] = (double)B;
    diag[1] = (double)tau * 0x1p-48;
    diag[2] = ((double)tau * 0x1p-48) * sps[B];
    diag[3] = (double)taken;
  }
  free(cs);
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Zero-overhead scheduling, [P1] §5.2: the serving scheduler sets the next   */
/* capacity K from confidences two steps old and then takes, among the        */
/* current candidates, the top K by current survival -- so it never waits    */
/* for this step's scheduling.  When K is predicted from the past, the early  */
/* stop of Algorithm 1 is left out (to avoid a local optimum at a throughput  */
/* cliff of an irregular SPS curve).                                          */
/* Capacity: the candidates of the given (old) confidences in Algorithm 1's   */
/* order, Theta_i = tau_i * SPS(R + i) for i = 0..R gamma taken candidates    */
/* (same exact fixed-point tau and exact product comparison as Algorithm 1);  */
/* K = the smallest i at which Theta_i is the global maximum.                 */
/* Selection: l_r = number of candidates of r among the first min(K, R gamma) */
/* of the current confidences' order.                                         */
/* ------------------------------------------------------------------------- */
int oracle_schedule_capacity(int R, int gamma, const float* c_old, const double* sps, int sps_len,
                             int32_t* K, double* diag /* [4]: B*, tau*, Theta*, K (may be NULL) */) {
  if (R < 1 || gamma < 1) return 1;
  if (sps_len < R * (1 + gamma) + 1) return 1;
  const int n = R * gamma;
  cand* cs = sorted_candidates(R, gamma, c_old, NULL);
  if (!rates_ok(R, gamma, sps)) {
    free(cs);
    return 3;
  }
  int64_t tau = (int64_t)R << 48, best_tau = tau;
  int best = 0;
  for (int i = 0; i < n; ++i) {
    tau += (int64_t)nearbyint((double)cs[i].a * 0x1p48);
    if (exact_greater(tau, sps[R + i + 1], best_tau, sps[R + best])) { /* strictly: first maximum */
      best = i + 1;
      best_tau = tau;
    }
  }
  *K = best;
  if (diag) {
    diag[0] = (double)(R + best);
    diag[1] = (double)best_tau * 0x1p-48;
    diag[2] = ((double)best_tau * 0x1p-48) * sps[R + best];
    diag[3] = (double)best;
  }
  free(cs);
  return 0;
}

int oracle_schedule_topk(int R, int gamma, const float* c_now, int K, int32_t* ell) {
  if (R < 1 || gamma < 1 || K < 0) return 1;
  const int n = R * gamma;
  cand* cs = sorted_candidates(R, gamma, c_now, NULL);
  for (int r = 0; r < R; ++r) ell[r] = 0;
  for (int i = 0; i < n && i < K; ++i) ell[cs[i].r] += 1;
  free(cs);
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Verification: standard rejection sampling over the scheduled prefix       */
/* ([P1] summary, §3; [P2] "배경"), plus the soft label of [P1] §3.2.1.       */
/*   p^t_j = softmax(Z_j / T) (target), p^d_j = exp(s_j - lse_j) (draft).     */
/*   For j = 1..l: c*_j = sum_v min(p^d_j(v), p^t_j(v)).                     */
/*   Accept x_j iff u_j < p^t_j(x_j) / p^d_j(x_j), tested as                  */
/*     ln u_j < (Z_j[x_j]/T - LSE^t_j) - logp_j    (fp32 decision),          */
/*   u_j = U01(seed, request, j, ACCEPT, 0).  n = number of leading accepts.  */
/*   n < l: the token at row n+1 is drawn from norm(max(0, p^t - p^d)) by     */
/*   two-level Gumbel-max (groups G(seed, request, n+1, RESAMPLE_GROUP, j),   */
/*   ids G(seed, request, n+1, RESAMPLE, v)); if that residual is identically */
/*   zero it is drawn from p^t instead.                                       */
/*   n = l: the bonus token at row l+1 is drawn from p^t the same way.        */
/*   Emitted: x_1..x_n then that token; n_emit = n + 1 ([P1] §3: tau counts   */
/*   the bonus token).  c*_j for j > l and LSE^t_j for j > l are NaN.         */
/* ------------------------------------------------------------------------- */
typedef struct {
  int n_req, gamma, V;
  double T;
  uint64_t seed;
  const int32_t* req_ids;
  const int32_t* x;
  const double *logp, *lse, *scores, *Z;
  const int32_t* ell;
  int32_t *n_acc, *tokens, *n_emit, *stop_kind;
  double *cstar, *lse_t, *acc_margin, *res_margin;
} verify_job;

static void verify_one(const verify_job* J, int i, double* buf, double* key) {
  const int g = J->gamma, V = J->V;
  const uint32_t req = (uint32_t)J->req_ids[i];
  int L = J->ell[i];
  if (L < 0) L = 0;
  if (L > g) L = g;
  const double* Zi = J->Z + (size_t)i * (g + 1) * V;
  const double* Si = J->scores + (size_t)i * g * V;
  double lse_t[1024];
  for (int j = 1; j <= g + 1; ++j) {
    double val = NAN;
    if (j <= L) {
      const double* z = Zi + (size_t)(j - 1) * V;
      for (int v = 0; v < V; ++v) buf[v] = z[v] / J->T;
      val = logsumexp(buf, V);
    }
    if (j <= 1023) lse_t[j] = val;
    if (J->lse_t) J->lse_t[(size_t)i * (g + 1) + (j - 1)] = val;
  }
  for (int j = 1; j <= g; ++j) {
    double cs = NAN;
    if (j <= L) {
      const double* z = Zi + (size_t)(j - 1) * V;
      const double* s = Si + (size_t)(j - 1) * V;
      const double ld = J->lse[(size_t)i * g + (j - 1)];
      cs = 0.0;
      for (int v = 0; v < V; ++v) {
        const double pd = exp(s[v] - ld);
        const double pt = exp(z[v] / J->T - lse_t[j]);
        cs += pd < pt ? pd : pt;
      }
    }
    J->cstar[(size_t)i * g + (j - 1)] = cs;
  }
  int n = 0;
  for (int j = 1; j <= g; ++j) {
    if (J->acc_margin) J->acc_margin[(size_t)i * g + (j - 1)] = NAN;
  }
  for (int j = 1; j <= L; ++j) {
    const int32_t xj = J->x[(size_t)i * g + (j - 1)];
    const double* z = Zi + (size_t)(j - 1) * V;
    const double u = oracle_uniform(oracle_rng_word(J->seed, req, (uint32_t)j,
                                                    ORACLE_PURPOSE_ACCEPT, 0u));
    const double lhs = log(u);
    const double rhs = (z[xj] / J->T - lse_t[j]) - J->logp[(size_t)i * g + (j - 1)];
    if (J->acc_margin) J->acc_margin[(size_t)i * g + (j - 1)] = fabs(lhs - rhs);
    if (!((float)lhs < (float)rhs)) break;
    n += 1;
  }
  int tok = -1, kind = 0;
  double margin = 0.0;
  if (n < L) {
    const int row = n + 1;
    const double* z = Zi + (size_t)(row - 1) * V;
    const double* s = Si + (size_t)(row - 1) * V;
    const double ld = J->lse[(size_t)i * g + (row - 1)];
    /* log-weights of norm(max(0, p^t - p^d)) (its normaliser does not change the draw) */
    for (int v = 0; v < V; ++v) {
      const double pt = exp(z[v] / J->T - lse_t[row]);
      const double pd = exp(s[v] - ld);
      const double res = pt - pd;
      key[v] = res > 0.0 ? log(res) : -INFINITY;
    }
    kind = 1;
    tok = two_level_argmax(key, V, J->seed, req, (uint32_t)row, ORACLE_PURPOSE_RESAMPLE_GROUP,
                           ORACLE_PURPOSE_RESAMPLE, buf, &margin);
    if (tok < 0) { /* the residual is zero everywhere: draw from p^t */
      kind = 2;
      for (int v = 0; v < V; ++v) key[v] = z[v] / J->T;
      tok = two_level_argmax(key, V, J->seed, req, (uint32_t)row, ORACLE_PURPOSE_RESAMPLE_GROUP,
                             ORACLE_PURPOSE_RESAMPLE, buf, &margin);
    }
  } else {
    const int row = L + 1;
    const double* z = Zi + (size_t)(row - 1) * V;
    for (int v = 0; v < V; ++v) key[v] = z[v] / J->T;  /* bonus token from p^t */
    tok = two_level_argmax(key, V, J->seed, req, (uint32_t)row, ORACLE_PURPOSE_RESAMPLE_GROUP,
                           ORACLE_PURPOSE_RESAMPLE, buf, &margin);
  }
  int32_t* t = J->tokens + (size_t)i * (g + 1);
  for (int j = 0; j < g + 1; ++j) t[j] = -1;
  for (int j = 0; j < n; ++j) t[j] = J->x[(size_t)i * g + j];
  t[n] = tok;
  J->n_acc[i] = n;
  J->n_emit[i] = n + 1;
  if (J->stop_kind) J->stop_kind[i] = kind;
  if (J->res_margin) J->res_margin[i] = margin;
}

static void verify_fn(const void* job, int i, double* a, double* b) {
  verify_one((const verify_job*)job, i, a, b);
}

int oracle_verify(int n_req, const int32_t* req_ids, int gamma, int V, double T, uint64_t seed,
                  const int32_t* x, const double* logp, const double* lse, const double* scores,
                  const double* Z, const int32_t* ell, int32_t* n_acc, int32_t* tokens,
                  int32_t* n_emit, double* cstar, double* lse_t, double* acc_margin,
                  double* res_margin, int32_t* stop_kind, int nthreads) {
  if (n_req < 0 || gamma < 1 || gamma > 1022 || V < 1 || !(T > 0.0)) return 1;
  for (int i = 0; i < n_req; ++i)
    for (int j = 0; j < gamma && j < ell[i]; ++j)
      if (x[(size_t)i * gamma + j] < 0 || x[(size_t)i * gamma + j] >= V) return 2;
  verify_job J = {n_req,  gamma, V,    T,     seed,      req_ids, x,         logp,
                  lse,    scores, Z,   ell,   n_acc,     tokens,  n_emit,    stop_kind,
                  cstar,  lse_t, acc_margin, res_margin};
  run_parallel(&J, n_req, nthreads, (size_t)V, verify_fn);
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Sequential Temperature Scaling, [P1] §3.2.1: on held-out data, the          */
/* cumulative prefix survival is calibrated by a left-to-right 1-D grid search */
/* that minimises each position's Expected Calibration Error with the earlier  */
/* positions' calibration held fixed.                                          */
/*   Sample s, position k: raw confidence c_{s,k}, outcome y_{s,k} in {0,1}    */
/*   (position k accepted given the prefix accepted); the survival label is    */
/*   Y_{s,k} = prod_{i<=k} y_{s,i}.                                            */
/*   Temperature scaling: chat(c; T) = sigmoid(logit(c) / T) (0 and 1 stay,     */
/*   T = 1 returns c itself).                                                  */
/*   Calibrated survival: ahat_{s,k} = prod_{i<=k} chat(c_{s,i}; T_i).         */
/*   ECE_k = (1/N) sum_b | sum_{s in bin b} (ahat_{s,k} - Y_{s,k}) |, with     */
/*   M equal-width bins on [0, 1], b = min(floor(ahat M), M - 1).              */
/*   T_k = the grid temperature with the smallest ECE_k (ties: the earlier     */
/*   grid entry), given T_1 .. T_{k-1}.                                        */
/* Static-threshold pruning, [P1] §4.3.3: l_r = the number of leading          */
/* positions whose calibrated survival is at least theta (the survival does    */
/* not increase along a request, so this is a prefix).                         */
/* ------------------------------------------------------------------------- */
double oracle_temper(double c, double T) {
  if (!(c > 0.0)) return 0.0;
  if (!(c < 1.0)) return 1.0;
  if (T == 1.0) return c; /* sigmoid(logit(c)) = c */
  const double z = (log(c) - log1p(-c)) / T;
  return 1.0 / (1.0 + exp(-z));
}

int oracle_sts_calibrate(int N, int gamma, const float* c, const uint8_t* y, const double* grid,
                         int G, int M, double* temps, double* ece_out /* [gamma] or NULL */) {
  if (N < 1 || gamma < 1 || G < 1 || M < 1) return 1;
  for (int g = 0; g < G; ++g)
    if (!(grid[g] > 0.0) || !isfinite(grid[g])) return 1;
  double* ahat = (double*)malloc(sizeof(double) * (size_t)N);
  uint8_t* Y = (uint8_t*)malloc((size_t)N);
  double* bins = (double*)malloc(sizeof(double) * (size_t)M);
  for (int s = 0; s < N; ++s) {
    ahat[s] = 1.0;
    Y[s] = 1;
  }
  for (int k = 0; k < gamma; ++k) {
    int best = 0;
    double best_ece = INFINITY;
    for (int g = 0; g < G; ++g) {
      for (int b = 0; b < M; ++b) bins[b] = 0.0;
      for (int s = 0; s < N; ++s) {
        const double a = ahat[s] * oracle_temper((double)c[(size_t)s * gamma + k], grid[g]);
        const int yk = Y[s] && y[(size_t)s * gamma + k];
        int b = (int)floor(a * M);
        if (b > M - 1) b = M - 1;
        if (b < 0) b = 0;
        bins[b] += a - (double)yk;
      }
      double e = 0.0;
      for (int b = 0; b < M; ++b) e += fabs(bins[b]);
      e /= (double)N;
      if (e < best_ece) {
        best_ece = e;
        best = g;
      }
    }
    temps[k] = grid[best];
    if (ece_out) ece_out[k] = best_ece;
    for (int s = 0; s < N; ++s) {
      ahat[s] *= oracle_temper((double)c[(size_t)s * gamma + k], grid[best]);
      Y[s] = Y[s] && y[(size_t)s * gamma + k];
    }
  }
  free(ahat);
  free(Y);
  free(bins);
  return 0;
}

/* ECE of given temperatures at every position (the objective above). */
int oracle_sts_ece(int N, int gamma, const float* c, const uint8_t* y, const double* temps, int M,
                   double* ece_out) {
  if (N < 1 || gamma < 1 || M < 1) return 1;
  double* bins = (double*)malloc(sizeof(double) * (size_t)M);
  double* ahat = (double*)malloc(sizeof(double) * (size_t)N);
  uint8_t* Y = (uint8_t*)malloc((size_t)N);
  for (int s = 0; s < N; ++s) {
    ahat[s] = 1.0;
    Y[s] = 1;
  }
  for (int k = 0; k < gamma; ++k) {
    for (int b = 0; b < M; ++b) bins[b] = 0.0;
    for (int s = 0; s < N; ++s) {
      ahat[s] *= oracle_temper((double)c[(size_t)s * gamma + k], temps[k]);
      Y[s] = Y[s] && y[(size_t)s * gamma + k];
      int b = (int)floor(ahat[s] * M);
      if (b > M - 1) b = M - 1;
      if (b < 0) b = 0;
      bins[b] += ahat[s] - (double)Y[s];
    }
    double e = 0.0;
    for (int b = 0; b < M; ++b) e += fabs(bins[b]);
    ece_out[k] = e / (double)N;
  }
  free(bins);
  free(ahat);
  free(Y);
  return 0;
}

int oracle_schedule_threshold(int R, int gamma, const float* c, const double* temps /* or NULL */,
                              double theta, int32_t* ell) {
  if (R < 1 || gamma < 1) return 1;
  for (int r = 0; r < R; ++r) {
    double a = 1.0;
    int l = 0;
    for (int j = 0; j < gamma; ++j) {
      a *= oracle_temper((double)c[(size_t)r * gamma + j], temps ? temps[j] : 1.0); /* T = 1: c */
      if (!(a >= theta)) break;
      l = j + 1;
    }
    ell[r] = l;
  }
  return 0;
}
