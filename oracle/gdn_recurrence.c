/*
 * Oracle O1: the Gated DeltaNet recurrence, token by token, in fp64 on the CPU.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this code. The GPU library never calls it and shares
 * no code, header or constant with it.
 *
 * What it computes (plain definition, no chunking, no reordering):
 *
 *   For every sequence b and value head hv, with h = floor(hv / (HV/H)):
 *     S <- state_pool[cache_indices[b], hv]                      (V x K, fp64)
 *     for each token t of the sequence, in order:
 *       q^ = q[t,h] / sqrt(|q[t,h]|^2 + 1e-6),  k^ likewise
 *       log alpha = -exp(A_log[hv]) * softplus(a[t,hv] + dt_bias[hv])
 *       beta      = 1 / (1 + exp(-b[t,hv]))
 *       S <- alpha * S (I - beta k^ k^T) + beta v[t,hv] k^T
 *       o[t,hv] = scale * S q^                (the token reads after its write)
 *     state_out <- S
 *
 * Sources:
 *  - the state transition S_t = S_{t-1}(alpha_t (I - beta_t k_t k_t^T)) + beta_t v_t k_t^T,
 *    S in R^{d_v x d_k}: "Simple math to speed up GDN prefill", section "Reminder";
 *  - the gate inputs ("raw decay-gate input (before softplus/exp)", "raw update-gate
 *    input (before sigmoid)"), A_log and dt_bias per value head, q not pre-normalised,
 *    shapes [total_tokens, H, K] / [total_tokens, HV, V], state_pool [pool, HV, V, K]
 *    updated in place, cache_indices and cu_seqlens: pymllm
 *    "pymllm.layers.attention.gdn_chunkwise", gdn_extend_chunkwise, Parameters;
 *  - a token sees its own write (read after write): "nrm-training-kernels",
 *    section "General implementation", item 4 (level 0 writes before the read).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - log alpha = -exp(A_log) * softplus(a + dt_bias), softplus(x) = max(x,0) + log1p(exp(-|x|));
 *  - both q and k are L2-normalised with epsilon 1e-6 inside the square root;
 *  - GQA: value head hv reads q/k head floor(hv / (HV/H)); HV must be a multiple of H;
 *  - o = scale * S q^ with scale = 1 unless the caller passes another value;
 *  - a zero-length sequence leaves its slot untouched.
 *
 * Since alpha is a scalar, S alpha (I - beta k k^T) + beta v k^T equals
 * alpha S + beta (v - alpha S k) k^T; the code applies it in that order
 * (decay, then the rank-one delta write), which is the same matrix product.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_INDEX 2
#define ORACLE_ERR_NOMEM 3

/* ---- element widening (exact) ------------------------------------------ */

/* bfloat16 is the top 16 bits of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double fp16_bits_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double x;
  if (e == 0)
    x = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
  else if (e == 31)
    x = m ? NAN : INFINITY;
  else
    x = ldexp((double)(m + 1024), e - 25); /* (1 + m/1024) * 2^(e-15) */
  return sign ? -x : x;
}

static double widen(const uint16_t *p, int64_t i, int is_fp16) {
  return is_fp16 ? fp16_bits_to_double(p[i]) : bf16_bits_to_double(p[i]);
}

/* ---- gates ---------------------------------------------------------------- */

double oracle_softplus(double x) { return fmax(x, 0.0) + log1p(exp(-fabs(x))); }

/* log alpha = -exp(A_log) * softplus(a + dt_bias). */
double oracle_log_alpha(double a, double A_log, double dt_bias) {
  return -exp(A_log) * oracle_softplus(a + dt_bias);
}

/* beta = sigmoid(b). */
double oracle_beta(double b) { return 1.0 / (1.0 + exp(-b)); }

/* ---- one token of the recurrence ------------------------------------------ */

/*
 * One step on a V x K row-major state S (S[i*K + j], i over d_v, j over d_k):
 *   S <- alpha S;  u = beta (v - S k);  S <- S + u k^T;  o = scale * S q.
 * qn and kn are already normalised. work must hold V doubles.
 */
void oracle_delta_step(double *S, const double *qn, const double *kn, const double *v,
                       double alpha, double beta, double scale, int K, int V, double *o,
                       double *work) {
  for (int i = 0; i < V; ++i)
    for (int j = 0; j < K; ++j) S[(int64_t)i * K + j] *= alpha;
  for (int i = 0; i < V; ++i) {
    double sk = 0.0;
    for (int j = 0; j < K; ++j) sk += S[(int64_t)i * K + j] * kn[j];
    work[i] = beta * (v[i] - sk);
  }
  for (int i = 0; i < V; ++i)
    for (int j = 0; j < K; ++j) S[(int64_t)i * K + j] += work[i] * kn[j];
  for (int i = 0; i < V; ++i) {
    double sq = 0.0;
    for (int j = 0; j < K; ++j) sq += S[(int64_t)i * K + j] * qn[j];
    o[i] = scale * sq;
  }
}

/*
 * The recurrence over T tokens with explicit alpha and beta and pre-normalised
 * q/k (row-major [T][K]); v is [T][V]. S (V x K) is updated in place; out is [T][V].
 * Used directly by the pins that choose alpha and beta by hand.
 */
int oracle_delta_rule(const double *qn, const double *kn, const double *v, const double *alpha,
                      const double *beta, int64_t T, int K, int V, double scale, double *S,
                      double *out) {
  if (K <= 0 || V <= 0 || T < 0) return ORACLE_ERR_ARG;
  double *work = (double *)malloc(sizeof(double) * (size_t)V);
  if (!work) return ORACLE_ERR_NOMEM;
  for (int64_t t = 0; t < T; ++t)
    oracle_delta_step(S, qn + t * K, kn + t * K, v + t * V, alpha[t], beta[t], scale, K, V,
                      out + t * V, work);
  free(work);
  return ORACLE_OK;
}

/* x / sqrt(|x|^2 + eps) */
static void l2_normalise(double *x, int n) {
  double ss = 0.0;
  for (int j = 0; j < n; ++j) ss += x[j] * x[j];
  double r = 1.0 / sqrt(ss + 1e-6);
  for (int j = 0; j < n; ++j) x[j] *= r;
}

/* ---- the full call: many (sequence, value head) chains on threads ------------ */

typedef struct {
  const uint16_t *q, *k, *v;
  int is_fp16;
  const float *a, *b, *A_log, *dt_bias;
  const float *state_pool;
  const int64_t *cache_indices, *cu_seqlens;
  int64_t total_tokens;
  int H, HV, K, V;
  double scale;
  const int32_t *chain_seq, *chain_hv; /* chain c is (chain_seq[c], chain_hv[c]) */
  const int64_t *out_offset;           /* first output row of chain c in out */
  const int32_t *order;                /* chains, longest first */
  int n_chains;
  double *out;       /* packed [sum of chain lengths][V] */
  double *state_out; /* [n_chains][V][K] */
  int next;          /* next index into order, taken under the lock */
  pthread_mutex_t lock;
  int failed;
} job_t;

static int run_chain(job_t *J, int c) {
  const int K = J->K, V = J->V, H = J->H, HV = J->HV;
  const int seq = J->chain_seq[c], hv = J->chain_hv[c];
  const int h = hv / (HV / H);
  const int64_t t0 = J->cu_seqlens[seq], t1 = J->cu_seqlens[seq + 1];
  const int64_t slot = J->cache_indices[seq];
  double *S = J->state_out + (int64_t)c * V * K;
  double *buf = (double *)malloc(sizeof(double) * (size_t)(2 * K + 2 * V));
  if (!buf) return ORACLE_ERR_NOMEM;
  double *qn = buf, *kn = buf + K, *vv = buf + 2 * K, *work = buf + 2 * K + V;
  const float *S0 = J->state_pool + (slot * HV + hv) * (int64_t)V * K;
  for (int64_t i = 0; i < (int64_t)V * K; ++i) S[i] = (double)S0[i];
  const double A_log = J->A_log[hv], dt_bias = J->dt_bias[hv];
  double *o = J->out + J->out_offset[c] * V;
  for (int64_t t = t0; t < t1; ++t) {
    for (int j = 0; j < K; ++j) {
      qn[j] = widen(J->q, (t * H + h) * K + j, J->is_fp16);
      kn[j] = widen(J->k, (t * H + h) * K + j, J->is_fp16);
    }
    for (int i = 0; i < V; ++i) vv[i] = widen(J->v, (t * HV + hv) * (int64_t)V + i, J->is_fp16);
    l2_normalise(qn, K);
    l2_normalise(kn, K);
    const double alpha = exp(oracle_log_alpha((double)J->a[t * HV + hv], A_log, dt_bias));
    const double beta = oracle_beta((double)J->b[t * HV + hv]);
    oracle_delta_step(S, qn, kn, vv, alpha, beta, J->scale, K, V, o + (t - t0) * V, work);
  }
  free(buf);
  return ORACLE_OK;
}

static void *worker(void *arg) {
  job_t *J = (job_t *)arg;
  for (;;) {
    pthread_mutex_lock(&J->lock);
    int i = J->next++;
    pthread_mutex_unlock(&J->lock);
    if (i >= J->n_chains) break;
    if (run_chain(J, J->order[i]) != ORACLE_OK) {
      pthread_mutex_lock(&J->lock);
      J->failed = 1;
      pthread_mutex_unlock(&J->lock);
    }
  }
  return NULL;
}

static const int64_t *g_len_for_sort;
static int cmp_longest_first(const void *x, const void *y) {
  int64_t lx = g_len_for_sort[*(const int32_t *)x], ly = g_len_for_sort[*(const int32_t *)y];
  if (lx != ly) return lx > ly ? -1 : 1;
  return *(const int32_t *)x - *(const int32_t *)y;
}

/*
 * Run the recurrence for a list of chains (chain_seq[c], chain_hv[c]).
 * If chain_seq is NULL every (sequence, value head) pair is run, sequence-major
 * (c = seq * HV + hv). Outputs for chain c are packed contiguously, in chain
 * order, as [len(seq)][V] doubles in out; final states go to state_out[c] (V x K).
 * n_threads <= 0 uses every online core. Returns the number of threads used
 * (>= 1) on success, or minus an ORACLE_ERR_* code.
 */
int oracle_gdn_forward(const uint16_t *q, const uint16_t *k, const uint16_t *v, int is_fp16,
                       const float *a, const float *b, const float *A_log, const float *dt_bias,
                       const float *state_pool, int64_t pool_size, const int64_t *cache_indices,
                       const int64_t *cu_seqlens, int batch, int64_t total_tokens, int H, int HV,
                       int K, int V, double scale, const int32_t *chain_seq,
                       const int32_t *chain_hv, int n_chains, double *out, double *state_out,
                       int n_threads) {
  if (H <= 0 || HV <= 0 || HV % H != 0 || K <= 0 || V <= 0 || batch < 0) return -ORACLE_ERR_ARG;
  if (cu_seqlens[0] != 0 || cu_seqlens[batch] != total_tokens) return -ORACLE_ERR_ARG;
  for (int s = 0; s < batch; ++s) {
    if (cu_seqlens[s + 1] < cu_seqlens[s]) return -ORACLE_ERR_ARG;
    if (cache_indices[s] < 0 || cache_indices[s] >= pool_size) return -ORACLE_ERR_INDEX;
    for (int r = 0; r < s; ++r)
      if (cache_indices[r] == cache_indices[s]) return -ORACLE_ERR_INDEX;
  }
  int32_t *own_seq = NULL, *own_hv = NULL;
  if (!chain_seq) {
    n_chains = batch * HV;
    own_seq = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n_chains ? n_chains : 1));
    own_hv = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n_chains ? n_chains : 1));
    if (!own_seq || !own_hv) return -ORACLE_ERR_NOMEM;
    for (int c = 0; c < n_chains; ++c) {
      own_seq[c] = c / HV;
      own_hv[c] = c % HV;
    }
    chain_seq = own_seq;
    chain_hv = own_hv;
  }
  for (int c = 0; c < n_chains; ++c)
    if (chain_seq[c] < 0 || chain_seq[c] >= batch || chain_hv[c] < 0 || chain_hv[c] >= HV)
      return -ORACLE_ERR_ARG;
  size_t nc = (size_t)(n_chains ? n_chains : 1);
  int64_t *len = (int64_t *)malloc(sizeof(int64_t) * nc);
  int64_t *off = (int64_t *)malloc(sizeof(int64_t) * nc);
  int32_t *order = (int32_t *)malloc(sizeof(int32_t) * nc);
  if (!len || !off || !order) return -ORACLE_ERR_NOMEM;
  int64_t acc = 0;
  for (int c = 0; c < n_chains; ++c) {
    len[c] = cu_seqlens[chain_seq[c] + 1] - cu_seqlens[chain_seq[c]];
    off[c] = acc;
    acc += len[c];
    order[c] = c;
  }
  g_len_for_sort = len;
  qsort(order, (size_t)n_chains, sizeof(int32_t), cmp_longest_first);

  if (n_threads <= 0) n_threads = (int)sysconf(_SC_NPROCESSORS_ONLN);
  if (n_threads < 1) n_threads = 1;
  if (n_threads > n_chains) n_threads = n_chains > 0 ? n_chains : 1;

  job_t J;
  memset(&J, 0, sizeof J);
  J.q = q; J.k = k; J.v = v; J.is_fp16 = is_fp16;
  J.a = a; J.b = b; J.A_log = A_log; J.dt_bias = dt_bias;
  J.state_pool = state_pool; J.cache_indices = cache_indices; J.cu_seqlens = cu_seqlens;
  J.total_tokens = total_tokens; J.H = H; J.HV = HV; J.K = K; J.V = V; J.scale = scale;
  J.chain_seq = chain_seq; J.chain_hv = chain_hv; J.out_offset = off; J.order = order;
  J.n_chains = n_chains; J.out = out; J.state_out = state_out;
  pthread_mutex_init(&J.lock, NULL);

  pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
  int started = 0;
  for (int i = 0; i < n_threads; ++i)
    if (pthread_create(&th[i], NULL, worker, &J) == 0) ++started;
  if (started == 0) worker(&J);
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  pthread_mutex_destroy(&J.lock);
  free(th);
  free(len);
  free(off);
  free(order);
  free(own_seq);
  free(own_hv);
  if (J.failed) return -ORACLE_ERR_NOMEM;
  return started > 0 ? started : 1;
}

/* Widening helpers exposed so tests can pin them against numpy/torch. */
double oracle_bf16_to_double(uint16_t h) { return bf16_bits_to_double(h); }
double oracle_fp16_to_double(uint16_t h) { return fp16_bits_to_double(h); }
