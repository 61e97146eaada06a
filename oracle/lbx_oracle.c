/*
 * lbx_oracle.c -- plain, slow, fp64 CPU oracle for the tree-verify step of a
 * hybrid model's gated-DeltaNet layers.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the package's smoke check and the bench's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA library; the only thing both sides share is the seeded input
 * generator, which holds none of the method's arithmetic.
 *
 * What it computes (sources: Lucebox hub README, section "02 DFlash DDtree",
 * list "Implemented here" -- the three tree-aware state-rollback ops
 * ggml_ssm_conv_tree, ggml_gated_delta_net_tree and
 * ggml_gated_delta_net_tree_persist -- and list "Algorithms used", which names
 * DDTree's tree-structured verify; the recurrence itself is the gated delta
 * rule S_n = a_n S_parent(n) (I - b_n k_n k_n^T) + b_n v_n k_n^T, o_n = S_n q_n):
 *
 *   1. tree conv: each draft node's depthwise causal conv runs along the
 *      node's ancestor path instead of token order; past the root it reads
 *      the conv cache (K-1 raw prior inputs, oldest first).  Then SiLU, then
 *      q and k are L2-normalised per key head (v is not).
 *   2. tree recurrence: every node's state is the plain sequential delta-rule
 *      recurrence over its root-to-node path, started from the cached state
 *      of the request's slot.  Computed here literally, per node, by walking
 *      that path (O(depth * d^2) per node: slow by design).
 *   3. persist: the accepted node's state and the last K-1 raw inputs of the
 *      path ending at the accepted node (continuing into the old cache) are
 *      written back to the request's slot.
 *
 * Readings where the pages are silent:
 *   - value head h reads key head h / (Hv/Hk) (contiguous GQA groups);
 *   - conv channels are ordered q | k | v, conv has no bias, tap K-1
 *     multiplies the current node;
 *   - L2 normalisation is x / sqrt(sum x^2 + eps) after SiLU;
 *   - gates a, b arrive already activated;
 *   - node 0 is the root (the last accepted token), parent[0] = -1 and
 *     parent[i] < i; the accepted path runs from node 0 to accepted[b];
 *   - state is stored [d_v][d_k] (row = value dimension);
 *   - o_n = q_scale * S_n q_n (q_scale = 1 unless stated).
 *
 * All arithmetic is double.  bf16 inputs are widened exactly.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define LBXO_OK 0
#define LBXO_EINVAL (-1)
#define LBXO_ETREE (-3)
#define LBXO_ENOMEM (-4)

typedef struct {
  int L, Bq, N, Hk, Hv, d, K, n_slots;
  double l2_eps, q_scale;
} lbxo_cfg;

/* Exact widening of a bf16 bit pattern. */
static double bf16_to_double(uint16_t u) {
  uint32_t w = (uint32_t)u << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

static int channels(const lbxo_cfg *c) { return 2 * c->Hk * c->d + c->Hv * c->d; }

static int cfg_ok(const lbxo_cfg *c) {
  if (!c) return 0;
  if (c->L < 1 || c->Bq < 1 || c->N < 1 || c->Hk < 1 || c->Hv < 1 || c->d < 1 || c->K < 1)
    return 0;
  if (c->Hv % c->Hk != 0) return 0;
  if (c->n_slots < c->Bq) return 0;
  return 1;
}

/* A tree is valid when node 0 is the root and every other node's parent has
 * a smaller index (topological numbering). */
int lbxo_check_tree(const int32_t *parent, int N) {
  if (N < 1 || parent[0] != -1) return LBXO_ETREE;
  for (int i = 1; i < N; ++i)
    if (parent[i] < 0 || parent[i] >= i) return LBXO_ETREE;
  return LBXO_OK;
}

static int is_chain(const int32_t *parent, int N) {
  for (int i = 0; i < N; ++i)
    if (parent[i] != i - 1) return 0;
  return 1;
}

/* ------------------------------------------------------------------------ */
/* 1. Tree conv + SiLU (+ L2 for q and k).                                    */
/* ------------------------------------------------------------------------ */

/* The j-th element of node n's conv window (j = 0 is n itself, j = 1 its
 * parent, ...).  Past the root the window continues into the cache, most
 * recent cached row (index K-2) first. */
static double window_value(int n, int j, int c, int C, int K, const uint16_t *x_lb,
                           const float *cache, const int32_t *parent) {
  int m = n;
  int steps = 0;
  while (steps < j && m >= 0) {
    m = parent[m];
    ++steps;
  }
  if (m >= 0) return bf16_to_double(x_lb[(size_t)m * C + c]);
  /* m fell off the root after (steps) moves; the remaining (j - steps) moves,
   * plus the move that left the root, walk back through the cache. */
  int past = j - steps + 1; /* 1 = most recent cached row */
  return (double)cache[(size_t)(K - 1 - past) * C + c];
}

/* Conv + SiLU of one channel of one node, before any normalisation:
 * y = sum_{j=0}^{K-1} w[c][K-1-j] * xhat_j[c];  out = y * sigmoid(y). */
static double conv_silu(int n, int c, int C, int K, const uint16_t *x_lb,
                        const uint16_t *w_l, const float *cache, const int32_t *parent) {
  double y = 0.0;
  for (int j = 0; j < K; ++j)
    y += bf16_to_double(w_l[(size_t)c * K + (K - 1 - j)]) *
         window_value(n, j, c, C, K, x_lb, cache, parent);
  return y / (1.0 + exp(-y));
}

static void l2_normalise(double *v, int d, double eps) {
  double ss = 0.0;
  for (int i = 0; i < d; ++i) ss += v[i] * v[i];
  double s = 1.0 / sqrt(ss + eps);
  for (int i = 0; i < d; ++i) v[i] *= s;
}

/* Conv output of one (layer, request): qkv [N][C], q and k normalised. */
int lbxo_conv_lb(int N, int Hk, int Hv, int d, int K, double l2_eps, const uint16_t *x_lb,
                 const uint16_t *w_l, const float *cache, const int32_t *parent, double *qkv) {
  if (lbxo_check_tree(parent, N) != LBXO_OK) return LBXO_ETREE;
  int C = 2 * Hk * d + Hv * d;
  for (int n = 0; n < N; ++n) {
    double *row = qkv + (size_t)n * C;
    for (int c = 0; c < C; ++c) row[c] = conv_silu(n, c, C, K, x_lb, w_l, cache, parent);
    for (int g = 0; g < 2 * Hk; ++g) l2_normalise(row + (size_t)g * d, d, l2_eps);
  }
  return LBXO_OK;
}

/* Whole-batch tree conv: qkv [L][Bq][N][C].  lb_mask [L][Bq] may be NULL. */
int lbxo_tree_conv(const lbxo_cfg *cfg, const uint16_t *x, const uint16_t *conv_w,
                   const float *conv_cache, const int32_t *parent, const int32_t *slot,
                   const uint8_t *lb_mask, double *qkv) {
  if (!cfg_ok(cfg)) return LBXO_EINVAL;
  int L = cfg->L, Bq = cfg->Bq, N = cfg->N, K = cfg->K, C = channels(cfg);
  for (int b = 0; b < Bq; ++b) {
    if (lbxo_check_tree(parent + (size_t)b * N, N) != LBXO_OK) return LBXO_ETREE;
    if (slot[b] < 0 || slot[b] >= cfg->n_slots) return LBXO_EINVAL;
  }
  for (int l = 0; l < L; ++l)
    for (int b = 0; b < Bq; ++b) {
      if (lb_mask && !lb_mask[(size_t)l * Bq + b]) continue;
      const uint16_t *x_lb = x + ((size_t)l * Bq + b) * N * C;
      const float *cache = conv_cache + ((size_t)l * cfg->n_slots + slot[b]) * (K - 1) * C;
      int rc = lbxo_conv_lb(N, cfg->Hk, cfg->Hv, cfg->d, K, cfg->l2_eps, x_lb,
                            conv_w + (size_t)l * C * K, cache, parent + (size_t)b * N,
                            qkv + ((size_t)l * Bq + b) * N * C);
      if (rc) return rc;
    }
  return LBXO_OK;
}

/* ------------------------------------------------------------------------ */
/* 2. Gated delta-rule recurrence.                                           */
/* ------------------------------------------------------------------------ */

/* One step of the gated delta rule, rank-1 form:
 * S <- a S (I - b k k^T) + b v k^T = a (S - b (S k) k^T) + b v k^T. */
static void delta_step(double *S, int d, double a, double b, const double *k, const double *v,
                       double *Sk) {
  for (int i = 0; i < d; ++i) {
    double acc = 0.0;
    for (int j = 0; j < d; ++j) acc += S[(size_t)i * d + j] * k[j];
    Sk[i] = acc;
  }
  for (int i = 0; i < d; ++i)
    for (int j = 0; j < d; ++j)
      S[(size_t)i * d + j] = a * (S[(size_t)i * d + j] - b * Sk[i] * k[j]) + b * v[i] * k[j];
}

/* The same step with the transition matrix written out: M = I - b k k^T,
 * S <- a (S M) + b v k^T, with S M a plain d x d matrix product.  Used only
 * as a brute-force cross-check on small d. */
static void delta_step_matrix(double *S, int d, double a, double b, const double *k,
                              const double *v, double *M, double *T) {
  for (int r = 0; r < d; ++r)
    for (int c = 0; c < d; ++c) M[(size_t)r * d + c] = (r == c ? 1.0 : 0.0) - b * k[r] * k[c];
  for (int i = 0; i < d; ++i)
    for (int c = 0; c < d; ++c) {
      double acc = 0.0;
      for (int r = 0; r < d; ++r) acc += S[(size_t)i * d + r] * M[(size_t)r * d + c];
      T[(size_t)i * d + c] = acc;
    }
  for (int i = 0; i < d; ++i)
    for (int j = 0; j < d; ++j)
      S[(size_t)i * d + j] = a * T[(size_t)i * d + j] + b * v[i] * k[j];
}

/* Per-head inputs of one (layer, request, value head h), from the conv
 * output: q_n, k_n (key head h / G) and v_n (value head h). */
static const double *q_of(const double *qkv, int n, int C, int d, int kh) {
  return qkv + (size_t)n * C + (size_t)kh * d;
}
static const double *k_of(const double *qkv, int n, int C, int d, int Hk, int kh) {
  return qkv + (size_t)n * C + (size_t)Hk * d + (size_t)kh * d;
}
static const double *v_of(const double *qkv, int n, int C, int d, int Hk, int h) {
  return qkv + (size_t)n * C + (size_t)2 * Hk * d + (size_t)h * d;
}

enum { FORM_PATH = 0, FORM_MATRIX = 1, FORM_SEQUENTIAL = 2 };

/*
 * Recurrence of one (layer, request, value head).
 *   qkv  [N][C]   conv output of this (layer, request)
 *   a, b [N][Hv]  bf16 gates of this (layer, request)
 *   S0   [d][d]   fp32 cached state of the request's slot, head h
 * Outputs (each may be NULL):
 *   o           [N][d]     o_n = q_scale * S_n q_n
 *   node_states [N][d][d]  S_n
 *   S_acc       [d][d]     S_accepted
 * form: FORM_PATH walks each node's root-to-node path with the rank-1 step;
 * FORM_MATRIX does the same with explicit d x d transition matrices;
 * FORM_SEQUENTIAL requires a chain and runs one state through the tokens in
 * order, the textbook sequential recurrence.
 */
int lbxo_deltanet_head(int N, int Hk, int Hv, int d, int h, double q_scale, int form,
                       const double *qkv, const uint16_t *a, const uint16_t *b, const float *S0,
                       const int32_t *parent, int accepted, double *o, double *node_states,
                       double *S_acc) {
  if (lbxo_check_tree(parent, N) != LBXO_OK) return LBXO_ETREE;
  if (h < 0 || h >= Hv || Hv % Hk) return LBXO_EINVAL;
  if (S_acc && (accepted < 0 || accepted >= N)) return LBXO_EINVAL;
  if (form == FORM_SEQUENTIAL && !is_chain(parent, N)) return LBXO_ETREE;
  int C = 2 * Hk * d + Hv * d;
  int kh = h / (Hv / Hk);
  size_t dd = (size_t)d * d;
  double *S = malloc(dd * sizeof *S);
  double *M = malloc(dd * sizeof *M);
  double *T = malloc(dd * sizeof *T);
  double *Sk = malloc((size_t)d * sizeof *Sk);
  int *path = malloc((size_t)N * sizeof *path);
  if (!S || !M || !T || !Sk || !path) {
    free(S), free(M), free(T), free(Sk), free(path);
    return LBXO_ENOMEM;
  }

  if (form == FORM_SEQUENTIAL) {
    for (size_t e = 0; e < dd; ++e) S[e] = (double)S0[e];
    for (int t = 0; t < N; ++t) {
      delta_step(S, d, bf16_to_double(a[(size_t)t * Hv + h]),
                 bf16_to_double(b[(size_t)t * Hv + h]), k_of(qkv, t, C, d, Hk, kh),
                 v_of(qkv, t, C, d, Hk, h), Sk);
      if (o) {
        const double *q = q_of(qkv, t, C, d, kh);
        for (int i = 0; i < d; ++i) {
          double acc = 0.0;
          for (int j = 0; j < d; ++j) acc += S[(size_t)i * d + j] * q[j];
          o[(size_t)t * d + i] = q_scale * acc;
        }
      }
      if (node_states) memcpy(node_states + (size_t)t * dd, S, dd * sizeof *S);
      if (S_acc && t == accepted) memcpy(S_acc, S, dd * sizeof *S);
    }
  } else {
    for (int n = 0; n < N; ++n) {
      /* root-to-node path, root first */
      int len = 0;
      for (int m = n; m >= 0; m = parent[m]) path[len++] = m;
      for (size_t e = 0; e < dd; ++e) S[e] = (double)S0[e];
      for (int s = len - 1; s >= 0; --s) {
        int m = path[s];
        double am = bf16_to_double(a[(size_t)m * Hv + h]);
        double bm = bf16_to_double(b[(size_t)m * Hv + h]);
        const double *k = k_of(qkv, m, C, d, Hk, kh);
        const double *v = v_of(qkv, m, C, d, Hk, h);
        if (form == FORM_MATRIX)
          delta_step_matrix(S, d, am, bm, k, v, M, T);
        else
          delta_step(S, d, am, bm, k, v, Sk);
      }
      if (o) {
        const double *q = q_of(qkv, n, C, d, kh);
        for (int i = 0; i < d; ++i) {
          double acc = 0.0;
          for (int j = 0; j < d; ++j) acc += S[(size_t)i * d + j] * q[j];
          o[(size_t)n * d + i] = q_scale * acc;
        }
      }
      if (node_states) memcpy(node_states + (size_t)n * dd, S, dd * sizeof *S);
      if (S_acc && n == accepted) memcpy(S_acc, S, dd * sizeof *S);
    }
  }
  free(S), free(M), free(T), free(Sk), free(path);
  return LBXO_OK;
}

/* ------------------------------------------------------------------------ */
/* 3. Persist.                                                               */
/* ------------------------------------------------------------------------ */

/* New conv window of one (layer, request): the last K-1 entries of the
 * sequence [old cache rows (oldest first), x of the path root..accepted].
 * Values are copied, not computed, so the result is exact. */
int lbxo_persist_conv_lb(int N, int C, int K, const uint16_t *x_lb, const float *cache_old,
                         const int32_t *parent, int accepted, float *cache_new) {
  if (lbxo_check_tree(parent, N) != LBXO_OK) return LBXO_ETREE;
  if (accepted < 0 || accepted >= N) return LBXO_EINVAL;
  int *path = malloc((size_t)N * sizeof *path);
  if (!path) return LBXO_ENOMEM;
  int len = 0;
  for (int m = accepted; m >= 0; m = parent[m]) path[len++] = m; /* accepted first */
  /* sequence index s (0 = oldest) over K-1 + len entries */
  int total = (K - 1) + len;
  for (int r = 0; r < K - 1; ++r) {
    int s = total - (K - 1) + r;
    for (int c = 0; c < C; ++c) {
      float val;
      if (s < K - 1) {
        val = cache_old[(size_t)s * C + c];
      } else {
        int node = path[len - 1 - (s - (K - 1))];
        uint32_t w = (uint32_t)x_lb[(size_t)node * C + c] << 16;
        memcpy(&val, &w, sizeof val);
      }
      cache_new[(size_t)r * C + c] = val;
    }
  }
  free(path);
  return LBXO_OK;
}

/* ------------------------------------------------------------------------ */
/* Whole-step drivers (threads over independent (layer, request, head)).    */
/* ------------------------------------------------------------------------ */

typedef struct {
  const lbxo_cfg *cfg;
  const uint16_t *x, *conv_w, *a, *b;
  const float *state, *conv_cache;
  const int32_t *parent, *slot, *accepted;
  const int32_t *items; /* [n_items][3] = (l, b, h) */
  int n_items, form;
  double *o_items;    /* [n_items][N][d] or NULL */
  double *sacc_items; /* [n_items][d][d] or NULL */
  int next;
  int rc;
  pthread_mutex_t mu;
} heads_job;

/* q/k/v of one (layer, request) for the channels of value head h only: the
 * conv output restricted to those channels, laid out as a full [N][C] row so
 * the head function can index it. */
static int head_conv(const heads_job *J, int l, int b, int h, double *qkv) {
  const lbxo_cfg *c = J->cfg;
  int N = c->N, K = c->K, d = c->d, Hk = c->Hk, C = channels(c);
  int kh = h / (c->Hv / Hk);
  const uint16_t *x_lb = J->x + ((size_t)l * c->Bq + b) * N * C;
  const uint16_t *w_l = J->conv_w + (size_t)l * C * K;
  const float *cache = J->conv_cache + ((size_t)l * c->n_slots + J->slot[b]) * (K - 1) * C;
  const int32_t *par = J->parent + (size_t)b * N;
  int base[3] = {kh * d, Hk * d + kh * d, 2 * Hk * d + h * d};
  for (int n = 0; n < N; ++n)
    for (int g = 0; g < 3; ++g) {
      double *row = qkv + (size_t)n * C + base[g];
      for (int i = 0; i < d; ++i) row[i] = conv_silu(n, base[g] + i, C, K, x_lb, w_l, cache, par);
      if (g < 2) l2_normalise(row, d, c->l2_eps);
    }
  return LBXO_OK;
}

static void *heads_worker(void *arg) {
  heads_job *J = arg;
  const lbxo_cfg *c = J->cfg;
  int N = c->N, d = c->d, C = channels(c);
  double *qkv = malloc((size_t)N * C * sizeof *qkv);
  if (!qkv) {
    pthread_mutex_lock(&J->mu);
    J->rc = LBXO_ENOMEM;
    pthread_mutex_unlock(&J->mu);
    return NULL;
  }
  for (;;) {
    pthread_mutex_lock(&J->mu);
    int it = J->next++;
    int stop = J->rc != LBXO_OK;
    pthread_mutex_unlock(&J->mu);
    if (stop || it >= J->n_items) break;
    int l = J->items[3 * it], b = J->items[3 * it + 1], h = J->items[3 * it + 2];
    head_conv(J, l, b, h, qkv);
    const float *S0 =
        J->state + (((size_t)l * c->n_slots + J->slot[b]) * c->Hv + h) * (size_t)d * d;
    int rc = lbxo_deltanet_head(
        N, c->Hk, c->Hv, d, h, c->q_scale, J->form, qkv, J->a + ((size_t)l * c->Bq + b) * N * c->Hv,
        J->b + ((size_t)l * c->Bq + b) * N * c->Hv, S0, J->parent + (size_t)b * N,
        J->accepted ? J->accepted[b] : -1, J->o_items ? J->o_items + (size_t)it * N * d : NULL,
        NULL, J->sacc_items ? J->sacc_items + (size_t)it * d * d : NULL);
    if (rc) {
      pthread_mutex_lock(&J->mu);
      J->rc = rc;
      pthread_mutex_unlock(&J->mu);
    }
  }
  free(qkv);
  return NULL;
}

/*
 * Full verify step (conv -> recurrence -> accepted state) for a list of
 * heads.  items [n_items][3] = (layer, request, value head).  For each item
 * writes o_items[it] = o of that head for all N nodes ([N][d]) and
 * sacc_items[it] = the accepted node's state ([d][d]); either may be NULL.
 * form: 0 path walk, 1 explicit matrices, 2 sequential (chains only).
 * n_threads <= 0 uses every online core.  Returns the thread count used via
 * *threads_used (may be NULL).
 */
int lbxo_verify_heads(const lbxo_cfg *cfg, const uint16_t *x, const uint16_t *conv_w,
                      const uint16_t *a, const uint16_t *b, const float *state,
                      const float *conv_cache, const int32_t *parent, const int32_t *slot,
                      const int32_t *accepted, const int32_t *items, int n_items, int form,
                      double *o_items, double *sacc_items, int n_threads, int *threads_used) {
  if (!cfg_ok(cfg) || n_items < 0) return LBXO_EINVAL;
  for (int bb = 0; bb < cfg->Bq; ++bb) {
    if (lbxo_check_tree(parent + (size_t)bb * cfg->N, cfg->N) != LBXO_OK) return LBXO_ETREE;
    if (slot[bb] < 0 || slot[bb] >= cfg->n_slots) return LBXO_EINVAL;
    if (accepted && (accepted[bb] < 0 || accepted[bb] >= cfg->N)) return LBXO_EINVAL;
  }
  for (int it = 0; it < n_items; ++it) {
    const int32_t *e = items + 3 * it;
    if (e[0] < 0 || e[0] >= cfg->L || e[1] < 0 || e[1] >= cfg->Bq || e[2] < 0 || e[2] >= cfg->Hv)
      return LBXO_EINVAL;
  }
  if (n_threads <= 0) n_threads = (int)sysconf(_SC_NPROCESSORS_ONLN);
  if (n_threads < 1) n_threads = 1;
  if (n_threads > n_items && n_items > 0) n_threads = n_items;
  heads_job J = {cfg, x, conv_w, a, b, state, conv_cache, parent, slot, accepted, items,
                 n_items, form, o_items, sacc_items, 0, LBXO_OK, PTHREAD_MUTEX_INITIALIZER};
  pthread_t *th = malloc((size_t)n_threads * sizeof *th);
  if (!th) return LBXO_ENOMEM;
  int started = 0;
  for (int t = 1; t < n_threads; ++t)
    if (pthread_create(&th[started], NULL, heads_worker, &J) == 0) ++started;
  /* the calling thread works too */
  heads_worker(&J);
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  free(th);
  if (threads_used) *threads_used = started + 1;
  return J.rc;
}

/* Whole-batch recurrence from a given conv output (for checking the
 * unfused recurrence on its own).  qkv [L][Bq][N][C] double,
 * o [L][Bq][N][Hv][d], node_states [L][Bq][N][Hv][d][d] (may be NULL). */
int lbxo_tree_deltanet(const lbxo_cfg *cfg, const double *qkv, const uint16_t *a,
                       const uint16_t *b, const float *state, const int32_t *parent,
                       const int32_t *slot, int form, double *o, double *node_states) {
  if (!cfg_ok(cfg)) return LBXO_EINVAL;
  int L = cfg->L, Bq = cfg->Bq, N = cfg->N, Hv = cfg->Hv, d = cfg->d, C = channels(cfg);
  size_t dd = (size_t)d * d;
  double *oh = malloc((size_t)N * d * sizeof *oh);
  double *ns = node_states ? malloc((size_t)N * dd * sizeof *ns) : NULL;
  if (!oh || (node_states && !ns)) {
    free(oh), free(ns);
    return LBXO_ENOMEM;
  }
  int rc = LBXO_OK;
  for (int bb = 0; bb < Bq && rc == LBXO_OK; ++bb)
    if (slot[bb] < 0 || slot[bb] >= cfg->n_slots) rc = LBXO_EINVAL;
  for (int l = 0; l < L && rc == LBXO_OK; ++l)
    for (int bb = 0; bb < Bq && rc == LBXO_OK; ++bb)
      for (int h = 0; h < Hv && rc == LBXO_OK; ++h) {
        const float *S0 = state + (((size_t)l * cfg->n_slots + slot[bb]) * Hv + h) * dd;
        rc = lbxo_deltanet_head(N, cfg->Hk, Hv, d, h, cfg->q_scale, form,
                                qkv + ((size_t)l * Bq + bb) * N * C,
                                a + ((size_t)l * Bq + bb) * N * Hv,
                                b + ((size_t)l * Bq + bb) * N * Hv, S0,
                                parent + (size_t)bb * N, -1, oh, ns, NULL);
        if (rc) break;
        for (int n = 0; n < N; ++n) {
          memcpy(o + ((((size_t)l * Bq + bb) * N + n) * Hv + h) * d, oh + (size_t)n * d,
                 (size_t)d * sizeof *oh);
          if (node_states)
            memcpy(node_states + ((((size_t)l * Bq + bb) * N + n) * Hv + h) * dd,
                   ns + (size_t)n * dd, dd * sizeof *ns);
        }
      }
  free(oh), free(ns);
  return rc;
}

/* Persist from per-node fp32 snapshots (the unfused write-back): for every
 * (layer, request) copy node_states[accepted] into the slot's state and
 * rewrite the slot's conv window.  state and conv_cache are updated in place;
 * slots no request names are left untouched.
 * node_states [L][Bq][N][Hv][d][d] fp32. */
int lbxo_tree_persist(const lbxo_cfg *cfg, const uint16_t *x, const float *node_states,
                      const int32_t *parent, const int32_t *slot, const int32_t *accepted,
                      float *state, float *conv_cache) {
  if (!cfg_ok(cfg)) return LBXO_EINVAL;
  int L = cfg->L, Bq = cfg->Bq, N = cfg->N, Hv = cfg->Hv, d = cfg->d, K = cfg->K,
      C = channels(cfg);
  size_t dd = (size_t)d * d;
  for (int bb = 0; bb < Bq; ++bb) {
    if (lbxo_check_tree(parent + (size_t)bb * N, N) != LBXO_OK) return LBXO_ETREE;
    if (slot[bb] < 0 || slot[bb] >= cfg->n_slots) return LBXO_EINVAL;
    if (accepted[bb] < 0 || accepted[bb] >= N) return LBXO_EINVAL;
  }
  float *tmp = malloc((size_t)(K > 1 ? K - 1 : 1) * C * sizeof *tmp);
  if (!tmp) return LBXO_ENOMEM;
  for (int l = 0; l < L; ++l)
    for (int bb = 0; bb < Bq; ++bb) {
      int s = slot[bb], acc = accepted[bb];
      for (int h = 0; h < Hv; ++h)
        memcpy(state + (((size_t)l * cfg->n_slots + s) * Hv + h) * dd,
               node_states + ((((size_t)l * Bq + bb) * N + acc) * Hv + h) * dd,
               dd * sizeof *state);
      float *cache = conv_cache + ((size_t)l * cfg->n_slots + s) * (K - 1) * C;
      lbxo_persist_conv_lb(N, C, K, x + ((size_t)l * Bq + bb) * N * C, cache,
                           parent + (size_t)bb * N, acc, tmp);
      memcpy(cache, tmp, (size_t)(K - 1) * C * sizeof *tmp);
    }
  free(tmp);
  return LBXO_OK;
}

/* ---- verify argmax and greedy acceptance walk -------------------------------
 *
 * Sources: Lucebox hub README, section "GPU draft top-K & verify-argmax
 * (DFlash)" (the target's per-node argmax over the vocabulary, taken on the
 * device from the logits buffer, decides acceptance), and the same README's
 * serving notes (temperature 0, greedy decoding, gives the highest acceptance).
 * The pages print no rule; the plain greedy reading is taken:
 *   - the target's choice at node n is the argmax of its logits row n: the
 *     largest value; NaN ranks below every number; among equal values (and
 *     in an all-NaN row) the lowest index;
 *   - the walk starts at the root (node 0, the last accepted token, always
 *     kept); at node u it moves to the lowest-index child c of u whose draft
 *     token equals the target's choice at u, and stops when there is none;
 *   - accepted[b] = the node where it stops; next[b] = the target's choice at
 *     that node (the token that follows the accepted path).
 * logits [Bq][N][V] fp32, draft [Bq][N] int32 (draft[b][0] is not read),
 * parent [Bq][N] int32; argmax [Bq][N], accepted [Bq], next [Bq] int32 out.
 */

/* 1 if value a at index ia ranks above value b at index ib. */
static int ranks_above(float a, int ia, float b, int ib) {
  int na = isnan(a), nb = isnan(b);
  if (na && nb) return ia < ib;
  if (na) return 0;
  if (nb) return 1;
  if (a > b) return 1;
  if (a < b) return 0;
  return ia < ib;
}

int lbxo_accept_walk(int Bq, int N, int V, const float *logits, const int32_t *draft,
                     const int32_t *parent, int32_t *argmax_out, int32_t *accepted_out,
                     int32_t *next_out) {
  if (Bq < 1 || N < 1 || V < 1) return LBXO_EINVAL;
  for (int bb = 0; bb < Bq; ++bb)
    if (lbxo_check_tree(parent + (size_t)bb * N, N) != LBXO_OK) return LBXO_ETREE;
  for (int bb = 0; bb < Bq; ++bb) {
    int32_t *am = argmax_out + (size_t)bb * N;
    for (int n = 0; n < N; ++n) {
      const float *row = logits + ((size_t)bb * N + n) * V;
      int best = 0;
      for (int v = 1; v < V; ++v)
        if (ranks_above(row[v], v, row[best], best)) best = v;
      am[n] = best;
    }
    const int32_t *par = parent + (size_t)bb * N, *dr = draft + (size_t)bb * N;
    int u = 0;
    for (;;) {
      int next = -1;
      for (int c = u + 1; c < N; ++c)
        if (par[c] == u && dr[c] == am[u]) {
          next = c;
          break;
        }
      if (next < 0) break;
      u = next;
    }
    accepted_out[bb] = u;
    next_out[bb] = am[u];
  }
  return LBXO_OK;
}

/* ---- DDTree construction from draft top-K scores ----------------------------
 *
 * Sources: Lucebox hub README, "Algorithms used" (DDTree: a tree-structured
 * verify that beats chain verify at the same budget), "Implemented here"
 * (budget 22 on the RTX 3090) and "GPU draft top-K & verify-argmax (DFlash)"
 * (the draft's top-K tokens, K in 1..8, and their log-sum-exp, per position).
 * The pages print no construction rule; the plain reading taken:
 *   - the draft gives, for each of the D positions after the root, its top-K
 *     tokens tok[d][k] with log-probabilities logp[d][k];
 *   - a node at depth d >= 1 is a choice of one of those K tokens at every
 *     position 0..d-1 along its path; its score is the sum of the path's
 *     log-probabilities, summed in fp32 from the root down (score(child) =
 *     score(parent) + logp[depth(parent)][k]);
 *   - the tree of budget B is built best first: starting from the root
 *     (score 0), repeatedly add the not-yet-added child of an added node with
 *     the highest score (ties: the lower parent index, then the lower k),
 *     until B nodes or no candidate is left; nodes are numbered in the order
 *     they are added, so parent[i] < i.  This keeps the B highest-scoring
 *     nodes, the tree that maximises the summed path probability when the
 *     draft's positions are taken as independent.
 * logp [Bq][D][K] fp32, tok [Bq][D][K] int32, root_tok [Bq] int32;
 * out: parent [Bq][B], token [Bq][B], depth [Bq][B] int32, score [Bq][B]
 * fp32, n_nodes [Bq] int32; unused node slots get parent -1, token -1,
 * depth -1, score 0.
 */
int lbxo_ddtree_build(int Bq, int D, int K, int B, const float *logp, const int32_t *tok,
                      const int32_t *root_tok, int32_t *parent, int32_t *token, int32_t *depth,
                      float *score, int32_t *n_nodes) {
  if (Bq < 1 || D < 0 || K < 1 || B < 1) return LBXO_EINVAL;
  int *slot = malloc((size_t)B * sizeof *slot); /* the k each node was chosen with */
  if (!slot) return LBXO_ENOMEM;
  for (int bb = 0; bb < Bq; ++bb) {
    const float *lp = logp + (size_t)bb * D * K;
    const int32_t *tk = tok + (size_t)bb * D * K;
    int32_t *par = parent + (size_t)bb * B, *tn = token + (size_t)bb * B,
            *dp = depth + (size_t)bb * B;
    float *sc = score + (size_t)bb * B;
    for (int i = 0; i < B; ++i) par[i] = -1, tn[i] = -1, dp[i] = -1, sc[i] = 0.0f, slot[i] = -1;
    tn[0] = root_tok[bb], dp[0] = 0;
    int n = 1;
    while (n < B) {
      /* every child (u, k) of an added node u that is not added yet */
      int bu = -1, bk = -1;
      float bs = 0.0f;
      for (int u = 0; u < n; ++u) {
        if (dp[u] >= D) continue;
        for (int k = 0; k < K; ++k) {
          int added = 0;
          for (int c = 1; c < n; ++c)
            if (par[c] == u && slot[c] == k) added = 1;
          if (added) continue;
          const float s = sc[u] + lp[dp[u] * K + k]; /* fp32, root down */
          /* scan order is (u, k) ascending: a strict > keeps the first of a tie */
          if (bu < 0 || s > bs) bu = u, bk = k, bs = s;
        }
      }
      if (bu < 0) break;
      par[n] = bu, slot[n] = bk, tn[n] = tk[dp[bu] * K + bk], dp[n] = dp[bu] + 1, sc[n] = bs;
      ++n;
    }
    n_nodes[bb] = n;
  }
  free(slot);
  return LBXO_OK;
}

/* ---- Tree-masked attention of the full-attention layers ---------------------
 *
 * Sources: Lucebox hub README -- DDTree verifies the whole draft tree in one
 * target forward ("Algorithms used": a tree-structured verify), and the
 * target is a hybrid whose full-attention layers keep a KV cache (flags
 * "--max-ctx N", the KV cache size, and "--fa-window N", default 0 = full
 * attention; a finite window drops the system prompt from the full-attention
 * layers).  The pages print no formula; the plain reading taken:
 *   - in the verify forward draft node n sits one position after its parent,
 *     so its query sees the request's cached context (positions
 *     0..ctx_len[b]-1) and the tree nodes on its own root path (its
 *     ancestors and itself), nothing else (full attention, no window);
 *   - query head hq reads KV head hq / (Hq/Hkv) (contiguous GQA groups);
 *   - o[n][hq] = sum_j softmax_j(scale * q.k_j) v_j over that key set.
 * Layers are a batch dimension sharing the tree and the context lengths:
 * q [L][Bq][N][Hq][dh], k_cache and v_cache [L][Bq][T][Hkv][dh], k_tree and
 * v_tree [L][Bq][N][Hkv][dh] (bf16 bit patterns); ctx_len [Bq] in 0..T,
 * parent [Bq][N]; o [L][Bq][N][Hq][dh] double out.
 */
int lbxo_tree_attention(int L, int Bq, int N, int Hq, int Hkv, int dh, int T,
                        const int32_t *ctx_len, double scale, const uint16_t *q,
                        const uint16_t *k_cache, const uint16_t *v_cache, const uint16_t *k_tree,
                        const uint16_t *v_tree, const int32_t *parent, double *o) {
  if (L < 1 || Bq < 1 || N < 1 || Hq < 1 || Hkv < 1 || dh < 1 || T < 0 || Hq % Hkv) return LBXO_EINVAL;
  for (int bb = 0; bb < Bq; ++bb) {
    if (ctx_len[bb] < 0 || ctx_len[bb] > T) return LBXO_EINVAL;
    if (lbxo_check_tree(parent + (size_t)bb * N, N) != LBXO_OK) return LBXO_ETREE;
  }
  const int G = Hq / Hkv;
  int *path = malloc((size_t)N * sizeof *path);
  double *s = malloc(((size_t)T + N) * sizeof *s);
  if (!path || !s) {
    free(path);
    free(s);
    return LBXO_ENOMEM;
  }
  for (int l = 0; l < L; ++l)
    for (int bb = 0; bb < Bq; ++bb) {
      const size_t lb = (size_t)l * Bq + bb;
      const int C = ctx_len[bb];
      const int32_t *par = parent + (size_t)bb * N;
      for (int n = 0; n < N; ++n) {
        int P = 0; /* the tree keys of node n: itself and its ancestors */
        for (int j = n; j >= 0; j = par[j]) path[P++] = j;
        for (int hq = 0; hq < Hq; ++hq) {
          const int g = hq / G;
          const uint16_t *qv = q + ((lb * N + n) * Hq + hq) * (size_t)dh;
          /* scores of the context keys, then of the path keys */
          for (int t = 0; t < C + P; ++t) {
            const uint16_t *kv = t < C ? k_cache + ((lb * T + t) * Hkv + g) * (size_t)dh
                                       : k_tree + ((lb * N + path[t - C]) * Hkv + g) * (size_t)dh;
            double dot = 0.0;
            for (int i = 0; i < dh; ++i) dot += bf16_to_double(qv[i]) * bf16_to_double(kv[i]);
            s[t] = scale * dot;
          }
          double mx = s[0];
          for (int t = 1; t < C + P; ++t)
            if (s[t] > mx) mx = s[t];
          double sum = 0.0;
          for (int t = 0; t < C + P; ++t) {
            s[t] = exp(s[t] - mx);
            sum += s[t];
          }
          double *out = o + ((lb * N + n) * Hq + hq) * (size_t)dh;
          for (int i = 0; i < dh; ++i) out[i] = 0.0;
          for (int t = 0; t < C + P; ++t) {
            const uint16_t *vv = t < C ? v_cache + ((lb * T + t) * Hkv + g) * (size_t)dh
                                       : v_tree + ((lb * N + path[t - C]) * Hkv + g) * (size_t)dh;
            const double p = s[t] / sum;
            for (int i = 0; i < dh; ++i) out[i] += p * bf16_to_double(vv[i]);
          }
        }
      }
    }
  free(path);
  free(s);
  return LBXO_OK;
}
