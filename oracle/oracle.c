/*
 * oracle.c -- plain, slow, fp64 CPU oracle for target-model tree verification.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header, table or helper
 * with the CUDA path.
 *
 * Sources (four web pages on speculative decoding; titles abbreviated):
 *   [EC]  "端云协同推测解码中草稿模型动态生成与验证并行化：探究树形注意力机制与显存碎片整理联合加速"
 *         (edge-cloud speculative decoding, tree attention and KV defragmentation)
 *   [LLM] "端侧大模型推测解码草稿模型动态剪枝策略：详解基于重要性采样的树形验证并行加速机制"
 *         (on-device LLM draft pruning with importance-sampling correction)
 *   [MM]  "端侧多模态大模型推测解码草稿模型动态剪枝：详解基于重要性采样的树形验证并行加速策略"
 *         (on-device multimodal draft pruning, importance-sampled tree verification)
 *
 * Two functions:
 *
 *   oracle_tree_attention_rows  -- dense masked attention in fp64, row by row:
 *       every query row (sequence b, tree node i, query head h) attends to all
 *       prefix keys of its sequence (gathered through the block table; [MM] §3.2
 *       "common-prefix merging": the prefix KV is stored once and reached through
 *       an index mapping) and to the tree keys j allowed by the tree mask of
 *       [EC] §2.2.2: M_tree[i,j] = 0 iff j is an ancestor of i or j == i, else
 *       -inf.  Ancestry is decided literally, by walking parent pointers up from
 *       i (parent = -1 at the root, [EC] appendix B "Tree_Parent_Idx").
 *       Softmax with max subtraction and the weighted sum of V, all in fp64.
 *       Inputs are bf16, or E4M3 codes with one fp32 scale per row of D
 *       elements (the FP8 KV cache with per-block scales that [EC] §9.3 and
 *       [LLM] §9.1 mention; one block = one row of a token and head): each
 *       element is decoded from the E4M3 definition (1 sign, 4 exponent bits
 *       with bias 7, 3 mantissa bits; exponent field 0 is subnormal; the
 *       all-ones pattern S.1111.111 is NaN; no infinities) and multiplied by
 *       its row's scale, exactly, in fp64.
 *
 *   oracle_accept -- the fused accept pass, one tree at a time:
 *       1. p, q of node i taken from the rows of its parent (the distribution
 *          the target/draft model produced after the parent token).
 *       2. pruning renormalisation ([LLM] §2.2.1-§2.2.2 and §7.1): on the
 *          retained set R_j the target and draft probabilities are divided by
 *          Z_j, the retained draft mass; off R_j both are zero (log space: add
 *          log(1/Z) on R, -inf elsewhere).  Z_j is the exact sum of the draft
 *          probabilities quantised to 2^-40, rounded once to fp32.
 *       3. per-node test u < min(1, p/q) ([EC] §2.2.3 step 1-2), evaluated as
 *          fl32(u*q) < p (strict; NaN rejects); variants: a calibration
 *          factor g, fl32(u*q) < fl32(g*p) ([MM] §3.3), and the log-space
 *          clamped test of [LLM] §10.2 (fp32, as the page states it).
 *       4. literal walk: depth-first from the root, children in increasing
 *          index order, descending only into accepted children ([EC] §2.2.3
 *          step 3: cut at the first rejection, keep the longest accepted
 *          path); the deepest node wins, ties to the smallest index.
 *       5. bonus token: a draw from the residual max(0, p - q) of the cut node
 *          when it has children, else from p (the resampling at rejection of
 *          [LLM] §1.2 step 3), with an exact fixed-point inverse CDF
 *          (quanta 2^-40, 64-bit sums, t = floor(u0 * S) in 128-bit integer).
 *   test 2 replaces steps 3-5 with the multi-candidate walk (siblings tried
 *       in order with residual updates, the multi-step speculative sampling
 *       of SpecInfer, which the pages cite among their sources; the pages
 *       themselves only say "resample at the rejection"): from the root, the
 *       children c of the current node j are tested in increasing index
 *       order against the current target distribution cur (at first p~_j):
 *       accept c iff fl32(u_c q~_j(x_c)) < fl32(g cur(x_c)); the first
 *       accepted child becomes the current node.  Each rejection replaces cur
 *       by its normalised residual: r = max(0, fl32(cur - q~_j)), S = sum of
 *       the 2^-40 quanta of r (exact), N = fp32(S 2^-40), cur = fl32(r / N)
 *       (cur kept when S = 0).  When every child is rejected the bonus is
 *       drawn from the last residual r (from cur when its S is 0); at a leaf
 *       from p~ of the leaf.  On a chain this is exactly steps 3-5.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared -pthread (no fast
 * math, no contraction: every fp32 product below is rounded once).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_TREE 5

/* ------------------------------------------------------------------------ */
/* bf16 -> fp64: a bf16 value is the upper half of an fp32 bit pattern, so   */
/* widening is exact.                                                         */
static double bf16_to_f64(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* E4M3 -> fp64 from the definition. */
static double e4m3_to_f64(uint8_t c) {
  const int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);          /* subnormal: 2^-6 * m/8 */
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7); /* normal: 2^(e-7) * (1 + m/8) */
  return sign ? -v : v;
}

/* Is j an ancestor of i, or i itself?  Literal parent-pointer walk. */
static int visible_tree_key(const int32_t *parent_local, int i, int j) {
  int k = i;
  while (k >= 0) {
    if (k == j) return 1;
    k = parent_local[k];
  }
  return 0;
}

typedef struct {
  int batch, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq;
  double scale;
  const void *q;              /* [total_nodes][Hq][D] bf16 bits (or E4M3) */
  const void *k_prefix;       /* [num_blocks][Hkv][block_size][D]        */
  const void *v_prefix;
  const int32_t *block_table; /* [batch][max_blocks_per_seq]             */
  const void *k_nodes;        /* [total_nodes][Hkv][D]                   */
  const void *v_nodes;
  const int32_t *parent;      /* [total_nodes], local, -1 at the root    */
  const int32_t *prefix_lens; /* [batch]                                 */
  const int32_t *node_offsets;/* [batch+1]                               */
  int dtype;                  /* 0: bf16; 1: E4M3 codes with row scales  */
  /* E4M3 only: one fp32 scale per row of D elements, indexed like the rows:
   * q [total_nodes][Hq], k/v prefix [num_blocks][Hkv][block_size],
   * k/v nodes [total_nodes][Hkv].  q, k_prefix, ... then point to uint8. */
  const float *q_scale, *k_prefix_scale, *v_prefix_scale, *k_nodes_scale, *v_nodes_scale;
} oracle_attn_args;

/* Row `row` (D elements) of an input tensor, widened to fp64. */
static void load_row(const oracle_attn_args *a, const void *base, const float *scales, size_t row,
                     double *dst) {
  const int D = a->head_dim;
  if (a->dtype == 0) {
    const uint16_t *p = (const uint16_t *)base + row * (size_t)D;
    for (int d = 0; d < D; ++d) dst[d] = bf16_to_f64(p[d]);
  } else {
    const uint8_t *p = (const uint8_t *)base + row * (size_t)D;
    const double sc = (double)scales[row];
    for (int d = 0; d < D; ++d) dst[d] = e4m3_to_f64(p[d]) * sc;
  }
}

typedef struct {
  const oracle_attn_args *a;
  const int32_t *rows; /* [nrows][3] = (b, local node i, q head h) */
  int nrows;
  double *out;         /* [nrows][D] */
  int next;            /* shared work counter */
  pthread_mutex_t lock;
} attn_job;

static void attn_one_row(const oracle_attn_args *a, int b, int i, int h, double *o) {
  const int D = a->head_dim, Hq = a->num_q_heads, Hkv = a->num_kv_heads;
  const int g = Hq / Hkv;
  const int kvh = h / g; /* query head h reads KV head floor(h/g) */
  const int L = a->prefix_lens[b];
  const int n0 = a->node_offsets[b], N = a->node_offsets[b + 1] - n0;
  const int nkeys = L + N;
  double *s = (double *)malloc(sizeof(double) * (size_t)(nkeys > 0 ? nkeys : 1));
  unsigned char *vis = (unsigned char *)malloc((size_t)(nkeys > 0 ? nkeys : 1));
  double qd[512], kv[512];
  load_row(a, a->q, a->q_scale, (size_t)(n0 + i) * Hq + h, qd);

  /* 1. key list [prefix 0..L-1 ; tree nodes 0..N-1] and dense scores */
  for (int t = 0; t < nkeys; ++t) {
    if (t < L) {
      int page = a->block_table[(size_t)b * a->max_blocks_per_seq + t / a->block_size];
      int slot = t % a->block_size;
      load_row(a, a->k_prefix, a->k_prefix_scale, ((size_t)page * Hkv + kvh) * a->block_size + slot, kv);
      vis[t] = 1; /* the committed prefix is visible to every node */
    } else {
      int j = t - L;
      load_row(a, a->k_nodes, a->k_nodes_scale, (size_t)(n0 + j) * Hkv + kvh, kv);
      vis[t] = (unsigned char)visible_tree_key(a->parent + n0, i, j);
    }
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += qd[d] * kv[d];
    s[t] = acc * a->scale;
  }
  /* 2. softmax over the visible keys (mask = -inf elsewhere) */
  double m = -INFINITY;
  for (int t = 0; t < nkeys; ++t)
    if (vis[t] && s[t] > m) m = s[t];
  double l = 0.0;
  for (int t = 0; t < nkeys; ++t) {
    s[t] = vis[t] ? exp(s[t] - m) : 0.0;
    l += s[t];
  }
  /* 3. o = sum_t softmax_t * v_t */
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  for (int t = 0; t < nkeys; ++t) {
    if (!vis[t]) continue;
    if (t < L) {
      int page = a->block_table[(size_t)b * a->max_blocks_per_seq + t / a->block_size];
      int slot = t % a->block_size;
      load_row(a, a->v_prefix, a->v_prefix_scale, ((size_t)page * Hkv + kvh) * a->block_size + slot, kv);
    } else {
      load_row(a, a->v_nodes, a->v_nodes_scale, (size_t)(n0 + (t - L)) * Hkv + kvh, kv);
    }
    double w = s[t] / l;
    for (int d = 0; d < D; ++d) o[d] += w * kv[d];
  }
  free(s);
  free(vis);
}

static void *attn_worker(void *arg) {
  attn_job *job = (attn_job *)arg;
  for (;;) {
    pthread_mutex_lock(&job->lock);
    int r = job->next++;
    pthread_mutex_unlock(&job->lock);
    if (r >= job->nrows) break;
    const int32_t *row = job->rows + 3 * (size_t)r;
    attn_one_row(job->a, row[0], row[1], row[2], job->out + (size_t)r * job->a->head_dim);
  }
  return NULL;
}

/* Computes the listed output rows.  Returns 0, or -1 on an unsupported size. */
int oracle_tree_attention_rows(const oracle_attn_args *a, int nrows, const int32_t *rows,
                               double *out, int nthreads) {
  if (a->head_dim > 512 || a->num_kv_heads <= 0 || a->num_q_heads % a->num_kv_heads) return -1;
  if (a->dtype != 0 && a->dtype != 1) return -1;
  if (a->dtype == 1 && (!a->q_scale || !a->k_prefix_scale || !a->v_prefix_scale ||
                        !a->k_nodes_scale || !a->v_nodes_scale))
    return -1;
  attn_job job;
  job.a = a;
  job.rows = rows;
  job.nrows = nrows;
  job.out = out;
  job.next = 0;
  pthread_mutex_init(&job.lock, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, attn_worker, &job);
  attn_worker(&job);
  for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
  pthread_mutex_destroy(&job.lock);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Accept.                                                                    */

typedef struct {
  int batch, vocab, kind; /* kind: 0 = probabilities, 1 = logits (target only) */
  int max_nodes;
  const float *target;          /* [total_nodes][V] */
  const float *draft_probs;     /* [total_nodes][V] */
  const int32_t *draft_tokens;  /* [total_nodes]    */
  const int32_t *parent;        /* [total_nodes]    */
  const int32_t *node_offsets;  /* [batch+1]        */
  const float *uniforms;        /* [total_nodes]    */
  const uint32_t *retained_mask;/* NULL or [total_nodes][ceil(V/32)] */
  int32_t *accepted_len;        /* [batch] */
  int32_t *path;                /* [batch][max_nodes] */
  int32_t *bonus_token;         /* [batch] */
  int32_t *status;              /* [batch] */
  float *pq_out;                /* NULL or [total_nodes][2] */
  int test;                     /* 0: ratio test, 1: log-space clamped test, 2: multi-candidate */
  float log_clamp;              /* L of the clamped test */
  const float *gamma;           /* NULL or [batch] calibration factors */
} oracle_accept_args;

static const double TWO40 = 1099511627776.0; /* 2^40 */

/* Target probability row j of tree (base row n0+j): probs as given, or the
 * fp64 softmax of the logits rounded once to fp32. */
static void target_prob_row(const oracle_accept_args *a, size_t row, float *dst) {
  const int V = a->vocab;
  const float *t = a->target + row * (size_t)V;
  if (a->kind == 0) {
    memcpy(dst, t, sizeof(float) * (size_t)V);
    return;
  }
  double m = -INFINITY;
  for (int v = 0; v < V; ++v)
    if ((double)t[v] > m) m = (double)t[v];
  double s = 0.0;
  for (int v = 0; v < V; ++v) s += exp((double)t[v] - m);
  double lse = m + log(s);
  for (int v = 0; v < V; ++v) dst[v] = (float)exp((double)t[v] - lse);
}

static int in_retained(const oracle_accept_args *a, size_t row, int v) {
  if (!a->retained_mask) return 1;
  const int W = (a->vocab + 31) / 32;
  return (int)((a->retained_mask[row * (size_t)W + (size_t)(v / 32)] >> (v % 32)) & 1u);
}

/* Z_j = fp32_RN( sum_{v in R_j} floor(q_{j,v} * 2^40) * 2^-40 ): the sum is
 * an exact 64-bit integer, converted to fp32 with one rounding. */
static float retained_mass(const oracle_accept_args *a, size_t row) {
  const int V = a->vocab;
  const float *q = a->draft_probs + row * (size_t)V;
  uint64_t s = 0;
  for (int v = 0; v < V; ++v)
    if (in_retained(a, row, v)) {
      float x = q[v];
      if (!(x > 0.0f)) continue;      /* negative, zero or NaN mass counts 0 */
      if (x > 32.0f) x = 32.0f;
      s += (uint64_t)((double)x * TWO40);
    }
  float z = (float)s; /* integer -> fp32, round to nearest even */
  return z * 0x1p-40f; /* exact power-of-two scaling */
}

/* The fixed-point quantum of a residual mass: clamp to [0, 32] (NaN -> 0),
 * then floor(r * 2^40). */
static uint64_t quantise(float r) {
  if (!(r > 0.0f)) return 0;
  if (r > 32.0f) r = 32.0f;
  return (uint64_t)((double)r * TWO40);
}

/* t = floor(u * S) exactly, for u an fp32 in [0,1) and S < 2^64. */
static uint64_t scaled_draw(float u, uint64_t S) {
  if (!(u > 0.0f)) return 0;
  int e;
  float fr = frexpf(u, &e);                     /* u = fr * 2^e, fr in [0.5, 1) */
  uint64_t m = (uint64_t)ldexpf(fr, 24);        /* 24-bit integer mantissa */
  int sh = 24 - e;                              /* u = m * 2^-sh, sh >= 24 */
  unsigned __int128 prod = (unsigned __int128)m * (unsigned __int128)S;
  if (sh >= 128) return 0;
  return (uint64_t)(prod >> sh);
}

typedef struct {
  const oracle_accept_args *a;
  int next;
  pthread_mutex_t lock;
} accept_job;

static void dfs_deepest(const int32_t *parent, const unsigned char *acc, int N, int node, int depth,
                        int *best, int *best_depth) {
  if (depth > *best_depth || (depth == *best_depth && node < *best)) {
    *best = node;
    *best_depth = depth;
  }
  for (int c = node + 1; c < N; ++c)
    if (parent[c] == node && acc[c]) dfs_deepest(parent, acc, N, c, depth + 1, best, best_depth);
}

/* p~ and q~ of row `row` (whole vocabulary): renormalised on the retained set
 * when a mask is given (0 off it), else as given. */
static void tilde_rows(const oracle_accept_args *a, size_t row, float *prow, float *ptil, float *qtil) {
  const int V = a->vocab;
  target_prob_row(a, row, prow);
  const float *qrow = a->draft_probs + row * (size_t)V;
  const float z = a->retained_mask ? retained_mass(a, row) : 1.0f;
  for (int v = 0; v < V; ++v) {
    if (a->retained_mask) {
      if (in_retained(a, row, v)) {
        ptil[v] = prow[v] / z;
        qtil[v] = qrow[v] / z;
      } else {
        ptil[v] = 0.0f;
        qtil[v] = 0.0f;
      }
    } else {
      ptil[v] = prow[v];
      qtil[v] = qrow[v];
    }
  }
}

/* The exact fixed-point inverse-CDF draw over quanta of w[0..V) with u0;
 * -1 when all quanta are 0. */
static int draw_quanta(const float *w, int V, float u0) {
  uint64_t S = 0;
  for (int v = 0; v < V; ++v) S += quantise(w[v]);
  if (S == 0) return -1;
  uint64_t t = scaled_draw(u0, S), cum = 0;
  for (int v = 0; v < V; ++v) {
    cum += quantise(w[v]);
    if (cum > t) return v;
  }
  return -1;
}

/* Smallest index of the largest entry (NaN ignored). */
static int argmax_row(const float *w, int V) {
  int token = 0;
  float best = -INFINITY;
  for (int v = 0; v < V; ++v)
    if (w[v] > best) {
      best = w[v];
      token = v;
    }
  return token;
}

/* Multi-candidate walk (test 2), the tree already validated. */
static void accept_one_tree_multi(const oracle_accept_args *a, int b, float g) {
  const int V = a->vocab;
  const int n0 = a->node_offsets[b];
  const int N = a->node_offsets[b + 1] - n0;
  const int32_t *par = a->parent + n0;
  const int32_t *tok = a->draft_tokens + n0;
  int32_t *path = a->path + (size_t)b * a->max_nodes;
  float *prow = (float *)malloc(sizeof(float) * (size_t)V);
  float *cur = (float *)malloc(sizeof(float) * (size_t)V);
  float *qtil = (float *)malloc(sizeof(float) * (size_t)V);
  float *res = (float *)malloc(sizeof(float) * (size_t)V);
  if (a->pq_out)
    for (int i = 0; i < N; ++i) {
      a->pq_out[2 * (size_t)(n0 + i) + 0] = 0.0f;
      a->pq_out[2 * (size_t)(n0 + i) + 1] = 0.0f;
    }
  int j = 0, len = 0, token = -1;
  for (;;) {
    tilde_rows(a, (size_t)(n0 + j), prow, cur, qtil);  /* cur = p~_j */
    int next = -1, rejected = 0;
    uint64_t last_S = 0;
    for (int c = j + 1; c < N && next < 0; ++c) {
      if (par[c] != j) continue;
      const float p = cur[tok[c]], q = qtil[tok[c]];
      if (a->pq_out) {
        a->pq_out[2 * (size_t)(n0 + c) + 0] = p;
        a->pq_out[2 * (size_t)(n0 + c) + 1] = q;
      }
      const float uq = a->uniforms[n0 + c] * q;
      const float gp = g * p;
      if (uq < gp) {
        next = c;
        break;
      }
      /* rejected: cur <- its normalised residual */
      uint64_t S = 0;
      for (int v = 0; v < V; ++v) {
        const float d = cur[v] - qtil[v];
        res[v] = d > 0.0f ? d : 0.0f;
        S += quantise(res[v]);
      }
      rejected = 1;
      last_S = S;
      if (S > 0) {
        const float Nf = (float)S * 0x1p-40f;
        for (int v = 0; v < V; ++v) cur[v] = res[v] / Nf;
      }
    }
    if (next >= 0) {
      path[len++] = next;
      j = next;
      continue;
    }
    const float u0 = a->uniforms[n0];
    if (rejected && last_S > 0) token = draw_quanta(res, V, u0);
    if (token < 0) token = draw_quanta(cur, V, u0);  /* a leaf, or an empty residual */
    if (token < 0) token = argmax_row(cur, V);
    break;
  }
  a->accepted_len[b] = len;
  a->bonus_token[b] = token;
  a->status[b] = ORACLE_OK;
  free(prow);
  free(cur);
  free(qtil);
  free(res);
}

static void accept_one_tree(const oracle_accept_args *a, int b) {
  const int V = a->vocab;
  const int n0 = a->node_offsets[b];
  const int N = a->node_offsets[b + 1] - n0;
  const int32_t *par = a->parent + n0;
  const int32_t *tok = a->draft_tokens + n0;
  int32_t *path = a->path + (size_t)b * a->max_nodes;
  for (int k = 0; k < a->max_nodes; ++k) path[k] = -1;

  /* validation of the tree and the tokens */
  int bad = (N < 1 || N > a->max_nodes);
  if (!bad && par[0] != -1) bad = 1;
  const float g = a->gamma ? a->gamma[b] : 1.0f;
  if (!(g > 0.0f && g <= 3.0e38f)) bad = 1; /* the calibration factor must be positive, finite */
  for (int i = 1; !bad && i < N; ++i)
    if (par[i] < 0 || par[i] >= i || tok[i] < 0 || tok[i] >= V) bad = 1;
  if (bad) {
    a->status[b] = ORACLE_BAD_TREE;
    a->accepted_len[b] = -1;
    a->bonus_token[b] = -1;
    return;
  }
  if (a->test == 2) {
    accept_one_tree_multi(a, b, g);
    return;
  }

  float *prow = (float *)malloc(sizeof(float) * (size_t)V);
  size_t prow_of = (size_t)-1; /* which row prow holds (logits mode) */
  float *pt = (float *)malloc(sizeof(float) * (size_t)N);
  float *qt = (float *)malloc(sizeof(float) * (size_t)N);
  unsigned char *acc = (unsigned char *)calloc((size_t)N, 1);

  /* 1.-3. per tested node i >= 1: p~, q~ from the parent's rows, then the test */
  for (int i = 1; i < N; ++i) {
    const size_t row = (size_t)(n0 + par[i]);
    const int x = tok[i];
    float p, q;
    if (a->kind == 0) {
      p = a->target[row * (size_t)V + (size_t)x];
    } else {
      if (prow_of != row) target_prob_row(a, row, prow);
      prow_of = row;
      p = prow[x];
    }
    q = a->draft_probs[row * (size_t)V + (size_t)x];
    if (a->retained_mask) {
      if (in_retained(a, row, x)) {
        float z = retained_mass(a, row);
        p = p / z;
        q = q / z;
      } else {
        p = 0.0f;
        q = 0.0f;
      }
    }
    pt[i] = p;
    qt[i] = q;
    const float u = a->uniforms[n0 + i];
    if (a->test == 0) {
      /* u < min(1, g p/q) ([MM] §3.3 calibration factor g; g = 1 is the
       * plain test), as fl32(u q) < fl32(g p) */
      float uq = u * q;
      float gp = g * p;
      acc[i] = (unsigned char)(uq < gp);
    } else {
      /* [LLM] §10.2 log-space test: r = clamp(log p - log q + log g, -L, L),
       * accept iff u < (r >= 0 ? 1 : exp(r)); p = 0 or a NaN r rejects */
      float r = (logf(p) - logf(q)) + logf(g);
      if (!(p > 0.0f) || r != r) {
        acc[i] = 0;
      } else {
        float rc = fmaxf(fminf(r, a->log_clamp), -a->log_clamp);
        acc[i] = (unsigned char)(u < (rc >= 0.0f ? 1.0f : expf(rc)));
      }
    }
  }
  if (a->pq_out) {
    a->pq_out[2 * (size_t)n0 + 0] = 0.0f;
    a->pq_out[2 * (size_t)n0 + 1] = 0.0f;
    for (int i = 1; i < N; ++i) {
      a->pq_out[2 * (size_t)(n0 + i) + 0] = pt[i];
      a->pq_out[2 * (size_t)(n0 + i) + 1] = qt[i];
    }
  }

  /* 4. the walk */
  int best = 0, best_depth = 0;
  dfs_deepest(par, acc, N, 0, 0, &best, &best_depth);
  a->accepted_len[b] = best_depth;
  for (int k = best_depth - 1, v = best; k >= 0; --k, v = par[v]) path[k] = v;

  /* 5. bonus token at the cut node */
  const size_t crow = (size_t)(n0 + best);
  int has_children = 0;
  for (int i = best + 1; i < N; ++i)
    if (par[i] == best) has_children = 1;
  target_prob_row(a, crow, prow);
  const float *qrow = a->draft_probs + crow * (size_t)V;
  float z = a->retained_mask ? retained_mass(a, crow) : 1.0f;
  float *ptil = (float *)malloc(sizeof(float) * (size_t)V);
  float *qtil = (float *)malloc(sizeof(float) * (size_t)V);
  for (int v = 0; v < V; ++v) {
    if (a->retained_mask) {
      if (in_retained(a, crow, v)) {
        ptil[v] = prow[v] / z;
        qtil[v] = qrow[v] / z;
      } else {
        ptil[v] = 0.0f;
        qtil[v] = 0.0f;
      }
    } else {
      ptil[v] = prow[v];
      qtil[v] = qrow[v];
    }
  }
  const float u0 = a->uniforms[n0];
  int token = -1;
  for (int pass = has_children ? 0 : 1; pass < 2 && token < 0; ++pass) {
    /* pass 0: residual max(0, p~ - q~); pass 1: p~ itself */
    uint64_t S = 0;
    for (int v = 0; v < V; ++v) S += quantise(pass == 0 ? ptil[v] - qtil[v] : ptil[v]);
    if (S == 0) continue;
    uint64_t t = scaled_draw(u0, S);
    uint64_t cum = 0;
    for (int v = 0; v < V; ++v) {
      cum += quantise(pass == 0 ? ptil[v] - qtil[v] : ptil[v]);
      if (cum > t) {
        token = v;
        break;
      }
    }
  }
  if (token < 0) { /* no mass at all: smallest index of the largest p~ (NaN ignored) */
    token = 0;
    float bestp = -INFINITY;
    for (int v = 0; v < V; ++v)
      if (ptil[v] > bestp) {
        bestp = ptil[v];
        token = v;
      }
  }
  a->bonus_token[b] = token;
  a->status[b] = ORACLE_OK;
  free(prow);
  free(pt);
  free(qt);
  free(acc);
  free(ptil);
  free(qtil);
}

static void *accept_worker(void *arg) {
  accept_job *job = (accept_job *)arg;
  for (;;) {
    pthread_mutex_lock(&job->lock);
    int b = job->next++;
    pthread_mutex_unlock(&job->lock);
    if (b >= job->a->batch) break;
    accept_one_tree(job->a, b);
  }
  return NULL;
}

int oracle_accept(const oracle_accept_args *a, int nthreads) {
  if (a->vocab <= 0 || a->max_nodes <= 0) return -1;
  accept_job job;
  job.a = a;
  job.next = 0;
  pthread_mutex_init(&job.lock, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, accept_worker, &job);
  accept_worker(&job);
  for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
  pthread_mutex_destroy(&job.lock);
  return 0;
}

/* Exposed for the pins: the fixed-point pieces on their own. */
uint64_t oracle_quantise(float r) { return quantise(r); }
double oracle_e4m3_to_f64(uint8_t c) { return e4m3_to_f64(c); }
uint64_t oracle_scaled_draw(float u, uint64_t S) { return scaled_draw(u, S); }
float oracle_retained_mass_row(const float *q, const uint32_t *mask, int vocab) {
  oracle_accept_args a;
  memset(&a, 0, sizeof a);
  a.vocab = vocab;
  a.draft_probs = q;
  a.retained_mask = mask;
  return retained_mass(&a, 0);
}

/* ------------------------------------------------------------------------
 * oracle_retained_set_row -- the retained set R of one draft row, the step
 * before the accept pass ([LLM] §2.1.2 "soft truncation" by cumulative
 * probability mass: tokens in descending draft probability, mass Q summed
 * until Q >= 1 - Prune_Ratio, the crossing token kept; [LLM] §7.1 the same
 * decision in log space).  Read exactly: tokens ordered by key desc, id asc,
 * with key = q if q > 0 else 0 (NaN and negatives count as 0); the set is the
 * shortest prefix of that order whose exact fixed-point mass sum of
 * quantise(q) reaches T (T = floor(mass * 2^40) >= 1, computed by the
 * caller); if no prefix does, every token.  Z = the set's fixed-point sum.
 * Writes the packed mask (bit v%32 of word v/32), *z_fixed, *z (Z rounded
 * once to fp32, times 2^-40) and *kept.
 * ------------------------------------------------------------------------ */
typedef struct {
  float key;
  int id;
} rs_item;

static int rs_cmp(const void *a, const void *b) {
  const rs_item *x = (const rs_item *)a, *y = (const rs_item *)b;
  if (x->key > y->key) return -1;
  if (x->key < y->key) return 1;
  return (x->id > y->id) - (x->id < y->id);
}

int oracle_retained_set_row(const float *q, int vocab, uint64_t T, uint32_t *mask,
                            uint64_t *z_fixed, float *z, int *kept) {
  if (vocab < 1 || T < 1) return 1;
  rs_item *it = (rs_item *)malloc(sizeof(rs_item) * (size_t)vocab);
  if (!it) return 1;
  for (int v = 0; v < vocab; ++v) {
    it[v].key = (q[v] > 0.0f) ? q[v] : 0.0f;
    it[v].id = v;
  }
  qsort(it, (size_t)vocab, sizeof(rs_item), rs_cmp);
  const int words = (vocab + 31) / 32;
  memset(mask, 0, sizeof(uint32_t) * (size_t)words);
  uint64_t cum = 0;
  int n = 0;
  while (n < vocab) {
    cum += quantise(it[n].key);
    const int id = it[n].id;
    mask[id >> 5] |= 1u << (id & 31);
    ++n;
    if (cum >= T) break;
  }
  *z_fixed = cum;
  *z = (float)cum * 0x1p-40f; /* one rounding of the sum, then exact scaling */
  *kept = n;
  free(it);
  return 0;
}
