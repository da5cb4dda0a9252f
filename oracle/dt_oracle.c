/*
 * dt_oracle.c -- plain CPU oracle of the DominoTree per-round conditional
 * draft-tree builder and of Domino's chain decoder (orc_chain, at the end).
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load, call or link this file. The CUDA
 * product path never does, and the two share no code: this file has its own
 * bf16 decoding, dot products, GRU cell, softmax, selection and search.
 *
 * Sources (page title, then section):
 *  [DOM]  "Domino：在投机解码中将因果建模与自回归草稿解耦" (Domino: decoupling
 *         causal modelling from autoregressive drafting; paper.rainbus.top/paper/2605.29707): core method (GRU causal state
 *         S_{i-1} = GRU(E_{<=i-1}), correction dL_i = W2 SiLU(W1 [H_i; S_{i-1}]),
 *         r = 256, final logits L_i = L_base^i + dL_i); method steps (block
 *         [x_t, MASK, ...] of size B, base logits for i = t+1 .. t+B-1).
 *  [TREE] "Riassunto Tecnico: DominoTree" (gist.science/it/paper/2607.08642):
 *         Componenti Core 1 (best-first max-heap on cumulative path
 *         log-probability, children scored by re-running the correction along
 *         the node's path, H_i shared), 2 (correction restricted to the top-M
 *         marginal candidates of each depth, then top-k children), 4 (fixed
 *         node budget), 5 (ancestor attention mask).
 *  [SUM]  "DominoTree：条件树草稿生成加速大模型推测解码" (aimsg.uk summary):
 *         core content (pick the best-scoring leaf, add its candidate children).
 *
 * Numerics (fixed definition, documented with the build):
 *  - values are stored as fp32; bf16 weights are decoded exactly;
 *  - every dot product is accumulated in fp64 and rounded once to fp32;
 *  - every elementwise expression is evaluated in fp64 from fp32 operands and
 *    rounded once to fp32;
 *  - the log-sum-exp is summed in fp64 in candidate order;
 *  - all decisions (top-M, top-k, heap order) compare fp32 values, the
 *    precision the CUDA path decides in.
 *
 * Readings of points the pages leave open (each one also listed with the build's
 * design notes):
 *  - log-probabilities are the log-softmax over the M corrected candidates;
 *  - the root state is GRU(state0, E[anchor]) (block position 0 is the anchor);
 *  - GRU gates follow the usual r, z, n convention, rows ordered r, z, n;
 *  - N counts non-root nodes; the N-th pop and depth-D nodes are not expanded;
 *  - ties: top-M and top-k prefer the lower token id; the frontier prefers the
 *    earlier push (push order = parent order, then child rank);
 *  - temperature divides the corrected logits; T == 0 builds with T = 1.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_BF16 1

#define ORC_OK 0
#define ORC_EINVAL (-1)
#define ORC_ENONFINITE (-4)
#define ORC_ENOMEM (-6)

typedef struct {
  int V, d, d_s, r, D, M, k, N, wdtype;
  const void *E;      /* [V][d]        */
  const void *W_ih;   /* [3 d_s][d]    */
  const void *W_hh;   /* [3 d_s][d_s]  */
  const float *b_ih;  /* [3 d_s] or NULL */
  const float *b_hh;  /* [3 d_s] or NULL */
  const void *W1;     /* [r][d + d_s]  */
  const void *W2;     /* [V][r]        */
} orc_model;

typedef struct {
  const float *base;    /* [D][V] base logits of depths 1..D */
  const float *H;       /* [D][d] backbone states of depths 1..D */
  const float *state0;  /* [d_s] initial GRU state */
  int32_t anchor;
  float temperature;
} orc_request;

typedef struct {
  int32_t *tokens, *parents, *depths; /* [N+1] */
  float *scores;                      /* [N+1] */
  uint8_t *mask;                      /* [(N+1)*(N+1)] or NULL */
  int32_t *topm;                      /* [D][M] or NULL */
  int32_t n_nodes;                    /* out: rows filled, root included */
  int32_t n_expanded;                 /* out: expansions performed */
} orc_tree;

/* ---------------------------------------------------------------- helpers */

static float bf16_decode(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

static float weight_at(const void *w, int wdtype, size_t i) {
  return wdtype == ORC_BF16 ? bf16_decode(((const uint16_t *)w)[i]) : ((const float *)w)[i];
}

/* fl32( sum_i w[off + i] * x[i] ), accumulated in fp64 */
static float dot_w(const void *w, int wdtype, size_t off, const float *x, int n) {
  double acc = 0.0;
  if (wdtype == ORC_BF16) {
    const uint16_t *p = (const uint16_t *)w + off;
    for (int i = 0; i < n; ++i) acc += (double)bf16_decode(p[i]) * (double)x[i];
  } else {
    const float *p = (const float *)w + off;
    for (int i = 0; i < n; ++i) acc += (double)p[i] * (double)x[i];
  }
  return (float)acc;
}

static double sigmoid64(double x) { return 1.0 / (1.0 + exp(-x)); }

/* ------------------------------------------------------------- top-M (a1) */

static _Thread_local const float *g_sort_row; /* qsort has no context argument */

/* (value desc, id asc); -0.0 and +0.0 compare equal as floats. */
static int cmp_value_desc_id_asc(const void *pa, const void *pb) {
  int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
  float va = g_sort_row[a], vb = g_sort_row[b];
  if (va > vb) return -1;
  if (va < vb) return 1;
  return (a < b) ? -1 : (a > b);
}

/* Top-M marginal candidates of one depth ([TREE] Componenti Core 2): the M
 * token ids of `row` sorted by (value desc, id asc). Returns ORC_ENONFINITE
 * when the row holds a NaN or +inf. */
int orc_topm(const float *row, int V, int M, int32_t *ids_out) {
  if (!row || !ids_out || V <= 0 || M <= 0 || M > V) return ORC_EINVAL;
  for (int v = 0; v < V; ++v)
    if (isnan(row[v]) || (isinf(row[v]) && row[v] > 0)) return ORC_ENONFINITE;
  int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * (size_t)V);
  if (!idx) return ORC_ENOMEM;
  for (int v = 0; v < V; ++v) idx[v] = v;
  g_sort_row = row;
  qsort(idx, (size_t)V, sizeof(int32_t), cmp_value_desc_id_asc);
  memcpy(ids_out, idx, sizeof(int32_t) * (size_t)M);
  free(idx);
  return ORC_OK;
}

/* -------------------------------------------------------- GRU cell (a3/a5) */

/* s_out = GRU(s, x) with gates r, z, n ([DOM] core method names the causal
 * encoder a GRU; the gate convention is the standard one):
 *   r  = sigma(W_ir x + b_ir + W_hr s + b_hr)
 *   z  = sigma(W_iz x + b_iz + W_hz s + b_hz)
 *   n  = tanh(W_in x + b_in + r * (W_hn s + b_hn))
 *   s' = (1 - z) * n + z * s                                                  */
void orc_gru_step(int d, int d_s, int wdtype, const void *W_ih, const void *W_hh,
                  const float *b_ih, const float *b_hh, const float *x, const float *s,
                  float *s_out) {
  for (int i = 0; i < d_s; ++i) {
    float gi[3], gh[3];
    double bi[3], bh[3];
    for (int g = 0; g < 3; ++g) {
      size_t row = (size_t)g * d_s + i;
      gi[g] = dot_w(W_ih, wdtype, row * (size_t)d, x, d);
      gh[g] = dot_w(W_hh, wdtype, row * (size_t)d_s, s, d_s);
      bi[g] = b_ih ? (double)b_ih[row] : 0.0;
      bh[g] = b_hh ? (double)b_hh[row] : 0.0;
    }
    float r = (float)sigmoid64((double)gi[0] + bi[0] + (double)gh[0] + bh[0]);
    float z = (float)sigmoid64((double)gi[1] + bi[1] + (double)gh[1] + bh[1]);
    float n = (float)tanh((double)gi[2] + bi[2] + (double)r * ((double)gh[2] + bh[2]));
    s_out[i] = (float)((1.0 - (double)z) * (double)n + (double)z * (double)s[i]);
  }
}

static void embed(const orc_model *m, int32_t tok, float *x) {
  for (int i = 0; i < m->d; ++i) x[i] = weight_at(m->E, m->wdtype, (size_t)tok * m->d + i);
}

/* ------------------------------------------------ scoring one expansion */

typedef struct {
  const orc_model *m;
  const orc_request *q;
  int32_t *cand;   /* [D][M]  top-M ids, depth j at row j-1 */
  float *U;        /* [D][r]  W1[:, :d] . H_j               */
  float *x, *h, *p, *L, *lp;
  int32_t *order;
  float Teff;
} orc_ctx;

static void ctx_free(orc_ctx *c) {
  free(c->cand); free(c->U); free(c->x); free(c->h); free(c->p); free(c->L); free(c->lp);
  free(c->order);
}

static int ctx_init(orc_ctx *c, const orc_model *m, const orc_request *q) {
  memset(c, 0, sizeof *c);
  c->m = m; c->q = q;
  if (!(q->temperature >= 0.0f) || isinf(q->temperature)) return ORC_EINVAL;
  c->Teff = (q->temperature == 0.0f) ? 1.0f : q->temperature; /* T = 0: greedy reading */
  c->cand = (int32_t *)malloc(sizeof(int32_t) * (size_t)m->D * m->M);
  c->U = (float *)malloc(sizeof(float) * (size_t)m->D * m->r);
  c->x = (float *)malloc(sizeof(float) * (size_t)m->d);
  c->h = (float *)malloc(sizeof(float) * (size_t)m->r);
  c->p = (float *)malloc(sizeof(float) * (size_t)m->r);
  c->L = (float *)malloc(sizeof(float) * (size_t)m->M);
  c->lp = (float *)malloc(sizeof(float) * (size_t)m->M);
  c->order = (int32_t *)malloc(sizeof(int32_t) * (size_t)m->M);
  if (!c->cand || !c->U || !c->x || !c->h || !c->p || !c->L || !c->lp || !c->order) {
    ctx_free(c);
    return ORC_ENOMEM;
  }
  /* (a1) candidates of every depth */
  for (int j = 0; j < m->D; ++j) {
    int rc = orc_topm(q->base + (size_t)j * m->V, m->V, m->M, c->cand + (size_t)j * m->M);
    if (rc) { ctx_free(c); return rc; }
  }
  /* (a2) path-independent half of the correction, once per depth:
   * U_j = W1[:, :d] . H_j  ([TREE] Componenti Core 1: H_i is shared) */
  for (int j = 0; j < m->D; ++j)
    for (int t = 0; t < m->r; ++t)
      c->U[(size_t)j * m->r + t] = dot_w(m->W1, m->wdtype, (size_t)t * (m->d + m->d_s),
                                         q->H + (size_t)j * m->d, m->d);
  return ORC_OK;
}

static _Thread_local const float *g_sort_L;
static _Thread_local const int32_t *g_sort_cand;
/* children order: (corrected logit desc, token id asc) */
static int cmp_child(const void *pa, const void *pb) {
  int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
  float la = g_sort_L[a], lb = g_sort_L[b];
  if (la > lb) return -1;
  if (la < lb) return 1;
  int32_t ta = g_sort_cand[a], tb = g_sort_cand[b];
  return (ta < tb) ? -1 : (ta > tb);
}

/* Score the M candidates of child depth j (1-based) for a node whose GRU state
 * is S, ([DOM] core method, [TREE] Componenti Core 2):
 *   h      = SiLU(U_j + W1[:, d:] . S)
 *   L_c    = (L_base^j[c] + W2[c, :] . h) / T        for c in C_j
 *   lp_c   = L_c - logsumexp_{c in C_j} L_c
 * On return c->L and c->lp hold L and lp in candidate order and c->order holds
 * the candidate positions sorted by (L desc, id asc). */
static void score_children(orc_ctx *c, int j, const float *S) {
  const orc_model *m = c->m;
  const int32_t *C = c->cand + (size_t)(j - 1) * m->M;
  const float *Uj = c->U + (size_t)(j - 1) * m->r;
  const float *base = c->q->base + (size_t)(j - 1) * m->V;
  for (int t = 0; t < m->r; ++t) {
    c->p[t] = dot_w(m->W1, m->wdtype, (size_t)t * (m->d + m->d_s) + m->d, S, m->d_s);
    double a = (double)Uj[t] + (double)c->p[t];
    c->h[t] = (float)(a * sigmoid64(a));
  }
  double mx = -INFINITY;
  for (int i = 0; i < m->M; ++i) {
    float dl = dot_w(m->W2, m->wdtype, (size_t)C[i] * m->r, c->h, m->r);
    c->L[i] = (float)(((double)base[C[i]] + (double)dl) / (double)c->Teff);
    if ((double)c->L[i] > mx) mx = (double)c->L[i];
  }
  float lse;
  if (mx == -INFINITY) {
    lse = -INFINITY;
  } else {
    double sum = 0.0;
    for (int i = 0; i < m->M; ++i) sum += exp((double)c->L[i] - mx);
    lse = (float)(mx + log(sum));
  }
  for (int i = 0; i < m->M; ++i)
    c->lp[i] = (lse == -INFINITY) ? -INFINITY : (float)((double)c->L[i] - (double)lse);
  for (int i = 0; i < m->M; ++i) c->order[i] = i;
  g_sort_L = c->L;
  g_sort_cand = C;
  qsort(c->order, (size_t)m->M, sizeof(int32_t), cmp_child);
}

/* ------------------------------------------------------- best-first search */

typedef struct {
  float score;
  int64_t seq;   /* push order */
  int32_t token, parent, depth;
} orc_entry;

/* (score desc, push order asc) */
static int entry_before(const orc_entry *a, const orc_entry *b) {
  if (a->score > b->score) return 1;
  if (a->score < b->score) return 0;
  return a->seq < b->seq;
}

static void fill_empty(const orc_model *m, orc_tree *t, int from) {
  for (int i = from; i <= m->N; ++i) {
    t->tokens[i] = -1; t->parents[i] = -1; t->depths[i] = -1; t->scores[i] = -INFINITY;
  }
}

static void emit_mask(const orc_model *m, orc_tree *t) {
  if (!t->mask) return;
  int n1 = m->N + 1;
  memset(t->mask, 0, (size_t)n1 * n1);
  for (int i = 0; i < t->n_nodes; ++i)               /* ancestor-or-self closure */
    for (int a = i; a >= 0; a = t->parents[a]) t->mask[(size_t)i * n1 + a] = 1;
}

static int check_model(const orc_model *m) {
  if (!m || !m->E || !m->W_ih || !m->W_hh || !m->W1 || !m->W2) return ORC_EINVAL;
  if (m->V <= 0 || m->d <= 0 || m->d_s <= 0 || m->r <= 0 || m->D <= 0 || m->M <= 0 ||
      m->k <= 0 || m->N < 0 || m->M > m->V || m->k > m->M)
    return ORC_EINVAL;
  if (m->wdtype != ORC_F32 && m->wdtype != ORC_BF16) return ORC_EINVAL;
  return ORC_OK;
}

/* Build one request's tree ([TREE] Componenti Core 1, 2, 4, 5; [SUM] core
 * content). Node 0 is the root (anchor, parent -1, depth 0, score 0). Then N
 * times: pop the frontier maximum, append it, and -- unless it is at depth D
 * or is the N-th pop -- advance its GRU state and push its top-k children with
 * score(parent) + lp. Rows after the last pop (frontier exhausted) are filled
 * with token/parent/depth -1 and score -inf. */
int orc_build_tree(const orc_model *m, const orc_request *q, orc_tree *t) {
  int rc = check_model(m);
  if (rc) return rc;
  if (!q || !q->base || !q->H || !q->state0 || !t || !t->tokens || !t->parents || !t->depths ||
      !t->scores)
    return ORC_EINVAL;
  if (q->anchor < 0 || q->anchor >= m->V) return ORC_EINVAL;
  t->n_nodes = 0;
  t->n_expanded = 0;
  fill_empty(m, t, 0);

  orc_ctx c;
  rc = ctx_init(&c, m, q);
  if (rc) { emit_mask(m, t); return rc; }
  if (t->topm) memcpy(t->topm, c.cand, sizeof(int32_t) * (size_t)m->D * m->M);

  const size_t ds = (size_t)m->d_s;
  float *S = (float *)malloc(sizeof(float) * ds * (size_t)(m->N + 1)); /* state per node */
  size_t cap = (size_t)m->k * (size_t)(m->N + 1);
  orc_entry *front = (orc_entry *)malloc(sizeof(orc_entry) * cap);
  if (!S || !front) { free(S); free(front); ctx_free(&c); return ORC_ENOMEM; }
  size_t nfront = 0;
  int64_t seq = 0;

  /* root: S_root = GRU(state0, E[anchor]) */
  embed(m, q->anchor, c.x);
  orc_gru_step(m->d, m->d_s, m->wdtype, m->W_ih, m->W_hh, m->b_ih, m->b_hh, c.x, q->state0, S);
  t->tokens[0] = q->anchor; t->parents[0] = -1; t->depths[0] = 0; t->scores[0] = 0.0f;
  t->n_nodes = 1;

  int node = 0; /* node to expand next */
  for (int pop = 0; pop <= m->N; ++pop) {
    /* expand `node` (root on the first pass) unless it is a leaf or the N-th pop */
    if (t->depths[node] < m->D && (node < m->N)) {
      int j = t->depths[node] + 1;
      score_children(&c, j, S + (size_t)node * ds);
      const int32_t *C = c.cand + (size_t)(j - 1) * m->M;
      for (int rnk = 0; rnk < m->k; ++rnk) {
        int i = c.order[rnk];
        orc_entry e;
        e.score = t->scores[node] + c.lp[i]; /* fp32 add */
        e.seq = seq++;
        e.token = C[i];
        e.parent = node;
        e.depth = j;
        front[nfront++] = e;
      }
      t->n_expanded++;
    }
    if (pop == m->N || nfront == 0) break;
    /* pop the frontier maximum */
    size_t best = 0;
    for (size_t f = 1; f < nfront; ++f)
      if (entry_before(&front[f], &front[best])) best = f;
    orc_entry e = front[best];
    front[best] = front[--nfront];
    int n = t->n_nodes++;
    t->tokens[n] = e.token; t->parents[n] = e.parent; t->depths[n] = e.depth;
    t->scores[n] = e.score;
    /* advance the GRU along the new node's path when it will be expanded */
    if (e.depth < m->D && n < m->N) {
      embed(m, e.token, c.x);
      orc_gru_step(m->d, m->d_s, m->wdtype, m->W_ih, m->W_hh, m->b_ih, m->b_hh, c.x,
                   S + (size_t)e.parent * ds, S + (size_t)n * ds);
    }
    node = n;
  }
  emit_mask(m, t);
  free(S); free(front); ctx_free(&c);
  return ORC_OK;
}

/* Children of the node reached by `path` (tokens at depths 1..len below the
 * anchor): the k best (token, lp) and, when all_lp is given, lp of every
 * candidate of depth len+1 in C_{len+1} order. Used by the brute-force check. */
int orc_children(const orc_model *m, const orc_request *q, const int32_t *path, int len,
                 int32_t *child_tokens, float *child_lp, float *all_lp, int32_t *cand_out) {
  int rc = check_model(m);
  if (rc) return rc;
  if (len < 0 || len >= m->D) return ORC_EINVAL;
  orc_ctx c;
  rc = ctx_init(&c, m, q);
  if (rc) return rc;
  float *s = (float *)malloc(sizeof(float) * m->d_s);
  float *s2 = (float *)malloc(sizeof(float) * m->d_s);
  embed(m, q->anchor, c.x);
  orc_gru_step(m->d, m->d_s, m->wdtype, m->W_ih, m->W_hh, m->b_ih, m->b_hh, c.x, q->state0, s);
  for (int i = 0; i < len; ++i) {
    embed(m, path[i], c.x);
    orc_gru_step(m->d, m->d_s, m->wdtype, m->W_ih, m->W_hh, m->b_ih, m->b_hh, c.x, s, s2);
    memcpy(s, s2, sizeof(float) * m->d_s);
  }
  score_children(&c, len + 1, s);
  const int32_t *C = c.cand + (size_t)len * m->M;
  for (int rnk = 0; rnk < m->k; ++rnk) {
    child_tokens[rnk] = C[c.order[rnk]];
    child_lp[rnk] = c.lp[c.order[rnk]];
  }
  if (all_lp) memcpy(all_lp, c.lp, sizeof(float) * m->M);
  if (cand_out) memcpy(cand_out, C, sizeof(int32_t) * m->M);
  free(s); free(s2); ctx_free(&c);
  return ORC_OK;
}

/* Score of a path: sum of the fp32 lp of each token under its prefix, added in
 * path order in fp32. *in_tree = 1 when every token is among the top-k
 * children of its prefix, 0 when one is a candidate outside the top-k, and -1
 * when one is not a top-M candidate of its depth. */
int orc_score_path(const orc_model *m, const orc_request *q, const int32_t *path, int len,
                   float *score, int32_t *in_tree) {
  int rc = check_model(m);
  if (rc) return rc;
  if (len < 0 || len > m->D) return ORC_EINVAL;
  orc_ctx c;
  rc = ctx_init(&c, m, q);
  if (rc) return rc;
  float *s = (float *)malloc(sizeof(float) * m->d_s);
  float *s2 = (float *)malloc(sizeof(float) * m->d_s);
  embed(m, q->anchor, c.x);
  orc_gru_step(m->d, m->d_s, m->wdtype, m->W_ih, m->W_hh, m->b_ih, m->b_hh, c.x, q->state0, s);
  float acc = 0.0f;
  int32_t ok = 1;
  for (int i = 0; i < len; ++i) {
    score_children(&c, i + 1, s);
    const int32_t *C = c.cand + (size_t)i * m->M;
    int pos = -1;
    for (int a = 0; a < m->M; ++a)
      if (C[a] == path[i]) pos = a;
    if (pos < 0) { ok = -1; acc = -INFINITY; break; }
    int rank = 0;
    while (c.order[rank] != pos) ++rank;
    if (rank >= m->k && ok == 1) ok = 0;
    acc = acc + c.lp[pos];
    if (i + 1 < len) {
      embed(m, path[i], c.x);
      orc_gru_step(m->d, m->d_s, m->wdtype, m->W_ih, m->W_hh, m->b_ih, m->b_hh, c.x, s, s2);
      memcpy(s, s2, sizeof(float) * m->d_s);
    }
  }
  *score = acc;
  *in_tree = ok;
  free(s); free(s2); ctx_free(&c);
  return ORC_OK;
}

/* ------------------------------------------------- Domino chain decoding */

/* One request of Domino's chain decoder ([DOM] method steps, inference: the
 * parallel backbone gives the base logits, the head updates the causal state
 * from the previously drawn draft token, corrects the logits and each draft
 * token is drawn from the corrected logits; [DOM] core method for the state
 * and the correction; [TREE] Definizione del Problema: the released decoder
 * follows this single chain). With the same readings as the tree builder
 * (root state, GRU gates, temperature divides the corrected logits):
 *
 *   S_0 = GRU(state0, E[anchor])
 *   for i = 1..D:
 *     h   = SiLU(W1[:, :d] . H_i + W1[:, d:] . S_{i-1})
 *     x_v = (L_base^i[v] + W2[v, :] . h) / Teff          every v in [0, V)
 *     m   = max_v x_v,  Z = sum_v exp(x_v - m)            (fp64, id order)
 *     T = 0 (greedy):  d_i = argmax_v x_v, lowest id among equal values
 *     T > 0 (sampled): d_i = min { v : sum_{w <= v} exp(x_w - m) > u_i Z },
 *                      the inverse CDF of softmax(x) in token-id order at the
 *                      caller's uniform draw u_i (clamped into [0, 1); NaN
 *                      reads as 0); the last v with exp(x_v - m) > 0 if the
 *                      sum never exceeds u_i Z
 *     t_i = forced[i-1] when `forced` is given, else d_i
 *     lp_i = x_{t_i} - (m + log Z)
 *     S_i = GRU(S_{i-1}, E[t_i])
 * Teff = T, or 1 when T = 0. A depth whose x values are all -inf gives
 * d_i = 0 and lp_i = -inf.
 *
 * Per step i (arrays of D): decided = d_i, tokens = t_i, lp = lp_i, and margin
 * = how close the decision was: greedy, x_(1) - x_(2) (best minus second-best
 * value, 0 on a tie); sampled, the distance of u_i Z from the nearer end of
 * d_i's CDF interval divided by Z. `forced` lets a caller replay the oracle
 * along another decoder's tokens and judge every step on its own.
 * Returns ORC_ENONFINITE when a base logit is NaN or +inf, ORC_EINVAL for a
 * temperature < 0 or not finite, or a token out of range. */
int orc_chain(const orc_model *m, const orc_request *q, const float *u, const int32_t *forced,
              int32_t *decided, int32_t *tokens, float *lp, float *margin) {
  int rc = check_model(m);
  if (rc) return rc;
  if (!q || !q->base || !q->H || !q->state0 || !decided || !tokens || !lp || !margin)
    return ORC_EINVAL;
  if (q->anchor < 0 || q->anchor >= m->V) return ORC_EINVAL;
  if (!(q->temperature >= 0.0f) || isinf(q->temperature)) return ORC_EINVAL;
  for (size_t i = 0; i < (size_t)m->D * m->V; ++i)
    if (isnan(q->base[i]) || (isinf(q->base[i]) && q->base[i] > 0)) return ORC_ENONFINITE;
  const int greedy = q->temperature == 0.0f;
  const double Teff = greedy ? 1.0 : (double)q->temperature;
  const int V = m->V, ds = m->d_s, r = m->r;
  float *s = (float *)malloc(sizeof(float) * ds);
  float *s2 = (float *)malloc(sizeof(float) * ds);
  float *x = (float *)malloc(sizeof(float) * m->d);
  float *h = (float *)malloc(sizeof(float) * r);
  float *xv = (float *)malloc(sizeof(float) * V);
  if (!s || !s2 || !x || !h || !xv) {
    free(s); free(s2); free(x); free(h); free(xv);
    return ORC_ENOMEM;
  }
  embed(m, q->anchor, x);
  orc_gru_step(m->d, ds, m->wdtype, m->W_ih, m->W_hh, m->b_ih, m->b_hh, x, q->state0, s);
  rc = ORC_OK;
  for (int i = 0; i < m->D && rc == ORC_OK; ++i) {
    const float *base = q->base + (size_t)i * V;
    for (int t = 0; t < r; ++t) {
      const size_t row = (size_t)t * (m->d + ds);
      float U = dot_w(m->W1, m->wdtype, row, q->H + (size_t)i * m->d, m->d);
      float P = dot_w(m->W1, m->wdtype, row + m->d, s, ds);
      double a = (double)U + (double)P;
      h[t] = (float)(a * sigmoid64(a));
    }
    double mx = -INFINITY;
    for (int v = 0; v < V; ++v) {
      float dl = dot_w(m->W2, m->wdtype, (size_t)v * r, h, r);
      xv[v] = (float)(((double)base[v] + (double)dl) / Teff);
      if ((double)xv[v] > mx) mx = (double)xv[v];
    }
    int d = 0;
    double Z = 0.0, mg = 0.0;
    if (mx == -INFINITY) {
      d = 0;
      mg = 0.0;
    } else {
      for (int v = 0; v < V; ++v) Z += exp((double)xv[v] - mx);
      if (greedy) {
        float best = xv[0], second = -INFINITY;
        int arg = 0;
        for (int v = 1; v < V; ++v) {
          if (xv[v] > best) { second = best; best = xv[v]; arg = v; }
          else if (xv[v] > second) second = xv[v];   /* a tie with best makes the gap 0 */
        }
        d = arg;
        mg = (double)best - (double)second;
      } else {
        float uu = u ? u[i] : 0.0f;
        double uc = (uu >= 0.0f) ? (uu < 1.0f ? (double)uu : (double)nextafterf(1.0f, 0.0f)) : 0.0;
        const double target = uc * Z;
        double cum = 0.0, lo_end = 0.0, hi_end = 0.0;
        int last_pos = 0;
        d = -1;
        for (int v = 0; v < V; ++v) {
          const double e = exp((double)xv[v] - mx);
          if (e > 0.0) last_pos = v;
          if (cum + e > target) { d = v; lo_end = cum; hi_end = cum + e; break; }
          cum += e;
        }
        if (d < 0) { d = last_pos; lo_end = hi_end = cum; }
        const double a = target - lo_end, b = hi_end - target;
        mg = (a < b ? a : b) / Z;
      }
    }
    const int32_t t = forced ? forced[i] : d;
    if (t < 0 || t >= V) { rc = ORC_EINVAL; break; }
    decided[i] = d;
    tokens[i] = t;
    margin[i] = (float)mg;
    lp[i] = (mx == -INFINITY) ? -INFINITY : (float)((double)xv[t] - (mx + log(Z)));
    if (i + 1 < m->D) {
      embed(m, t, x);
      orc_gru_step(m->d, ds, m->wdtype, m->W_ih, m->W_hh, m->b_ih, m->b_hh, x, s, s2);
      memcpy(s, s2, sizeof(float) * ds);
    }
  }
  free(s); free(s2); free(x); free(h); free(xv);
  return rc;
}
