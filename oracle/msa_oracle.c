/*
 * msa_oracle.c — plain, slow, fp64 CPU oracle for MInference-style dynamic
 * sparse prefill attention.  TEST INFRASTRUCTURE ONLY: it is loaded by the
 * test suite, by the package's smoke check and by the benchmark's CPU-baseline
 * leg, never by the library's compute path.  It shares no code, header, table
 * or constant with the CUDA library.
 *
 * Sources (web pages, cited by title and section/equation):
 *  [MI]  PaperTrace 2.1.2 "MInference: 按 head 模式加速长上下文 Prefill"
 *        eq.(1)-(2) dense causal attention; eq.(3)-(4) A-shape; eq.(5)
 *        Vertical-Slash; eq.(6) Block-Sparse; §3.1 proxy column/diagonal
 *        aggregation and top-k; §4 worked examples eq.(9)-(12); §6.2 proxy
 *        estimator (Ã = causal softmax of sampled rows, c_j and r_d sums).
 *  [BL]  "LLM模型之MInference" blog, §2.3.2 (last_q x K proxy; mean pooling for
 *        block-sparse) and §2.3.3 (Vertical-Slash index: verticals ascending,
 *        slashes descending, per-block ranges and uncovered columns).
 *  [CM]  PaperTrace 1.1.1 "成本模型" §1.2 causal edge counts, §2.1 window edges.
 *
 * Inputs Q, K, V are float arrays holding the exact bf16 input values; every
 * computation is done in double.  Readings where the pages are silent:
 *  - proxy aggregation is the SUM of causal-softmax probabilities for both
 *    columns and diagonals ([MI] §6.2 formulas);
 *  - top-k ties go to the lower index; k >= candidates takes all;
 *  - a slash offset δ covers, for query block u = [a, e], the key interval
 *    [a-δ, e-δ] clipped to [0, e] (a 64x64 tile on that diagonal, [MI] §2.1);
 *    verticals are single columns (a 1x64 strip); a row attends the union of
 *    its block's intervals and columns, restricted to j <= i;
 *  - block-sparse: the diagonal block is always kept and counts toward k_b,
 *    J_u = {u} ∪ top_{k_b-1}{v < u} by the raw dot product of block means.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------ threading */
static int g_threads = 0;

int ora_num_threads(void) {
  if (g_threads > 0) return g_threads;
  const char* env = getenv("MSA_ORACLE_THREADS");
  if (env && atoi(env) > 0) return atoi(env);
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}
void ora_set_threads(int t) { g_threads = t; }

typedef void (*ora_body)(void* ctx, int64_t item);
typedef struct {
  ora_body body;
  void* ctx;
  int64_t n;
  int64_t next;
  pthread_mutex_t mu;
} ora_pool;

static void* ora_worker(void* arg) {
  ora_pool* p = (ora_pool*)arg;
  for (;;) {
    pthread_mutex_lock(&p->mu);
    int64_t it = p->next++;
    pthread_mutex_unlock(&p->mu);
    if (it >= p->n) break;
    p->body(p->ctx, it);
  }
  return NULL;
}

/* Run body(ctx, item) for item in [0, n) on the oracle's threads. */
static void ora_parallel_for(int64_t n, ora_body body, void* ctx) {
  int nt = ora_num_threads();
  if (nt > n) nt = (int)(n > 0 ? n : 1);
  ora_pool p;
  p.body = body;
  p.ctx = ctx;
  p.n = n;
  p.next = 0;
  pthread_mutex_init(&p.mu, NULL);
  if (nt <= 1) {
    ora_worker(&p);
  } else {
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nt);
    for (int t = 0; t < nt; ++t) pthread_create(&th[t], NULL, ora_worker, &p);
    for (int t = 0; t < nt; ++t) pthread_join(th[t], NULL);
    free(th);
  }
  pthread_mutex_destroy(&p.mu);
}

static int cmp_i64(const void* a, const void* b) {
  int64_t x = *(const int64_t*)a, y = *(const int64_t*)b;
  return (x > y) - (x < y);
}

/* Sort and drop duplicates; returns the new length. */
static int64_t sort_unique(int64_t* v, int64_t m) {
  if (m <= 1) return m;
  qsort(v, (size_t)m, sizeof(int64_t), cmp_i64);
  int64_t w = 1;
  for (int64_t r = 1; r < m; ++r)
    if (v[r] != v[w - 1]) v[w++] = v[r];
  return w;
}

/* ------------------------------------------------------------ candidate sets */

/* [MI] eq.(3): N_A(i) = {0..min(g-1,i)} ∪ {max(0,i-w+1)..i}.  Keys ascending,
 * each once; returns |N_A(i)|. */
int64_t ora_ashape_set(int64_t i, int64_t g, int64_t w, int64_t* out) {
  int64_t m = 0;
  int64_t sink_hi = (g - 1 < i) ? g - 1 : i; /* inclusive */
  int64_t win_lo = (i - w + 1 > 0) ? i - w + 1 : 0;
  for (int64_t j = 0; j <= sink_hi; ++j) out[m++] = j;
  for (int64_t j = win_lo; j <= i; ++j)
    if (j > sink_hi) out[m++] = j; /* the union counts each key once */
  return m;
}

/* [MI] eq.(5): N_VS(i) = {j in C, j <= i} ∪ {i - δ : δ in D, 0 <= i - δ <= i}. */
int64_t ora_vs_logical_set(int64_t i, const int32_t* C, int64_t nc, const int32_t* D, int64_t nd, int64_t* out) {
  int64_t m = 0;
  for (int64_t t = 0; t < nc; ++t)
    if (C[t] >= 0 && C[t] <= i) out[m++] = C[t];
  for (int64_t t = 0; t < nd; ++t)
    if (D[t] >= 0 && i - D[t] >= 0) out[m++] = i - D[t];
  return sort_unique(out, m);
}

typedef struct {
  int64_t lo, hi;
} ora_range;

static int cmp_range_lo(const void* a, const void* b) {
  const ora_range* x = (const ora_range*)a;
  const ora_range* y = (const ora_range*)b;
  if (x->lo != y->lo) return (x->lo > y->lo) - (x->lo < y->lo);
  return (x->hi > y->hi) - (x->hi < y->hi);
}

/* Vertical-Slash index of query block u ([MI] §2.1 and §4.1 last paragraphs;
 * [BL] §2.3.3 "获取 Vertical-Slash Index"): rows a = u*b .. e = min(a+b,n)-1.
 * Each slash offset δ (taken in descending order, so ranges come out with
 * ascending starts) covers keys [a-δ, e-δ] ∩ [0, e]; an offset with e-δ < 0
 * covers nothing.  Overlapping or adjacent ranges are merged.  Columns are the
 * verticals c <= e (ascending) that no merged range contains.
 * ranges[2*r], ranges[2*r+1] = inclusive [lo, hi] of merged range r.
 * Returns nranges + ncols. */
int64_t ora_vs_block_index(int64_t u, int64_t n, int64_t b, const int32_t* C, int64_t nc, const int32_t* D,
                           int64_t nd, int64_t* ranges, int64_t* nranges, int64_t* cols, int64_t* ncols) {
  int64_t a = u * b;
  int64_t e = (a + b < n ? a + b : n) - 1;
  ora_range* rr = (ora_range*)malloc(sizeof(ora_range) * (size_t)(nd > 0 ? nd : 1));
  int64_t m = 0;
  /* δ descending: sort a copy of D */
  int64_t* dd = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nd > 0 ? nd : 1));
  for (int64_t t = 0; t < nd; ++t) dd[t] = D[t];
  int64_t ndu = sort_unique(dd, nd);
  for (int64_t t = ndu - 1; t >= 0; --t) {
    int64_t delta = dd[t];
    if (delta < 0) continue;
    int64_t hi = e - delta;
    if (hi < 0) continue;
    int64_t lo = a - delta;
    if (lo < 0) lo = 0;
    rr[m].lo = lo;
    rr[m].hi = hi;
    ++m;
  }
  qsort(rr, (size_t)m, sizeof(ora_range), cmp_range_lo); /* already ascending; keeps it explicit */
  int64_t nr = 0;
  for (int64_t t = 0; t < m; ++t) {
    if (nr > 0 && rr[t].lo <= ranges[2 * (nr - 1) + 1] + 1) {
      if (rr[t].hi > ranges[2 * (nr - 1) + 1]) ranges[2 * (nr - 1) + 1] = rr[t].hi;
    } else {
      ranges[2 * nr] = rr[t].lo;
      ranges[2 * nr + 1] = rr[t].hi;
      ++nr;
    }
  }
  /* columns: verticals ascending, c <= e, not inside a merged range */
  int64_t* cc = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nc > 0 ? nc : 1));
  for (int64_t t = 0; t < nc; ++t) cc[t] = C[t];
  int64_t ncu = sort_unique(cc, nc);
  int64_t k = 0;
  for (int64_t t = 0; t < ncu; ++t) {
    int64_t c = cc[t];
    if (c < 0 || c > e) continue;
    int covered = 0;
    for (int64_t r = 0; r < nr; ++r)
      if (c >= ranges[2 * r] && c <= ranges[2 * r + 1]) {
        covered = 1;
        break;
      }
    if (!covered) cols[k++] = c;
  }
  *nranges = nr;
  *ncols = k;
  free(rr);
  free(dd);
  free(cc);
  return nr + k;
}

/* Physical Vertical-Slash set of row i with query block size b:
 * (merged ranges of i's block ∪ its uncovered columns) ∩ [0, i].
 * With b = 1 it equals the logical set of eq.(5). */
int64_t ora_vs_physical_set(int64_t i, int64_t n, int64_t b, const int32_t* C, int64_t nc, const int32_t* D,
                            int64_t nd, int64_t* out) {
  int64_t u = i / b;
  int64_t* ranges = (int64_t*)malloc(sizeof(int64_t) * 2 * (size_t)(nd > 0 ? nd : 1));
  int64_t* cols = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nc > 0 ? nc : 1));
  int64_t nr = 0, ncol = 0;
  ora_vs_block_index(u, n, b, C, nc, D, nd, ranges, &nr, cols, &ncol);
  int64_t m = 0;
  for (int64_t r = 0; r < nr; ++r)
    for (int64_t j = ranges[2 * r]; j <= ranges[2 * r + 1] && j <= i; ++j) out[m++] = j;
  for (int64_t t = 0; t < ncol; ++t)
    if (cols[t] <= i) out[m++] = cols[t];
  free(ranges);
  free(cols);
  return sort_unique(out, m);
}

/* Block-sparse set of row i ([MI] eq.(6)): keys of the blocks v in J_u (u = i/b)
 * restricted to j <= i (the diagonal block gets the causal triangle). */
int64_t ora_bs_set(int64_t i, int64_t n, int64_t b, const int32_t* J, const int32_t* cnt, int64_t kb, int64_t* out) {
  int64_t u = i / b;
  int64_t m = 0;
  for (int64_t t = 0; t < cnt[u]; ++t) {
    int64_t v = J[u * kb + t];
    for (int64_t j = v * b; j < (v + 1) * b && j < n && j <= i; ++j) out[m++] = j;
  }
  return sort_unique(out, m);
}

/* ------------------------------------------------------------ proxy scores */

/* [MI] §6.2: causal softmax of the last L query rows against all keys,
 * Ã_ij = softmax_{j<=i}(scale * q_i.k_j), rows i = n-L .. n-1 ([BL] §2.3.2:
 * Q[-last_q:] x K).  A is [L][n]; entries with j > i are 0. */
typedef struct {
  int64_t n, d, L;
  double scale;
  const float *q, *k;
  double* A;
} proxy_ctx;

static void proxy_row(void* vctx, int64_t t) {
  proxy_ctx* c = (proxy_ctx*)vctx;
  int64_t i = c->n - c->L + t;
  double* row = c->A + t * c->n;
  const float* qi = c->q + i * c->d;
  double mx = -INFINITY;
  for (int64_t j = 0; j <= i; ++j) {
    const float* kj = c->k + j * c->d;
    double s = 0.0;
    for (int64_t x = 0; x < c->d; ++x) s += (double)qi[x] * (double)kj[x];
    s *= c->scale;
    row[j] = s;
    if (s > mx) mx = s;
  }
  double z = 0.0;
  for (int64_t j = 0; j <= i; ++j) z += exp(row[j] - mx);
  for (int64_t j = 0; j <= i; ++j) row[j] = exp(row[j] - mx) / z;
  for (int64_t j = i + 1; j < c->n; ++j) row[j] = 0.0;
}

void ora_vs_proxy_probs(int64_t n, int64_t d, int64_t L, double scale, const float* q, const float* k, double* A) {
  if (L > n) L = n;
  proxy_ctx c = {n, d, L, scale, q, k, A};
  ora_parallel_for(L, proxy_row, &c);
}

/* [MI] §3.1 and §6.2 aggregation of a proxy matrix whose row t is query
 * position pos[t]: column scores c_j = Σ_t A[t][j] and slash scores
 * r_d = Σ_t A[t][pos[t] - d] over the rows with pos[t] - d >= 0.
 * mode bit 0: column score = the maximum over the rows instead of the sum
 * ([MI] §3.1: one strong response kept, sensitive to spikes); mode bit 1:
 * slash score = the mean over its legal pairs (rows with pos[t] - d >= 0)
 * instead of the sum ([MI] §6.2: a sum favours short offsets, which have
 * more pairs); an offset with no legal pair scores 0. */
void ora_proxy_aggregate(const double* A, int64_t rows, int64_t n, const int64_t* pos, double* c, double* r,
                         int32_t mode) {
  int64_t* cnt = (int64_t*)calloc((size_t)n, sizeof(int64_t));
  for (int64_t j = 0; j < n; ++j) c[j] = 0.0;
  for (int64_t dd = 0; dd < n; ++dd) r[dd] = 0.0;
  for (int64_t t = 0; t < rows; ++t) {
    const double* row = A + t * n;
    for (int64_t j = 0; j < n; ++j) {
      if (mode & 1) {
        if (row[j] > c[j]) c[j] = row[j];
      } else {
        c[j] += row[j];
      }
      int64_t dd = pos[t] - j; /* the slash through (pos[t], j) */
      if (dd >= 0 && dd < n) {
        r[dd] += row[j];
        ++cnt[dd];
      }
    }
  }
  if (mode & 2)
    for (int64_t dd = 0; dd < n; ++dd) r[dd] = cnt[dd] ? r[dd] / (double)cnt[dd] : 0.0;
  free(cnt);
}

/* Full Vertical-Slash proxy: Ã for rows [n-L, n), then c and r. */
void ora_vs_proxy(int64_t n, int64_t d, int64_t L, double scale, const float* q, const float* k, double* c, double* r,
                  int32_t mode) {
  if (L > n) L = n;
  double* A = (double*)malloc(sizeof(double) * (size_t)(L * n));
  int64_t* pos = (int64_t*)malloc(sizeof(int64_t) * (size_t)L);
  ora_vs_proxy_probs(n, d, L, scale, q, k, A);
  for (int64_t t = 0; t < L; ++t) pos[t] = n - L + t;
  ora_proxy_aggregate(A, L, n, pos, c, r, mode);
  free(A);
  free(pos);
}

/* ------------------------------------------------------------ top-k */
typedef struct {
  double s;
  int64_t idx;
} scored;

static int cmp_scored(const void* a, const void* b) {
  const scored* x = (const scored*)a;
  const scored* y = (const scored*)b;
  if (x->s > y->s) return -1;
  if (x->s < y->s) return 1;
  return (x->idx > y->idx) - (x->idx < y->idx);
}

/* The k largest of score[0..n): higher score first, equal scores to the lower
 * index; k >= n takes all.  Writes the chosen indices in that order and
 * returns min(k, n). */
int64_t ora_topk(const double* score, int64_t n, int64_t k, int32_t* out) {
  if (k > n) k = n;
  if (k <= 0) return 0;
  scored* v = (scored*)malloc(sizeof(scored) * (size_t)n);
  for (int64_t j = 0; j < n; ++j) {
    v[j].s = score[j];
    v[j].idx = j;
  }
  qsort(v, (size_t)n, sizeof(scored), cmp_scored);
  for (int64_t t = 0; t < k; ++t) out[t] = (int32_t)v[t].idx;
  free(v);
  return k;
}

/* ------------------------------------------------------------ block-sparse index */

/* [BL] §2.3.2 Block-Sparse step 1: mean of the real tokens of each block of b
 * rows (the last block may be partial).  xbar is [ceil(n/b)][d]. */
void ora_bs_pool(const float* x, int64_t n, int64_t d, int64_t b, double* xbar) {
  int64_t nb = (n + b - 1) / b;
  for (int64_t u = 0; u < nb; ++u) {
    int64_t a = u * b, e = (a + b < n ? a + b : n);
    for (int64_t t = 0; t < d; ++t) {
      double s = 0.0;
      for (int64_t i = a; i < e; ++i) s += (double)x[i * d + t];
      xbar[u * d + t] = s / (double)(e - a);
    }
  }
}

typedef struct {
  const double *qb, *kb_;
  int64_t d, k;
  int32_t *J, *cnt;
} bs_ctx;

static void bs_row(void* vctx, int64_t u) {
  bs_ctx* c = (bs_ctx*)vctx;
  int32_t* Ju = c->J + u * c->k;
  int64_t m = 0;
  if (c->k >= 1) Ju[m++] = (int32_t)u; /* the diagonal block is always kept */
  if (u > 0 && c->k > 1) {
    double* score = (double*)malloc(sizeof(double) * (size_t)u);
    for (int64_t v = 0; v < u; ++v) {
      double s = 0.0;
      for (int64_t t = 0; t < c->d; ++t) s += c->qb[u * c->d + t] * c->kb_[v * c->d + t];
      score[v] = s; /* [BL] §2.3.2 step 2: Q̄ K̄^T block score */
    }
    int32_t* pick = (int32_t*)malloc(sizeof(int32_t) * (size_t)u);
    int64_t got = ora_topk(score, u, c->k - 1, pick);
    for (int64_t t = 0; t < got; ++t) Ju[m++] = pick[t];
    free(score);
    free(pick);
  }
  /* ascending block ids */
  int64_t* tmp = (int64_t*)malloc(sizeof(int64_t) * (size_t)(m > 0 ? m : 1));
  for (int64_t t = 0; t < m; ++t) tmp[t] = Ju[t];
  qsort(tmp, (size_t)m, sizeof(int64_t), cmp_i64);
  for (int64_t t = 0; t < m; ++t) Ju[t] = (int32_t)tmp[t];
  for (int64_t t = m; t < c->k; ++t) Ju[t] = -1;
  free(tmp);
  c->cnt[u] = (int32_t)m;
}

/* [MI] eq.(6) with [BL] §2.3.2: J_u = {u} ∪ top_{k_b-1}{v < u} of Q̄_u.K̄_v.
 * J is [N_b][k_b] ascending with -1 padding, cnt[u] = min(k_b, u+1). */
void ora_bs_index(const float* q, const float* k, int64_t n, int64_t d, int64_t b, int64_t kb, int32_t* J,
                  int32_t* cnt) {
  int64_t nb = (n + b - 1) / b;
  double* qb = (double*)malloc(sizeof(double) * (size_t)(nb * d));
  double* kbar = (double*)malloc(sizeof(double) * (size_t)(nb * d));
  ora_bs_pool(q, n, d, b, qb);
  ora_bs_pool(k, n, d, b, kbar);
  bs_ctx c = {qb, kbar, d, kb, J, cnt};
  ora_parallel_for(nb, bs_row, &c);
  free(qb);
  free(kbar);
}

/* ------------------------------------------------------------ attention */

/* [MI] eq.(1)-(2) with the sum restricted to the set: s_j = scale*q_i.k_j,
 * o_i = Σ_j exp(s_j - m) v_j / Σ_j exp(s_j - m) (m = max s_j), and
 * lse_i = m + log Σ_j exp(s_j - m).  An empty set gives o = 0, lse = -inf. */
void ora_attend(const float* q, const float* k, const float* v, int64_t d, double scale, int64_t i,
                const int64_t* set, int64_t m, double* o, double* lse) {
  for (int64_t x = 0; x < d; ++x) o[x] = 0.0;
  if (m == 0) {
    *lse = -INFINITY;
    return;
  }
  double* s = (double*)malloc(sizeof(double) * (size_t)m);
  const float* qi = q + i * d;
  double mx = -INFINITY;
  for (int64_t t = 0; t < m; ++t) {
    const float* kj = k + set[t] * d;
    double acc = 0.0;
    for (int64_t x = 0; x < d; ++x) acc += (double)qi[x] * (double)kj[x];
    s[t] = acc * scale;
    if (s[t] > mx) mx = s[t];
  }
  double z = 0.0;
  for (int64_t t = 0; t < m; ++t) {
    double p = exp(s[t] - mx);
    z += p;
    const float* vj = v + set[t] * d;
    for (int64_t x = 0; x < d; ++x) o[x] += p * (double)vj[x];
  }
  for (int64_t x = 0; x < d; ++x) o[x] /= z;
  *lse = mx + log(z);
  free(s);
}

/* ------------------------------------------------------------ one head */

enum { ORA_ASHAPE = 0, ORA_VS = 1, ORA_BLOCK = 2, ORA_DENSE = 3 };

typedef struct {
  int32_t pattern; /* ORA_* */
  int32_t sink, window;
  int32_t block;
  int32_t topk;
} ora_head;

typedef struct {
  const ora_head* cfg;
  int64_t n, d;
  double scale;
  const float *q, *k, *v;
  const int32_t *C, *D, *J, *cnt;
  int64_t nc, nd;
  const int64_t* rows;
  double *o, *lse;
  int64_t* size;
} head_ctx;

/* Candidate set N_h(i) of row i for the head's pattern. */
static int64_t head_set(const head_ctx* c, int64_t i, int64_t* buf) {
  switch (c->cfg->pattern) {
    case ORA_ASHAPE:
      return ora_ashape_set(i, c->cfg->sink, c->cfg->window, buf);
    case ORA_VS:
      return ora_vs_physical_set(i, c->n, c->cfg->block, c->C, c->nc, c->D, c->nd, buf);
    case ORA_BLOCK:
      return ora_bs_set(i, c->n, c->cfg->block, c->J, c->cnt, c->cfg->topk, buf);
    default: {
      for (int64_t j = 0; j <= i; ++j) buf[j] = j;
      return i + 1;
    }
  }
}

static void head_row(void* vctx, int64_t t) {
  head_ctx* c = (head_ctx*)vctx;
  int64_t i = c->rows[t];
  int64_t* buf = (int64_t*)malloc(sizeof(int64_t) * (size_t)(c->n + c->nc + c->nd + 1));
  int64_t m = head_set(c, i, buf);
  if (c->size) c->size[t] = m;
  if (c->o) ora_attend(c->q, c->k, c->v, c->d, c->scale, i, buf, m, c->o + t * c->d, c->lse + t);
  free(buf);
}

/* Output rows `rows` of one head: o [nrows][d], lse [nrows], size[t] = |N(i)|.
 * q, k, v are that head's [n][d] matrices.  o/lse may be NULL (sizes only). */
void ora_head_rows(const ora_head* cfg, int64_t n, int64_t d, double scale, const float* q, const float* k,
                   const float* v, const int32_t* C, int64_t nc, const int32_t* D, int64_t nd, const int32_t* J,
                   const int32_t* cnt, const int64_t* rows, int64_t nrows, double* o, double* lse, int64_t* size) {
  head_ctx c = {cfg, n, d, scale, q, k, v, C, D, J, cnt, nc, nd, rows, o, lse, size};
  ora_parallel_for(nrows, head_row, &c);
}

/* E_h = Σ_i |N_h(i)| over all rows ([MI] eq.(4) generalised to any pattern).
 * For Vertical-Slash heads the count per block is taken from the merged
 * ranges and columns of that block. */
typedef struct {
  const ora_head* cfg;
  int64_t n;
  const int32_t *C, *D, *J, *cnt;
  int64_t nc, nd;
  int64_t* per_block;
} edge_ctx;

static void edge_block(void* vctx, int64_t u) {
  edge_ctx* c = (edge_ctx*)vctx;
  int64_t b = c->cfg->pattern == ORA_ASHAPE || c->cfg->pattern == ORA_DENSE ? 64 : c->cfg->block;
  int64_t a = u * b, e = (a + b < c->n ? a + b : c->n) - 1;
  int64_t total = 0;
  if (c->cfg->pattern == ORA_VS) {
    int64_t* ranges = (int64_t*)malloc(sizeof(int64_t) * 2 * (size_t)(c->nd > 0 ? c->nd : 1));
    int64_t* cols = (int64_t*)malloc(sizeof(int64_t) * (size_t)(c->nc > 0 ? c->nc : 1));
    int64_t nr = 0, ncol = 0;
    ora_vs_block_index(u, c->n, b, c->C, c->nc, c->D, c->nd, ranges, &nr, cols, &ncol);
    for (int64_t i = a; i <= e; ++i) {
      int64_t m = 0;
      for (int64_t r = 0; r < nr; ++r) {
        int64_t lo = ranges[2 * r], hi = ranges[2 * r + 1] < i ? ranges[2 * r + 1] : i;
        if (hi >= lo) m += hi - lo + 1;
      }
      for (int64_t t = 0; t < ncol; ++t)
        if (cols[t] <= i) ++m;
      total += m;
    }
    free(ranges);
    free(cols);
  } else if (c->cfg->pattern == ORA_BLOCK) {
    for (int64_t i = a; i <= e; ++i) {
      int64_t m = 0;
      for (int64_t t = 0; t < c->cnt[u]; ++t) {
        int64_t v = c->J[u * c->cfg->topk + t];
        int64_t lo = v * b, hi = (v + 1) * b - 1;
        if (hi > i) hi = i;
        if (hi > c->n - 1) hi = c->n - 1;
        if (hi >= lo) m += hi - lo + 1;
      }
      total += m;
    }
  } else {
    int64_t* buf = (int64_t*)malloc(sizeof(int64_t) * (size_t)(c->n + 1));
    for (int64_t i = a; i <= e; ++i) {
      if (c->cfg->pattern == ORA_ASHAPE)
        total += ora_ashape_set(i, c->cfg->sink, c->cfg->window, buf);
      else
        total += i + 1;
    }
    free(buf);
  }
  c->per_block[u] = total;
}

int64_t ora_head_edges(const ora_head* cfg, int64_t n, const int32_t* C, int64_t nc, const int32_t* D, int64_t nd,
                       const int32_t* J, const int32_t* cnt) {
  int64_t b = cfg->pattern == ORA_ASHAPE || cfg->pattern == ORA_DENSE ? 64 : cfg->block;
  int64_t nb = (n + b - 1) / b;
  int64_t* per = (int64_t*)calloc((size_t)nb, sizeof(int64_t));
  edge_ctx c = {cfg, n, C, D, J, cnt, nc, nd, per};
  ora_parallel_for(nb, edge_block, &c);
  int64_t total = 0;
  for (int64_t u = 0; u < nb; ++u) total += per[u];
  free(per);
  return total;
}
