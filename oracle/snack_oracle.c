/*
 * CPU oracle for the truly sparse linear layer.
 *
 * TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the
 * benchmark's CPU-baseline leg load this library; the CUDA library never
 * does, and the two share no code, headers or tables.
 *
 * Source: "Beyond Masked Sparsity: SNACK Enables Truly Sparse Neural Networks
 * on GPU" (abstract).  The abstract describes a layer that keeps only the
 * weights that exist (COO) and computes with those alone, takes its
 * gradients in that same sparse form, and rewires its connections during
 * Dynamic Sparse Training.  It prints no formula, so every function below writes out the
 * plain definition of the operation its name gives:
 *
 *   W is out_f x in_f, held as COO triples (row[k], col[k], val[k]),
 *   sorted strictly by (row, col).  X is [batch, in_f] and Y is
 *   [batch, out_f], row-major (Y = X W^T + b, the torch Linear convention).
 *
 * Arithmetic is IEEE double.  Every output sums its terms in storage order
 * (increasing k, or increasing b for the batch sums), and every output also
 * gets T = sum of |terms|, which scales the tolerance of a comparison.
 *
 * Threads (pthreads) only split independent outputs; results do not depend
 * on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------------- */
/* a plain parallel-for over independent outputs                           */

static int g_threads = 1;

void oracle_set_threads(int n) { g_threads = n < 1 ? 1 : (n > 256 ? 256 : n); }
int oracle_get_threads(void) { return g_threads; }

typedef void (*range_fn)(void *ctx, int64_t lo, int64_t hi);

typedef struct {
  range_fn fn;
  void *ctx;
  int64_t lo, hi;
} range_job;

static void *range_thread(void *p) {
  range_job *j = (range_job *)p;
  j->fn(j->ctx, j->lo, j->hi);
  return NULL;
}

static void parallel_for(int64_t n, range_fn fn, void *ctx) {
  int t = g_threads;
  if (t <= 1 || n < 2) {
    fn(ctx, 0, n);
    return;
  }
  if ((int64_t)t > n) t = (int)n;
  pthread_t th[256];
  range_job jobs[256];
  int started[256];
  for (int i = 0; i < t; ++i) {
    jobs[i].fn = fn;
    jobs[i].ctx = ctx;
    jobs[i].lo = n * i / t;
    jobs[i].hi = n * (i + 1) / t;
    started[i] = (i > 0) && pthread_create(&th[i], NULL, range_thread, &jobs[i]) == 0;
  }
  fn(ctx, jobs[0].lo, jobs[0].hi);
  for (int i = 1; i < t; ++i) {
    if (started[i])
      pthread_join(th[i], NULL);
    else
      fn(ctx, jobs[i].lo, jobs[i].hi); /* thread could not start: run inline */
  }
}

/* ---------------------------------------------------------------------- */
/* pattern check                                                           */

/* 0: valid.  1: an index out of range.  2: not strictly increasing in (row, col). */
int oracle_check_coo(int64_t out_f, int64_t in_f, int64_t nnz, const int32_t *row,
                     const int32_t *col) {
  for (int64_t k = 0; k < nnz; ++k)
    if (row[k] < 0 || row[k] >= out_f || col[k] < 0 || col[k] >= in_f) return 1;
  for (int64_t k = 1; k < nnz; ++k) {
    int64_t a = (int64_t)row[k - 1] * in_f + col[k - 1];
    int64_t b = (int64_t)row[k] * in_f + col[k];
    if (!(a < b)) return 2;
  }
  return 0;
}

/* ---------------------------------------------------------------------- */
/* forward: Y[b,r] = bias[r] + sum_{k : row[k]=r} val[k] * X[b,col[k]]     */

typedef struct {
  int64_t out_f, in_f, nnz;
  const int32_t *row, *col;
  const double *val, *x, *bias;
  double *y, *t;
} fwd_ctx;

static void fwd_range(void *p, int64_t b0, int64_t b1) {
  fwd_ctx *c = (fwd_ctx *)p;
  for (int64_t b = b0; b < b1; ++b) {
    double *yb = c->y + b * c->out_f;
    double *tb = c->t ? c->t + b * c->out_f : NULL;
    const double *xb = c->x + b * c->in_f;
    for (int64_t r = 0; r < c->out_f; ++r) {
      yb[r] = c->bias ? c->bias[r] : 0.0;
      if (tb) tb[r] = c->bias ? fabs(c->bias[r]) : 0.0;
    }
    for (int64_t k = 0; k < c->nnz; ++k) {
      double term = c->val[k] * xb[c->col[k]];
      yb[c->row[k]] += term;
      if (tb) tb[c->row[k]] += fabs(term);
    }
  }
}

int oracle_fwd(int64_t out_f, int64_t in_f, int64_t nnz, const int32_t *row, const int32_t *col,
               const double *val, int64_t batch, const double *x, const double *bias, double *y,
               double *t) {
  if (oracle_check_coo(out_f, in_f, nnz, row, col) == 1) return 1;
  fwd_ctx c = {out_f, in_f, nnz, row, col, val, x, bias, y, t};
  parallel_for(batch, fwd_range, &c);
  return 0;
}

/* ---------------------------------------------------------------------- */
/* input gradient: dX[b,c] = sum_{k : col[k]=c} val[k] * dY[b,row[k]]      */

typedef struct {
  int64_t out_f, in_f, nnz;
  const int32_t *row, *col;
  const double *val, *dy;
  double *dx, *t;
} dx_ctx;

static void dx_range(void *p, int64_t b0, int64_t b1) {
  dx_ctx *c = (dx_ctx *)p;
  for (int64_t b = b0; b < b1; ++b) {
    double *o = c->dx + b * c->in_f;
    double *tb = c->t ? c->t + b * c->in_f : NULL;
    const double *g = c->dy + b * c->out_f;
    for (int64_t i = 0; i < c->in_f; ++i) {
      o[i] = 0.0;
      if (tb) tb[i] = 0.0;
    }
    for (int64_t k = 0; k < c->nnz; ++k) {
      double term = c->val[k] * g[c->row[k]];
      o[c->col[k]] += term;
      if (tb) tb[c->col[k]] += fabs(term);
    }
  }
}

int oracle_dx(int64_t out_f, int64_t in_f, int64_t nnz, const int32_t *row, const int32_t *col,
              const double *val, int64_t batch, const double *dy, double *dx, double *t) {
  if (oracle_check_coo(out_f, in_f, nnz, row, col) == 1) return 1;
  dx_ctx c = {out_f, in_f, nnz, row, col, val, dy, dx, t};
  parallel_for(batch, dx_range, &c);
  return 0;
}

/* ---------------------------------------------------------------------- */
/* weight gradient at the stored positions only (sampled dense-dense        */
/* product):  dW[k] = sum_b dY[b,row[k]] * X[b,col[k]]                      */
/* bias gradient:  db[r] = sum_b dY[b,r]                                    */

typedef struct {
  int64_t out_f, in_f, nnz, batch;
  const int32_t *row, *col;
  const double *x, *dy;
  double *dw, *t, *db;
} dw_ctx;

static void dw_range(void *p, int64_t k0, int64_t k1) {
  dw_ctx *c = (dw_ctx *)p;
  for (int64_t k = k0; k < k1; ++k) {
    double s = 0.0, a = 0.0;
    for (int64_t b = 0; b < c->batch; ++b) {
      double term = c->dy[b * c->out_f + c->row[k]] * c->x[b * c->in_f + c->col[k]];
      s += term;
      a += fabs(term);
    }
    c->dw[k] = s;
    if (c->t) c->t[k] = a;
  }
}

static void db_range(void *p, int64_t r0, int64_t r1) {
  dw_ctx *c = (dw_ctx *)p;
  for (int64_t r = r0; r < r1; ++r) {
    double s = 0.0;
    for (int64_t b = 0; b < c->batch; ++b) s += c->dy[b * c->out_f + r];
    c->db[r] = s;
  }
}

int oracle_dw(int64_t out_f, int64_t in_f, int64_t nnz, const int32_t *row, const int32_t *col,
              int64_t batch, const double *x, const double *dy, double *dw, double *t, double *db) {
  if (oracle_check_coo(out_f, in_f, nnz, row, col) == 1) return 1;
  dw_ctx c = {out_f, in_f, nnz, batch, row, col, x, dy, dw, t, db};
  parallel_for(nnz, dw_range, &c);
  if (db) parallel_for(out_f, db_range, &c);
  return 0;
}

/* ---------------------------------------------------------------------- */
/* GELU (exact, erf form) and its derivative                                */

double oracle_gelu(double x) { return 0.5 * x * (1.0 + erf(x / sqrt(2.0))); }

double oracle_gelu_grad(double x) {
  /* d/dx [x * Phi(x)] = Phi(x) + x * phi(x) */
  const double inv_sqrt_2pi = 0.39894228040143267794;
  return 0.5 * (1.0 + erf(x / sqrt(2.0))) + x * inv_sqrt_2pi * exp(-0.5 * x * x);
}

void oracle_gelu_vec(int64_t n, const double *x, double *y) {
  for (int64_t i = 0; i < n; ++i) y[i] = oracle_gelu(x[i]);
}

void oracle_gelu_grad_vec(int64_t n, const double *x, double *y) {
  for (int64_t i = 0; i < n; ++i) y[i] = oracle_gelu_grad(x[i]);
}

/* ---------------------------------------------------------------------- */
/* DST restructure: prune the n_prune smallest |w|, regrow as many at       */
/* uniformly random positions that were empty, with value +0.               */
/*                                                                          */
/* The random stream is SplitMix64 (Steele, Lea and Flood, "Fast splittable */
/* pseudorandom number generators", OOPSLA 2014): state advances by the     */
/* golden-ratio increment and each state goes through the published 64-bit  */
/* finaliser.  Draw i maps to a position by the multiply-high range          */
/* reduction of Lemire ("Fast random integer generation in an interval",    */
/* 2019): p = floor(u * n_pos / 2^64).                                      */

static const uint64_t SM64_GAMMA = 0x9E3779B97F4A7C15ULL;

uint64_t oracle_splitmix64_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* state before the first draw of (seed, step) */
uint64_t oracle_regrow_base(uint64_t seed, uint64_t step) {
  return oracle_splitmix64_mix(seed ^ oracle_splitmix64_mix(step));
}

/* position of draw i (i = 0, 1, 2, ...) in [0, n_pos) */
uint64_t oracle_regrow_draw(uint64_t seed, uint64_t step, uint64_t i, uint64_t n_pos) {
  uint64_t u = oracle_splitmix64_mix(oracle_regrow_base(seed, step) + (i + 1) * SM64_GAMMA);
  return (uint64_t)(((unsigned __int128)u * (unsigned __int128)n_pos) >> 64);
}

typedef struct {
  double mag; /* |val|; NaN is ordered above every number, all NaNs alike */
  int is_nan;
  int64_t k;
} prune_key;

static int prune_key_cmp(const void *pa, const void *pb) {
  const prune_key *a = (const prune_key *)pa, *b = (const prune_key *)pb;
  if (a->is_nan != b->is_nan) return a->is_nan < b->is_nan ? -1 : 1;
  if (!a->is_nan && a->mag != b->mag) return a->mag < b->mag ? -1 : 1;
  return a->k < b->k ? -1 : (a->k > b->k ? 1 : 0);
}

static int cmp_u64(const void *pa, const void *pb) {
  uint64_t a = *(const uint64_t *)pa, b = *(const uint64_t *)pb;
  return a < b ? -1 : (a > b ? 1 : 0);
}

static int sorted_contains(const uint64_t *a, int64_t n, uint64_t v) {
  int64_t lo = 0, hi = n;
  while (lo < hi) {
    int64_t mid = lo + (hi - lo) / 2;
    if (a[mid] < v)
      lo = mid + 1;
    else
      hi = mid;
  }
  return lo < n && a[lo] == v;
}

/* open-addressing set of positions (stored as p + 1, 0 = empty slot) */
typedef struct {
  uint64_t *slot;
  uint64_t mask;
} pos_set;

static int pos_set_insert(pos_set *s, uint64_t p) { /* 1 if newly inserted */
  uint64_t key = p + 1;
  uint64_t h = oracle_splitmix64_mix(key) & s->mask;
  for (;;) {
    if (s->slot[h] == 0) {
      s->slot[h] = key;
      return 1;
    }
    if (s->slot[h] == key) return 0;
    h = (h + 1) & s->mask;
  }
}

/*
 * Steps, in order:
 *  1. rank the stored weights by (|val|, k) ascending; the first n_prune are pruned;
 *  2. survivors keep their storage order and their values;
 *  3. O = every position of the input pattern (pruned ones included), so a
 *     position freed in this call is not regrown in the same call;
 *  4. draws i = 0, 1, ... give positions p_i; p_i is accepted when it is not in
 *     O and not equal to an already accepted position; stop at n_prune accepted
 *     (error if max_draws draws do not suffice);
 *  5. a regrown entry is (p / in_f, p mod in_f) with value +0;
 *  6. the output is survivors and regrown merged by position row*in_f+col;
 *     src_out[j] is the old index k of a survivor, -1 for a regrown entry.
 * Values of the output are val[src_out[j]] or +0; the caller gathers them.
 *
 * Returns the number of draws consumed (>= n_prune), or a negative error:
 *  -1 bad pattern, -2 n_prune out of range, -3 too few empty positions,
 *  -4 max_draws exhausted, -5 out of memory.
 */
int64_t oracle_restructure(int64_t out_f, int64_t in_f, int64_t nnz, const int32_t *row,
                           const int32_t *col, const double *val, int64_t n_prune, uint64_t seed,
                           uint64_t step, int64_t max_draws, int32_t *row_out, int32_t *col_out,
                           int64_t *src_out) {
  if (oracle_check_coo(out_f, in_f, nnz, row, col) != 0) return -1;
  if (n_prune < 0 || n_prune > nnz) return -2;
  uint64_t n_pos = (uint64_t)out_f * (uint64_t)in_f;
  if ((uint64_t)n_prune > n_pos - (uint64_t)nnz) return -3;

  int64_t rc = -5;
  prune_key *keys = (prune_key *)malloc(sizeof(prune_key) * (size_t)(nnz > 0 ? nnz : 1));
  unsigned char *pruned = (unsigned char *)calloc((size_t)(nnz > 0 ? nnz : 1), 1);
  uint64_t *pos = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)(nnz > 0 ? nnz : 1));
  uint64_t *grown = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)(n_prune > 0 ? n_prune : 1));
  uint64_t cap = 16;
  while (cap < 2 * (uint64_t)n_prune + 16) cap <<= 1;
  pos_set acc = {(uint64_t *)calloc((size_t)cap, sizeof(uint64_t)), cap - 1};
  if (!keys || !pruned || !pos || !grown || !acc.slot) goto done;

  /* 1. rank by magnitude, ties by storage index */
  for (int64_t k = 0; k < nnz; ++k) {
    keys[k].is_nan = isnan(val[k]) ? 1 : 0;
    keys[k].mag = keys[k].is_nan ? 0.0 : fabs(val[k]);
    keys[k].k = k;
  }
  qsort(keys, (size_t)nnz, sizeof(prune_key), prune_key_cmp);
  for (int64_t i = 0; i < n_prune; ++i) pruned[keys[i].k] = 1;

  /* 3. the old pattern O as sorted linear positions */
  for (int64_t k = 0; k < nnz; ++k) pos[k] = (uint64_t)row[k] * (uint64_t)in_f + (uint64_t)col[k];

  /* 4. draw until n_prune positions are accepted */
  int64_t n_acc = 0, i = 0;
  while (n_acc < n_prune) {
    if (i >= max_draws) {
      rc = -4;
      goto done;
    }
    uint64_t p = oracle_regrow_draw(seed, step, (uint64_t)i, n_pos);
    ++i;
    if (sorted_contains(pos, nnz, p)) continue;
    if (!pos_set_insert(&acc, p)) continue;
    grown[n_acc++] = p;
  }
  qsort(grown, (size_t)n_prune, sizeof(uint64_t), cmp_u64);

  /* 6. merge survivors (already in position order) with the regrown ones */
  {
    int64_t a = 0, g = 0, j = 0;
    for (;;) {
      while (a < nnz && pruned[a]) ++a;
      int have_a = a < nnz, have_g = g < n_prune;
      if (!have_a && !have_g) break;
      if (have_a && (!have_g || pos[a] < grown[g])) {
        row_out[j] = row[a];
        col_out[j] = col[a];
        src_out[j] = a;
        ++a;
      } else {
        row_out[j] = (int32_t)(grown[g] / (uint64_t)in_f);
        col_out[j] = (int32_t)(grown[g] % (uint64_t)in_f);
        src_out[j] = -1;
        ++g;
      }
      ++j;
    }
  }
  rc = i;

done:
  free(keys);
  free(pruned);
  free(pos);
  free(grown);
  free(acc.slot);
  return rc;
}

/* ---------------------------------------------------------------------- */
/* Per-row (constant fan-in) restructure: the structured DST variant in     */
/* which every output row keeps its number of stored weights (Structured    */
/* RigL imposes a constant fan-in; with equal row counts this preserves     */
/* it).  Row r prunes its p_r = min(n_per_row, len_r) smallest |w| by      */
/* (|w|, k) and regrows p_r columns of the same row that were empty before  */
/* the call, drawn from the row's own stream:                               */
/*   base_r = mix(seed ^ mix(step ^ (r * K))),  K = 0xD1B54A32D192ED03      */
/*   draw i: u = mix(base_r + (i + 1) * gamma), column = floor(u * in_f / 2^64) */
/* A draw is accepted when its column was empty in the row and is not       */
/* already accepted; the row stops at p_r accepted (error when             */
/* max_draws_per_row draws do not suffice).  Survivors and regrown columns  */
/* are merged by column; row r's output stays at the row's input offsets.  */
/* Row 0's stream is the unstructured restructure's stream, so a one-row    */
/* layer gives the same result as oracle_restructure.                        */
/*                                                                          */
/* Returns the total number of draws, or a negative error: -1 bad pattern,  */
/* -2 n_per_row negative, -3 a row has fewer empty columns than p_r,        */
/* -4 a row's draw budget is exhausted, -5 out of memory.                   */

static const uint64_t ROW_STREAM_K = 0xD1B54A32D192ED03ULL;

uint64_t oracle_row_base(uint64_t seed, uint64_t step, uint64_t r) {
  return oracle_splitmix64_mix(seed ^ oracle_splitmix64_mix(step ^ (r * ROW_STREAM_K)));
}

int64_t oracle_restructure_rows(int64_t out_f, int64_t in_f, int64_t nnz, const int32_t *row,
                                const int32_t *col, const double *val, int64_t n_per_row, uint64_t seed,
                                uint64_t step, int64_t max_draws_per_row, int32_t *row_out, int32_t *col_out,
                                int64_t *src_out) {
  if (oracle_check_coo(out_f, in_f, nnz, row, col) != 0) return -1;
  if (n_per_row < 0) return -2;
  int64_t *rp = (int64_t *)calloc((size_t)out_f + 1, sizeof(int64_t));
  prune_key *keys = (prune_key *)malloc(sizeof(prune_key) * (size_t)(nnz > 0 ? nnz : 1));
  unsigned char *pruned = (unsigned char *)calloc((size_t)(nnz > 0 ? nnz : 1), 1);
  uint64_t *grown = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)(nnz > 0 ? nnz : 1));
  uint64_t *rowpos = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)(nnz > 0 ? nnz : 1));
  int64_t rc = -5, draws = 0;
  if (!rp || !keys || !pruned || !grown || !rowpos) goto done;
  for (int64_t k = 0; k < nnz; ++k) rp[row[k] + 1]++;
  for (int64_t r = 0; r < out_f; ++r) rp[r + 1] += rp[r];
  for (int64_t r = 0; r < out_f; ++r) {
    const int64_t k0 = rp[r], len = rp[r + 1] - rp[r];
    const int64_t p = n_per_row < len ? n_per_row : len;
    if (p > in_f - len) {
      rc = -3;
      goto done;
    }
    /* prune: the p smallest (|w|, k) of the row */
    for (int64_t j = 0; j < len; ++j) {
      keys[j].is_nan = isnan(val[k0 + j]) ? 1 : 0;
      keys[j].mag = keys[j].is_nan ? 0.0 : fabs(val[k0 + j]);
      keys[j].k = k0 + j;
    }
    qsort(keys, (size_t)len, sizeof(prune_key), prune_key_cmp);
    for (int64_t j = 0; j < p; ++j) pruned[keys[j].k] = 1;
    /* regrow: the row's own draws; the old row's columns as sorted positions */
    for (int64_t j = 0; j < len; ++j) rowpos[j] = (uint64_t)col[k0 + j];
    uint64_t base = oracle_row_base(seed, step, (uint64_t)r);
    int64_t n_acc = 0, i = 0;
    while (n_acc < p) {
      if (i >= max_draws_per_row) {
        rc = -4;
        goto done;
      }
      uint64_t u = oracle_splitmix64_mix(base + ((uint64_t)i + 1) * SM64_GAMMA);
      uint64_t c = (uint64_t)(((unsigned __int128)u * (unsigned __int128)(uint64_t)in_f) >> 64);
      ++i;
      if (sorted_contains(rowpos, len, c)) continue;
      int dup = 0;
      for (int64_t a = 0; a < n_acc; ++a)
        if (grown[a] == c) {
          dup = 1;
          break;
        }
      if (dup) continue;
      grown[n_acc++] = c;
    }
    draws += i;
    qsort(grown, (size_t)p, sizeof(uint64_t), cmp_u64);
    /* merge the row's survivors with its regrown columns */
    int64_t a = k0, g = 0, j = k0;
    for (;;) {
      while (a < k0 + len && pruned[a]) ++a;
      int have_a = a < k0 + len, have_g = g < p;
      if (!have_a && !have_g) break;
      if (have_a && (!have_g || (uint64_t)col[a] < grown[g])) {
        row_out[j] = (int32_t)r;
        col_out[j] = col[a];
        src_out[j] = a;
        ++a;
      } else {
        row_out[j] = (int32_t)r;
        col_out[j] = (int32_t)grown[g];
        src_out[j] = -1;
        ++g;
      }
      ++j;
    }
  }
  rc = draws;

done:
  free(rp);
  free(keys);
  free(pruned);
  free(grown);
  free(rowpos);
  return rc;
}
