/*
 * swin_oracle.c -- plain fp64 CPU oracle for shifted-window multi-head
 * self-attention (SW-MSA) over a lat-lon(-depth) token grid.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the package smoke check and
 * the CPU-baseline leg of the benchmark may load this library. It shares no
 * code, header, table or helper with the CUDA path, and it includes nothing
 * from it. Arithmetic is fp64 throughout; inputs arrive as float32 (every
 * bf16 value is exact in float32, so the oracle sees exactly what the GPU
 * path sees).
 *
 * What it computes (sources, by page title and section):
 *  - "TERRA: A Hierarchical Parallel Training and Memory Orchestration
 *    Framework for High-Resolution AI-based Earth Modeling", Sec. IV.D
 *    (Differentiable Token Routes): every token is addressed by its global
 *    grid coordinate; its attention window is the coordinate divided (floor)
 *    by the window size and its place inside the window is the remainder.
 *    Shifting the windows changes the token's coordinate, which fixes its new
 *    window and offset; the backward of a route applies the inverse map.
 *  - "4D Parallelism Unlocks Exascale Bayesian Neural Networks for
 *    High-Fidelity Atmospheric Modeling", Model Architecture: between two
 *    attention layers the whole domain is rolled by floor(window/2) along the
 *    spatial dimensions, and attention runs inside non-overlapping windows the
 *    way Swin Transformer does it (Swin is reference [12] of TERRA and [34] of
 *    this page): softmax(Q K^T / sqrt(hd) + B) V per window and head, with a
 *    learned relative-position bias B of prod(2 w_d - 1) rows.
 *
 * Readings taken where the pages are silent (each one is also listed in the
 * design notes of the repository):
 *  - roll direction: position in the rolled frame p_d = (u_d - s_d) mod G_d
 *    (a roll by -s, as Swin does before window attention);
 *  - ragged windows: roll on the true extent G_d, then tile from the rolled
 *    origin; the last window along a dimension may be short and its missing
 *    slots are pads (no token, never a key, never stored);
 *  - shift mask: along a non-periodic dimension with s_d > 0 a token carries
 *    region bit d = [p_d >= G_d - s_d] (it wrapped across the edge); a key is
 *    visible only to queries with the same region bits; periodic dimensions
 *    (longitude) carry no bit;
 *  - land: land tokens are never keys; a land query's output is 0 and its
 *    log-sum-exp is -inf;
 *  - masked keys are excluded exactly (probability 0), not by a finite
 *    additive penalty;
 *  - logits: scale hd^-1/2 on q.k first, then the bias is added;
 *  - bias table row of a slot pair (i, j): sum over dims of
 *    (sig_i,d - sig_j,d + w_d - 1) * prod_{e>d} (2 w_e - 1), outermost first;
 *    table layout [rows][heads], row-major.
 *
 * Parity note: the absolute values of attention outputs have no worked
 * numeric example on the pages; the oracle is pinned by the tests through
 * independent derivations (token-pair brute force, library attention on the
 * special cases, closed forms, invariants and finite differences).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
  int32_t ndim;       /* 2 or 3 */
  int32_t pad0;
  int64_t batch;
  int32_t grid[3];    /* outermost first: (lat, lon) or (depth, lat, lon) */
  int32_t window[3];
  int32_t shift[3];
  int32_t periodic[3];
  int32_t heads;
  int32_t head_dim;
  int32_t has_land;
  int32_t pad1;
} oracle_desc;

#define ORACLE_OK 0
#define ORACLE_BAD_ARG (-1)
#define ORACLE_NO_MEMORY (-2)

/* ---- sizes -------------------------------------------------------------- */

static int check_desc(const oracle_desc *d) {
  if (!d) return ORACLE_BAD_ARG;
  if (d->ndim != 2 && d->ndim != 3) return ORACLE_BAD_ARG;
  if (d->batch < 1 || d->heads < 1 || d->head_dim < 1) return ORACLE_BAD_ARG;
  for (int a = 0; a < d->ndim; ++a) {
    if (d->grid[a] < 1 || d->window[a] < 1) return ORACLE_BAD_ARG;
    if (d->shift[a] < 0 || d->shift[a] >= d->window[a]) return ORACLE_BAD_ARG;
    if (d->shift[a] >= d->grid[a] && d->shift[a] > 0) return ORACLE_BAD_ARG;
  }
  return ORACLE_OK;
}

/* Windows per dimension: ceil(G_d / w_d). */
static int64_t windows_along(const oracle_desc *d, int a) {
  return (d->grid[a] + d->window[a] - 1) / d->window[a];
}

static int64_t windows_per_image(const oracle_desc *d) {
  int64_t m = 1;
  for (int a = 0; a < d->ndim; ++a) m *= windows_along(d, a);
  return m;
}

static int64_t tokens_per_image(const oracle_desc *d) {
  int64_t m = 1;
  for (int a = 0; a < d->ndim; ++a) m *= d->grid[a];
  return m;
}

static int slots_per_window(const oracle_desc *d) {
  int m = 1;
  for (int a = 0; a < d->ndim; ++a) m *= d->window[a];
  return m;
}

static int bias_rows(const oracle_desc *d) {
  int m = 1;
  for (int a = 0; a < d->ndim; ++a) m *= 2 * d->window[a] - 1;
  return m;
}

int oracle_sizes(const oracle_desc *d, int64_t *nwin, int64_t *tokens,
                 int32_t *slots, int32_t *rows) {
  int rc = check_desc(d);
  if (rc) return rc;
  if (nwin) *nwin = windows_per_image(d);
  if (tokens) *tokens = tokens_per_image(d);
  if (slots) *slots = slots_per_window(d);
  if (rows) *rows = bias_rows(d);
  return ORACLE_OK;
}

/* ---- routing, written from the token's side ------------------------------
 * For a token with grid coordinate u: rolled position p_d = (u_d - s_d) mod
 * G_d; window coordinate p_d / w_d; in-window offset p_d mod w_d; region bit
 * d set when dimension d is not periodic, s_d > 0 and p_d >= G_d - s_d.
 * Window and slot are flattened row-major, outermost dimension first. */
static void route_token(const oracle_desc *d, int64_t tok, int64_t *win,
                        int *slot, int *reg) {
  int u[3];
  int64_t rest = tok;
  for (int a = d->ndim - 1; a >= 0; --a) {
    u[a] = (int)(rest % d->grid[a]);
    rest /= d->grid[a];
  }
  int64_t wf = 0;
  int sf = 0, r = 0;
  for (int a = 0; a < d->ndim; ++a) {
    int G = d->grid[a], w = d->window[a], s = d->shift[a];
    int p = ((u[a] - s) % G + G) % G;
    wf = wf * windows_along(d, a) + p / w;
    sf = sf * w + p % w;
    if (!d->periodic[a] && s > 0 && p >= G - s) r |= 1 << a;
  }
  *win = wf;
  *slot = sf;
  *reg = r;
}

/* Bias-table row of the slot pair (query slot i, key slot j). */
static int rel_row(const oracle_desc *d, int i, int j) {
  int si[3], sj[3];
  for (int a = d->ndim - 1; a >= 0; --a) {
    si[a] = i % d->window[a];
    i /= d->window[a];
    sj[a] = j % d->window[a];
    j /= d->window[a];
  }
  int row = 0;
  for (int a = 0; a < d->ndim; ++a)
    row = row * (2 * d->window[a] - 1) + (si[a] - sj[a] + d->window[a] - 1);
  return row;
}

/* Routing tables for one image.
 *   win_src[w*n + s]  token index feeding slot s of window w, -1 for a pad slot
 *   region[w*n + s]   region bits of that token (0 for a pad slot)
 *   tok_dst[t]        w*n + s of token t (the inverse route)
 *   relidx[i*n + j]   bias-table row of the slot pair (i, j)
 * Any pointer may be NULL. */
int oracle_tables(const oracle_desc *d, int32_t *win_src, uint8_t *region,
                  int32_t *tok_dst, int32_t *relidx) {
  int rc = check_desc(d);
  if (rc) return rc;
  int64_t nw = windows_per_image(d), N = tokens_per_image(d);
  int n = slots_per_window(d);
  if (win_src)
    for (int64_t x = 0; x < nw * n; ++x) win_src[x] = -1;
  if (region) memset(region, 0, (size_t)(nw * n));
  for (int64_t t = 0; t < N; ++t) {
    int64_t w;
    int s, r;
    route_token(d, t, &w, &s, &r);
    if (win_src) win_src[w * n + s] = (int32_t)t;
    if (region) region[w * n + s] = (uint8_t)r;
    if (tok_dst) tok_dst[t] = (int32_t)(w * n + s);
  }
  if (relidx)
    for (int i = 0; i < n; ++i)
      for (int j = 0; j < n; ++j) relidx[i * n + j] = rel_row(d, i, j);
  return ORACLE_OK;
}

/* ---- one window, one head ------------------------------------------------ */

typedef struct {
  int n;
  const int32_t *src;  /* [n] token of each slot, -1 pad */
  const uint8_t *reg;  /* [n] region bits */
  const uint8_t *lnd;  /* [n] land flag of each slot's token (0 for pads) */
} window_view;

/* visible(i, j): key slot j takes part in the softmax of query slot i. */
static int visible(const window_view *wv, int i, int j) {
  return wv->src[j] >= 0 && !wv->lnd[j] && wv->reg[j] == wv->reg[i];
}

/* Probabilities P[i*n + j] of one window and head; rows of pad and land
 * queries are left at 0. lse[i] receives the natural-log log-sum-exp
 * (-inf for land queries, NaN for pads). */
static void window_probs(const oracle_desc *d, const window_view *wv,
                         const float *q, const float *k, const float *bias,
                         int64_t img_off, int h, double *S, double *P,
                         double *lse) {
  int n = wv->n, hd = d->head_dim, C = d->heads * d->head_dim, H = d->heads;
  double scale = 1.0 / sqrt((double)hd);
  for (int x = 0; x < n * n; ++x) P[x] = 0.0;
  for (int i = 0; i < n; ++i) {
    if (wv->src[i] < 0) {
      if (lse) lse[i] = NAN;
      continue;
    }
    if (wv->lnd[i]) {
      if (lse) lse[i] = -INFINITY;
      continue;
    }
    const float *qi = q + (img_off + wv->src[i]) * C + (int64_t)h * hd;
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) {
      if (!visible(wv, i, j)) continue;
      const float *kj = k + (img_off + wv->src[j]) * C + (int64_t)h * hd;
      double dot = 0.0;
      for (int c = 0; c < hd; ++c) dot += (double)qi[c] * (double)kj[c];
      double s = scale * dot + (double)bias[(int64_t)rel_row(d, i, j) * H + h];
      S[i * n + j] = s;
      if (s > m) m = s;
    }
    double l = 0.0;
    for (int j = 0; j < n; ++j)
      if (visible(wv, i, j)) l += exp(S[i * n + j] - m);
    for (int j = 0; j < n; ++j)
      if (visible(wv, i, j)) P[i * n + j] = exp(S[i * n + j] - m) / l;
    if (lse) lse[i] = m + log(l);
  }
}

typedef struct {
  int32_t *src;
  uint8_t *reg;
  uint8_t *lnd;
} window_tables;

static int load_tables(const oracle_desc *d, window_tables *t) {
  int64_t nw = windows_per_image(d);
  int n = slots_per_window(d);
  t->src = (int32_t *)malloc(sizeof(int32_t) * nw * n);
  t->reg = (uint8_t *)malloc((size_t)(nw * n));
  t->lnd = NULL;
  if (!t->src || !t->reg) return ORACLE_NO_MEMORY;
  oracle_tables(d, t->src, t->reg, NULL, NULL);
  return ORACLE_OK;
}

static void free_tables(window_tables *t) {
  free(t->src);
  free(t->reg);
}

static void make_view(const oracle_desc *d, const window_tables *t,
                      const uint8_t *land, int64_t gid, uint8_t *lnd_buf,
                      window_view *wv) {
  int64_t nw = windows_per_image(d), N = tokens_per_image(d);
  int n = slots_per_window(d);
  int64_t b = gid / nw, w = gid % nw;
  wv->n = n;
  wv->src = t->src + w * n;
  wv->reg = t->reg + w * n;
  for (int s = 0; s < n; ++s)
    lnd_buf[s] = (land && wv->src[s] >= 0) ? (land[b * N + wv->src[s]] != 0) : 0;
  wv->lnd = lnd_buf;
}

/* Forward over a list of windows.
 *   win_ids  global window ids b*nwin + w (NULL: every window of every image)
 *   o_win    [n_ids][n][C]  output rows per slot (0 for pad and land slots)
 *   lse_win  [n_ids][heads][n] natural-log LSE (-inf land, NaN pad); may be NULL
 * Inputs q, k, v: [B, grid..., C] float32; bias [rows][heads] float32;
 * land [B, grid...] uint8 or NULL. */
int oracle_fwd(const oracle_desc *d, const float *q, const float *k,
               const float *v, const float *bias, const uint8_t *land,
               const int64_t *win_ids, int64_t n_ids, double *o_win,
               double *lse_win) {
  int rc = check_desc(d);
  if (rc) return rc;
  if (!q || !k || !v || !bias || !o_win) return ORACLE_BAD_ARG;
  if (d->has_land && !land) return ORACLE_BAD_ARG;
  int64_t nw = windows_per_image(d), N = tokens_per_image(d);
  if (!win_ids) n_ids = d->batch * nw;
  int n = slots_per_window(d), H = d->heads, hd = d->head_dim, C = H * hd;
  window_tables t;
  if (load_tables(d, &t)) {
    free_tables(&t);
    return ORACLE_NO_MEMORY;
  }
  int failed = 0;
#pragma omp parallel
  {
    double *S = (double *)malloc(sizeof(double) * n * n);
    double *P = (double *)malloc(sizeof(double) * n * n);
    double *lse = (double *)malloc(sizeof(double) * n);
    uint8_t *lnd = (uint8_t *)malloc((size_t)n);
    if (!S || !P || !lse || !lnd) {
#pragma omp atomic write
      failed = 1;
    } else {
#pragma omp for schedule(dynamic, 4)
      for (int64_t it = 0; it < n_ids * H; ++it) {
        int64_t x = it / H;
        int h = (int)(it % H);
        int64_t gid = win_ids ? win_ids[x] : x;
        int64_t b = gid / nw;
        window_view wv;
        make_view(d, &t, land, gid, lnd, &wv);
        window_probs(d, &wv, q, k, bias, b * N, h, S, P, lse);
        for (int i = 0; i < n; ++i) {
          double *oi = o_win + (x * n + i) * C + (int64_t)h * hd;
          for (int c = 0; c < hd; ++c) {
            double acc = 0.0;
            for (int j = 0; j < n; ++j) {
              if (P[i * n + j] == 0.0) continue;
              acc += P[i * n + j] *
                     (double)v[(b * N + wv.src[j]) * C + (int64_t)h * hd + c];
            }
            oi[c] = acc;
          }
          if (lse_win) lse_win[(x * H + h) * n + i] = lse[i];
        }
      }
    }
    free(S);
    free(P);
    free(lse);
    free(lnd);
  }
  free_tables(&t);
  return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/* Backward over a list of windows: exact derivatives of L = sum(O * dO).
 *   dout      [B, grid..., C] float32, upstream gradient of O
 *   dq/dk/dv_win  [n_ids][n][C] (0 for pad slots); any may be NULL
 *   dbias     [rows][heads], OVERWRITTEN with the sum over the listed windows;
 *             may be NULL
 * The textbook softmax derivative is used:
 *   dV_j = sum_i P_ij dO_i,  dP_ij = dO_i . v_j,
 *   dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik),
 *   dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i,
 *   dBias[row(i,j)] += dS_ij. */
int oracle_bwd(const oracle_desc *d, const float *q, const float *k,
               const float *v, const float *bias, const uint8_t *land,
               const float *dout, const int64_t *win_ids, int64_t n_ids,
               double *dq_win, double *dk_win, double *dv_win, double *dbias) {
  int rc = check_desc(d);
  if (rc) return rc;
  if (!q || !k || !v || !bias || !dout) return ORACLE_BAD_ARG;
  if (d->has_land && !land) return ORACLE_BAD_ARG;
  int64_t nw = windows_per_image(d), N = tokens_per_image(d);
  if (!win_ids) n_ids = d->batch * nw;
  int n = slots_per_window(d), H = d->heads, hd = d->head_dim, C = H * hd;
  int R = bias_rows(d);
  double scale = 1.0 / sqrt((double)hd);
  window_tables t;
  if (load_tables(d, &t)) {
    free_tables(&t);
    return ORACLE_NO_MEMORY;
  }
  if (dbias)
    for (int64_t x = 0; x < (int64_t)R * H; ++x) dbias[x] = 0.0;
  int failed = 0;
#pragma omp parallel
  {
    double *S = (double *)malloc(sizeof(double) * n * n);
    double *P = (double *)malloc(sizeof(double) * n * n);
    double *dP = (double *)malloc(sizeof(double) * n * n);
    double *dS = (double *)malloc(sizeof(double) * n * n);
    double *db = (double *)calloc((size_t)R * H, sizeof(double));
    uint8_t *lnd = (uint8_t *)malloc((size_t)n);
    if (!S || !P || !dP || !dS || !db || !lnd) {
#pragma omp atomic write
      failed = 1;
    } else {
#pragma omp for schedule(dynamic, 4)
      for (int64_t it = 0; it < n_ids * H; ++it) {
        int64_t x = it / H;
        int h = (int)(it % H);
        int64_t gid = win_ids ? win_ids[x] : x;
        int64_t b = gid / nw, off = b * N;
        window_view wv;
        make_view(d, &t, land, gid, lnd, &wv);
        window_probs(d, &wv, q, k, bias, off, h, S, P, NULL);
#define ROW(ptr, slot) ((ptr) + (off + wv.src[slot]) * C + (int64_t)h * hd)
        /* dP and dS, query by query */
        for (int i = 0; i < n; ++i) {
          double delta = 0.0;
          for (int j = 0; j < n; ++j) {
            dP[i * n + j] = 0.0;
            if (P[i * n + j] == 0.0) continue;
            const float *go = ROW(dout, i), *vj = ROW(v, j);
            double acc = 0.0;
            for (int c = 0; c < hd; ++c) acc += (double)go[c] * (double)vj[c];
            dP[i * n + j] = acc;
            delta += P[i * n + j] * acc;
          }
          for (int j = 0; j < n; ++j)
            dS[i * n + j] = P[i * n + j] * (dP[i * n + j] - delta);
        }
        for (int s = 0; s < n && (dq_win || dk_win || dv_win); ++s) {
          double *gq = dq_win ? dq_win + (x * n + s) * C + (int64_t)h * hd : NULL;
          double *gk = dk_win ? dk_win + (x * n + s) * C + (int64_t)h * hd : NULL;
          double *gv = dv_win ? dv_win + (x * n + s) * C + (int64_t)h * hd : NULL;
          for (int c = 0; c < hd; ++c) {
            double aq = 0.0, ak = 0.0, av = 0.0;
            if (wv.src[s] >= 0) {
              for (int j = 0; j < n; ++j) /* s as query */
                if (dS[s * n + j] != 0.0) aq += dS[s * n + j] * (double)ROW(k, j)[c];
              for (int i = 0; i < n; ++i) { /* s as key */
                if (dS[i * n + s] != 0.0) ak += dS[i * n + s] * (double)ROW(q, i)[c];
                if (P[i * n + s] != 0.0) av += P[i * n + s] * (double)ROW(dout, i)[c];
              }
            }
            if (gq) gq[c] = scale * aq;
            if (gk) gk[c] = scale * ak;
            if (gv) gv[c] = av;
          }
        }
#undef ROW
        if (dbias)
          for (int i = 0; i < n; ++i)
            for (int j = 0; j < n; ++j)
              if (dS[i * n + j] != 0.0)
                db[(int64_t)rel_row(d, i, j) * H + h] += dS[i * n + j];
      }
      if (dbias) {
#pragma omp critical
        for (int64_t x = 0; x < (int64_t)R * H; ++x) dbias[x] += db[x];
      }
    }
    free(S);
    free(P);
    free(dP);
    free(dS);
    free(db);
    free(lnd);
  }
  free_tables(&t);
  return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/* ---- sampled rows, for windows too large for the per-window form --------
 * One query's attention depends on its own window alone, so the quantities of
 * oracle_fwd / oracle_bwd can be had token by token without any n x n
 * matrix (memory O(n) per thread). Tokens are listed by their flat index
 * b*N + t; outputs are rows in the order listed.
 *
 * oracle_route: window, slot and region bits of each listed token (the
 * token-side route above).
 */
int oracle_route(const oracle_desc *d, const int64_t *tok, int64_t n_tok,
                 int64_t *gid, int32_t *slot, int32_t *reg) {
  int rc = check_desc(d);
  if (rc) return rc;
  int64_t N = tokens_per_image(d), nw = windows_per_image(d);
  for (int64_t x = 0; x < n_tok; ++x) {
    if (tok[x] < 0 || tok[x] >= d->batch * N) return ORACLE_BAD_ARG;
    int64_t w;
    int s, r;
    route_token(d, tok[x] % N, &w, &s, &r);
    if (gid) gid[x] = (tok[x] / N) * nw + w;
    if (slot) slot[x] = s;
    if (reg) reg[x] = r;
  }
  return ORACLE_OK;
}

/* Logits of query slot i against every slot of its window for head h:
 * s[j] = scale q_i.k_j + bias(i, j) for visible keys, -inf otherwise.
 * Returns the log-sum-exp over the visible keys (-inf if there is none). */
static double query_logits(const oracle_desc *d, const window_view *wv,
                           const float *q, const float *k, const float *bias,
                           int64_t img_off, int h, int i, double *s) {
  int n = wv->n, hd = d->head_dim, C = d->heads * d->head_dim, H = d->heads;
  double scale = 1.0 / sqrt((double)hd), m = -INFINITY;
  const float *qi = q + (img_off + wv->src[i]) * C + (int64_t)h * hd;
  for (int j = 0; j < n; ++j) {
    s[j] = -INFINITY;
    if (!visible(wv, i, j)) continue;
    const float *kj = k + (img_off + wv->src[j]) * C + (int64_t)h * hd;
    double dot = 0.0;
    for (int c = 0; c < hd; ++c) dot += (double)qi[c] * (double)kj[c];
    s[j] = scale * dot + (double)bias[(int64_t)rel_row(d, i, j) * H + h];
    if (s[j] > m) m = s[j];
  }
  if (m == -INFINITY) return -INFINITY;
  double l = 0.0;
  for (int j = 0; j < n; ++j)
    if (s[j] != -INFINITY) l += exp(s[j] - m);
  return m + log(l);
}

/* delta_i = sum_j P_ij dP_ij, dP_ij = dout_i . v_j, over the visible keys
 * whose logits are in s (P_ij = exp(s[j] - lse)). */
static double query_delta(const oracle_desc *d, const window_view *wv,
                          const float *v, const float *dout, int64_t img_off,
                          int h, int i, const double *s, double lse) {
  int n = wv->n, hd = d->head_dim, C = d->heads * d->head_dim;
  const float *go = dout + (img_off + wv->src[i]) * C + (int64_t)h * hd;
  double delta = 0.0;
  for (int j = 0; j < n; ++j) {
    if (s[j] == -INFINITY) continue;
    const float *vj = v + (img_off + wv->src[j]) * C + (int64_t)h * hd;
    double dp = 0.0;
    for (int c = 0; c < hd; ++c) dp += (double)go[c] * (double)vj[c];
    delta += exp(s[j] - lse) * dp;
  }
  return delta;
}

/* Query rows: for each listed token, O [n_tok][C], LSE [n_tok][heads]
 * (natural log; -inf for land) and, when dout and dq_rows are given,
 * dQ [n_tok][C] = scale sum_j P_ij (dP_ij - delta_i) k_j. Land tokens get
 * zero rows. lse_rows and dq_rows may be NULL. */
int oracle_query_rows(const oracle_desc *d, const float *q, const float *k,
                      const float *v, const float *bias, const uint8_t *land,
                      const float *dout, const int64_t *tok, int64_t n_tok,
                      double *o_rows, double *lse_rows, double *dq_rows) {
  int rc = check_desc(d);
  if (rc) return rc;
  if (!q || !k || !v || !bias || !tok || !o_rows) return ORACLE_BAD_ARG;
  if (d->has_land && !land) return ORACLE_BAD_ARG;
  if (dq_rows && !dout) return ORACLE_BAD_ARG;
  int64_t N = tokens_per_image(d), nw = windows_per_image(d);
  for (int64_t x = 0; x < n_tok; ++x)
    if (tok[x] < 0 || tok[x] >= d->batch * N) return ORACLE_BAD_ARG;
  int n = slots_per_window(d), H = d->heads, hd = d->head_dim, C = H * hd;
  double scale = 1.0 / sqrt((double)hd);
  window_tables t;
  if (load_tables(d, &t)) {
    free_tables(&t);
    return ORACLE_NO_MEMORY;
  }
  int failed = 0;
#pragma omp parallel
  {
    double *s = (double *)malloc(sizeof(double) * n);
    uint8_t *lnd = (uint8_t *)malloc((size_t)n);
    if (!s || !lnd) {
#pragma omp atomic write
      failed = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t it = 0; it < n_tok * H; ++it) {
        int64_t x = it / H;
        int h = (int)(it % H);
        int64_t b = tok[x] / N, w;
        int i, reg;
        route_token(d, tok[x] % N, &w, &i, &reg);
        window_view wv;
        make_view(d, &t, land, b * nw + w, lnd, &wv);
        double *oi = o_rows + x * C + (int64_t)h * hd;
        double *gq = dq_rows ? dq_rows + x * C + (int64_t)h * hd : NULL;
        for (int c = 0; c < hd; ++c) {
          oi[c] = 0.0;
          if (gq) gq[c] = 0.0;
        }
        if (wv.lnd[i]) {
          if (lse_rows) lse_rows[x * H + h] = -INFINITY;
          continue;
        }
        double lse = query_logits(d, &wv, q, k, bias, b * N, h, i, s);
        if (lse_rows) lse_rows[x * H + h] = lse;
        for (int j = 0; j < n; ++j) {
          if (s[j] == -INFINITY) continue;
          double p = exp(s[j] - lse);
          const float *vj = v + (b * N + wv.src[j]) * C + (int64_t)h * hd;
          for (int c = 0; c < hd; ++c) oi[c] += p * (double)vj[c];
        }
        if (!gq) continue;
        double delta = query_delta(d, &wv, v, dout, b * N, h, i, s, lse);
        const float *go = dout + (b * N + wv.src[i]) * C + (int64_t)h * hd;
        for (int j = 0; j < n; ++j) {
          if (s[j] == -INFINITY) continue;
          const float *vj = v + (b * N + wv.src[j]) * C + (int64_t)h * hd;
          const float *kj = k + (b * N + wv.src[j]) * C + (int64_t)h * hd;
          double dp = 0.0;
          for (int c = 0; c < hd; ++c) dp += (double)go[c] * (double)vj[c];
          double ds = exp(s[j] - lse) * (dp - delta);
          for (int c = 0; c < hd; ++c) gq[c] += scale * ds * (double)kj[c];
        }
      }
    }
    free(s);
    free(lnd);
  }
  free_tables(&t);
  return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/* Key rows: for each listed token as a key, dK [n_tok][C] and dV [n_tok][C]:
 *   dV_j = sum_i P_ij dout_i,  dK_j = scale sum_i P_ij (dP_ij - delta_i) q_i
 * over the queries i that see key j (live queries of its window with its
 * region bits). These need the LSE and delta of every such query, so the
 * work is O(n_r^2 hd) per (window, head) for a window whose sampled keys'
 * regions hold n_r queries. Land tokens get zero rows. Either output may be
 * NULL. */
int oracle_key_rows(const oracle_desc *d, const float *q, const float *k,
                    const float *v, const float *bias, const uint8_t *land,
                    const float *dout, const int64_t *tok, int64_t n_tok,
                    double *dk_rows, double *dv_rows) {
  int rc = check_desc(d);
  if (rc) return rc;
  if (!q || !k || !v || !bias || !dout || !tok) return ORACLE_BAD_ARG;
  if (d->has_land && !land) return ORACLE_BAD_ARG;
  int64_t N = tokens_per_image(d), nw = windows_per_image(d);
  for (int64_t x = 0; x < n_tok; ++x)
    if (tok[x] < 0 || tok[x] >= d->batch * N) return ORACLE_BAD_ARG;
  int n = slots_per_window(d), H = d->heads, hd = d->head_dim, C = H * hd;
  double scale = 1.0 / sqrt((double)hd);
  window_tables t;
  if (load_tables(d, &t)) {
    free_tables(&t);
    return ORACLE_NO_MEMORY;
  }
  int64_t *gid = (int64_t *)malloc(sizeof(int64_t) * (n_tok > 0 ? n_tok : 1));
  int *slot = (int *)malloc(sizeof(int) * (n_tok > 0 ? n_tok : 1));
  double *lse = (double *)malloc(sizeof(double) * n);
  double *delta = (double *)malloc(sizeof(double) * n);
  uint8_t *lnd = (uint8_t *)malloc((size_t)n);
  uint8_t *done = (uint8_t *)calloc((size_t)(n_tok > 0 ? n_tok : 1), 1);
  int failed = !gid || !slot || !lse || !delta || !lnd || !done;
  for (int64_t x = 0; !failed && x < n_tok; ++x) {
    int64_t w;
    int reg;
    route_token(d, tok[x] % N, &w, &slot[x], &reg);
    gid[x] = (tok[x] / N) * nw + w;
    for (int c = 0; c < C; ++c) {
      if (dk_rows) dk_rows[x * C + c] = 0.0;
      if (dv_rows) dv_rows[x * C + c] = 0.0;
    }
  }
  /* one window at a time: the window of the first key not yet done */
  for (int64_t x0 = 0; !failed && x0 < n_tok; ++x0) {
    if (done[x0]) continue;
    int64_t g = gid[x0], b = g / nw;
    window_view wv;
    make_view(d, &t, land, g, lnd, &wv);
    /* regions of this window's listed keys */
    int need[8] = {0};
    for (int64_t x = x0; x < n_tok; ++x)
      if (gid[x] == g && wv.src[slot[x]] >= 0) need[wv.reg[slot[x]] & 7] = 1;
    for (int h = 0; h < H && !failed; ++h) {
      /* LSE and delta of every live query of those regions */
#pragma omp parallel
      {
        double *s = (double *)malloc(sizeof(double) * n);
        if (!s) {
#pragma omp atomic write
          failed = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
          for (int i = 0; i < n; ++i) {
            lse[i] = -INFINITY;
            delta[i] = 0.0;
            if (wv.src[i] < 0 || wv.lnd[i] || !need[wv.reg[i] & 7]) continue;
            lse[i] = query_logits(d, &wv, q, k, bias, b * N, h, i, s);
            delta[i] = query_delta(d, &wv, v, dout, b * N, h, i, s, lse[i]);
          }
        }
        free(s);
      }
      if (failed) break;
      /* each listed key of this window, against every query that sees it */
#pragma omp parallel for schedule(dynamic, 1)
      for (int64_t x = x0; x < n_tok; ++x) {
        if (gid[x] != g) continue;
        int j = slot[x];
        double *gk = dk_rows ? dk_rows + x * C + (int64_t)h * hd : NULL;
        double *gv = dv_rows ? dv_rows + x * C + (int64_t)h * hd : NULL;
        const float *kj = k + (b * N + wv.src[j]) * C + (int64_t)h * hd;
        const float *vj = v + (b * N + wv.src[j]) * C + (int64_t)h * hd;
        for (int i = 0; i < n; ++i) {
          if (lse[i] == -INFINITY || !visible(&wv, i, j)) continue;
          const float *qi = q + (b * N + wv.src[i]) * C + (int64_t)h * hd;
          const float *go = dout + (b * N + wv.src[i]) * C + (int64_t)h * hd;
          double dot = 0.0, dp = 0.0;
          for (int c = 0; c < hd; ++c) {
            dot += (double)qi[c] * (double)kj[c];
            dp += (double)go[c] * (double)vj[c];
          }
          double p = exp(scale * dot + (double)bias[(int64_t)rel_row(d, i, j) * H + h] - lse[i]);
          for (int c = 0; c < hd; ++c) {
            if (gv) gv[c] += p * (double)go[c];
            if (gk) gk[c] += scale * p * (dp - delta[i]) * (double)qi[c];
          }
        }
      }
    }
    for (int64_t x = x0; x < n_tok; ++x)
      if (gid[x] == g) done[x] = 1;
  }
  free(gid);
  free(slot);
  free(lse);
  free(delta);
  free(lnd);
  free(done);
  free_tables(&t);
  return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
