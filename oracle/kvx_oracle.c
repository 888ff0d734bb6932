/*
 * kvx_oracle.c -- plain fp64 CPU oracle of the cross-model KV-cache transfer.
 *
 * TEST INFRASTRUCTURE ONLY (tests, smoke check, CPU baseline leg of the
 * benchmark).  Every function is the plain definition written out as nested
 * loops in double precision; there is no blocking, fusion or reordering.
 * The sources and readings are listed in kvx_oracle.h.
 */
#include "kvx_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* [HIR] "Why carrying the cache across is the hard part": the position is
 * folded into a key as a rotation.  [QKV] "Линейного моста...": strip the
 * source RoPE, apply the target RoPE.  Half-split pairing (i, i + d/2) with
 * frequency theta^(-2i/d). */
void kvxo_rope(const double *x, int d, double pos, double theta, int sign,
               double *out) {
  int half = d / 2;
  for (int i = 0; i < half; ++i) {
    double w = pow(theta, -2.0 * (double)i / (double)d);
    double a = (double)sign * pos * w;
    double c = cos(a), s = sin(a);
    double x0 = x[i], x1 = x[i + half];
    out[i] = x0 * c - x1 * s;
    out[i + half] = x0 * s + x1 * c;
  }
}

/* One token of one (target layer, head): [HIR] steps 1-3, [QKV] feature
 * concatenation and the per-(layer, head) map x @ w + b. */
void kvxo_map_token(int d, int k, double theta_src, double theta_tgt,
                    const double *const *src_k_rows,
                    const double *const *src_v_rows,
                    const double *Wk, const double *Wv,
                    const double *bk, const double *bv,
                    double p_src, double p_tgt,
                    double *out_k, double *out_v) {
  int kd = k * d;
  double *xk = (double *)malloc(sizeof(double) * (size_t)kd);
  double *xv = (double *)malloc(sizeof(double) * (size_t)kd);
  double *yk = (double *)malloc(sizeof(double) * (size_t)d);

  /* step 1 + concatenation: un-rotate each selected key, keep values */
  for (int j = 0; j < k; ++j) {
    kvxo_rope(src_k_rows[j], d, p_src, theta_src, -1, xk + j * d);
    for (int c = 0; c < d; ++c) xv[j * d + c] = src_v_rows[j][c];
  }
  /* step 2: y = x W + b, separately for keys and values.  Each output
   * element is summed as b[n] + x[0] W[0][n] + x[1] W[1][n] + ... in order. */
  for (int n = 0; n < d; ++n) {
    yk[n] = bk[n];
    out_v[n] = bv[n];
  }
  for (int q = 0; q < kd; ++q) {
    const double *wk_row = Wk + (size_t)q * d;
    const double *wv_row = Wv + (size_t)q * d;
    for (int n = 0; n < d; ++n) {
      yk[n] += xk[q] * wk_row[n];
      out_v[n] += xv[q] * wv_row[n];
    }
  }
  /* step 3: re-rotate the mapped key into its target position */
  kvxo_rope(yk, d, p_tgt, theta_tgt, +1, out_k);

  free(xk);
  free(xv);
  free(yk);
}

/* Cache install.  Contiguous: one [capacity] slab per request.  Paged
 * ([KNLP] inject through a block table): logical block p'/bs of request r is
 * physical block block_table[r][p'/bs], slot p' % bs. */
int64_t kvxo_dst_row(int layout, int64_t r, int64_t p_tgt,
                     int64_t dst_capacity, int64_t block_size,
                     int64_t num_blocks, const int32_t *block_table,
                     int64_t max_blocks_per_req, int *bad) {
  *bad = 0;
  if (layout == KVXO_CONTIGUOUS) {
    if (p_tgt >= dst_capacity) {
      *bad = KVXO_BAD_ROW;
      return -1;
    }
    return r * dst_capacity + p_tgt;
  }
  int64_t logical = p_tgt / block_size;
  if (logical >= max_blocks_per_req) {
    *bad = KVXO_BAD_BLOCK;
    return -1;
  }
  int64_t phys = block_table[r * max_blocks_per_req + logical];
  if (phys < 0 || phys >= num_blocks) {
    *bad = KVXO_BAD_BLOCK;
    return -1;
  }
  return phys * block_size + p_tgt % block_size;
}

/* Reading the pilot's own paged cache: the same block-table rule as the
 * target install, applied to the source position. */
int64_t kvxo_src_row(int layout, int64_t g, int64_t r, int64_t p, int64_t block_size,
                     int64_t num_blocks, const int32_t *block_table,
                     int64_t max_blocks_per_req, int *bad) {
  *bad = 0;
  if (layout == KVXO_CONTIGUOUS) return g;
  int64_t logical = p / block_size;
  if (logical >= max_blocks_per_req) {
    *bad = KVXO_BAD_SRC_BLOCK;
    return -1;
  }
  int64_t phys = block_table[r * max_blocks_per_req + logical];
  if (phys < 0 || phys >= num_blocks) {
    *bad = KVXO_BAD_SRC_BLOCK;
    return -1;
  }
  return phys * block_size + p % block_size;
}

static int64_t kvxo_src_rows(const kvxo_problem *P) {
  return P->src_layout == KVXO_PAGED ? P->src_num_blocks * P->src_block_size : P->ntok;
}

int kvxo_transfer(const kvxo_problem *P, double *dst_k, double *dst_v) {
  const int64_t Ls = P->src_layers, Lt = P->tgt_layers, H = P->kv_heads;
  const int64_t d = P->head_dim, k = P->k, kd = k * d;
  const int64_t ntok = P->ntok, src_rows = kvxo_src_rows(P);
  const int64_t rows = P->layout == KVXO_CONTIGUOUS
                           ? (int64_t)P->num_requests * P->dst_capacity
                           : P->num_blocks * P->block_size;
  int status = 0;

  /* a malformed request table invalidates the whole transfer */
  if (P->cu_seqlens) {
    int ok = P->cu_seqlens[0] == 0 && P->cu_seqlens[P->num_requests] == ntok;
    for (int64_t r = 0; r < P->num_requests; ++r)
      if (P->cu_seqlens[r + 1] < P->cu_seqlens[r]) ok = 0;
    if (!ok) return KVXO_BAD_SEQLENS;
  }

  const double **krows = (const double **)malloc(sizeof(double *) * (size_t)k);
  const double **vrows = (const double **)malloc(sizeof(double *) * (size_t)k);
  double *ok = (double *)malloc(sizeof(double) * (size_t)d);
  double *ov = (double *)malloc(sizeof(double) * (size_t)d);

  /* target layers whose selection row holds an index outside [0, Ls) */
  char *layer_ok = (char *)malloc((size_t)Lt);
  for (int64_t lt = 0; lt < Lt; ++lt) {
    layer_ok[lt] = 1;
    for (int64_t j = 0; j < k; ++j) {
      int32_t s = P->layer_idx[lt * k + j];
      if (s < 0 || s >= Ls) layer_ok[lt] = 0;
    }
    if (!layer_ok[lt]) status |= KVXO_BAD_LAYER_INDEX;
  }

  for (int64_t r = 0; r < P->num_requests; ++r) {
    int64_t beg = P->cu_seqlens ? P->cu_seqlens[r] : 0;
    int64_t end = P->cu_seqlens ? P->cu_seqlens[r + 1] : ntok;
    for (int64_t g = beg; g < end; ++g) {
      int64_t p = P->src_pos ? P->src_pos[g] : g - beg;
      int64_t off = P->tgt_offset ? P->tgt_offset[r] : 0;
      int64_t pt = P->tgt_pos ? P->tgt_pos[g] : p + off;
      if (p < 0 || p >= P->max_position || pt < 0 || pt >= P->max_position) {
        status |= KVXO_BAD_POSITION;
        continue;
      }
      int bad = 0;
      int64_t srow = kvxo_src_row(P->src_layout, g, r, p, P->src_block_size,
                                  P->src_num_blocks, P->src_block_table,
                                  P->src_max_blocks_per_req, &bad);
      if (srow < 0) {
        status |= bad;
        continue;
      }
      int64_t row = kvxo_dst_row(P->layout, r, pt, P->dst_capacity,
                                 P->block_size, P->num_blocks, P->block_table,
                                 P->max_blocks_per_req, &bad);
      if (row < 0) {
        status |= bad;
        continue;
      }
      for (int64_t lt = 0; lt < Lt; ++lt) {
        if (!layer_ok[lt]) continue;
        for (int64_t h = 0; h < H; ++h) {
          for (int64_t j = 0; j < k; ++j) {
            int64_t s = P->layer_idx[lt * k + j];
            krows[j] = P->src_k + ((s * src_rows + srow) * H + h) * d;
            vrows[j] = P->src_v + ((s * src_rows + srow) * H + h) * d;
          }
          const double *Wk = P->w + ((lt * H + h) * 2 + 0) * kd * d;
          const double *Wv = P->w + ((lt * H + h) * 2 + 1) * kd * d;
          const double *bk = P->b + ((lt * H + h) * 2 + 0) * d;
          const double *bv = P->b + ((lt * H + h) * 2 + 1) * d;
          kvxo_map_token((int)d, (int)k, P->theta_src, P->theta_tgt, krows,
                         vrows, Wk, Wv, bk, bv, (double)p, (double)pt, ok, ov);
          double *dk = dst_k + ((lt * rows + row) * H + h) * d;
          double *dv = dst_v + ((lt * rows + row) * H + h) * d;
          memcpy(dk, ok, sizeof(double) * (size_t)d);
          memcpy(dv, ov, sizeof(double) * (size_t)d);
        }
      }
    }
  }
  free(layer_ok);
  free(krows);
  free(vrows);
  free(ok);
  free(ov);
  return status;
}

/* Wide-feature mapper (definition in kvx_oracle.h): one dense map per
 * target layer over all heads' keys and values of the selected layers. */
void kvxo_map_token_wide(int H, int d, int k, double theta_src, double theta_tgt,
                         const double *const *src_k_rows,
                         const double *const *src_v_rows, const double *W,
                         const double *b, double p_src, double p_tgt,
                         double *out_k, double *out_v) {
  int64_t F = (int64_t)k * 2 * H * d, N = (int64_t)H * 2 * d;
  double *x = (double *)malloc(sizeof(double) * (size_t)F);
  double *y = (double *)malloc(sizeof(double) * (size_t)N);

  /* features in (j, m, h, i) order: un-rotated keys, then values as stored */
  for (int j = 0; j < k; ++j)
    for (int h = 0; h < H; ++h) {
      kvxo_rope(src_k_rows[j] + (int64_t)h * d, d, p_src, theta_src, -1,
                x + ((int64_t)(j * 2 + 0) * H + h) * d);
      for (int i = 0; i < d; ++i)
        x[((int64_t)(j * 2 + 1) * H + h) * d + i] = src_v_rows[j][(int64_t)h * d + i];
    }
  /* y = x W + b, summed in feature order */
  for (int64_t n = 0; n < N; ++n) y[n] = b[n];
  for (int64_t q = 0; q < F; ++q) {
    const double *w_row = W + q * N;
    for (int64_t n = 0; n < N; ++n) y[n] += x[q] * w_row[n];
  }
  /* outputs (h, m, i): keys re-rotated into the target position */
  for (int h = 0; h < H; ++h) {
    kvxo_rope(y + (int64_t)(h * 2 + 0) * d, d, p_tgt, theta_tgt, +1, out_k + (int64_t)h * d);
    memcpy(out_v + (int64_t)h * d, y + (int64_t)(h * 2 + 1) * d, sizeof(double) * (size_t)d);
  }
  free(x);
  free(y);
}

int kvxo_transfer_wide(const kvxo_problem *P, double *dst_k, double *dst_v) {
  const int64_t Ls = P->src_layers, Lt = P->tgt_layers, H = P->kv_heads;
  const int64_t d = P->head_dim, k = P->k, ntok = P->ntok, src_rows = kvxo_src_rows(P);
  const int64_t F = k * 2 * H * d, N = H * 2 * d;
  const int64_t rows = P->layout == KVXO_CONTIGUOUS
                           ? (int64_t)P->num_requests * P->dst_capacity
                           : P->num_blocks * P->block_size;
  int status = 0;

  if (P->cu_seqlens) {
    int ok = P->cu_seqlens[0] == 0 && P->cu_seqlens[P->num_requests] == ntok;
    for (int64_t r = 0; r < P->num_requests; ++r)
      if (P->cu_seqlens[r + 1] < P->cu_seqlens[r]) ok = 0;
    if (!ok) return KVXO_BAD_SEQLENS;
  }

  const double **krows = (const double **)malloc(sizeof(double *) * (size_t)k);
  const double **vrows = (const double **)malloc(sizeof(double *) * (size_t)k);
  double *ok = (double *)malloc(sizeof(double) * (size_t)(H * d));
  double *ov = (double *)malloc(sizeof(double) * (size_t)(H * d));
  char *layer_ok = (char *)malloc((size_t)Lt);
  for (int64_t lt = 0; lt < Lt; ++lt) {
    layer_ok[lt] = 1;
    for (int64_t j = 0; j < k; ++j) {
      int32_t s = P->layer_idx[lt * k + j];
      if (s < 0 || s >= Ls) layer_ok[lt] = 0;
    }
    if (!layer_ok[lt]) status |= KVXO_BAD_LAYER_INDEX;
  }

  for (int64_t r = 0; r < P->num_requests; ++r) {
    int64_t beg = P->cu_seqlens ? P->cu_seqlens[r] : 0;
    int64_t end = P->cu_seqlens ? P->cu_seqlens[r + 1] : ntok;
    for (int64_t g = beg; g < end; ++g) {
      int64_t p = P->src_pos ? P->src_pos[g] : g - beg;
      int64_t off = P->tgt_offset ? P->tgt_offset[r] : 0;
      int64_t pt = P->tgt_pos ? P->tgt_pos[g] : p + off;
      if (p < 0 || p >= P->max_position || pt < 0 || pt >= P->max_position) {
        status |= KVXO_BAD_POSITION;
        continue;
      }
      int bad = 0;
      int64_t srow = kvxo_src_row(P->src_layout, g, r, p, P->src_block_size,
                                  P->src_num_blocks, P->src_block_table,
                                  P->src_max_blocks_per_req, &bad);
      if (srow < 0) {
        status |= bad;
        continue;
      }
      int64_t row = kvxo_dst_row(P->layout, r, pt, P->dst_capacity,
                                 P->block_size, P->num_blocks, P->block_table,
                                 P->max_blocks_per_req, &bad);
      if (row < 0) {
        status |= bad;
        continue;
      }
      for (int64_t lt = 0; lt < Lt; ++lt) {
        if (!layer_ok[lt]) continue;
        for (int64_t j = 0; j < k; ++j) {
          int64_t s = P->layer_idx[lt * k + j];
          krows[j] = P->src_k + (s * src_rows + srow) * H * d;
          vrows[j] = P->src_v + (s * src_rows + srow) * H * d;
        }
        kvxo_map_token_wide((int)H, (int)d, (int)k, P->theta_src, P->theta_tgt,
                            krows, vrows, P->w + lt * F * N, P->b + lt * N,
                            (double)p, (double)pt, ok, ov);
        memcpy(dst_k + (lt * rows + row) * H * d, ok, sizeof(double) * (size_t)(H * d));
        memcpy(dst_v + (lt * rows + row) * H * d, ov, sizeof(double) * (size_t)(H * d));
      }
    }
  }
  free(layer_ok);
  free(krows);
  free(vrows);
  free(ok);
  free(ov);
  return status;
}

/* KV cosine of [HIR] ("Reading the retention score") and explained variance
 * of [QKV] ("Линейного моста, как ни странно, хватает"), accumulated over
 * the tokens a transfer writes; definitions in kvx_oracle.h. */
int kvxo_kv_diagnostics(const kvxo_problem *P, const double *mapped_k,
                        const double *mapped_v, const double *ref_k,
                        const double *ref_v, double *stats) {
  const int64_t Lt = P->tgt_layers, H = P->kv_heads, d = P->head_dim;
  const int64_t ntok = P->ntok, F = d + 4;
  const int64_t rows = P->layout == KVXO_CONTIGUOUS
                           ? (int64_t)P->num_requests * P->dst_capacity
                           : P->num_blocks * P->block_size;
  int status = 0;
  for (int64_t i = 0; i < Lt * H * 2 * F; ++i) stats[i] = 0.0;
  if (P->cu_seqlens) {
    int ok = P->cu_seqlens[0] == 0 && P->cu_seqlens[P->num_requests] == ntok;
    for (int64_t r = 0; r < P->num_requests; ++r)
      if (P->cu_seqlens[r + 1] < P->cu_seqlens[r]) ok = 0;
    if (!ok) return KVXO_BAD_SEQLENS;
  }
  double *content = (double *)malloc(sizeof(double) * (size_t)d);
  for (int64_t r = 0; r < P->num_requests; ++r) {
    int64_t beg = P->cu_seqlens ? P->cu_seqlens[r] : 0;
    int64_t end = P->cu_seqlens ? P->cu_seqlens[r + 1] : ntok;
    for (int64_t g = beg; g < end; ++g) {
      int64_t p = P->src_pos ? P->src_pos[g] : g - beg;
      int64_t off = P->tgt_offset ? P->tgt_offset[r] : 0;
      int64_t pt = P->tgt_pos ? P->tgt_pos[g] : p + off;
      if (p < 0 || p >= P->max_position || pt < 0 || pt >= P->max_position) {
        status |= KVXO_BAD_POSITION;
        continue;
      }
      int bad = 0;
      int64_t row = kvxo_dst_row(P->layout, r, pt, P->dst_capacity,
                                 P->block_size, P->num_blocks, P->block_table,
                                 P->max_blocks_per_req, &bad);
      if (row < 0) {
        status |= bad;
        continue;
      }
      for (int64_t lt = 0; lt < Lt; ++lt) {
        for (int64_t h = 0; h < H; ++h) {
          for (int m = 0; m < 2; ++m) {
            const double *a = (m == 0 ? mapped_k : mapped_v) + ((lt * rows + row) * H + h) * d;
            const double *y = (m == 0 ? ref_k : ref_v) + ((lt * rows + row) * H + h) * d;
            double dot = 0.0, aa = 0.0, yy = 0.0, res = 0.0;
            for (int64_t i = 0; i < d; ++i) {
              dot += a[i] * y[i];
              aa += a[i] * a[i];
              yy += y[i] * y[i];
              res += (y[i] - a[i]) * (y[i] - a[i]);
            }
            double *st = stats + ((lt * H + h) * 2 + m) * F;
            st[0] += 1.0;
            if (aa > 0.0 && yy > 0.0) st[1] += dot / sqrt(aa * yy);
            st[2] += res;
            st[3] += yy;
            if (m == 0)
              kvxo_rope(y, (int)d, (double)pt, P->theta_tgt, -1, content);
            else
              memcpy(content, y, sizeof(double) * (size_t)d);
            for (int64_t i = 0; i < d; ++i) st[4 + i] += content[i];
          }
        }
      }
    }
  }
  free(content);
  return status;
}

/* Ridge demo of [QKV] ("Линейного моста, как ни странно, хватает"): centre
 * X and Y on their column means, solve (XcT Xc + lam I) W = XcT Yc, and set
 * b = ybar - xbar W.  The solve is a plain Cholesky factorisation. */
int kvxo_ridge_fit(const double *X, const double *Y, int64_t n, int p, int q,
                   double lam, double *W, double *b) {
  double *xm = (double *)calloc((size_t)p, sizeof(double));
  double *ym = (double *)calloc((size_t)q, sizeof(double));
  double *A = (double *)calloc((size_t)p * p, sizeof(double));
  double *B = (double *)calloc((size_t)p * q, sizeof(double));
  int rc = 0;

  for (int64_t t = 0; t < n; ++t) {
    for (int i = 0; i < p; ++i) xm[i] += X[t * p + i];
    for (int i = 0; i < q; ++i) ym[i] += Y[t * q + i];
  }
  for (int i = 0; i < p; ++i) xm[i] /= (double)n;
  for (int i = 0; i < q; ++i) ym[i] /= (double)n;

  /* A = XcT Xc + lam I ; B = XcT Yc */
  for (int64_t t = 0; t < n; ++t) {
    for (int i = 0; i < p; ++i) {
      double xi = X[t * p + i] - xm[i];
      for (int j = 0; j < p; ++j) A[i * p + j] += xi * (X[t * p + j] - xm[j]);
      for (int j = 0; j < q; ++j) B[i * q + j] += xi * (Y[t * q + j] - ym[j]);
    }
  }
  for (int i = 0; i < p; ++i) A[i * p + i] += lam;

  /* Cholesky A = L LT, L stored in the lower triangle of A */
  for (int j = 0; j < p && rc == 0; ++j) {
    double s = A[j * p + j];
    for (int m = 0; m < j; ++m) s -= A[j * p + m] * A[j * p + m];
    if (!(s > 0.0)) {
      rc = -1;
      break;
    }
    double ljj = sqrt(s);
    A[j * p + j] = ljj;
    for (int i = j + 1; i < p; ++i) {
      double v = A[i * p + j];
      for (int m = 0; m < j; ++m) v -= A[i * p + m] * A[j * p + m];
      A[i * p + j] = v / ljj;
    }
  }
  if (rc == 0) {
    /* forward solve L Z = B, then back solve LT W = Z, column by column */
    for (int c = 0; c < q; ++c) {
      for (int i = 0; i < p; ++i) {
        double v = B[i * q + c];
        for (int m = 0; m < i; ++m) v -= A[i * p + m] * W[m * q + c];
        W[i * q + c] = v / A[i * p + i];
      }
      for (int i = p - 1; i >= 0; --i) {
        double v = W[i * q + c];
        for (int m = i + 1; m < p; ++m) v -= A[m * p + i] * W[m * q + c];
        W[i * q + c] = v / A[i * p + i];
      }
    }
    for (int c = 0; c < q; ++c) {
      double v = ym[c];
      for (int i = 0; i < p; ++i) v -= xm[i] * W[i * q + c];
      b[c] = v;
    }
  }
  free(xm);
  free(ym);
  free(A);
  free(B);
  return rc;
}

/* Layer-selection scores (definition and readings in kvx_oracle.h): for
 * every (target layer, head, K|V) the content-space target vectors are
 * regressed with the ridge demo on one source layer's (or a set's) content
 * vectors, and the in-sample explained variance is summed over dimensions. */
static double kvxo_score_fit(const double *X, const double *Y, int64_t n, int p, int d,
                             double lam) {
  double *W = (double *)malloc(sizeof(double) * (size_t)p * d);
  double *b = (double *)malloc(sizeof(double) * (size_t)d);
  double *ym = (double *)calloc((size_t)d, sizeof(double));
  double r2 = NAN;
  if (kvxo_ridge_fit(X, Y, n, p, d, lam, W, b) == 0) {
    for (int64_t g = 0; g < n; ++g)
      for (int i = 0; i < d; ++i) ym[i] += Y[g * d + i];
    for (int i = 0; i < d; ++i) ym[i] /= (double)n;
    double ss_res = 0.0, ss_tot = 0.0;
    for (int64_t g = 0; g < n; ++g) {
      for (int i = 0; i < d; ++i) {
        double pred = b[i];
        for (int f = 0; f < p; ++f) pred += X[g * p + f] * W[(int64_t)f * d + i];
        double e = Y[g * d + i] - pred;
        double c = Y[g * d + i] - ym[i];
        ss_res += e * e;
        ss_tot += c * c;
      }
    }
    if (ss_tot > 0.0) r2 = 1.0 - ss_res / ss_tot;
  }
  free(W);
  free(b);
  free(ym);
  return r2;
}

int kvxo_layer_scores(const kvxo_problem *P, const double *tgt_k, const double *tgt_v,
                      double lam, double *r2, double *r2_set) {
  const int64_t Ls = P->src_layers, Lt = P->tgt_layers, H = P->kv_heads, d = P->head_dim;
  const int64_t ntok = P->ntok, k = P->k;
  const int want_set = r2_set != NULL && P->layer_idx != NULL;
  for (int64_t i = 0; i < Lt * Ls * H * 2; ++i) r2[i] = NAN;
  if (want_set)
    for (int64_t i = 0; i < Lt * H * 2; ++i) r2_set[i] = NAN;
  if (P->cu_seqlens) {
    int ok = P->cu_seqlens[0] == 0 && P->cu_seqlens[P->num_requests] == ntok;
    for (int64_t r = 0; r < P->num_requests; ++r)
      if (P->cu_seqlens[r + 1] < P->cu_seqlens[r]) ok = 0;
    if (!ok) return KVXO_BAD_SEQLENS;
  }
  /* every token's position */
  int64_t *pos = (int64_t *)malloc(sizeof(int64_t) * (size_t)(ntok > 0 ? ntok : 1));
  for (int64_t r = 0; r < P->num_requests; ++r) {
    int64_t beg = P->cu_seqlens ? P->cu_seqlens[r] : 0;
    int64_t end = P->cu_seqlens ? P->cu_seqlens[r + 1] : ntok;
    for (int64_t g = beg; g < end; ++g) {
      pos[g] = P->src_pos ? P->src_pos[g] : g - beg;
      if (pos[g] < 0 || pos[g] >= P->max_position) {
        free(pos);
        return KVXO_BAD_POSITION;
      }
    }
  }
  int status = 0;
  double *Y = (double *)malloc(sizeof(double) * (size_t)(ntok * d + 1));
  double *X = (double *)malloc(sizeof(double) * (size_t)(ntok * d + 1));
  double *Xs = want_set ? (double *)malloc(sizeof(double) * (size_t)(ntok * k * d + 1)) : NULL;
  for (int64_t lt = 0; lt < Lt; ++lt) {
    for (int64_t h = 0; h < H; ++h) {
      for (int m = 0; m < 2; ++m) {
        /* the target's content vectors of (lt, h, m) */
        for (int64_t g = 0; g < ntok; ++g) {
          const double *y = (m == 0 ? tgt_k : tgt_v) + ((lt * ntok + g) * H + h) * d;
          if (m == 0) kvxo_rope(y, (int)d, (double)pos[g], P->theta_tgt, -1, Y + g * d);
          else memcpy(Y + g * d, y, sizeof(double) * (size_t)d);
        }
        /* one source layer at a time */
        for (int64_t s = 0; s < Ls; ++s) {
          for (int64_t g = 0; g < ntok; ++g) {
            const double *x = (m == 0 ? P->src_k : P->src_v) + ((s * ntok + g) * H + h) * d;
            if (m == 0) kvxo_rope(x, (int)d, (double)pos[g], P->theta_src, -1, X + g * d);
            else memcpy(X + g * d, x, sizeof(double) * (size_t)d);
          }
          r2[((lt * Ls + s) * H + h) * 2 + m] = kvxo_score_fit(X, Y, ntok, (int)d, (int)d, lam);
        }
        /* the set of the layer table, concatenated in table order */
        if (want_set) {
          int ok = 1;
          for (int64_t j = 0; j < k; ++j) {
            int32_t s = P->layer_idx[lt * k + j];
            if (s < 0 || s >= Ls) ok = 0;
          }
          if (!ok) {
            status |= KVXO_BAD_LAYER_INDEX;
            continue;
          }
          for (int64_t g = 0; g < ntok; ++g) {
            for (int64_t j = 0; j < k; ++j) {
              int64_t s = P->layer_idx[lt * k + j];
              const double *x = (m == 0 ? P->src_k : P->src_v) + ((s * ntok + g) * H + h) * d;
              double *dst = Xs + (g * k + j) * d;
              if (m == 0) kvxo_rope(x, (int)d, (double)pos[g], P->theta_src, -1, dst);
              else memcpy(dst, x, sizeof(double) * (size_t)d);
            }
          }
          r2_set[(lt * H + h) * 2 + m] = kvxo_score_fit(Xs, Y, ntok, (int)(k * d), (int)d, lam);
        }
      }
    }
  }
  free(pos);
  free(Y);
  free(X);
  free(Xs);
  return status;
}

int kvxo_ridge_features(const kvxo_problem *P, const double *tgt_k, const double *tgt_v,
                        double *x, double *y) {
  const int64_t Ls = P->src_layers, Lt = P->tgt_layers, H = P->kv_heads, d = P->head_dim;
  const int64_t ntok = P->ntok, k = P->k;
  const int64_t B = Lt * H * 2;
  const int want_y = y != NULL && tgt_k != NULL && tgt_v != NULL;
  for (int64_t e = 0; e < B * ntok * k * d; ++e) x[e] = 0.0;
  if (want_y)
    for (int64_t e = 0; e < B * ntok * d; ++e) y[e] = 0.0;
  if (P->cu_seqlens) {
    int ok = P->cu_seqlens[0] == 0 && P->cu_seqlens[P->num_requests] == ntok;
    for (int64_t r = 0; r < P->num_requests; ++r)
      if (P->cu_seqlens[r + 1] < P->cu_seqlens[r]) ok = 0;
    if (!ok) return KVXO_BAD_SEQLENS;
  }
  int status = 0;
  for (int64_t r = 0; r < P->num_requests; ++r) {
    const int64_t beg = P->cu_seqlens ? P->cu_seqlens[r] : 0;
    const int64_t end = P->cu_seqlens ? P->cu_seqlens[r + 1] : ntok;
    for (int64_t g = beg; g < end; ++g) {
      const int64_t p = P->src_pos ? P->src_pos[g] : g - beg;
      if (p < 0 || p >= P->max_position) {
        status |= KVXO_BAD_POSITION;
        continue;                               /* the token's rows stay zero */
      }
      for (int64_t lt = 0; lt < Lt; ++lt) {
        int row_ok = 1;
        for (int64_t j = 0; j < k; ++j) {
          const int32_t s = P->layer_idx[lt * k + j];
          if (s < 0 || s >= Ls) row_ok = 0;
        }
        if (!row_ok) status |= KVXO_BAD_LAYER_INDEX;
        for (int64_t h = 0; h < H; ++h) {
          for (int m = 0; m < 2; ++m) {
            const int64_t b = (lt * H + h) * 2 + m;
            /* the selected layers' content, concatenated in table order */
            for (int64_t j = 0; row_ok && j < k; ++j) {
              const int64_t s = P->layer_idx[lt * k + j];
              const double *v = (m == 0 ? P->src_k : P->src_v) + ((s * ntok + g) * H + h) * d;
              double *o = x + (b * ntok + g) * k * d + j * d;
              if (m == 0) kvxo_rope(v, (int)d, (double)p, P->theta_src, -1, o);
              else memcpy(o, v, sizeof(double) * (size_t)d);
            }
            /* the target layer's content at the same position */
            if (want_y) {
              const double *v = (m == 0 ? tgt_k : tgt_v) + ((lt * ntok + g) * H + h) * d;
              double *o = y + (b * ntok + g) * d;
              if (m == 0) kvxo_rope(v, (int)d, (double)p, P->theta_tgt, -1, o);
              else memcpy(o, v, sizeof(double) * (size_t)d);
            }
          }
        }
      }
    }
  }
  return status;
}
