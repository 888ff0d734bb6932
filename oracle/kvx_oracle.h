/*
 * kvx_oracle.h -- plain fp64 CPU oracle of the cross-model KV-cache transfer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load or call this code.  It shares no
 * code, header, table or helper with the CUDA library: it is an independent
 * restatement of what the transfer computes, written for a reader to check by
 * eye against the sources it cites, and deliberately slow (nested loops,
 * double precision, one thread).
 *
 * Sources (page title, then section):
 *  [HIR] "Helm Intelligent Routing" (docs.iterate.ai), section
 *        "Why carrying the cache across is the hard part", steps 1-3:
 *        un-rotate the pilot's keys into content space, apply a per-layer,
 *        per-head linear map fitted offline, re-rotate into the position the
 *        entry will occupy in the target sequence (re-rotation cannot be
 *        skipped).  Section "Current limitation": the mapped cache is
 *        installed into the engine's paged cache.
 *  [QKV] "Перенос KV-кэша между моделями Qwen3 вместо повторного префилла"
 *        (reactapp.top), section "Линейного моста, как ни странно, хватает":
 *        pick, per target layer, the source layers that best predict it and
 *        concatenate their features; one ridge regression per target
 *        (layer, head), one for keys and one for values; strip the source
 *        RoPE before mapping keys and apply the target RoPE afterwards; the
 *        ridge demo fits Y ~ XW + b on centred X, Y with (XcT Xc + lam I).
 *  [KNLP] knlp.io "routing" page, the connector flow's inject step: selected
 *        entries are written into the paged cache through a block table.
 *
 * Readings where the sources are silent (the same readings the CUDA library
 * documents):
 *  - RoPE is half-split: pairs (i, i + d/2), frequency w_i = theta^(-2i/d).
 *    rotate multiplies (x_i + j x_{i+d/2}) by exp(+j p w_i); unrotate is
 *    rotate at -p.  Only keys carry RoPE; values are mapped as stored.
 *  - The feature vector of target head h is the concatenation, in index-table
 *    order, of the k selected source layers' head-h vectors (width k*d);
 *    W[lt][h][m] is [k*d][d] row-major, m = 0 for K and 1 for V.
 *  - Request r owns source rows [cu_seqlens[r], cu_seqlens[r+1]).  The
 *    request table must start at 0, never decrease and end at ntok; if it
 *    does not, nothing is written and only KVXO_BAD_SEQLENS is returned.
 *  - The target position p' sets both the re-rotation angle and the cache
 *    row.  p' = tgt_pos[g] if given, else p + tgt_offset[r] (0 if absent).
 *    Source and target positions must lie in [0, max_position).
 *  - Contiguous target: row = r * dst_capacity + p' (needs p' < capacity).
 *    Paged target: row = block_table[r][p' / bs] * bs + p' % bs (needs
 *    p' / bs < max_blocks_per_req and the block id in [0, num_blocks)).
 *  - A row whose layer index, position, block or row is out of range is not
 *    written; the matching KVXO_BAD_* bit is OR-ed into the return value.
 */
#ifndef KVX_ORACLE_H
#define KVX_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return bits of kvxo_transfer (rows that trip one are skipped). */
#define KVXO_BAD_LAYER_INDEX 1
#define KVXO_BAD_POSITION    2
#define KVXO_BAD_BLOCK       4
#define KVXO_BAD_ROW         8
#define KVXO_BAD_SEQLENS     32
#define KVXO_BAD_SRC_BLOCK   64   /* paged source: p / bs beyond the table or a
                                     block id outside the source pool */

#define KVXO_CONTIGUOUS 0
#define KVXO_PAGED      1

/* Half-split RoPE of one head vector x[d] (d even) at position pos with base
 * theta.  sign = +1 rotates (applies RoPE), sign = -1 un-rotates.  out may
 * not alias x. */
void kvxo_rope(const double *x, int d, double pos, double theta, int sign,
               double *out);

/* One token, one (target layer, head): gather the k selected source rows,
 * un-rotate the keys at p_src with theta_src, concatenate, map with
 * Wk/Wv ([k*d][d] row-major) and bk/bv ([d]), re-rotate the mapped key at
 * p_tgt with theta_tgt.  src_k_rows[j] / src_v_rows[j] point at the head
 * vector [d] of the j-th selected source layer. */
void kvxo_map_token(int d, int k, double theta_src, double theta_tgt,
                    const double *const *src_k_rows,
                    const double *const *src_v_rows,
                    const double *Wk, const double *Wv,
                    const double *bk, const double *bv,
                    double p_src, double p_tgt,
                    double *out_k, double *out_v);

/* Row of the target cache that token (request r, target position p_tgt)
 * lands in, or -1 with *bad set to the KVXO_BAD_* reason. */
int64_t kvxo_dst_row(int layout, int64_t r, int64_t p_tgt,
                     int64_t dst_capacity, int64_t block_size,
                     int64_t num_blocks, const int32_t *block_table,
                     int64_t max_blocks_per_req, int *bad);

typedef struct {
  int32_t src_layers, tgt_layers, kv_heads, head_dim, k;
  double theta_src, theta_tgt;
  int64_t max_position;        /* positions must lie in [0, max_position) */
  int32_t num_requests;
  int64_t ntok;                /* source rows */
  const int64_t *cu_seqlens;   /* [R+1] or NULL (then R == 1, all ntok rows) */
  const double *src_k;         /* [Ls][ntok][H][d] */
  const double *src_v;
  const int32_t *layer_idx;    /* [Lt][k] */
  const double *w;             /* [Lt][H][2][k*d][d] */
  const double *b;             /* [Lt][H][2][d] */
  const int64_t *src_pos;      /* [ntok] or NULL: 0..len_r-1 per request */
  const int64_t *tgt_pos;      /* [ntok] or NULL: src_pos + tgt_offset[r] */
  const int64_t *tgt_offset;   /* [R] or NULL: 0 */
  int32_t layout;              /* KVXO_CONTIGUOUS or KVXO_PAGED */
  int64_t dst_capacity;        /* contiguous: rows per request */
  int64_t block_size, num_blocks, max_blocks_per_req;
  const int32_t *block_table;  /* [R][max_blocks_per_req] (paged) */
  /* Source layout.  KVXO_CONTIGUOUS: src_k / src_v are [Ls][ntok][H][d] and
   * token g is row g.  KVXO_PAGED: they are [Ls][src_num_blocks *
   * src_block_size][H][d], the pilot's own paged cache, and token g of
   * request r at source position p is row kvxo_src_row(...). */
  int32_t src_layout;
  int64_t src_block_size, src_num_blocks, src_max_blocks_per_req;
  const int32_t *src_block_table;  /* [R][src_max_blocks_per_req] (paged) */
} kvxo_problem;

/* Source row of packed token g (request r, source position p): g for a
 * contiguous source; src_block_table[r][p / bs] * bs + p % bs for a paged
 * one (the pilot's cache holds its tokens at their positions, like the
 * target cache of [KNLP]'s inject step), or -1 with *bad = KVXO_BAD_SRC_BLOCK
 * when p / bs >= max_blocks_per_req or the block id is outside
 * [0, num_blocks).  Per token the checks run in the order: positions, source
 * row, destination row; the first that fails names the skip. */
int64_t kvxo_src_row(int layout, int64_t g, int64_t r, int64_t p, int64_t block_size,
                     int64_t num_blocks, const int32_t *block_table,
                     int64_t max_blocks_per_req, int *bad);

/* Whole transfer.  dst_k / dst_v are [Lt][rows][H][d] with rows =
 * R * dst_capacity (contiguous) or num_blocks * block_size (paged); rows not
 * written keep their contents.  Returns the OR of KVXO_BAD_* bits. */
int kvxo_transfer(const kvxo_problem *prob, double *dst_k, double *dst_v);

/* Wide-feature mapper: the reading of the 14B -> 32B mapper size in [QKV]
 * section "Ограничения, важные в продакшене" (about 1.07e9 parameters, 4 GB
 * per direction, which is 2^30 = Lt * F * N fp32 weights for Lt = 64,
 * F = 8192, N = 2048): every target layer maps ALL heads' keys and values
 * of its k selected source layers to all its heads' keys and values with
 * one dense map.  Per token and target layer lt:
 *   x (width F = k * 2 * H * d), feature (j, m, h, i) at
 *     ((j * 2 + m) * H + h) * d + i:  m = 0 the key of source layer
 *     idx[lt][j], head h, un-rotated at p (theta_src); m = 1 that layer's
 *     value of head h as stored;
 *   y = x W[lt] + b[lt], W[lt] [F][N] row-major, N = H * 2 * d, output
 *     (h, m, i) at (h * 2 + m) * d + i, i.e. b keeps the per-head layout
 *     [Lt][H][2][d];
 *   key outputs (m = 0) re-rotated at p' (theta_tgt), then installed as in
 *     kvxo_transfer.
 * Each output element is summed as b[n] + x[0] W[0][n] + x[1] W[1][n] + ...
 * in feature order.  With W[lt] zero outside the blocks (h, m) -> (h, m) it
 * is the per-head transfer (same sums, same order).
 * src_k_rows[j] / src_v_rows[j] point at the [H][d] head vectors of the
 * j-th selected source layer; out_k / out_v are [H][d]. */
void kvxo_map_token_wide(int H, int d, int k, double theta_src, double theta_tgt,
                         const double *const *src_k_rows,
                         const double *const *src_v_rows, const double *W,
                         const double *b, double p_src, double p_tgt,
                         double *out_k, double *out_v);

/* Whole wide-feature transfer: as kvxo_transfer with prob->w read as
 * [Lt][k * 2 * H * d][H * 2 * d]. */
int kvxo_transfer_wide(const kvxo_problem *prob, double *dst_k, double *dst_v);

/* Fidelity diagnostics of a transfer: how close the mapped cache is to the
 * target model's own cache for the same tokens.
 *  [HIR] section "Reading the retention score": "KV cosine" -- the closeness
 *        of the mapped cache to the target's own, a diagnostic read beside
 *        retention.
 *  [QKV] section "Линейного моста, как ни странно, хватает": the share of
 *        the target keys' / values' variance that the selected source layers
 *        explain (one best layer ~56 % / 32 %, a set ~79 % / 65 %).
 * Readings: the cosine is taken per (target layer, token, head) between the
 * two d-vectors as stored (both keys carry the target RoPE at p', which a
 * cosine does not see) and is 0 when either vector is zero; the explained
 * variance is the centred R^2 of the mapped vectors as predictions of the
 * target's, summed over the d dimensions, in content space: keys are
 * un-rotated at p' (theta_tgt) before the mean is taken; the residual and
 * the norms are the same in either space.
 * For each (lt, h, m), m = 0 keys and 1 values, the d + 4 doubles at
 * stats[((lt * H + h) * 2 + m) * (d + 4)] are set to
 *   [0] n, tokens compared;          [1] sum of the cosines;
 *   [2] sum |ref - mapped|^2;        [3] sum |ref|^2;
 *   [4 + i] sum of ref_i in content space.
 * Mean cosine = [1] / [0]; R^2 = 1 - [2] / ([3] - |[4..]|^2 / [0]).
 * The tokens are the ones a transfer with the same problem writes: the same
 * position and row rules (prob's source arrays, W and layer table are not
 * used); caches are [Lt][rows][H][d] as for kvxo_transfer.  Returns the OR
 * of the KVXO_BAD_* bits of the skipped tokens (KVXO_BAD_SEQLENS: nothing
 * compared, all stats 0). */
int kvxo_kv_diagnostics(const kvxo_problem *prob, const double *mapped_k,
                        const double *mapped_v, const double *ref_k,
                        const double *ref_v, double *stats);

/* Centred ridge regression with intercept, as in the ridge demo of [QKV]:
 * X [n][p], Y [n][q] row-major; W [p][q] = (XcT Xc + lam I)^-1 XcT Yc,
 * b [q] = ybar - xbar W.  Solved by Cholesky.  Returns 0, or -1 if the
 * normal matrix is not positive definite. */
int kvxo_ridge_fit(const double *X, const double *Y, int64_t n, int p, int q,
                   double lam, double *W, double *b);

/* Layer-selection scores: how much of a target layer's key / value variance
 * one source layer, or a set of source layers, explains through the ridge
 * bridge.  [QKV] section "Линейного моста, как ни странно, хватает": the
 * method picks, per target layer, the source layers whose KV states best
 * predict it; for Qwen3 14B -> 32B the best single layer explains about 56 %
 * of the target keys' variance and 32 % of the values', a set about 79 % and
 * 65 %.  Readings:
 *  - Both caches hold the same tokens (calibration prefills both models on
 *    the same text), packed the same way: token g is row g of src_k / src_v
 *    ([Ls][ntok][H][d]) and of tgt_k / tgt_v ([Lt][ntok][H][d]), at the
 *    same position p (src_pos[g], else g - cu_seqlens[r]).
 *  - Keys are compared in content space: source keys un-rotated at p with
 *    theta_src, target keys at p with theta_tgt; values as stored.
 *  - The predictor of target (lt, h, m) from source layer s is the ridge
 *    demo's fit (kvxo_ridge_fit, centred, intercept, lam unscaled) of the
 *    target head-h vectors on the source head-h vectors of layer s; the set
 *    predictor concatenates the k layers of layer_idx[lt] in table order
 *    (the transfer's feature vector).
 *  - The score is the in-sample explained variance summed over the d
 *    dimensions: R^2 = 1 - sum_g |y_g - (x_g W + b)|^2 / sum_g |y_g - ybar|^2.
 * r2 [Lt][Ls][H][2] (m = 0 keys, 1 values); r2_set [Lt][H][2], computed when
 * both it and prob->layer_idx are given.  Every token must have a position
 * in [0, max_position): otherwise nothing is scored, every output is NaN and
 * KVXO_BAD_POSITION is returned (KVXO_BAD_SEQLENS likewise for a malformed
 * request table).  A set row with a layer index outside [0, Ls) gives NaN
 * scores for that target layer and KVXO_BAD_LAYER_INDEX; a fit whose normal
 * matrix is not positive definite, or a target with no variance, gives NaN.
 * prob's transfer-only fields (W, b, target positions, layouts) are unused;
 * the source must be packed (KVXO_CONTIGUOUS). */
int kvxo_layer_scores(const kvxo_problem *prob, const double *tgt_k,
                      const double *tgt_v, double lam, double *r2, double *r2_set);

/* The inputs of the ridge fits of the maps, in content space ("Перенос
 * KV-кэша между моделями Qwen3 вместо повторного префилла", section
 * "Линейного моста, как ни странно, хватает": strip the source RoPE,
 * concatenate the selected layers' features, fit one ridge map per target
 * (layer, head), one for keys and one for values).  For every target layer
 * lt, head h and m (0 keys, 1 values), batch b = (lt H + h) 2 + m:
 *   x[b][g][j d + i] = dim i of source layer layer_idx[lt][j], head h, token
 *                      g; keys un-rotated at the token's position with
 *                      theta_src, values as stored;
 *   y[b][g][i]       = dim i of target layer lt, head h, token g; keys
 *                      un-rotated at the same position with theta_tgt.
 * x is [Lt][H][2][ntok][k d], y [Lt][H][2][ntok][d] (y and the target caches
 * may be NULL).  Positions come from the request table or src_pos as for the
 * transfer.  A token whose position lies outside [0, max_position) gets zero
 * rows (KVXO_BAD_POSITION); a table row with a layer outside [0, Ls) leaves
 * that target layer's x rows zero (KVXO_BAD_LAYER_INDEX); a malformed request
 * table leaves everything zero (KVXO_BAD_SEQLENS).  The source must be packed
 * (KVXO_CONTIGUOUS); W, b, target positions and layouts are unused. */
int kvxo_ridge_features(const kvxo_problem *prob, const double *tgt_k, const double *tgt_v,
                        double *x, double *y);

#ifdef __cplusplus
}
#endif
#endif /* KVX_ORACLE_H */
