/*
 * kvx.h -- C ABI of the GB300 cross-model KV-cache transfer library.
 *
 * What it computes.  A pilot (source) model has filled its KV cache for a
 * prompt; a larger target model of the same family is to continue from it
 * without re-reading the prompt.  For every target layer lt, KV head h and
 * token, the library
 *   1. gathers the head-h key and value vectors of the k source layers
 *      idx[lt][0..k-1] selected for lt,
 *   2. un-rotates each key out of the source model's RoPE at its source
 *      position p (half-split pairs (i, i + d/2), frequency
 *      theta_src^(-2i/d)),
 *   3. concatenates the k content vectors (width k*d, index-table order),
 *   4. applies the per-(target layer, head) linear map y = x W + b, one map
 *      for keys (m = 0) and one for values (m = 1),
 *   5. re-rotates the mapped key into the target RoPE (theta_tgt) at the
 *      position p' it will occupy in the target sequence,
 *   6. stores both into the target cache, contiguous or paged.
 * Sources: "Helm Intelligent Routing" (docs.iterate.ai), section "Why
 * carrying the cache across is the hard part", steps 1-3 (un-rotate, map,
 * re-rotate; re-rotation has no skip switch), section "Requirements" (the
 * pair must share KV-head count and head dimension; layer counts may differ)
 * and section "Current limitation" (install into the engine's paged cache);
 * "Перенос KV-кэша между моделями Qwen3 вместо повторного префилла"
 * (reactapp.top), section "Линейного моста, как ни странно, хватает"
 * (selected source layers' features concatenated; one ridge map per target
 * (layer, head), separately for keys and values; strip source RoPE, map,
 * apply target RoPE); knlp.io routing page, the connector's inject step
 * (writes into the paged cache through a block table).
 *
 * Execution model.  kvx_plan_create / kvx_plan_destroy may allocate, free
 * and synchronise.  kvx_transfer only validates its arguments on the host
 * and enqueues kernels on the given stream: it never synchronises and never
 * allocates.  A plan is immutable after creation.  All tensors are owned by
 * the caller.  A SIMT plan owns RoPE tables (read only; its transfers may
 * run concurrently on several streams).  A tensor-core plan computes RoPE
 * angles on the fly and owns a workspace that every transfer rewrites (the
 * bf16 image of W): transfers with the same tensor-core plan must be
 * ordered (same stream, or events).
 *
 * Errors.  Every call returns a kvx_status.  Host-detectable errors are
 * returned before anything is enqueued, and nothing is written.  Errors only
 * the device can see (an index-table entry outside [0, src_layers), a
 * position outside [0, max_position), a block id outside [0, num_blocks), a
 * contiguous row beyond the capacity, a malformed request table, a pipeline
 * wait that gave up) never trap: the affected rows are skipped (all rows,
 * for a malformed request table) and the matching KVX_FLAG_* bits are OR-ed
 * into the caller's status word.  When
 * that word is non-zero after the stream completes, the destination rows of
 * this transfer are unspecified and the caller falls back to a normal
 * prefill of the target ("What happens when a transfer cannot be used":
 * every refusal falls back to prefill).
 */
#ifndef KVX_H
#define KVX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KVX_OK = 0,
  KVX_ERR_INVALID_ARG = 1,    /* a NULL pointer, negative size, bad enum    */
  KVX_ERR_PAIR_MISMATCH = 2,  /* source/target KV heads or head_dim differ  */
  KVX_ERR_UNSUPPORTED = 3,    /* valid, but not supported by this build or
                                 device (e.g. not sm_103, kernel forced onto
                                 a shape it does not handle)                 */
  KVX_ERR_CUDA = 4,           /* a CUDA runtime call failed                  */
  KVX_ERR_NO_MEMORY = 5,      /* plan tables could not be allocated          */
  KVX_ERR_TOO_LARGE = 6       /* kvx_transfer_static: the RoPE tables of this
                                 descriptor do not fit its fixed device array */
} kvx_status;

/* Bits OR-ed into kvx_transfer_args.status by the device. */
#define KVX_FLAG_BAD_LAYER_INDEX 1u  /* idx[lt][j] outside [0, src_layers)    */
#define KVX_FLAG_BAD_POSITION    2u  /* p or p' outside [0, max_position)     */
#define KVX_FLAG_BAD_BLOCK       4u  /* p'/bs >= max_blocks_per_req, or the
                                        block id outside [0, num_blocks)     */
#define KVX_FLAG_BAD_ROW         8u  /* contiguous p' >= dst_capacity         */
#define KVX_FLAG_TIMEOUT        16u  /* a pipeline wait gave up              */
#define KVX_FLAG_BAD_SEQLENS    32u  /* cu_seqlens does not start at 0, runs
                                        backwards or does not end at ntok:
                                        nothing is written                   */
#define KVX_FLAG_BAD_SRC_BLOCK  64u  /* paged source: p/src_bs >=
                                        max_src_blocks_per_req, or the block
                                        id outside [0, src_num_blocks)       */
#define KVX_FLAG_NOT_SPD       128u  /* kvx_ridge_fit: XcT Xc + lam I has a
                                        non-positive pivot (W, b left NaN)   */

typedef enum { KVX_F32 = 0, KVX_BF16 = 1 } kvx_dtype;
typedef enum { KVX_CONTIGUOUS = 0, KVX_PAGED = 1 } kvx_layout;
typedef enum {
  KVX_KERNEL_AUTO = 0,        /* tensor-core path when the shape allows it  */
  KVX_KERNEL_SIMT = 1,        /* fp32 FMA contraction (any even head_dim)   */
  KVX_KERNEL_TCGEN05 = 2      /* tcgen05 tensor cores: bf16 K/V,
                                 head_dim 128, k <= 6 for the per-head map
                                 (W takes k x 32 KB of shared memory; AUTO
                                 picks SIMT beyond)                          */
} kvx_kernel;

/* Which map the transfer applies.
 * PER_HEAD: one map per (target layer, head, K|V) over that head's features
 *   of the k selected layers (width k*d); W is [Lt][H][2][k*d][d].
 * WIDE: one map per target layer over ALL heads' keys and values of the k
 *   selected layers (width F = k*2*H*d) to all heads' keys and values
 *   (N = H*2*d); W is [Lt][F][N], feature (j, m, h, i) at row
 *   ((j*2 + m)*H + h)*d + i (m = 0 the un-rotated key, 1 the value, of
 *   source layer idx[lt][j], head h), output (h, m, i) at column
 *   (h*2 + m)*d + i; b keeps the [Lt][H][2][d] layout.  This is the reading
 *   of the 14B -> 32B mapper size in "Перенос KV-кэша между моделями Qwen3
 *   вместо повторного префилла", section "Ограничения, важные в продакшене"
 *   (about 1.07e9 parameters, 4 GB: 64 x 8192 x 2048 fp32 weights). */
typedef enum { KVX_MAPPER_PER_HEAD = 0, KVX_MAPPER_WIDE = 1 } kvx_mapper;

/* Plan descriptor.  The source and target KV-head counts and head
 * dimensions are given separately so that an incompatible pair is refused
 * with KVX_ERR_PAIR_MISMATCH ("Requirements": same number of KV heads and
 * the same per-head dimension; layer counts may differ freely). */
typedef struct {
  int32_t src_layers;       /* Ls >= 1                                        */
  int32_t tgt_layers;       /* Lt >= 1                                        */
  int32_t src_kv_heads;     /* H, must equal tgt_kv_heads                     */
  int32_t tgt_kv_heads;
  int32_t src_head_dim;     /* d, even, 2..256; must equal tgt_head_dim       */
  int32_t tgt_head_dim;
  int32_t k;                /* selected source layers per target layer, >= 1 */
  double rope_theta_src;    /* RoPE base of the source model, finite, > 0     */
  double rope_theta_tgt;    /* RoPE base of the target model, finite, > 0     */
  int32_t kv_dtype;         /* kvx_dtype of source and target K/V             */
  int32_t w_dtype;          /* kvx_dtype of W                                 */
  int32_t b_dtype;          /* kvx_dtype of b                                 */
  int32_t dst_layout;       /* kvx_layout of the target cache                 */
  int32_t block_size;       /* tokens per block, PAGED only (>= 1)            */
  int32_t max_position;     /* every source and target position must lie in
                               [0, max_position); sizes the SIMT RoPE tables */
  int32_t kernel;           /* kvx_kernel                                    */
  int32_t tiles_per_item;   /* tensor-core path: token tiles (128 rows, or
                               256 for CTA pairs) per work item; W is loaded
                               once per item; 0 = default (32)              */
  int32_t flags;            /* KVX_PLAN_* bits; 0 for normal use            */
  int32_t mapper;           /* kvx_mapper; WIDE needs the tensor-core kernel
                               (bf16 K/V, head_dim 128)                     */
  int32_t max_tokens;       /* WIDE, or a PAGED source on the tensor-core
                               kernel: the most source tokens (ntok) one
                               transfer may carry; sizes the plan's buffers
                               of packed / un-rotated source rows
                               ([Ls][max_tokens][H][d] each); 0 =
                               max_position.  Ignored otherwise             */
  int32_t src_layout;       /* kvx_layout of the SOURCE cache: CONTIGUOUS
                               (packed rows) or PAGED (the pilot's own paged
                               cache, read through a source block table)    */
  int32_t src_block_size;   /* tokens per source block, PAGED source only   */
} kvx_plan_desc;

/* Failure-detection test hook (tensor-core path): the warps that fill the
 * MMA operand never signal it, so the pipeline waits run out (after 20 ms
 * instead of 2 s) and the transfer reports KVX_FLAG_TIMEOUT.  Nothing faults
 * or hangs; the kernel drains and exits.  Never set in production. */
#define KVX_PLAN_TEST_STALL 1

/* kvx_plan_desc.flags bit: run the tensor-core kernel on single CTAs even
 * where the device can co-schedule CTA pairs (by default a pair shares each
 * M = 256 MMA, every CTA holding half of W).  For testing both forms. */
#define KVX_PLAN_TC_SINGLE_CTA 2

typedef struct kvx_plan kvx_plan; /* opaque */

/* Arguments of one transfer.  All pointers are DEVICE pointers to memory of
 * the current device, except where noted; arrays are dense, row-major, with
 * the element type fixed by the plan.  ntok = total source tokens of all
 * requests, packed request after request. */
typedef struct {
  const void *src_k;          /* CONTIGUOUS source: [Ls][ntok][H][d] source keys
                                 (RoPE-rotated), token g at row g.  PAGED
                                 source: [Ls][src_num_blocks*src_bs][H][d],
                                 token g of request r at source position p at
                                 row src_block_table[r][p/src_bs]*src_bs +
                                 p % src_bs (the pilot's paged cache)        */
  const void *src_v;          /* source values, same layout as src_k; src_k
                                 and src_v may be NULL when ntok == 0        */
  int64_t ntok;               /* >= 0 (0: nothing to do)                      */
  int32_t num_requests;       /* R >= 1                                       */
  const int32_t *cu_seqlens;  /* [R+1] request r owns source rows
                                 [cu[r], cu[r+1]); must start at 0, never
                                 decrease and end at ntok (else nothing is
                                 written and KVX_FLAG_BAD_SEQLENS is set).
                                 NULL means R == 1 and the single request
                                 owns all ntok rows                          */
  const int32_t *layer_idx;   /* [Lt][k] selected source layers, in
                                 feature-concatenation order                 */
  const void *w;              /* PER_HEAD: [Lt][H][2][k*d][d] map, m = 0 keys,
                                 1 values; rows follow the concatenation
                                 order.  WIDE: [Lt][k*2*H*d][H*2*d] (see
                                 kvx_mapper)                                 */
  const void *b;              /* [Lt][H][2][d] bias                           */
  const int32_t *src_pos;     /* [ntok] source positions, or NULL: 0..len-1
                                 within each request                         */
  const int32_t *tgt_pos;     /* [ntok] target positions, or NULL:
                                 p' = p + tgt_offset[r]                      */
  const int32_t *tgt_offset;  /* [R] or NULL (offset 0)                       */
  void *dst_k;                /* CONTIGUOUS: [Lt][R*dst_capacity][H][d], row
                                 r*dst_capacity + p';  PAGED:
                                 [Lt][num_blocks*block_size][H][d], row
                                 block_table[r][p'/bs]*bs + p' % bs          */
  void *dst_v;                /* same layout as dst_k                         */
  int64_t dst_capacity;       /* CONTIGUOUS: rows per request (>= 1)          */
  int64_t num_blocks;         /* PAGED: blocks in the pool (>= 1)             */
  const int32_t *block_table; /* PAGED: [R][max_blocks_per_req]               */
  int32_t max_blocks_per_req; /* PAGED: >= 1                                  */
  uint32_t *status;           /* optional device word; KVX_FLAG_* bits are
                                 OR-ed in (never cleared by the library)     */
  int64_t src_num_blocks;     /* PAGED source: blocks in the source pool      */
  const int32_t *src_block_table; /* PAGED source: [R][max_src_blocks_per_req] */
  int32_t max_src_blocks_per_req; /* PAGED source: >= 1                        */
} kvx_transfer_args;

/* Validate the descriptor and prepare the plan on the current device: for
 * the SIMT kernel, RoPE tables (cos/sin of p * w_i for p in
 * [0, max_position), computed in double precision on the host and stored as
 * fp32); for the tensor-core kernel, the frequencies w_i / 2pi as 64-bit
 * fixed-point fractions of a turn (the kernel reduces p * w_i exactly in
 * integer arithmetic and evaluates sin/cos on [-pi, pi)) and the W-image
 * workspace.  Returns an opaque plan in *out.
 * Returns KVX_ERR_INVALID_ARG / KVX_ERR_PAIR_MISMATCH for a bad descriptor
 * (before touching the device), KVX_ERR_UNSUPPORTED if the current device
 * is not sm_103 or the forced kernel cannot handle the shape, KVX_ERR_CUDA or
 * KVX_ERR_NO_MEMORY if the device work fails (KVX_ERR_NO_MEMORY also when
 * the RoPE tables of max_position would not fit the device, or their host
 * staging buffer cannot be allocated).  On error *out is NULL. */
kvx_status kvx_plan_create(const kvx_plan_desc *desc, kvx_plan **out);

/* Enqueue one transfer on `stream` (a cudaStream_t; NULL is the legacy
 * default stream).  Asynchronous: no host synchronisation, no allocation.
 * Returns KVX_ERR_INVALID_ARG for a NULL plan/args or a missing required
 * pointer or size, and, for a tensor-core plan, for source bases that are
 * not 16-byte aligned or cache bases that are not 32-byte aligned, and, for a
 * WIDE plan or a tensor-core plan with a PAGED source, for ntok >
 * max_tokens; KVX_ERR_CUDA if a launch fails.
 * Device-detected errors are reported through args->status as described
 * above.  A WIDE plan's transfer runs three kernels: the source keys of all
 * layers un-rotated into the plan's buffer, W into a bf16 image, and the
 * map as one tensor-core contraction per (target layer, 256 tokens, head)
 * with bias, re-rotation and the cache install in its epilogue.  With a
 * PAGED source the SIMT kernel reads the source rows through the source
 * block table directly; the tensor-core kernels first pack the rows they
 * read (every layer's keys and values, or the values for WIDE, whose key
 * pre-pass reads the paged keys itself) into the plan's buffers, one more
 * launch. */
kvx_status kvx_transfer(const kvx_plan *plan, const kvx_transfer_args *args,
                        void *stream);

/* Free the plan's tables (synchronises the device).  NULL is a no-op. */
kvx_status kvx_plan_destroy(kvx_plan *plan);

/* Static, NUL-terminated description of a status code. */
const char *kvx_status_string(kvx_status status);

/* Which kernel the plan runs (KVX_KERNEL_SIMT or KVX_KERNEL_TCGEN05), or -1
 * for a NULL plan. */
int32_t kvx_plan_kernel(const kvx_plan *plan);

/* Number of kernel launches one kvx_transfer call enqueues with this plan
 * (0 when ntok == 0), or -1 for a NULL plan. */
int32_t kvx_plan_launches(const kvx_plan *plan);

/* CTAs that share each MMA in the plan's tensor-core kernel: 2 when the
 * device co-schedules CTA pairs (one M = 256 MMA per K step, each CTA holding
 * half of W), 1 for single CTAs (or KVX_PLAN_TC_SINGLE_CTA), 0 for a SIMT
 * plan, -1 for a NULL plan. */
int32_t kvx_plan_cta_group(const kvx_plan *plan);

/* Arguments of one fidelity-diagnostics call: a mapped cache (the output of a
 * transfer) and the target model's own cache for the same tokens, in the
 * plan's destination layout, plus the request table, positions and row
 * rules of that transfer.  DEVICE pointers, as for kvx_transfer_args. */
typedef struct {
  const void *mapped_k;       /* [Lt][rows][H][d] mapped keys (kv dtype)      */
  const void *mapped_v;       /* [Lt][rows][H][d] mapped values               */
  const void *ref_k;          /* [Lt][rows][H][d] the target's own keys       */
  const void *ref_v;          /* [Lt][rows][H][d] the target's own values     */
  int64_t ntok;               /* source tokens of the transfer, >= 0          */
  int32_t num_requests;       /* R >= 1                                       */
  const int32_t *cu_seqlens;  /* [R+1] or NULL (R == 1), as for kvx_transfer  */
  const int32_t *src_pos;     /* [ntok] or NULL, as for kvx_transfer          */
  const int32_t *tgt_pos;     /* [ntok] or NULL                               */
  const int32_t *tgt_offset;  /* [R] or NULL                                  */
  int64_t dst_capacity;       /* CONTIGUOUS: rows per request                 */
  int64_t num_blocks;         /* PAGED: blocks in the pool                    */
  const int32_t *block_table; /* PAGED: [R][max_blocks_per_req]               */
  int32_t max_blocks_per_req; /* PAGED                                        */
  double *stats;              /* [Lt][H][2][d + 4] output, overwritten        */
  uint32_t *status;           /* optional device word, KVX_FLAG_* OR-ed in    */
} kvx_diag_args;

/* Fidelity diagnostics of a transfer: how close the mapped cache is to the
 * target model's own cache for the same tokens.  "Helm Intelligent Routing",
 * section "Reading the retention score": the KV cosine between the mapped
 * cache and the target's own is read beside retention as a diagnostic.
 * "Перенос KV-кэша между моделями Qwen3 вместо повторного префилла", section
 * "Линейного моста, как ни странно, хватает": the share of the target keys'
 * and values' variance that the selected source layers explain.
 *
 * For each (target layer lt, head h, m), m = 0 keys and 1 values, the d + 4
 * doubles at stats[((lt * H + h) * 2 + m) * (d + 4)] are set to
 *   [0] n, the tokens compared;
 *   [1] the sum over them of cos(mapped, ref) of the two d-vectors as stored
 *       (0 for a token where either vector is zero);
 *   [2] sum |ref - mapped|^2;   [3] sum |ref|^2;
 *   [4 + i] sum of ref_i in content space (keys un-rotated at p' with the
 *       target RoPE base, values as stored).
 * Mean cosine = [1] / [0]; explained variance (centred R^2, summed over the
 * d dimensions) = 1 - [2] / ([3] - |[4..]|^2 / [0]).  The tokens compared are
 * the ones a transfer with the same request table, positions and destination
 * layout writes; rows it would skip for those reasons are skipped with the
 * same KVX_FLAG_* bits (a malformed request table: all stats 0 and
 * KVX_FLAG_BAD_SEQLENS).  The source side is not read (a paged source's block
 * table plays no part).  Sums are formed in fp32 per thread and
 * combined in fp64; the order of the fp64 additions is not fixed.
 * Asynchronous on `stream`, no allocation, two kernel launches (clear the
 * stats, accumulate).  Returns KVX_ERR_INVALID_ARG for a NULL plan/args, a
 * missing pointer or size, or a plan of another device; KVX_ERR_UNSUPPORTED
 * when target layers x row groups exceed 65,535 CTAs in the grid's y
 * dimension (nothing enqueued); KVX_ERR_CUDA if a launch fails. */
kvx_status kvx_kv_diagnostics(const kvx_plan *plan, const kvx_diag_args *args, void *stream);

/* Arguments of a batch of independent ridge fits (kvx_ridge_fit).  DEVICE
 * pointers; arrays dense and row-major. */
typedef struct {
  int32_t batch;            /* independent fits, 1..65535                     */
  int64_t n;                /* observations per fit, 1..65535*16384           */
  int32_t p;                /* features per observation, 1..4096              */
  int32_t q;                /* outputs per observation, 1..4096               */
  double lambda;            /* ridge strength, added unscaled to the diagonal */
  int32_t x_dtype;          /* kvx_dtype of x and y                           */
  const void *x;            /* [batch][n][p] features                         */
  const void *y;            /* [batch][n][q] targets                          */
  float *w;                 /* [batch][p][q] output: the map                  */
  float *b;                 /* [batch][q] output: the bias                    */
  void *workspace;          /* scratch of at least kvx_ridge_workspace_bytes(),
                               16-byte aligned                                */
  size_t workspace_bytes;
  uint32_t *status;         /* optional device word, KVX_FLAG_NOT_SPD OR-ed in */
} kvx_ridge_args;

/* Bytes of scratch a kvx_ridge_fit call with these sizes needs: fp64 column
 * sums, Gram blocks and cross products (8 * batch * (p + q + p*p + p*q)),
 * the split-precision planes of one chunk of 16,384 observations
 * (2 * 4 * batch * (p + q) * 16384 bytes), the inverses of the factor's
 * 64 x 64 diagonal blocks (8 * batch * ceil(p / 64) * 4096) and the columns'
 * shifts (8 * batch * (p + q)), each part but the last rounded up to 256
 * bytes; 0 for sizes outside the limits above. */
size_t kvx_ridge_workspace_bytes(int32_t batch, int32_t p, int32_t q);

/* Fit the maps: for each fit, W = (XcT Xc + lambda I)^-1 XcT Yc and
 * b = ybar - xbar W, with Xc, Yc the observations centred on their column
 * means.  "Перенос KV-кэша между моделями Qwen3 вместо повторного префилла",
 * section "Линейного моста, как ни странно, хватает": one ridge regression per
 * target (layer, head), one for keys and one for values, fitted on paired
 * source / target observations; its ridge demo centres X and Y and adds
 * lambda I unscaled (0.01 there).  A batch ordered (target layer, head, K|V)
 * with p = k*d and q = d writes W and b in exactly the layouts kvx_transfer
 * reads for a per-head plan with fp32 W and b.  The observations are first
 * shifted by a per-column fp32 value (the mean of 256 of the column's
 * observations spread evenly over all n) and the Gram blocks of the shifted values formed on the
 * tensor cores with each shifted fp32 value split into two tf32 values
 * (products hi*hi + hi*lo + lo*hi, about 22 significant bits; fp32 partial
 * sums over 256 observations, summed in fp32 over slices of 4,096, slices
 * added in fp64); the centring is then exact in fp64 as a rank-one
 * correction with the shifted values' column sums.  The Cholesky
 * factorisation and both triangular solves run in fp64, W and b are stored
 * as fp32; the factorisation is blocked by 64 and spread over CTAs.
 * Asynchronous on `stream`; no allocation (the caller passes the scratch);
 * 4 + 2 ceil(n / 16384) + 3 ceil(p / 64) - 1 kernel launches.  Returns KVX_ERR_INVALID_ARG for a NULL
 * pointer, sizes outside the limits, a non-finite lambda, or a workspace that
 * is too small or not 16-byte aligned; KVX_ERR_CUDA if a launch fails.  A fit
 * whose matrix is not positive definite gets NaN W and b and sets
 * KVX_FLAG_NOT_SPD. */
kvx_status kvx_ridge_fit(const kvx_ridge_args *args, void *stream);

/* Arguments of the layer-selection scores (kvx_layer_scores).  DEVICE
 * pointers unless noted; shapes come from the plan (Ls, Lt, H, d, k, the two
 * RoPE bases, max_position, the cache dtype).  Both caches hold the same
 * tokens in the same packed order (calibration prefills both models on the
 * same text): token g is row g of the source and of the target arrays. */
typedef struct {
  const void *src_k, *src_v;  /* [Ls][ntok][H][d] the pilot's cache (keys
                                 RoPE-rotated with rope_theta_src)           */
  const void *tgt_k, *tgt_v;  /* [Lt][ntok][H][d] the target's own cache of
                                 the same tokens (keys with rope_theta_tgt)  */
  int64_t ntok;               /* tokens, >= 2                                 */
  int32_t num_requests;       /* R >= 1                                       */
  const int32_t *cu_seqlens;  /* [R+1] or NULL (R == 1), as for kvx_transfer  */
  const int32_t *src_pos;     /* [ntok] positions, or NULL: 0..len-1 per
                                 request; both caches are at these positions */
  const int32_t *layer_idx;   /* [Lt][k] or NULL: also score each row's set  */
  double lambda;              /* ridge strength (> 0), added unscaled         */
  double *r2;                 /* [Lt][Ls][H][2] output, m = 0 keys, 1 values  */
  double *r2_set;             /* [Lt][H][2] output, or NULL (needs layer_idx) */
  void *workspace;            /* kvx_layer_scores_workspace_bytes(plan, ntok)
                                 bytes, 16-byte aligned                      */
  size_t workspace_bytes;
  uint32_t *status;           /* optional device word; KVX_FLAG_* OR-ed in    */
} kvx_score_args;

/* Bytes of scratch kvx_layer_scores needs for `ntok` tokens (content
 * features of one (head, K|V) at a time, the split-precision planes of one
 * chunk of up to 16,384 tokens, fp64 sums, Gram and cross blocks), or 0 if
 * the plan cannot score (head_dim not a multiple of 16 or above 128,
 * ntok < 2). */
size_t kvx_layer_scores_workspace_bytes(const kvx_plan *plan, int64_t ntok);

/* Layer-selection scores: how much of each target layer's key / value
 * variance one source layer, or the set of a layer-table row, explains
 * through the ridge bridge.  "Перенос KV-кэша между моделями Qwen3 вместо
 * повторного префилла", section "Линейного моста, как ни странно, хватает":
 * the method picks, per target layer, the source layers whose KV states best
 * predict it (for 14B -> 32B the best single layer explains ~56 % of the
 * keys' variance and ~32 % of the values', a set ~79 % and ~65 %), and fits
 * one ridge regression per target (layer, head), one for keys, one for
 * values.  For every (target layer lt, source layer s, head h, K|V): keys are
 * taken in content space (source keys un-rotated at their position with
 * rope_theta_src, target keys with rope_theta_tgt), the ridge demo's
 * centred fit of the target vectors on the source vectors is formed, and
 * r2 = 1 - sum |y - (x W + b)|^2 / sum |y - ybar|^2, summed over the d
 * dimensions (in-sample).  With layer_idx the set of row lt (its k layers
 * concatenated in table order, the transfer's feature vector) is scored the
 * same way into r2_set.  Computed from fp32 content features: the centred
 * Gram and cross blocks on the tensor cores with each centred value split
 * into two tf32 values (products hi*hi + hi*lo + lo*hi, fp32 partial sums
 * over 256 tokens added in fp64), an fp64 Cholesky of G + lambda I and fp64
 * triangular solves: r2 = (|L^-1 C|^2 + lambda |W|^2) / sum |y - ybar|^2.
 * Asynchronous on `stream`; no allocation (the caller passes the scratch).
 * Returns KVX_ERR_INVALID_ARG for a NULL pointer, lambda <= 0 or non-finite,
 * ntok < 2, or a workspace that is too small or not 16-byte aligned;
 * KVX_ERR_UNSUPPORTED for a head_dim the
 * scorer does not handle; KVX_ERR_CUDA if a launch fails.  Device-detected:
 * a token position outside [0, max_position) or a malformed request table
 * makes every score NaN (KVX_FLAG_BAD_POSITION / KVX_FLAG_BAD_SEQLENS); a
 * set row with a layer index outside [0, Ls) gives NaN set scores
 * (KVX_FLAG_BAD_LAYER_INDEX); a fit that is not positive definite or a
 * target without variance gives NaN (KVX_FLAG_NOT_SPD for the former). */
kvx_status kvx_layer_scores(const kvx_plan *plan, const kvx_score_args *args, void *stream);

/* Arguments of kvx_ridge_features.  DEVICE pointers, 16-byte aligned; shapes
 * come from the plan (Ls, Lt, H, d, k, the two RoPE bases, max_position, the
 * cache dtype).  As for kvx_score_args, both caches hold the same tokens in
 * the same packed order. */
typedef struct {
  const void *src_k, *src_v;  /* [Ls][ntok][H][d] the pilot's cache (keys
                                 RoPE-rotated with rope_theta_src)           */
  const void *tgt_k, *tgt_v;  /* [Lt][ntok][H][d] the target's own cache (keys
                                 with rope_theta_tgt); needed only with y    */
  int64_t ntok;               /* tokens, 0 .. 2^31 - 1                        */
  int32_t num_requests;       /* R >= 1                                       */
  const int32_t *cu_seqlens;  /* [R+1] or NULL (R == 1), as for kvx_transfer  */
  const int32_t *src_pos;     /* [ntok] positions, or NULL: 0..len-1 per
                                 request; both caches are at these positions */
  const int32_t *layer_idx;   /* [Lt][k] the layer table the maps will serve  */
  int32_t out_dtype;          /* kvx_dtype of x and y                         */
  void *x;                    /* [Lt][H][2][ntok][k d] output                 */
  void *y;                    /* [Lt][H][2][ntok][d] output, or NULL          */
  uint32_t *status;           /* optional device word; KVX_FLAG_* OR-ed in    */
} kvx_feature_args;

/* The observations of the ridge fits of a per-head plan's maps, in content
 * space.  "Перенос KV-кэша между моделями Qwen3 вместо повторного префилла",
 * section "Линейного моста, как ни странно, хватает": each target (layer,
 * head) gets one ridge map for keys and one for values, fitted on the
 * concatenated features of the source layers chosen for that target layer,
 * with the source RoPE stripped from the keys before the map and the target
 * RoPE applied after it.  For target layer lt, head h and m (0 keys,
 * 1 values), batch b = (lt H + h) 2 + m and token g at position p (from
 * src_pos, else its offset in its request):
 *   x[b][g][j d + i] = dim i of source layer layer_idx[lt][j], head h;
 *                      keys un-rotated at p with rope_theta_src;
 *   y[b][g][i]       = dim i of target layer lt, head h; keys un-rotated at
 *                      p with rope_theta_tgt.
 * Values are copied as stored.  x and y are exactly the x and y of one
 * kvx_ridge_fit batch (p = k d, q = d) whose W and b kvx_transfer then reads
 * for this plan.  The un-rotation runs in fp32 with angles from the plan's
 * fixed-point RoPE phases (about 1e-6 relative error); a bf16 output is the
 * fp32 result rounded to nearest.  Device-detected: a token whose position
 * lies outside [0, max_position) gets zero rows in x and y
 * (KVX_FLAG_BAD_POSITION); a table row naming a layer outside [0, Ls) leaves
 * that target layer's x rows zero (KVX_FLAG_BAD_LAYER_INDEX; y is still
 * written); a malformed request table leaves x and y all zero
 * (KVX_FLAG_BAD_SEQLENS).  Asynchronous on `stream`, no allocation, one kernel
 * launch (none for ntok == 0, when the caches and outputs may be NULL).
 * Returns KVX_ERR_INVALID_ARG for a NULL plan, args or required pointer, y
 * without both target caches, a pointer that is not 16-byte aligned, sizes
 * outside the limits, a bad out_dtype, or a plan of another device; KVX_ERR_UNSUPPORTED for a wide-mapper plan, a head_dim
 * that is not a multiple of 8 or exceeds 128, or 2 Lt H above 2^31 - 1;
 * KVX_ERR_CUDA if the launch fails. */
kvx_status kvx_ridge_features(const kvx_plan *plan, const kvx_feature_args *args, void *stream);

/* Allocation-free transfer.  The sources have no counterpart for this call:
 * it exists for callers that may not allocate device memory -- engines that
 * reserve nearly all of the GPU for their own paged KV-cache pool and forbid
 * later cudaMalloc calls, and latency-critical paths where cudaMalloc or
 * cudaFree (which may synchronise the device) are not acceptable.
 *
 * It performs the same transfer as a plan created from `desc` with
 * kernel = KVX_KERNEL_SIMT (fp32 FMA contraction) and takes the same
 * arguments, but needs no plan and calls no cudaMalloc, cudaFree or other
 * allocating routine.  Its RoPE tables live in one fixed device array of
 * 2^20 (cos, sin) pairs (8 MiB), compiled into the library and kept on every
 * GPU that loads it until the process exits; each call refills it on the
 * device before the transfer kernel runs.  Limits: max_position * head_dim/2
 * table entries, doubled when the two RoPE bases differ, must not exceed
 * 2^20, else KVX_ERR_TOO_LARGE is returned before anything is enqueued;
 * desc->kernel must be AUTO or SIMT, desc->flags 0 and desc->mapper PER_HEAD.
 *
 * All calls share the array: calls whose work overlaps on the GPU (two
 * streams, for instance) race on it and must be ordered by the caller.  The
 * first call on a device looks up the array's device address (once per
 * device and CUDA context, under a lock; a call after cudaDeviceReset looks
 * it up again in the new context); make that first call before any stream
 * capture.
 * Other errors as for kvx_transfer; `stream` as for kvx_transfer. */
kvx_status kvx_transfer_static(const kvx_plan_desc *desc, const kvx_transfer_args *args,
                               void *stream);

#ifdef __cplusplus
}
#endif
#endif /* KVX_H */
