/*
 * kvx_c_client.c -- a plain C99 client of the kvx C ABI (include/kvx.h).
 *
 * It shows that the header compiles as C and that a C program links against
 * libkvx.so, and it exercises the calls whose answers need no GPU: descriptor
 * and argument validation, the NULL-handle queries, the ridge scratch size and
 * the status strings.  Prints "ok" and exits 0 when every answer is the
 * documented one; otherwise exits with the number of the first check that
 * failed.
 */
#include <stdio.h>
#include <string.h>

#include "kvx.h"

static void pair_14b_32b(kvx_plan_desc *d) {
  memset(d, 0, sizeof *d);
  d->src_layers = 40;
  d->tgt_layers = 64;
  d->src_kv_heads = 8;
  d->tgt_kv_heads = 8;
  d->src_head_dim = 128;
  d->tgt_head_dim = 128;
  d->k = 4;
  d->rope_theta_src = 1e6;
  d->rope_theta_tgt = 1e6;
  d->kv_dtype = KVX_BF16;
  d->w_dtype = KVX_F32;
  d->b_dtype = KVX_BF16;
  d->dst_layout = KVX_CONTIGUOUS;
  d->max_position = 32768;
  d->kernel = KVX_KERNEL_AUTO;
  d->mapper = KVX_MAPPER_PER_HEAD;
  d->src_layout = KVX_CONTIGUOUS;
}

int main(void) {
  kvx_plan_desc d;
  kvx_plan *plan = (kvx_plan *)&d; /* must come back NULL on every error */
  kvx_ridge_args r;
  kvx_diag_args g;
  kvx_transfer_args a;
  kvx_feature_args f;
  int s;

  memset(&d, 0, sizeof d);
  if (kvx_plan_create(&d, &plan) != KVX_ERR_INVALID_ARG || plan != NULL) return 1;
  pair_14b_32b(&d);
  d.tgt_head_dim = 64; /* the pair must share the head dimension */
  plan = (kvx_plan *)&d;
  if (kvx_plan_create(&d, &plan) != KVX_ERR_PAIR_MISMATCH || plan != NULL) return 2;
  pair_14b_32b(&d);
  d.rope_theta_tgt = -1.0;
  if (kvx_plan_create(&d, &plan) != KVX_ERR_INVALID_ARG) return 3;
  if (kvx_plan_create(NULL, &plan) != KVX_ERR_INVALID_ARG) return 4;

  memset(&a, 0, sizeof a);
  if (kvx_transfer(NULL, &a, NULL) != KVX_ERR_INVALID_ARG) return 5;
  if (kvx_plan_destroy(NULL) != KVX_OK) return 6;
  if (kvx_plan_kernel(NULL) != -1 || kvx_plan_launches(NULL) != -1 ||
      kvx_plan_cta_group(NULL) != -1)
    return 7;

  if (kvx_ridge_workspace_bytes(16, 512, 128) == 0 || kvx_ridge_workspace_bytes(0, 512, 128) != 0)
    return 8;
  memset(&r, 0, sizeof r);
  if (kvx_ridge_fit(&r, NULL) != KVX_ERR_INVALID_ARG) return 9;
  if (kvx_layer_scores(NULL, NULL, NULL) != KVX_ERR_INVALID_ARG ||
      kvx_layer_scores_workspace_bytes(NULL, 4096) != 0)
    return 13;
  memset(&f, 0, sizeof f);
  if (kvx_ridge_features(NULL, &f, NULL) != KVX_ERR_INVALID_ARG ||
      kvx_ridge_features(NULL, NULL, NULL) != KVX_ERR_INVALID_ARG)
    return 14;
  memset(&g, 0, sizeof g);
  if (kvx_kv_diagnostics(NULL, &g, NULL) != KVX_ERR_INVALID_ARG) return 10;

  pair_14b_32b(&d);
  d.kernel = KVX_KERNEL_TCGEN05; /* the allocation-free call runs SIMT only */
  if (kvx_transfer_static(&d, &a, NULL) != KVX_ERR_INVALID_ARG) return 11;
  d.kernel = KVX_KERNEL_AUTO;
  d.rope_theta_tgt = 5e5; /* two tables of 32768 x 64 pairs exceed its array */
  if (kvx_transfer_static(&d, &a, NULL) != KVX_ERR_TOO_LARGE) return 12;

  for (s = KVX_OK; s <= KVX_ERR_TOO_LARGE; ++s)
    printf("%d %s\n", s, kvx_status_string((kvx_status)s));
  printf("ok\n");
  return 0;
}
