// kvx_internal.h -- plan object and kernel parameter block shared by the
// host API (kvx_api.cpp) and the kernels (kvx_simt.cu, kvx_tcgen05.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvx.h"

struct kvx_plan {
  kvx_plan_desc desc;
  int device;
  int kernel;            // KVX_KERNEL_SIMT or KVX_KERNEL_TCGEN05
  int num_sms;
  int half;              // head_dim / 2
  // RoPE tables: rope[p * half + i] = (cos, sin)(p * theta^(-2i/d)),
  // p in [0, max_position), computed in double on the host, stored fp32.
  float2 *rope_src;
  float2 *rope_tgt;      // aliases rope_src when the two thetas are equal
  // tensor-core path only: bf16 W image written by every transfer before the
  // main kernel reads it (transfers sharing a plan are stream-ordered on it)
  void *workspace;
  size_t workspace_bytes;
  int tiles_per_item;    // 128-token tiles per work item of the persistent kernel
  void *encode_tiled;    // driver entry point cuTensorMapEncodeTiled
  // tensor-core path: source RoPE table, position-major per quad of pairs
  // (i .. i+3), i % 4 == 0: tc_rope_src[i/4][p] = bf16x2 (cos_i, cos_i+1),
  // (sin_i, sin_i+1), (cos_i+2, cos_i+3), (sin_i+2, sin_i+3); target RoPE
  // frequencies as 64-bit fractions of a turn, round(w_i / 2pi * 2^64)
  // (set for every plan: the diagnostics kernel uses them too)
  void *tc_rope_src;
  unsigned long long turns_tgt[128];
  // source RoPE frequencies in the same fixed point (the wide path's
  // un-rotation pre-pass)
  unsigned long long turns_src[128];
  // wide-feature mapper: the workspace holds the bf16 W image, the fp32
  // bias and the un-rotated source keys [Ls][max_tokens][H][d]
  int64_t max_tokens;
  // tensor-core plans with a paged source: the rows the kernels read, packed
  // into [Ls][max_tokens][H][d] buffers (keys and values; values only for
  // the wide map, whose workspace already holds the un-rotated keys)
  void *packed_k, *packed_v;
  int stall_test;        // KVX_PLAN_TEST_STALL: failure-detection test hook
  int tc_pairs;          // tensor-core path: CTA pairs resident at once (0: single CTAs)
};

// Everything a kernel needs, passed by value.
struct KvxParams {
  const void *src_k, *src_v;
  const void *w, *b;
  void *dst_k, *dst_v;
  const int32_t *cu_seqlens, *layer_idx, *src_pos, *tgt_pos, *tgt_offset;
  const int32_t *block_table;
  uint32_t *status;
  const float2 *rope_src, *rope_tgt;
  int64_t ntok, dst_capacity, num_blocks, dst_rows;
  int32_t R, max_blocks;
  int32_t Ls, Lt, H, d, k, layout, block_size, max_position;
  // source layout: CONTIGUOUS (row g) or PAGED (through src_block_table);
  // src_rows = rows per source layer of the arrays src_k / src_v point at
  int32_t src_layout, src_block_size, src_max_blocks;
  int64_t src_num_blocks, src_rows;
  const int32_t *src_block_table;
};

// Per-kernel launchers; return cudaSuccess or the launch error.
cudaError_t kvx_simt_prepare(const kvx_plan *plan);
cudaError_t kvx_simt_launch(const kvx_plan *plan, const KvxParams &p, cudaStream_t s);
bool kvx_simt_supports(const kvx_plan_desc &d);

// Packs the source rows of a paged source into [Ls][out_rows][H][d]
// buffers (either may be NULL to skip it); rows whose position or source
// block is out of range are written as zeros.
cudaError_t kvx_pack_source(const KvxParams &p, void *out_k, void *out_v, int64_t out_rows,
                            int elem_bytes, cudaStream_t s);

bool kvx_wide_supports(const kvx_plan_desc &d);
size_t kvx_wide_workspace_bytes(const kvx_plan_desc &d, int64_t max_tokens);
cudaError_t kvx_wide_prepare(kvx_plan *plan);
cudaError_t kvx_wide_launch(const kvx_plan *plan, const KvxParams &p, cudaStream_t s);

bool kvx_tc_supports(const kvx_plan_desc &d);
size_t kvx_tc_workspace_bytes(const kvx_plan_desc &d);
void *kvx_tc_encoder();
cudaError_t kvx_tc_prepare(kvx_plan *plan);
cudaError_t kvx_tc_launch(const kvx_plan *plan, const KvxParams &p, cudaStream_t s);
