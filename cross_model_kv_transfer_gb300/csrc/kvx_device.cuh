// kvx_device.cuh -- per-request / per-token bookkeeping shared by the kernels:
// request ranges, source and target positions, cache rows, range checks.
//
// Cache install ("Helm Intelligent Routing", section "Current limitation":
// the mapped cache goes into the engine's paged cache; knlp.io routing page,
// inject step: entries are written through the block table):
//   contiguous  row = r * dst_capacity + p'
//   paged       row = block_table[r][p' / bs] * bs + p' % bs
// where p' is the position the entry will occupy in the target sequence
// ("re-rotated into the position it will occupy").
#pragma once

#include <stdint.h>

#include "kvx_internal.h"

namespace kvx {

// The request table must start at 0, never decrease and end at ntok; a
// malformed table invalidates the whole transfer (KVX_FLAG_BAD_SEQLENS, no
// writes).  Checked cooperatively by all `nthreads` threads of the CTA (every
// thread must call it).
__device__ __forceinline__ bool seqlens_ok(const KvxParams &p, int tid, int nthreads) {
  bool ok = true;
  if (p.cu_seqlens != nullptr) {
    for (int r = tid; r < p.R; r += nthreads)
      ok = ok && p.cu_seqlens[r + 1] >= p.cu_seqlens[r];
    if (tid == 0) ok = ok && p.cu_seqlens[0] == 0 && (int64_t)p.cu_seqlens[p.R] == p.ntok;
  }
  return __syncthreads_and(ok) != 0;
}

// Request owning packed source row g (a valid table is assumed): the largest
// r in [0, R) with cu[r] <= g.
__device__ __forceinline__ int request_of(const KvxParams &p, int64_t g) {
  if (p.cu_seqlens == nullptr) return 0;
  int lo = 0, hi = p.R - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((int64_t)p.cu_seqlens[mid] <= g) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Source position p, target position p' and destination row of packed
// source row g.  Returns 0 and sets row >= 0, or the KVX_FLAG_* reason with
// row = -1.
// Also sets srow, the row of token g in the source arrays: g for a
// contiguous source, src_block_table[r][p / bs] * bs + p % bs for a paged one
// (the pilot's own paged cache holds its tokens at their source positions).
// The checks run in the order positions, source row, destination row; the
// first that fails is returned (srow and row stay -1 from there on).
__device__ __forceinline__ uint32_t token_meta(const KvxParams &p, int64_t g, int32_t &ps,
                                               int32_t &pt, int64_t &row, int64_t &srow) {
  row = -1;
  srow = -1;
  const int r = request_of(p, g);
  const int64_t beg = p.cu_seqlens ? (int64_t)p.cu_seqlens[r] : 0;
  const int64_t sp = p.src_pos ? (int64_t)p.src_pos[g] : g - beg;
  const int64_t off = p.tgt_offset ? (int64_t)p.tgt_offset[r] : 0;
  const int64_t tp = p.tgt_pos ? (int64_t)p.tgt_pos[g] : sp + off;
  if (sp < 0 || sp >= p.max_position || tp < 0 || tp >= p.max_position)
    return KVX_FLAG_BAD_POSITION;
  ps = (int32_t)sp;
  pt = (int32_t)tp;
  if (p.src_layout == KVX_PAGED) {
    const int64_t logical = sp / p.src_block_size;
    if (logical >= p.src_max_blocks) return KVX_FLAG_BAD_SRC_BLOCK;
    const int64_t phys = p.src_block_table[(int64_t)r * p.src_max_blocks + logical];
    if (phys < 0 || phys >= p.src_num_blocks) return KVX_FLAG_BAD_SRC_BLOCK;
    srow = phys * p.src_block_size + sp % p.src_block_size;
  } else {
    srow = g;
  }
  if (p.layout == KVX_CONTIGUOUS) {
    if (tp >= p.dst_capacity) return KVX_FLAG_BAD_ROW;
    row = (int64_t)r * p.dst_capacity + tp;
    return 0;
  }
  const int64_t logical = tp / p.block_size;
  if (logical >= p.max_blocks) return KVX_FLAG_BAD_BLOCK;
  const int64_t phys = p.block_table[(int64_t)r * p.max_blocks + logical];
  if (phys < 0 || phys >= p.num_blocks) return KVX_FLAG_BAD_BLOCK;
  row = phys * p.block_size + tp % p.block_size;
  return 0;
}

__device__ __forceinline__ uint32_t token_meta(const KvxParams &p, int64_t g, int32_t &ps,
                                               int32_t &pt, int64_t &row) {
  int64_t srow;
  return token_meta(p, g, ps, pt, row, srow);
}

// True if every selected source layer of target layer lt lies in [0, Ls).
__device__ __forceinline__ bool layer_row_ok(const KvxParams &p, int lt) {
  bool ok = true;
  for (int j = 0; j < p.k; ++j) {
    const int s = p.layer_idx[lt * p.k + j];
    ok = ok && s >= 0 && s < p.Ls;
  }
  return ok;
}

__device__ __forceinline__ void report(const KvxParams &p, uint32_t bits) {
  if (bits && p.status) atomicOr(p.status, bits);
}

}  // namespace kvx
