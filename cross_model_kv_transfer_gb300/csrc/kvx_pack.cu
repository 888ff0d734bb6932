// kvx_pack.cu -- packing a paged source for the tensor-core kernels.
//
// The pilot's KV cache may itself be paged: token g of request r at source
// position p lives in row src_block_table[r][p / bs] * bs + p % bs of every
// source layer (the block-table rule of the knlp.io routing page's inject
// step, applied to the pilot's side).  The tensor-core kernels stage source
// tiles with TMA boxes of 128 consecutive rows, so for a paged source the
// rows they read are first gathered into [Ls][rows][H][d] buffers in packed
// order (row g = token g).  One thread moves one 16-byte word; rows whose
// position or source block is out of range are written as zeros (the
// transfer skips those tokens and flags them).
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvx_device.cuh"
#include "kvx_internal.h"

namespace {

__global__ void __launch_bounds__(256) pack_source_kernel(const __grid_constant__ KvxParams p,
                                                          uint4 *__restrict__ out_k,
                                                          uint4 *__restrict__ out_v,
                                                          int64_t out_rows, int words) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t g = e / words;
  if (g >= p.ntok) return;
  const int w = (int)(e - g * words);
  const int64_t s = blockIdx.y;
  int32_t ps = 0, pt = 0;
  int64_t row = -1, srow = -1;
  kvx::token_meta(p, g, ps, pt, row, srow);
  const int64_t o = (s * out_rows + g) * words + w;
  const int64_t i = (s * p.src_rows + srow) * words + w;
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  if (out_k) out_k[o] = srow >= 0 ? __ldcs(reinterpret_cast<const uint4 *>(p.src_k) + i) : zero;
  if (out_v) out_v[o] = srow >= 0 ? __ldcs(reinterpret_cast<const uint4 *>(p.src_v) + i) : zero;
}

}  // namespace

cudaError_t kvx_pack_source(const KvxParams &p, void *out_k, void *out_v, int64_t out_rows,
                            int elem_bytes, cudaStream_t s) {
  const int64_t row_bytes = (int64_t)p.H * p.d * elem_bytes;
  if (row_bytes % 16 != 0 || p.Ls > 65535) return cudaErrorInvalidValue;
  const int words = (int)(row_bytes / 16);
  const int64_t threads = p.ntok * words;
  if (threads == 0) return cudaSuccess;
  dim3 grid((unsigned)((threads + 255) / 256), (unsigned)p.Ls);
  pack_source_kernel<<<grid, 256, 0, s>>>(p, reinterpret_cast<uint4 *>(out_k),
                                          reinterpret_cast<uint4 *>(out_v), out_rows, words);
  return cudaGetLastError();
}
