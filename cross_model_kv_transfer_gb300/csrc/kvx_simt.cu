// kvx_simt.cu -- the transfer with an fp32 FMA contraction on the CUDA cores.
//
// Used for fp32 caches (where bf16 tensor-core operands would not meet an
// fp32 tolerance) and for head dimensions the tensor-core kernel does not
// take.  One CTA computes one (target layer lt, head h, K|V, tile of up to
// 8*G consecutive packed source rows, which may span requests):
//   1. gather the k selected source rows of each token into shared memory,
//      un-rotating keys out of the source RoPE ("Helm Intelligent Routing",
//      "Why carrying the cache across is the hard part", step 1; Qwen3
//      article, linear-bridge section: concatenate the selected layers'
//      features, strip source RoPE before mapping keys),
//   2. y = x W + b in fp32, thread (i, y) owning output channels i and
//      i + d/2 of 8 tokens, so the RoPE pair of step 3 stays in registers
//      (step 2: per-layer, per-head linear map),
//   3. re-rotate keys into the target RoPE at p' (step 3), store to the
//      contiguous or paged target cache.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kvx_device.cuh"
#include "kvx_internal.h"

namespace {

constexpr int kRowsPerThread = 8;
constexpr int kThreads = 128;

__device__ __forceinline__ float ldf(const float *p) { return __ldg(p); }
__device__ __forceinline__ float ldf(const __nv_bfloat16 *p) {
  return __bfloat162float(__ldg(p));
}
__device__ __forceinline__ void stf(float *p, float v) { *p = v; }
__device__ __forceinline__ void stf(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

int row_groups(int half) { return half >= kThreads ? 1 : kThreads / half; }

size_t smem_bytes(int half, int kd) {
  const int tt = kRowsPerThread * row_groups(half);
  return (size_t)tt * (kd + 1) * sizeof(float) + (size_t)tt * (sizeof(int64_t) + 2 * sizeof(int32_t));
}

template <typename KT, typename WT, typename BT>
__global__ void __launch_bounds__(kThreads) simt_transfer_kernel(KvxParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int half = p.d >> 1;
  const int G = blockDim.y;
  const int TT = kRowsPerThread * G;
  const int kd = p.k * p.d;
  const int ldx = kd + 1;
  float *X = reinterpret_cast<float *>(smem_raw);
  int64_t *s_row = reinterpret_cast<int64_t *>(X + (size_t)TT * ldx);
  int32_t *s_ps = reinterpret_cast<int32_t *>(s_row + TT);
  int32_t *s_pt = s_ps + TT;
  __shared__ uint32_t s_bits;
  __shared__ int s_layer_ok;

  const int tx = threadIdx.x, ty = threadIdx.y;
  const int tid = ty * blockDim.x + tx;
  const int z = blockIdx.z;
  const int m = z & 1;  // 0: keys, 1: values
  const int h = (z >> 1) % p.H;
  const int lt = (z >> 1) / p.H;

  if (!kvx::seqlens_ok(p, tid, blockDim.x * blockDim.y)) {
    if (blockIdx.x == 0 && z == 0 && tid == 0) kvx::report(p, KVX_FLAG_BAD_SEQLENS);
    return;
  }
  const int64_t t0 = (int64_t)blockIdx.x * TT;

  if (tid == 0) {
    s_bits = 0;
    s_layer_ok = kvx::layer_row_ok(p, lt);
  }
  __syncthreads();
  if (tid < TT) {
    const int64_t g = t0 + tid;
    int32_t ps = 0, pt = 0;
    int64_t row = -1;
    if (g < p.ntok) {
      const uint32_t bad = kvx::token_meta(p, g, ps, pt, row);
      if (bad) atomicOr(&s_bits, bad);
    }
    s_row[tid] = row;
    s_ps[tid] = ps;
    s_pt[tid] = pt;
  }
  __syncthreads();
  if (tid == 0) {
    // row errors are reported by the (lt 0, head 0, K) CTAs, layer errors by
    // the first token tile with head 0, K
    uint32_t bits = (lt == 0 && h == 0 && m == 0) ? s_bits : 0u;
    if (!s_layer_ok && blockIdx.x == 0 && h == 0 && m == 0) bits |= KVX_FLAG_BAD_LAYER_INDEX;
    kvx::report(p, bits);
  }
  if (!s_layer_ok) return;

  // ---- 1. gather + un-rotate (keys) into X[TT][k*d] -----------------------
  const KT *src = reinterpret_cast<const KT *>(m == 0 ? p.src_k : p.src_v);
  for (int q = ty; q < TT; q += G) {
    if (s_row[q] < 0) continue;
    const int64_t g = t0 + q;
    for (int i = tx; i < half; i += blockDim.x) {
      float c = 1.f, s = 0.f;
      if (m == 0) {
        const float2 cs = p.rope_src[(int64_t)s_ps[q] * half + i];
        c = cs.x;
        s = cs.y;
      }
      for (int j = 0; j < p.k; ++j) {
        const int sl = p.layer_idx[lt * p.k + j];
        const KT *v = src + (((int64_t)sl * p.ntok + g) * p.H + h) * p.d;
        const float x0 = ldf(v + i), x1 = ldf(v + i + half);
        // un-rotate: multiply (x0 + j x1) by exp(-j p w_i)
        X[q * ldx + j * p.d + i] = m == 0 ? fmaf(x0, c, x1 * s) : x0;
        X[q * ldx + j * p.d + i + half] = m == 0 ? fmaf(x1, c, -x0 * s) : x1;
      }
    }
  }
  __syncthreads();

  // ---- 2. y = x W + b (fp32) ----------------------------------------------
  const WT *W = reinterpret_cast<const WT *>(p.w) + (((int64_t)lt * p.H + h) * 2 + m) * kd * p.d;
  const BT *B = reinterpret_cast<const BT *>(p.b) + (((int64_t)lt * p.H + h) * 2 + m) * p.d;
  for (int i = tx; i < half; i += blockDim.x) {
    float acc0[kRowsPerThread], acc1[kRowsPerThread];
#pragma unroll
    for (int rr = 0; rr < kRowsPerThread; ++rr) acc0[rr] = acc1[rr] = 0.f;
    for (int qq = 0; qq < kd; ++qq) {
      const float w0 = ldf(W + (int64_t)qq * p.d + i);
      const float w1 = ldf(W + (int64_t)qq * p.d + i + half);
#pragma unroll
      for (int rr = 0; rr < kRowsPerThread; ++rr) {
        const float xv = X[(ty + rr * G) * ldx + qq];
        acc0[rr] = fmaf(xv, w0, acc0[rr]);
        acc1[rr] = fmaf(xv, w1, acc1[rr]);
      }
    }
    const float b0 = ldf(B + i), b1 = ldf(B + i + half);

    // ---- 3. bias, re-rotate keys at p', store -----------------------------
    KT *dst = reinterpret_cast<KT *>(m == 0 ? p.dst_k : p.dst_v);
#pragma unroll
    for (int rr = 0; rr < kRowsPerThread; ++rr) {
      const int q = ty + rr * G;
      const int64_t row = s_row[q];
      if (row < 0) continue;
      float y0 = acc0[rr] + b0, y1 = acc1[rr] + b1;
      if (m == 0) {
        const float2 cs = p.rope_tgt[(int64_t)s_pt[q] * half + i];
        const float r0 = fmaf(y0, cs.x, -y1 * cs.y);  // (y0 + j y1) exp(+j p' w_i)
        const float r1 = fmaf(y0, cs.y, y1 * cs.x);
        y0 = r0;
        y1 = r1;
      }
      KT *o = dst + (((int64_t)lt * p.dst_rows + row) * p.H + h) * p.d;
      stf(o + i, y0);
      stf(o + i + half, y1);
    }
  }
}

template <typename KT, typename WT, typename BT>
void *kernel_ptr() {
  return reinterpret_cast<void *>(&simt_transfer_kernel<KT, WT, BT>);
}

void *select_kernel(const kvx_plan_desc &d) {
  const bool kb = d.kv_dtype == KVX_BF16, wb = d.w_dtype == KVX_BF16, bb = d.b_dtype == KVX_BF16;
  using bf = __nv_bfloat16;
  if (kb) {
    if (wb) return bb ? kernel_ptr<bf, bf, bf>() : kernel_ptr<bf, bf, float>();
    return bb ? kernel_ptr<bf, float, bf>() : kernel_ptr<bf, float, float>();
  }
  if (wb) return bb ? kernel_ptr<float, bf, bf>() : kernel_ptr<float, bf, float>();
  return bb ? kernel_ptr<float, float, bf>() : kernel_ptr<float, float, float>();
}

constexpr size_t kMaxSmem = 227 * 1024;

}  // namespace

bool kvx_simt_supports(const kvx_plan_desc &d) {
  const int half = d.src_head_dim / 2;
  if ((int64_t)d.tgt_layers * d.src_kv_heads * 2 > 65535) return false;
  return smem_bytes(half, d.k * d.src_head_dim) + 64 <= kMaxSmem;
}

cudaError_t kvx_simt_prepare(const kvx_plan *plan) {
  const kvx_plan_desc &d = plan->desc;
  const size_t bytes = smem_bytes(plan->half, d.k * d.src_head_dim);
  return cudaFuncSetAttribute(select_kernel(d), cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)bytes);
}

cudaError_t kvx_simt_launch(const kvx_plan *plan, const KvxParams &p, cudaStream_t s) {
  const int half = plan->half;
  const int G = row_groups(half);
  const int tt = kRowsPerThread * G;
  dim3 block(half >= kThreads ? kThreads : half, G);
  dim3 grid((unsigned)((p.ntok + tt - 1) / tt), 1u, (unsigned)(p.Lt * p.H * 2));
  const size_t bytes = smem_bytes(half, p.k * p.d);
  void *fn = select_kernel(plan->desc);
  KvxParams pp = p;
  void *args[] = {&pp};
  return cudaLaunchKernel(fn, grid, block, args, bytes, s);
}
