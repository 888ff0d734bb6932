// kvx_features.cu -- content-space inputs of the ridge fits (kvx_ridge_features).
//
// The Qwen3 14B -> 32B article, section "Линейного моста, как ни странно,
// хватает", fits one ridge bridge per target (layer, head), one for keys and
// one for values, on the concatenated features of the source layers chosen
// for that target layer, with the source RoPE stripped from the keys before
// the map and the target RoPE applied after it: the fit sees keys in content
// space on both sides.  This file writes those observations from the paired
// caches of a calibration prefill.  For target layer lt, head h and m (0 keys,
// 1 values), batch b = (lt H + h) 2 + m:
//   x[b][g] = the table row's k source layers of token g side by side, keys
//             un-rotated at the token's position with the source base;
//   y[b][g] = target layer lt of token g, keys un-rotated with the target base;
// the batch order kvx_ridge_fit takes and the order kvx_transfer reads W in.
//
// One pass, bound by HBM writes (x is k rows per source row read).  A thread
// carries 4 RoPE pairs of one token (dims 4q .. 4q+3 and d/2 + 4q ..),
// computes each base's 4 angles once and reuses them for the k source rows,
// and consecutive threads write consecutive 16-byte (fp32) or 8-byte (bf16)
// pieces of a row.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvx_internal.h"
#include "kvx_ptx.cuh"

namespace {

constexpr int kFeatMaxD = 128;
constexpr int kFeatThreads = 256;

struct FeatParams {
  const void *src_k, *src_v, *tgt_k, *tgt_v;
  void *x, *y;
  const int32_t *cu, *src_pos, *layer_idx;
  uint32_t *status;
  int64_t n;
  int R, Ls, Lt, H, d, k, max_position;
  unsigned long long turns_src[kFeatMaxD / 2], turns_tgt[kFeatMaxD / 2];
};

__device__ __forceinline__ void load4(const float *p, float v[4]) {
  const float4 t = __ldg(reinterpret_cast<const float4 *>(p));
  v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16 *p, float v[4]) {
  const uint2 t = __ldg(reinterpret_cast<const uint2 *>(p));
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&t.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&t.y));
  v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}
__device__ __forceinline__ void store4(float *p, const float v[4]) {
  *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
__device__ __forceinline__ void store4(__nv_bfloat16 *p, const float v[4]) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
  const __nv_bfloat162 b = __floats2bfloat162_rn(v[2], v[3]);
  uint2 t;
  t.x = *reinterpret_cast<const uint32_t *>(&a);
  t.y = *reinterpret_cast<const uint32_t *>(&b);
  *reinterpret_cast<uint2 *>(p) = t;
}

// (x0 + j x1) e^{-j p w} for the 4 pairs, angles given.
__device__ __forceinline__ void unrotate(float lo[4], float hi[4], const float c[4],
                                         const float s[4]) {
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float a = lo[e] * c[e] + hi[e] * s[e];
    const float b = hi[e] * c[e] - lo[e] * s[e];
    lo[e] = a;
    hi[e] = b;
  }
}

// Request owning packed token g (a valid table assumed).
__device__ __forceinline__ int request_of(const int32_t *cu, int R, int64_t g) {
  if (!cu) return 0;
  int lo = 0, hi = R - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((int64_t)cu[mid] <= g) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Grid: x = (lt H + h) 2 + m, fastest, so that the CTAs of one group of
// 256 / (d / 8) tokens run together and share its source rows in L2; the
// token group is blockIdx.z * gridDim.y + blockIdx.y.  The k rows go one at a
// time (load, un-rotate, store): about 40 registers, 6 CTAs per SM, and the
// 48 warps of an SM keep enough loads in flight to stream the writes at HBM
// speed.  (Holding all k rows' loads in registers before the first store
// needs ~100 registers and 2 CTAs per SM, and ran at half the speed.)
template <typename T, typename O>
__global__ void __launch_bounds__(kFeatThreads, 6) features_kernel(const __grid_constant__ FeatParams p) {
  const int per_tok = p.d / 8;
  const int tpb = kFeatThreads / per_tok;
  const int m = blockIdx.x & 1, h = (blockIdx.x >> 1) % p.H, lt = (blockIdx.x >> 1) / p.H;
  const int64_t group = (int64_t)blockIdx.z * gridDim.y + blockIdx.y;
  const int tid = threadIdx.x;
  // every CTA checks the request table (a malformed one leaves only zeros);
  // without one there is nothing to check and no barrier
  bool table_ok = true;
  if (p.cu) {
    for (int r = tid; r < p.R; r += blockDim.x) table_ok = table_ok && p.cu[r + 1] >= p.cu[r];
    if (tid == 0) table_ok = table_ok && p.cu[0] == 0 && (int64_t)p.cu[p.R] == p.n;
    table_ok = __syncthreads_and(table_ok);
  }
  const int32_t *__restrict__ layers = p.layer_idx + (int64_t)lt * p.k;
  bool row_ok = true;
#pragma unroll 4
  for (int j = 0; j < p.k; ++j) {   // the row's loads issue together
    const int32_t s = __ldg(layers + j);
    row_ok = row_ok && s >= 0 && s < p.Ls;
  }
  if (tid == 0 && group == 0 && m == 0 && h == 0 && p.status) {
    if (!table_ok && lt == 0) atomicOr(p.status, KVX_FLAG_BAD_SEQLENS);
    if (table_ok && !row_ok) atomicOr(p.status, KVX_FLAG_BAD_LAYER_INDEX);
  }
  const int q = tid % per_tok;
  const int64_t g = group * tpb + tid / per_tok;
  if (g >= p.n) return;
  const int d = p.d, half = d / 2;
  const int64_t kd = (int64_t)p.k * d;
  const int64_t b = ((int64_t)lt * p.H + h) * 2 + m;
  O *__restrict__ xrow = reinterpret_cast<O *>(p.x) + (b * p.n + g) * kd + 4 * q;
  O *__restrict__ yrow = p.y ? reinterpret_cast<O *>(p.y) + (b * p.n + g) * d + 4 * q : nullptr;
  int64_t pos = -1;
  if (table_ok) {
    const int r = request_of(p.cu, p.R, g);
    pos = p.src_pos ? (int64_t)p.src_pos[g] : g - (p.cu ? (int64_t)p.cu[r] : 0);
  }
  const bool pos_ok = table_ok && pos >= 0 && pos < p.max_position;
  if (table_ok && !pos_ok && blockIdx.x == 0 && q == 0 && p.status)
    atomicOr(p.status, KVX_FLAG_BAD_POSITION);
  const float zero[4] = {0.f, 0.f, 0.f, 0.f};
  float c[4], s[4];
  if (m == 0 && pos_ok) {
#pragma unroll
    for (int e = 0; e < 4; ++e) rope_cs((uint32_t)pos, p.turns_src[4 * q + e], c[e], s[e]);
  }
  const T *__restrict__ src = reinterpret_cast<const T *>(m ? p.src_v : p.src_k);
  for (int j = 0; j < p.k; ++j) {
    if (!(pos_ok && row_ok)) {
      store4(xrow + (int64_t)j * d, zero);
      store4(xrow + (int64_t)j * d + half, zero);
      continue;
    }
    const T *row = src + (((int64_t)__ldg(layers + j) * p.n + g) * p.H + h) * d + 4 * q;
    float lo[4], hi[4];
    load4(row, lo);
    load4(row + half, hi);
    if (m == 0) unrotate(lo, hi, c, s);
    store4(xrow + (int64_t)j * d, lo);
    store4(xrow + (int64_t)j * d + half, hi);
  }
  if (!yrow) return;
  if (!pos_ok) {
    store4(yrow, zero);
    store4(yrow + half, zero);
    return;
  }
  const T *tgt = reinterpret_cast<const T *>(m ? p.tgt_v : p.tgt_k);
  const T *row = tgt + (((int64_t)lt * p.n + g) * p.H + h) * d + 4 * q;
  float lo[4], hi[4];
  load4(row, lo);
  load4(row + half, hi);
  if (m == 0) {
#pragma unroll
    for (int e = 0; e < 4; ++e) rope_cs((uint32_t)pos, p.turns_tgt[4 * q + e], c[e], s[e]);
    unrotate(lo, hi, c, s);
  }
  store4(yrow, lo);
  store4(yrow + half, hi);
}

template <typename T>
cudaError_t launch_t(const FeatParams &fp, bool out_bf16, dim3 grid, cudaStream_t s) {
  if (out_bf16)
    features_kernel<T, __nv_bfloat16><<<grid, kFeatThreads, 0, s>>>(fp);
  else
    features_kernel<T, float><<<grid, kFeatThreads, 0, s>>>(fp);
  return cudaGetLastError();
}

bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

}  // namespace

extern "C" kvx_status kvx_ridge_features(const kvx_plan *plan, const kvx_feature_args *a,
                                         void *stream) {
  if (!plan || !a) return KVX_ERR_INVALID_ARG;
  const kvx_plan_desc &d = plan->desc;
  const int D = d.src_head_dim;
  if (d.mapper != KVX_MAPPER_PER_HEAD || D % 8 != 0 || D > kFeatMaxD || d.k < 1 ||
      d.src_kv_heads != d.tgt_kv_heads || D != d.tgt_head_dim ||
      (d.kv_dtype != KVX_F32 && d.kv_dtype != KVX_BF16))
    return KVX_ERR_UNSUPPORTED;
  const bool with_y = a->y != nullptr;
  if (a->ntok < 0 || a->ntok > INT32_MAX || !a->layer_idx || a->num_requests < 1 ||
      (!a->cu_seqlens && a->num_requests != 1) ||
      (a->out_dtype != KVX_F32 && a->out_dtype != KVX_BF16))
    return KVX_ERR_INVALID_ARG;
  // the caches and outputs may be NULL when there are no tokens
  if (a->ntok > 0 && (!a->src_k || !a->src_v || !a->x || (with_y && (!a->tgt_k || !a->tgt_v))))
    return KVX_ERR_INVALID_ARG;
  if (!aligned16(a->src_k) || !aligned16(a->src_v) || !aligned16(a->x) ||
      (with_y && (!aligned16(a->tgt_k) || !aligned16(a->tgt_v) || !aligned16(a->y))))
    return KVX_ERR_INVALID_ARG;
  if ((int64_t)d.tgt_layers * d.src_kv_heads * 2 > INT32_MAX) return KVX_ERR_UNSUPPORTED;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return KVX_ERR_CUDA;
  if (cur != plan->device) return KVX_ERR_INVALID_ARG;
  if (a->ntok == 0) return KVX_OK;

  FeatParams fp;
  fp.src_k = a->src_k;
  fp.src_v = a->src_v;
  fp.tgt_k = with_y ? a->tgt_k : nullptr;
  fp.tgt_v = with_y ? a->tgt_v : nullptr;
  fp.x = a->x;
  fp.y = a->y;
  fp.cu = a->cu_seqlens;
  fp.src_pos = a->src_pos;
  fp.layer_idx = a->layer_idx;
  fp.status = a->status;
  fp.n = a->ntok;
  fp.R = a->num_requests;
  fp.Ls = d.src_layers;
  fp.Lt = d.tgt_layers;
  fp.H = d.src_kv_heads;
  fp.d = D;
  fp.k = d.k;
  fp.max_position = d.max_position;
  for (int i = 0; i < kFeatMaxD / 2; ++i) {
    fp.turns_src[i] = i < D / 2 ? plan->turns_src[i] : 0ull;
    fp.turns_tgt[i] = i < D / 2 ? plan->turns_tgt[i] : 0ull;
  }
  const int64_t tpb = kFeatThreads / (D / 8);
  const int64_t groups = (a->ntok + tpb - 1) / tpb;
  const int64_t gy = groups < 65535 ? groups : 65535;
  const dim3 grid((unsigned)(d.tgt_layers * d.src_kv_heads * 2), (unsigned)gy,
                  (unsigned)((groups + gy - 1) / gy));
  cudaStream_t s = (cudaStream_t)stream;
  const bool ob = a->out_dtype == KVX_BF16;
  const cudaError_t e = d.kv_dtype == KVX_BF16 ? launch_t<__nv_bfloat16>(fp, ob, grid, s)
                                               : launch_t<float>(fp, ob, grid, s);
  return e == cudaSuccess ? KVX_OK : KVX_ERR_CUDA;
}
