// kvx_scores.cu -- layer-selection scores (kvx_layer_scores).
//
// The Qwen3 14B -> 32B article, section "Линейного моста, как ни странно,
// хватает", chooses for every target layer the source layers whose KV states
// best predict it and fits one ridge bridge per target (layer, head), one for
// keys and one for values (its ridge demo: centre X and Y, solve
// (XcT Xc + lam I) W = XcT Yc, b = ybar - xbar W).  This file scores those
// choices on paired caches of the same tokens: for every (target layer lt,
// source layer s, head h, K|V) the in-sample explained variance of the ridge
// fit of the target's content vectors on the source's,
//   r2 = 1 - sum |y - (x W + b)|^2 / sum |y - ybar|^2   (summed over d),
// and, given a layer table, the same for each row's concatenated set.
//
// With G = XcT Xc + lam I = L L^T, C = XcT Yc, W = G^-1 C and Z = L^-1 C,
// the residual is sum |Yc|^2 - |Z|^2 - lam |W|^2, so
//   r2 = (|Z|^2 + lam |W|^2) / sum |Yc|^2.
// Per (head, K|V) one pass of launches:
//   1. content features (keys un-rotated at the token's position with each
//      model's base, values as stored) of every source and target layer,
//      fp32, with fp64 column sums and the targets' sums of squares;
//   2. centred Gram blocks G (upper triangle) and cross blocks C: fp32
//      products in register tiles, fp32 partial sums over 256 tokens, slices
//      of tokens added in fp64 with atomics; one batch per source layer (G
//      of that layer, C against every target layer at once), and with a
//      layer table one batch per target layer (its row's layers gathered as
//      the features, C against that target layer);
//   3. fp64 Cholesky of G + lam I, blocked by 64 (kvx_chol.cuh);
//   4. fp64 forward and back substitution per column, keeping only the
//      column's |z|^2 and |w|^2, summed per target layer;
//   5. the scores.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>

#include "kvx_chol.cuh"
#include "kvx_internal.h"

namespace {

constexpr int kTile = 64;              // Gram tile
constexpr int kChunkObs = 32;          // tokens staged per step
constexpr int kFlushObs = 256;         // fp32 partials flushed this often
constexpr int64_t kRowsPerSlice = 8192;  // tokens per CTA of the Gram kernel
constexpr int kMaxD = 128;
constexpr int kMaxK = 8;

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// Per-pass scratch (one head h and one of K|V), carved from the caller's
// workspace.
struct Pass {
  float *X;          // [Ls][n][d] source content
  float *Y;          // [n][Lt][d] target content (all target layers per token)
  double *xs;        // [Ls][d] column sums
  double *ys;        // [Lt][d]
  double *yss;       // [Lt] sums of squares
  double *G;         // [Ls][d][d]
  double *C;         // [Ls][d][Lt*d]
  double *zz, *ww;   // [Ls][Lt]
  double *Gs;        // [Lt][k*d][k*d]   (sets)
  double *Cs;        // [Lt][k*d][d]
  double *zzs, *wws; // [Lt]
  int *bad;          // [1]: the transfer-wide validity (positions, request table)
};

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

struct Layout {
  size_t X, Y, xs, ys, yss, G, C, zz, ww, Gs, Cs, zzs, wws, bad, total;
};

Layout layout_of(int64_t Ls, int64_t Lt, int64_t d, int64_t k, int64_t n) {
  Layout L;
  size_t at = 0;
  auto take = [&](size_t bytes) { const size_t o = at; at += round256(bytes); return o; };
  L.X = take((size_t)Ls * n * d * 4);
  L.Y = take((size_t)n * Lt * d * 4);
  L.xs = take((size_t)Ls * d * 8);
  L.ys = take((size_t)Lt * d * 8);
  L.yss = take((size_t)Lt * 8);
  L.G = take((size_t)Ls * d * d * 8);
  L.C = take((size_t)Ls * d * Lt * d * 8);
  L.zz = take((size_t)Ls * Lt * 8);
  L.ww = take((size_t)Ls * Lt * 8);
  L.Gs = take((size_t)Lt * k * d * k * d * 8);
  L.Cs = take((size_t)Lt * k * d * d * 8);
  L.zzs = take((size_t)Lt * 8);
  L.wws = take((size_t)Lt * 8);
  L.bad = take(16);
  L.total = at;
  return L;
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

// The request table: starts at 0, never decreases, ends at ntok.
__global__ void check_table_kernel(const int32_t *cu, int R, int64_t n, int *bad,
                                   uint32_t *status) {
  bool ok = true;
  if (cu) {
    for (int r = threadIdx.x; r < R; r += blockDim.x) ok = ok && cu[r + 1] >= cu[r];
    if (threadIdx.x == 0) ok = ok && cu[0] == 0 && (int64_t)cu[R] == n;
  }
  ok = __syncthreads_and(ok);
  if (threadIdx.x == 0) {
    bad[0] = ok ? 0 : 1;
    if (!ok && status) atomicOr(status, KVX_FLAG_BAD_SEQLENS);
  }
}

__global__ void clear_kernel(double *x, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    x[i] = 0.0;
}

// Angle of position p for a frequency stored as a 64-bit fraction of a turn
// (p * F mod 2^64, top 32 bits, in [-pi, pi)), as the transfer kernels use.
__device__ __forceinline__ void turn_cs(uint32_t pos, unsigned long long turns, float &c, float &s) {
  const uint32_t hi = (uint32_t)(turns >> 32), lo = (uint32_t)turns;
  const uint32_t top = __umulhi(pos, lo) + pos * hi;
  const float a = (float)(int32_t)top * 1.46291807926715968e-9f;   // 2 pi / 2^32
  __sincosf(a, &s, &c);
}

struct Turns {
  unsigned long long src[kMaxD / 2], tgt[kMaxD / 2];
};

// 1. Content features of one (head, K|V) for every source layer (blockIdx.y
// < Ls) and target layer, with column sums.  A thread handles 8 RoPE pairs
// of one token: dims 8q.. and d/2 + 8q..; a block covers 256 / (d / 16)
// tokens.  Keys are un-rotated at the token's position (source base for
// source layers, target base for target layers).
template <typename T>
__global__ void __launch_bounds__(256) content_kernel(
    const T *__restrict__ src, const T *__restrict__ tgt, int Ls, int Lt, int H, int d, int h,
    int is_key, int64_t n, const int32_t *__restrict__ cu, int R,
    const int32_t *__restrict__ src_pos, int max_position, const __grid_constant__ Turns turns,
    Pass ps, uint32_t *status) {
  __shared__ float ssum[kMaxD];
  __shared__ float sss;
  const int L = blockIdx.y;
  const bool is_src = L < Ls;
  const int layer = is_src ? L : L - Ls;
  const int per_tok = d / 16;                      // threads per token
  const int tpb = 256 / per_tok;                   // tokens per block
  const int tid = threadIdx.x;
  for (int i = tid; i < d; i += blockDim.x) ssum[i] = 0.f;
  if (tid == 0) sss = 0.f;
  __syncthreads();
  const int q = tid % per_tok;
  const int64_t g = (int64_t)blockIdx.x * tpb + tid / per_tok;
  const int half = d / 2;
  float lo[8], hi[8];
  bool valid = g < n;
  if (valid) {
    const T *row = (is_src ? src + (((int64_t)layer * n + g) * H + h) * d
                           : tgt + (((int64_t)layer * n + g) * H + h) * d);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      lo[e] = to_f<T>(row[8 * q + e]);
      hi[e] = to_f<T>(row[half + 8 * q + e]);
    }
    if (is_key) {
      const int r = request_of(cu, R, g);
      const int64_t p = src_pos ? (int64_t)src_pos[g] : g - (cu ? (int64_t)cu[r] : 0);
      if (p < 0 || p >= max_position) {
        if (L == 0 && q == 0) {
          ps.bad[0] = 1;
          if (status) atomicOr(status, KVX_FLAG_BAD_POSITION);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float c, s;
          turn_cs((uint32_t)p, is_src ? turns.src[8 * q + e] : turns.tgt[8 * q + e], c, s);
          // (x0 + j x1) * exp(-j p w)
          const float a = lo[e] * c + hi[e] * s;
          const float b = hi[e] * c - lo[e] * s;
          lo[e] = a;
          hi[e] = b;
        }
      }
    } else if (L == 0 && q == 0) {
      // values carry no position, but the positions are checked all the same
      const int r = request_of(cu, R, g);
      const int64_t p = src_pos ? (int64_t)src_pos[g] : g - (cu ? (int64_t)cu[r] : 0);
      if (p < 0 || p >= max_position) {
        ps.bad[0] = 1;
        if (status) atomicOr(status, KVX_FLAG_BAD_POSITION);
      }
    }
    float *out = is_src ? ps.X + ((int64_t)layer * n + g) * d
                        : ps.Y + (g * Lt + layer) * d;
    float sq = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      out[8 * q + e] = lo[e];
      out[half + 8 * q + e] = hi[e];
      atomicAdd(&ssum[8 * q + e], lo[e]);
      atomicAdd(&ssum[half + 8 * q + e], hi[e]);
      sq += lo[e] * lo[e] + hi[e] * hi[e];
    }
    if (!is_src) atomicAdd(&sss, sq);
  }
  __syncthreads();
  double *sums = is_src ? ps.xs + (int64_t)layer * d : ps.ys + (int64_t)layer * d;
  for (int i = tid; i < d; i += blockDim.x) atomicAdd(sums + i, (double)ssum[i]);
  if (!is_src && tid == 0) atomicAdd(ps.yss + layer, (double)sss);
}

// 2. Centred Gram (upper-triangle tiles) and cross blocks of a batch of
// fits.  Fit b has p = nsel * d features: feature j * d + i is dim i of
// source layer xl[b * nsel + j] (content X), and q target columns starting
// at column y0 + b * y_step of the [n][Lt * d] target content Y.
__global__ void __launch_bounds__(256) gram_kernel(
    const float *__restrict__ X, const float *__restrict__ Y, const double *__restrict__ xs,
    const double *__restrict__ ys, const int32_t *__restrict__ xl, int nsel, int d, int Lt,
    int64_t n, int q, int y0, int y_step, double *__restrict__ G, double *__restrict__ C,
    int tiles_p, int tiles_q) {
  __shared__ float sa[kChunkObs][kTile];
  __shared__ float sb[kChunkObs][kTile];
  __shared__ float mean_a[kTile], mean_b[kTile];
  __shared__ int src_a[kTile];                      // source layer of each a column
  __shared__ int src_b[kTile];                      // (Gram tiles) of each b column
  const int b = blockIdx.z;
  const int p = nsel * d;
  int ti, tj;
  {
    int t = blockIdx.x;
    const int n_upper = tiles_p * (tiles_p + 1) / 2;
    if (t < n_upper) {
      ti = 0;
      while (t >= tiles_p - ti) {
        t -= tiles_p - ti;
        ++ti;
      }
      tj = ti + t;
    } else {
      t -= n_upper;
      ti = t / tiles_q;
      tj = tiles_p + t % tiles_q;
    }
  }
  const bool is_c = tj >= tiles_p;
  const int i0 = ti * kTile;
  const int j0 = (is_c ? tj - tiles_p : tj) * kTile;
  const int ncols = is_c ? q : p;
  const int ycol0 = y0 + b * y_step;
  const double inv_n = 1.0 / (double)n;
  const int tid = threadIdx.x;
  if (tid < kTile) {
    const int f = i0 + tid;
    if (f < p) {
      const int s = xl[b * nsel + f / d];
      src_a[tid] = s;
      mean_a[tid] = (float)(xs[(int64_t)s * d + f % d] * inv_n);
    } else {
      src_a[tid] = -1;
      mean_a[tid] = 0.f;
    }
  } else if (tid < 2 * kTile) {
    const int c = tid - kTile;
    const int f = j0 + c;
    if (f < ncols) {
      if (is_c) {
        src_b[c] = -1;
        mean_b[c] = (float)(ys[(int64_t)(ycol0 + f)] * inv_n);   // ys is [Lt][d] = [Lt*d]
      } else {
        const int s = xl[b * nsel + f / d];
        src_b[c] = s;
        mean_b[c] = (float)(xs[(int64_t)s * d + f % d] * inv_n);
      }
    } else {
      src_b[c] = -2;
      mean_b[c] = 0.f;
    }
  }
  const int tx = tid & 15, ty = tid >> 4;
  const int64_t t0 = (int64_t)blockIdx.y * kRowsPerSlice;
  const int64_t t1 = t0 + kRowsPerSlice < n ? t0 + kRowsPerSlice : n;
  float acc[4][4], part[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[r][c] = 0.f, part[r][c] = 0.f;
  __syncthreads();
  int since_flush = 0;
  const int64_t yrow = (int64_t)Lt * d;
  for (int64_t t = t0; t < t1; t += kChunkObs) {
    for (int e = tid; e < kChunkObs * kTile; e += blockDim.x) {
      const int o = e / kTile, c = e % kTile;
      const int64_t u = t + o;
      const bool in = u < t1;
      const int fa = i0 + c, fb = j0 + c;
      sa[o][c] = (in && src_a[c] >= 0)
                     ? X[((int64_t)src_a[c] * n + u) * d + fa % d] - mean_a[c]
                     : 0.f;
      float vb = 0.f;
      if (in && src_b[c] != -2)
        vb = (is_c ? Y[u * yrow + ycol0 + fb] : X[((int64_t)src_b[c] * n + u) * d + fb % d]) -
             mean_b[c];
      sb[o][c] = vb;
    }
    __syncthreads();
#pragma unroll 8
    for (int o = 0; o < kChunkObs; ++o) {
      const float4 a4 = *reinterpret_cast<const float4 *>(&sa[o][4 * ty]);
      const float4 b4 = *reinterpret_cast<const float4 *>(&sb[o][4 * tx]);
      const float av[4] = {a4.x, a4.y, a4.z, a4.w};
      const float bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) part[r][c] = fmaf(av[r], bv[c], part[r][c]);
    }
    __syncthreads();
    since_flush += kChunkObs;
    if (since_flush >= kFlushObs) {
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] += part[r][c], part[r][c] = 0.f;
      since_flush = 0;
    }
  }
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = i0 + 4 * ty + r, j = j0 + 4 * tx + c;
      if (i >= p || j >= ncols) continue;
      const double v = (double)acc[r][c] + (double)part[r][c];
      if (is_c)
        atomicAdd(C + ((int64_t)b * p + i) * q + j, v);
      else
        atomicAdd(G + ((int64_t)b * p + i) * p + j, v);
    }
}

// 4. Per (fit b, nc columns): forward L z = c and back L^T w = z in fp64
// (chol_solve_cols), then |z|^2 and |w|^2 added into zz / ww
// [b][column / d] (the target layer of the column for the per-layer fits,
// the single output group for the sets).
__global__ void __launch_bounds__(kSolveThreads) solve_norms_kernel(
    const double *__restrict__ G, const double *__restrict__ C, int p, int q, int d, int nc,
    double *__restrict__ zz, double *__restrict__ ww, int groups) {
  extern __shared__ double cols[];   // [p][nc], then p reciprocals
  const int b = blockIdx.x;
  const double *A = G + (int64_t)b * p * p;
  if (isnan(A[0])) return;    // not positive definite: the scores stay NaN
  const int c0 = blockIdx.y * nc;
  const double *src = C + (int64_t)b * p * q;
  for (int e = threadIdx.x; e < p * nc; e += kSolveThreads) {
    const int i = e / nc, j = e % nc;
    cols[e] = c0 + j < q ? src[(int64_t)i * q + c0 + j] : 0.0;
  }
  double zn, wn;
  chol_solve_cols(A, p, cols, cols + (size_t)p * nc, nc, zn, wn);
  const int c = c0 + threadIdx.x;
  if (threadIdx.x < nc && c < q) {
    const int grp = groups > 1 ? c / d : 0;
    atomicAdd(zz + (int64_t)b * groups + grp, zn);
    atomicAdd(ww + (int64_t)b * groups + grp, wn);
  }
}

// 5. The scores of one pass: r2 = (|Z|^2 + lam |W|^2) / sum |Yc|^2.
__global__ void finalize_kernel(const Pass ps, int Ls, int Lt, int H, int d, int h, int m,
                                int64_t n, double lam, double *__restrict__ r2,
                                double *__restrict__ r2_set, const int32_t *__restrict__ idx,
                                int k, uint32_t *status) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  const bool bad = ps.bad[0] != 0;
  if (e < Lt) {
    // the set of row e
    if (r2_set) {
      bool ok = !bad;
      for (int j = 0; j < k; ++j) ok = ok && idx[e * k + j] >= 0 && idx[e * k + j] < Ls;
      double tot = ps.yss[e];
      for (int i = 0; i < d; ++i) tot -= ps.ys[(int64_t)e * d + i] * ps.ys[(int64_t)e * d + i] / (double)n;
      const bool spd = !isnan(ps.Gs[(int64_t)e * k * d * k * d]);
      double v = nan("");
      if (ok && spd && tot > 0.0) v = (ps.zzs[e] + lam * ps.wws[e]) / tot;
      r2_set[((int64_t)e * H + h) * 2 + m] = v;
    }
  }
  if (e < Ls * Lt) {
    const int s = e / Lt, lt = e % Lt;
    double tot = ps.yss[lt];
    for (int i = 0; i < d; ++i) tot -= ps.ys[(int64_t)lt * d + i] * ps.ys[(int64_t)lt * d + i] / (double)n;
    const bool spd = !isnan(ps.G[(int64_t)s * d * d]);
    double v = nan("");
    if (!bad && spd && tot > 0.0) v = (ps.zz[(int64_t)s * Lt + lt] + lam * ps.ww[(int64_t)s * Lt + lt]) / tot;
    r2[(((int64_t)lt * Ls + s) * H + h) * 2 + m] = v;
  }
  (void)status;
}

// Bad layer indices of the table (once).
__global__ void check_rows_kernel(const int32_t *idx, int Lt, int k, int Ls, uint32_t *status) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e < Lt * k && (idx[e] < 0 || idx[e] >= Ls) && status)
    atomicOr(status, KVX_FLAG_BAD_LAYER_INDEX);
}

// Identity list 0..Ls-1 for the per-layer fits; the set fits read the
// table, with out-of-range indices clamped (their scores are NaN anyway).
__global__ void layer_lists_kernel(int32_t *ident, int Ls, int32_t *sets, const int32_t *idx,
                                   int n_idx) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e < Ls) ident[e] = e;
  if (e < n_idx) {
    const int v = idx[e];
    sets[e] = v < 0 ? 0 : (v >= Ls ? Ls - 1 : v);
  }
}

bool plan_ok(const kvx_plan_desc &d) {
  return d.src_head_dim % 16 == 0 && d.src_head_dim <= kMaxD && d.k >= 1 && d.k <= kMaxK &&
         d.src_kv_heads == d.tgt_kv_heads && d.src_head_dim == d.tgt_head_dim &&
         (d.kv_dtype == KVX_F32 || d.kv_dtype == KVX_BF16);
}

size_t lists_bytes(const kvx_plan_desc &d) {
  return round256((size_t)d.src_layers * 4) + round256((size_t)d.tgt_layers * d.k * 4);
}

}  // namespace

extern "C" size_t kvx_layer_scores_workspace_bytes(const kvx_plan *plan, int64_t ntok) {
  if (!plan || ntok < 2 || !plan_ok(plan->desc)) return 0;
  const kvx_plan_desc &d = plan->desc;
  return layout_of(d.src_layers, d.tgt_layers, d.src_head_dim, d.k, ntok).total + lists_bytes(d);
}

extern "C" kvx_status kvx_layer_scores(const kvx_plan *plan, const kvx_score_args *a,
                                       void *stream) {
  if (!plan || !a) return KVX_ERR_INVALID_ARG;
  const kvx_plan_desc &d = plan->desc;
  if (!plan_ok(d)) return KVX_ERR_UNSUPPORTED;
  if (!a->src_k || !a->src_v || !a->tgt_k || !a->tgt_v || !a->r2 || !a->workspace ||
      a->ntok < 2 || a->num_requests < 1 || (!a->cu_seqlens && a->num_requests != 1) ||
      !(a->lambda > 0.0) || !std::isfinite(a->lambda) || (a->r2_set && !a->layer_idx))
    return KVX_ERR_INVALID_ARG;
  const int64_t n = a->ntok;
  if (a->workspace_bytes < kvx_layer_scores_workspace_bytes(plan, n)) return KVX_ERR_INVALID_ARG;
  const int64_t slices64 = (n + kRowsPerSlice - 1) / kRowsPerSlice;
  if (slices64 > 65535 || n > INT32_MAX) return KVX_ERR_INVALID_ARG;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return KVX_ERR_CUDA;
  if (cur != plan->device) return KVX_ERR_INVALID_ARG;

  const int Ls = d.src_layers, Lt = d.tgt_layers, H = d.src_kv_heads, D = d.src_head_dim, k = d.k;
  const bool sets = a->r2_set != nullptr;
  cudaStream_t s = (cudaStream_t)stream;
  const Layout lay = layout_of(Ls, Lt, D, k, n);
  unsigned char *ws = reinterpret_cast<unsigned char *>(a->workspace);
  Pass ps;
  ps.X = reinterpret_cast<float *>(ws + lay.X);
  ps.Y = reinterpret_cast<float *>(ws + lay.Y);
  ps.xs = reinterpret_cast<double *>(ws + lay.xs);
  ps.ys = reinterpret_cast<double *>(ws + lay.ys);
  ps.yss = reinterpret_cast<double *>(ws + lay.yss);
  ps.G = reinterpret_cast<double *>(ws + lay.G);
  ps.C = reinterpret_cast<double *>(ws + lay.C);
  ps.zz = reinterpret_cast<double *>(ws + lay.zz);
  ps.ww = reinterpret_cast<double *>(ws + lay.ww);
  ps.Gs = reinterpret_cast<double *>(ws + lay.Gs);
  ps.Cs = reinterpret_cast<double *>(ws + lay.Cs);
  ps.zzs = reinterpret_cast<double *>(ws + lay.zzs);
  ps.wws = reinterpret_cast<double *>(ws + lay.wws);
  ps.bad = reinterpret_cast<int *>(ws + lay.bad);
  int32_t *ident = reinterpret_cast<int32_t *>(ws + lay.total);
  int32_t *set_list = reinterpret_cast<int32_t *>(ws + lay.total + round256((size_t)Ls * 4));

  Turns turns;
  for (int i = 0; i < D / 2; ++i) {
    turns.src[i] = plan->turns_src[i];
    turns.tgt[i] = plan->turns_tgt[i];
  }
  check_table_kernel<<<1, 256, 0, s>>>(a->cu_seqlens, a->num_requests, n, ps.bad, a->status);
  const int n_idx = sets ? Lt * k : 0;
  layer_lists_kernel<<<(Ls + n_idx + 255) / 256 + 1, 256, 0, s>>>(ident, Ls, set_list,
                                                                 a->layer_idx, n_idx);
  if (sets) check_rows_kernel<<<(Lt * k + 255) / 256, 256, 0, s>>>(a->layer_idx, Lt, k, Ls, a->status);
  if (cudaGetLastError() != cudaSuccess) return KVX_ERR_CUDA;

  const int tiles_d = (D + kTile - 1) / kTile;
  const int q1 = Lt * D;
  const int tiles_q1 = (q1 + kTile - 1) / kTile;
  const int pk = k * D, tiles_pk = (pk + kTile - 1) / kTile;
  // the per-pass fp64 region: sums, yss, G, C, zz, ww, Gs, Cs, zzs, wws
  double *clear_from = ps.xs;
  const int64_t clear_words = (int64_t)(lay.bad - lay.xs) / 8;
  const int per_tok = D / 16, tpb = 256 / per_tok;
  dim3 cgrid((unsigned)((n + tpb - 1) / tpb), (unsigned)(Ls + Lt));
  const int cols1 = solve_cols_per_cta(D), colsk = solve_cols_per_cta(pk);
  for (int h = 0; h < H; ++h) {
    for (int m = 0; m < 2; ++m) {
      clear_kernel<<<1024, 256, 0, s>>>(clear_from, clear_words);
      if (d.kv_dtype == KVX_BF16)
        content_kernel<__nv_bfloat16><<<cgrid, 256, 0, s>>>(
            reinterpret_cast<const __nv_bfloat16 *>(m ? a->src_v : a->src_k),
            reinterpret_cast<const __nv_bfloat16 *>(m ? a->tgt_v : a->tgt_k), Ls, Lt, H, D, h,
            m == 0, n, a->cu_seqlens, a->num_requests, a->src_pos, d.max_position, turns, ps,
            a->status);
      else
        content_kernel<float><<<cgrid, 256, 0, s>>>(
            reinterpret_cast<const float *>(m ? a->src_v : a->src_k),
            reinterpret_cast<const float *>(m ? a->tgt_v : a->tgt_k), Ls, Lt, H, D, h, m == 0, n,
            a->cu_seqlens, a->num_requests, a->src_pos, d.max_position, turns, ps, a->status);
      // per-layer fits: batch s, features = source layer s, targets = every
      // target layer's columns
      gram_kernel<<<dim3((unsigned)(tiles_d * (tiles_d + 1) / 2 + tiles_d * tiles_q1),
                         (unsigned)slices64, (unsigned)Ls),
                    256, 0, s>>>(ps.X, ps.Y, ps.xs, ps.ys, ident, 1, D, Lt, n, q1, 0, 0, ps.G,
                                 ps.C, tiles_d, tiles_q1);
      if (chol_factor(ps.G, Ls, D, a->lambda, a->status, s) != cudaSuccess) return KVX_ERR_CUDA;
      solve_norms_kernel<<<dim3((unsigned)Ls, (unsigned)((q1 + cols1 - 1) / cols1)), kSolveThreads,
                           solve_smem_bytes(D, cols1), s>>>(ps.G, ps.C, D, q1, D, cols1, ps.zz,
                                                            ps.ww, Lt);
      if (sets) {
        // set fits: batch lt, features = the row's k layers, targets = lt
        gram_kernel<<<dim3((unsigned)(tiles_pk * (tiles_pk + 1) / 2 + tiles_pk * tiles_d),
                           (unsigned)slices64, (unsigned)Lt),
                      256, 0, s>>>(ps.X, ps.Y, ps.xs, ps.ys, set_list, k, D, Lt, n, D, 0, D,
                                   ps.Gs, ps.Cs, tiles_pk, tiles_d);
        if (chol_factor(ps.Gs, Lt, pk, a->lambda, a->status, s) != cudaSuccess)
          return KVX_ERR_CUDA;
        solve_norms_kernel<<<dim3((unsigned)Lt, (unsigned)((D + colsk - 1) / colsk)),
                             kSolveThreads, solve_smem_bytes(pk, colsk), s>>>(
            ps.Gs, ps.Cs, pk, D, D, colsk, ps.zzs, ps.wws, 1);
      }
      finalize_kernel<<<(Ls * Lt + 255) / 256 + 1, 256, 0, s>>>(
          ps, Ls, Lt, H, D, h, m, n, a->lambda, a->r2, a->r2_set, a->layer_idx, k, a->status);
      if (cudaGetLastError() != cudaSuccess) return KVX_ERR_CUDA;
    }
  }
  return KVX_OK;
}
