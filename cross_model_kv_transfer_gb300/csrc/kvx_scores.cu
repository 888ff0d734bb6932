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
//      fp32 [Ls + Lt][n][d], with fp64 column sums;
//   2. per chunk of 16,384 tokens: the centred features split into tf32 hi
//      and lo planes (kvx_moments.cuh), then on the tensor cores (products
//      hi*hi + hi*lo + lo*hi) the centred Gram blocks G of every source layer
//      and its cross blocks C against every target layer's columns, each
//      target layer's own Gram block (its trace is sum |Yc|^2), and with a
//      layer table the Gram blocks of each row's set (its layers gathered as
//      128-row blocks) and their cross blocks against that target layer;
//      fp32 partial sums over 256 tokens, summed in fp32 per slice of 4,096,
//      added in fp64;
//   3. per-layer fits: the fp64 Cholesky of G + lam I (kvx_chol.cuh), then
//      M = (G + lam I)^-1, N = M + lam M M = R R^T (a second Cholesky), and
//      |Z|^2 + lam |W|^2 = |R^T C|^2 per target layer as one triangular
//      product per source layer;
//   4. set fits: the Cholesky of each set's Gram block, the inverses of its
//      64 x 64 diagonal blocks, and fp64 forward and back substitution by
//      64-row blocks (kvx_chol.cuh), keeping only |z|^2 and |w|^2;
//   5. the scores.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>

#include "kvx_chol.cuh"
#include "kvx_moments.cuh"
#include "kvx_internal.h"

namespace {

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
  float *X;          // [Ls + Lt][n][d] content: source layers, then target layers
  float *planes;     // [2][(Ls + Lt) d][np] tf32 hi and lo of one chunk
  double *xs;        // [Ls][d] column sums (followed by ys)
  double *ys;        // [Lt][d]
  double *G;         // [Ls][d][d]
  double *C;         // [Ls][d][Lt*d]
  double *M;         // [Ls][d][d]  (G + lam I)^-1
  double *N;         // [Ls][d][d]  M + lam M M, then its Cholesky factor R
  double *Gy;        // [Lt][d][d]  centred Gram of each target layer (its trace: SS_tot)
  double *zz, *ww;   // [Ls][Lt]
  double *Gs;        // [Lt][k*d][k*d]   (sets)
  double *Cs;        // [Lt][k*d][d]
  double *zzs, *wws; // [Lt]
  double *Dinv;      // [Lt][k d / 64][64][64] inverse diagonal blocks of the sets' factors
  int *bad;          // [1]: the transfer-wide validity (positions, request table)
};

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

struct Layout {
  size_t X, planes, xs, ys, G, C, M, N, Gy, zz, ww, Gs, Cs, zzs, wws, Dinv, bad, total;
};

// Tokens per plane chunk, padded to the tensor-core block.
int64_t chunk_np(int64_t n) {
  const int64_t len = n < kMomChunk ? n : kMomChunk;
  return (len + kMomKB - 1) / kMomKB * kMomKB;
}

Layout layout_of(int64_t Ls, int64_t Lt, int64_t d, int64_t k, int64_t n) {
  Layout L;
  size_t at = 0;
  auto take = [&](size_t bytes) { const size_t o = at; at += round256(bytes); return o; };
  L.X = take((size_t)(Ls + Lt) * n * d * 4);
  L.planes = take((size_t)2 * (Ls + Lt) * d * chunk_np(n) * 4);
  L.xs = (size_t)at;
  at += (size_t)Ls * d * 8;                       // xs and ys adjacent: [Ls + Lt][d]
  L.ys = at;
  at += round256((size_t)Lt * d * 8);
  L.G = take((size_t)Ls * d * d * 8);
  L.C = take((size_t)Ls * d * Lt * d * 8);
  L.M = take((size_t)Ls * d * d * 8);
  L.N = take((size_t)Ls * d * d * 8);
  L.Gy = take((size_t)Lt * d * d * 8);
  L.zz = take((size_t)Ls * Lt * 8);
  L.ww = take((size_t)Ls * Lt * 8);
  L.Gs = take((size_t)Lt * k * d * k * d * 8);
  L.Cs = take((size_t)Lt * k * d * d * 8);
  L.zzs = take((size_t)Lt * 8);
  L.wws = take((size_t)Lt * 8);
  L.Dinv = take((size_t)Lt * ((k * d + 63) / 64) * 64 * 64 * 8);
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
  const int L = blockIdx.y;
  const bool is_src = L < Ls;
  const int layer = is_src ? L : L - Ls;
  const int per_tok = d / 16;                      // threads per token
  const int tpb = 256 / per_tok;                   // tokens per block
  const int tid = threadIdx.x;
  for (int i = tid; i < d; i += blockDim.x) ssum[i] = 0.f;
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
    float *out = ps.X + ((int64_t)L * n + g) * d;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      out[8 * q + e] = lo[e];
      out[half + 8 * q + e] = hi[e];
      atomicAdd(&ssum[8 * q + e], lo[e]);
      atomicAdd(&ssum[half + 8 * q + e], hi[e]);
    }
  }
  __syncthreads();
  double *sums = is_src ? ps.xs + (int64_t)layer * d : ps.ys + (int64_t)layer * d;
  for (int i = tid; i < d; i += blockDim.x) atomicAdd(sums + i, (double)ssum[i]);
}

// 2. Per chunk [n0, n0 + np): the centred content of plane row f (= layer
// f / d, dimension f % d, source layers first) as tf32 hi and lo planes,
// column t - n0 (tokens beyond n are zero); a CTA transposes 32 rows x 128
// tokens through shared memory (16 loads per thread in flight).
constexpr int kSplitObs = 128;
__global__ void __launch_bounds__(256) split_kernel(const float *__restrict__ X,
                                                    const double *__restrict__ sums, int64_t n,
                                                    int rows, int d, int64_t n0, int64_t np,
                                                    float *__restrict__ planes) {
  __shared__ float blk[kSplitObs][33];
  const int f0 = blockIdx.y * 32;
  const int64_t c0 = (int64_t)blockIdx.x * kSplitObs;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int f = f0 + tx;
  float mean = 0.f;
  if (f < rows) mean = (float)(sums[f] / (double)n);
  const float *col = X + (int64_t)(f / d) * n * d + f % d;
  float v[kSplitObs / 8];
#pragma unroll
  for (int i = 0; i < kSplitObs / 8; ++i) {
    const int64_t t = n0 + c0 + ty + 8 * i;
    v[i] = f < rows && t < n ? col[t * d] - mean : 0.f;
  }
#pragma unroll
  for (int i = 0; i < kSplitObs / 8; ++i) blk[ty + 8 * i][tx] = v[i];
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int fr = f0 + ty + 8 * i;
    if (fr >= rows) continue;
#pragma unroll
    for (int j = 0; j < kSplitObs / 32; ++j) {
      const int64_t c = c0 + tx + 32 * j;
      if (c < np) mom_put(planes, rows, np, fr, c, blk[tx + 32 * j][ty + 8 * i]);
    }
  }
}

// The tensor-core tiles of one pass.  Per source layer s: its Gram block
// (A = B = layer s) and ceil(Lt d / 128) cross tiles against the target
// columns.  Per target layer: its own Gram block (the trace is the centred
// total sum of squares).  Per target layer lt (with a table): the Gram blocks (j1 <= j2)
// of its set, A = layer sets[lt][j1], B = layer sets[lt][j2], and its k cross
// blocks against layer lt's d columns.  Plane row of layer L, dim i: L d + i
// (target layer lt is L = Ls + lt).  With d < 128 a block's extra rows are
// other layers' and are not stored.
struct ScoreTiles {
  int Ls, Lt, d, k, nq, layer_tiles;
  const int32_t *sets;
  double *G, *C, *Gy, *Gs, *Cs;
  __device__ MomTile tile(int t) const {
    MomTile m;
    m.m_valid = d;
    if (t >= layer_tiles && t < layer_tiles + Lt) {   // a target layer's own Gram block
      const int lt = t - layer_tiles;
      m.a_row = m.b_row = (Ls + lt) * d;
      m.n_split = m.n_valid = d;
      m.out0 = m.out1 = Gy + (int64_t)lt * d * d;
      m.ld0 = m.ld1 = d;
      return m;
    }
    if (t >= layer_tiles) t -= Lt;
    if (t < layer_tiles) {
      const int s = t / (1 + nq), j = t % (1 + nq);
      m.a_row = s * d;
      if (j == 0) {
        m.b_row = s * d;
        m.n_split = m.n_valid = d;
        m.out0 = m.out1 = G + (int64_t)s * d * d;
        m.ld0 = m.ld1 = d;
      } else {
        const int c0 = (j - 1) * kMomRows;
        m.b_row = Ls * d + c0;
        m.n_split = 0;
        m.n_valid = min(kMomRows, Lt * d - c0);
        m.out0 = m.out1 = C + (int64_t)s * d * Lt * d + c0;
        m.ld0 = m.ld1 = (int64_t)Lt * d;
      }
      return m;
    }
    const int pairs = k * (k + 1) / 2, per = pairs + k, p = k * d;
    int r = t - layer_tiles;
    const int lt = r / per;
    r -= lt * per;
    if (r < pairs) {
      int j1 = 0;
      while (r >= k - j1) {
        r -= k - j1;
        ++j1;
      }
      const int j2 = j1 + r;
      m.a_row = sets[lt * k + j1] * d;
      m.b_row = sets[lt * k + j2] * d;
      m.n_split = m.n_valid = d;
      m.out0 = m.out1 = Gs + (int64_t)lt * p * p + (int64_t)j1 * d * p + j2 * d;
      m.ld0 = m.ld1 = p;
    } else {
      const int j = r - pairs;
      m.a_row = sets[lt * k + j] * d;
      m.b_row = (Ls + lt) * d;
      m.n_split = 0;
      m.n_valid = d;
      m.out0 = m.out1 = Cs + (int64_t)lt * p * d + (int64_t)j * d * d;
      m.ld0 = m.ld1 = d;
    }
    return m;
  }
};

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

// 4'. The per-layer fits without per-column solves.  With G_lam = G + lam I,
// M = G_lam^-1 and W = M C, the explained sum of squares of a target block
// C is |L^-1 C|^2 + lam |W|^2 = tr(C^T (M + lam M M) C) = |R^T C|^2 for
// N = M + lam M M = R R^T.  Per source layer: M from the factor of G_lam
// (column solves against the identity), N, the Cholesky factor R of N, and
// then one triangular product R^T C over all Lt d target columns: half the
// multiply-adds of the forward and back solves, and no chain of dependent
// steps per column.

// a. Per (source layer s, nc columns): columns of M = G_lam^-1.
__global__ void __launch_bounds__(kSolveThreads) inverse_kernel(const double *__restrict__ G,
                                                                int d, int nc,
                                                                double *__restrict__ Minv) {
  extern __shared__ double cols[];   // [d][nc], then d reciprocals
  const int s = blockIdx.x, c0 = blockIdx.y * nc;
  const double *A = G + (int64_t)s * d * d;
  double *M = Minv + (int64_t)s * d * d;
  if (isnan(A[0])) {
    if (blockIdx.y == 0 && threadIdx.x == 0) M[0] = nan("");
    return;
  }
  for (int e = threadIdx.x; e < d * nc; e += kSolveThreads)
    cols[e] = e / nc == c0 + e % nc ? 1.0 : 0.0;
  double zn, wn;
  chol_solve_cols(A, d, cols, cols + (size_t)d * nc, nc, zn, wn);
  for (int e = threadIdx.x; e < d * nc; e += kSolveThreads)
    if (c0 + e % nc < d) M[(int64_t)(e / nc) * d + c0 + e % nc] = cols[e];
}

// b. N = M + lam M M per source layer, the full symmetric matrix, 64 x 64
// output tiles (4 x 4 per thread, 16 rows of K per step).
__global__ void __launch_bounds__(256) bridge_n_kernel(const double *__restrict__ Minv, int d,
                                                       double lam, double *__restrict__ N) {
  __shared__ double sa[16][65], sb[16][65];
  const int s = blockIdx.z, i0 = blockIdx.y * 64, j0 = blockIdx.x * 64;
  const double *M = Minv + (int64_t)s * d * d;
  double *O = N + (int64_t)s * d * d;
  if (isnan(M[0])) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) O[0] = nan("");
    return;
  }
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  double acc[4][4] = {};
  for (int k0 = 0; k0 < d; k0 += 16) {
    for (int e = tid; e < 16 * 64; e += 256) {
      const int kk = e / 64, ii = e % 64;
      sa[kk][ii] = i0 + ii < d ? M[(int64_t)(i0 + ii) * d + k0 + kk] : 0.0;   // M symmetric
      sb[kk][ii] = j0 + ii < d ? M[(int64_t)(k0 + kk) * d + j0 + ii] : 0.0;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      double a[4], b[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) a[r] = sa[kk][4 * ty + r], b[r] = sb[kk][4 * tx + r];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = fma(a[r], b[c], acc[r][c]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = i0 + 4 * ty + r, j = j0 + 4 * tx + c;
      if (i < d && j < d) O[(int64_t)i * d + j] = fma(lam, acc[r][c], M[(int64_t)i * d + j]);
    }
}

// c. Per (source layer s, 64 target columns), after the factorisation of N:
// Q = R^T C for the columns (row i of R^T = row i of the factor's upper
// triangle, k >= i), and |Q|^2 of each column added into zz[s][column / d].
// Warp w owns rows 16 w .. 16 w + 15 (a lane: 4 rows x 8 columns) and skips
// the blocks of K below its rows.
__global__ void __launch_bounds__(256) bridge_norms_kernel(const double *__restrict__ Nf,
                                                           const double *__restrict__ C, int d,
                                                           int q, int Lt,
                                                           double *__restrict__ zz) {
  __shared__ double sr[kMaxD][17];
  __shared__ double sc[16][64];
  __shared__ double red[8][64];
  const int s = blockIdx.y, c0 = blockIdx.x * 64;
  const double *A = Nf + (int64_t)s * d * d;
  if (isnan(A[0])) return;
  const double *Cs = C + (int64_t)s * d * q;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rq = lane >> 3, cg = lane & 7;
  const int i0 = warp * 16 + rq * 4;           // rows i0 .. i0 + 3 (d is a multiple of 16)
  const bool rows_ok = warp * 16 < d;
  double acc[4][8] = {};
  for (int k0 = 0; k0 < d; k0 += 16) {
    for (int e = tid; e < d * 16; e += 256) {
      const int i = e >> 4, k = k0 + (e & 15);
      sr[i][e & 15] = k >= i ? A[(int64_t)i * d + k] : 0.0;
    }
    for (int e = tid; e < 16 * 64; e += 256) {
      const int kk = e >> 6, j = e & 63;
      sc[kk][j] = c0 + j < q ? Cs[(int64_t)(k0 + kk) * q + c0 + j] : 0.0;
    }
    __syncthreads();
    if (rows_ok && k0 + 15 >= warp * 16) {
#pragma unroll 4
      for (int kk = 0; kk < 16; ++kk) {
        double r[4], cv[8];
#pragma unroll
        for (int a = 0; a < 4; ++a) r[a] = sr[i0 + a][kk];
#pragma unroll
        for (int c = 0; c < 8; ++c) cv[c] = sc[kk][8 * cg + c];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int c = 0; c < 8; ++c) acc[a][c] = fma(r[a], cv[c], acc[a][c]);
      }
    }
    __syncthreads();
  }
  double part[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    double v = 0.0;
#pragma unroll
    for (int a = 0; a < 4; ++a) v = fma(acc[a][c], acc[a][c], v);
    v += __shfl_xor_sync(0xffffffffu, v, 8);
    v += __shfl_xor_sync(0xffffffffu, v, 16);
    part[c] = rows_ok ? v : 0.0;
  }
  if (rq == 0) {
#pragma unroll
    for (int c = 0; c < 8; ++c) red[warp][8 * cg + c] = part[c];
  }
  __syncthreads();
  if (tid < 64 && c0 + tid < q) {
    double t = 0.0;
#pragma unroll
    for (int w = 0; w < 8; ++w) t += red[w][tid];
    atomicAdd(zz + (int64_t)s * Lt + (c0 + tid) / d, t);
  }
}

// Epilogue of the blocked set solves: |z|^2 and |w|^2 of each column.
struct NormsEpi {
  double *zz, *ww;
  int q;
  __device__ void operator()(int b, int c0, const double *, double zn, double wn) const {
    if (threadIdx.x < kBlkCols && c0 + (int)threadIdx.x < q) {
      atomicAdd(zz + b, zn);
      atomicAdd(ww + b, wn);
    }
  }
  __device__ void failed(int, int) const {}
};

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
      double tot = 0.0;
      for (int i = 0; i < d; ++i) tot += ps.Gy[((int64_t)e * d + i) * d + i];
      const bool spd = !isnan(ps.Gs[(int64_t)e * k * d * k * d]);
      double v = nan("");
      if (ok && spd && tot > 0.0) v = (ps.zzs[e] + lam * ps.wws[e]) / tot;
      r2_set[((int64_t)e * H + h) * 2 + m] = v;
    }
  }
  if (e < Ls * Lt) {
    const int s = e / Lt, lt = e % Lt;
    double tot = 0.0;
    for (int i = 0; i < d; ++i) tot += ps.Gy[((int64_t)lt * d + i) * d + i];
    const bool spd = !isnan(ps.G[(int64_t)s * d * d]) && !isnan(ps.N[(int64_t)s * d * d]);
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

// The layer table with entries outside [0, Ls) clamped (their rows are
// flagged and get NaN scores); the tiles read layers through it.
__global__ void layer_lists_kernel(int32_t *sets, const int32_t *idx, int n_idx, int Ls) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
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

size_t lists_bytes(const kvx_plan_desc &d) { return round256((size_t)d.tgt_layers * d.k * 4); }

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
  if (n > INT32_MAX || (reinterpret_cast<uintptr_t>(a->workspace) & 15u) != 0)
    return KVX_ERR_INVALID_ARG;
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
  ps.planes = reinterpret_cast<float *>(ws + lay.planes);
  ps.xs = reinterpret_cast<double *>(ws + lay.xs);
  ps.ys = reinterpret_cast<double *>(ws + lay.ys);
  ps.G = reinterpret_cast<double *>(ws + lay.G);
  ps.C = reinterpret_cast<double *>(ws + lay.C);
  ps.M = reinterpret_cast<double *>(ws + lay.M);
  ps.N = reinterpret_cast<double *>(ws + lay.N);
  ps.Gy = reinterpret_cast<double *>(ws + lay.Gy);
  ps.zz = reinterpret_cast<double *>(ws + lay.zz);
  ps.ww = reinterpret_cast<double *>(ws + lay.ww);
  ps.Gs = reinterpret_cast<double *>(ws + lay.Gs);
  ps.Cs = reinterpret_cast<double *>(ws + lay.Cs);
  ps.zzs = reinterpret_cast<double *>(ws + lay.zzs);
  ps.wws = reinterpret_cast<double *>(ws + lay.wws);
  ps.Dinv = reinterpret_cast<double *>(ws + lay.Dinv);
  ps.bad = reinterpret_cast<int *>(ws + lay.bad);
  int32_t *set_list = reinterpret_cast<int32_t *>(ws + lay.total);

  Turns turns;
  for (int i = 0; i < D / 2; ++i) {
    turns.src[i] = plan->turns_src[i];
    turns.tgt[i] = plan->turns_tgt[i];
  }
  check_table_kernel<<<1, 256, 0, s>>>(a->cu_seqlens, a->num_requests, n, ps.bad, a->status);
  const int n_idx = sets ? Lt * k : 0;
  if (sets)
    layer_lists_kernel<<<(n_idx + 255) / 256, 256, 0, s>>>(set_list, a->layer_idx, n_idx, Ls);
  if (sets) check_rows_kernel<<<(Lt * k + 255) / 256, 256, 0, s>>>(a->layer_idx, Lt, k, Ls, a->status);
  if (cudaGetLastError() != cudaSuccess) return KVX_ERR_CUDA;

  const int q1 = Lt * D;
  const int pk = k * D;
  const int rows = (Ls + Lt) * D;
  const int nq = (q1 + kMomRows - 1) / kMomRows;
  const ScoreTiles tiles{Ls, Lt, D, k, nq, Ls * (1 + nq), set_list, ps.G, ps.C, ps.Gy, ps.Gs,
                         ps.Cs};
  const int num_tiles = tiles.layer_tiles + Lt + (sets ? Lt * (k * (k + 1) / 2 + k) : 0);
  // the per-pass fp64 region: sums, G, C, M, N, Gy, zz, ww, Gs, Cs, zzs, wws
  double *clear_from = ps.xs;
  const int64_t clear_words = (int64_t)(lay.bad - lay.xs) / 8;
  const int per_tok = D / 16, tpb = 256 / per_tok;
  dim3 cgrid((unsigned)((n + tpb - 1) / tpb), (unsigned)(Ls + Lt));
  const int cols1 = solve_cols_per_cta(D, Ls, D), colsk = solve_cols_per_cta(pk, Lt, D);
  if (sets && pk <= kBlkMaxP &&
      cudaFuncSetAttribute(chol_solve_blocked_kernel<NormsEpi>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)blk_solve_smem_bytes(pk)) != cudaSuccess)
    return KVX_ERR_CUDA;
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
      // Gram and cross blocks of the per-layer and set fits, chunk by chunk
      for (int64_t n0 = 0; n0 < n; n0 += kMomChunk) {
        const int64_t len = n - n0 < kMomChunk ? n - n0 : kMomChunk;
        const int64_t np = (len + kMomKB - 1) / kMomKB * kMomKB;
        split_kernel<<<dim3((unsigned)((np + kSplitObs - 1) / kSplitObs),
                            (unsigned)((rows + 31) / 32)),
                       256, 0, s>>>(
            ps.X, ps.xs, n, rows, D, n0, np, ps.planes);
        if (cudaGetLastError() != cudaSuccess) return KVX_ERR_CUDA;
        if (mom_launch(ps.planes, rows, np, tiles, num_tiles, a->status, s) != cudaSuccess)
          return KVX_ERR_CUDA;
      }
      // per-layer fits: |R^T C|^2 with R R^T = M + lam M M, M = (G + lam I)^-1
      if (chol_factor(ps.G, Ls, D, a->lambda, a->status, s) != cudaSuccess) return KVX_ERR_CUDA;
      inverse_kernel<<<dim3((unsigned)Ls, (unsigned)((D + cols1 - 1) / cols1)), kSolveThreads,
                       solve_smem_bytes(D, cols1), s>>>(ps.G, D, cols1, ps.M);
      bridge_n_kernel<<<dim3((unsigned)((D + 63) / 64), (unsigned)((D + 63) / 64), (unsigned)Ls),
                        256, 0, s>>>(ps.M, D, a->lambda, ps.N);
      if (chol_factor(ps.N, Ls, D, 0.0, a->status, s) != cudaSuccess) return KVX_ERR_CUDA;
      bridge_norms_kernel<<<dim3((unsigned)((q1 + 63) / 64), (unsigned)Ls), 256, 0, s>>>(
          ps.N, ps.C, D, q1, Lt, ps.zz);
      if (sets) {
        if (chol_factor(ps.Gs, Lt, pk, a->lambda, a->status, s) != cudaSuccess)
          return KVX_ERR_CUDA;
        if (pk <= kBlkMaxP) {
          chol_block_inverse_kernel<<<dim3((unsigned)Lt, (unsigned)((pk + 63) / 64)), 64, 0, s>>>(
              ps.Gs, pk, ps.Dinv);
          chol_solve_blocked_kernel<NormsEpi>
              <<<dim3((unsigned)Lt, (unsigned)((D + kBlkCols - 1) / kBlkCols)), kBlkThreads,
                 blk_solve_smem_bytes(pk), s>>>(ps.Gs, ps.Dinv, ps.Cs, pk, D,
                                                NormsEpi{ps.zzs, ps.wws, D});
        } else {
          solve_norms_kernel<<<dim3((unsigned)Lt, (unsigned)((D + colsk - 1) / colsk)),
                               kSolveThreads, solve_smem_bytes(pk, colsk), s>>>(
              ps.Gs, ps.Cs, pk, D, D, colsk, ps.zzs, ps.wws, 1);
        }
      }
      finalize_kernel<<<(Ls * Lt + 255) / 256 + 1, 256, 0, s>>>(
          ps, Ls, Lt, H, D, h, m, n, a->lambda, a->r2, a->r2_set, a->layer_idx, k, a->status);
      if (cudaGetLastError() != cudaSuccess) return KVX_ERR_CUDA;
    }
  }
  return KVX_OK;
}
