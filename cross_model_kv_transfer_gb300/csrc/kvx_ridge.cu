// kvx_ridge.cu -- the ridge fit of the maps (kvx_ridge_fit), on the GPU.
//
// The Qwen3 14B -> 32B article, section "Линейного моста, как ни странно,
// хватает", fits one ridge regression per target (layer, head), one for
// keys and one for values, on paired source / target cache observations; its
// ridge demo centres X and Y on their column means, solves
// (XcT Xc + lam I) W = XcT Yc and sets b = ybar - xbar W.  For a batch of
// independent fits (X [n][p], Y [n][q] each) this runs as
// 4 + 2 ceil(n / 16384) + 3 ceil(p / 64) - 1 launches:
//   1. clear the fp64 workspace;
//   2. a shift per column of X and Y: the mean of 256 of its observations
//      spread evenly over all of them, rounded to fp32 (one short pass
//      instead of a pass over all observations for the exact means);
//   3. per chunk of 16,384 observations: the shifted values v = [X | Y] -
//      shift split into tf32 hi and lo planes, transposed so that each
//      feature's observations are contiguous, with the column sums of v
//      (fp32 per thread, fp64 atomics per CTA); then the Gram blocks
//      V_xT V_x (upper triangle of 128 x 128 tiles) and V_xT V_y on the
//      tensor cores as hi*hi + hi*lo + lo*hi (kvx_moments.cuh), fp32 partial
//      sums over 256 observations in tensor memory, summed in fp32 over
//      slices of 4,096 and added in fp64;
//   4. the centring as an exact rank-one correction, G = V_xT V_x - s_x s_xT / n
//      and C = V_xT V_y - s_x s_yT / n with s the column sums of v (the
//      shifted-data form of the centred moments: the shift leaves each column
//      within a fraction of its spread of its mean, so the correction is small
//      against G and cancels nothing), and the column sums n shift + s;
//   5. G + lam I mirrored to full, then a Cholesky factorisation in fp64
//      blocked by 64 (per diagonal block: factor it, solve the panel below,
//      update the trailing blocks, each step spread over CTAs);
//   6. per (fit, nc output columns), one CTA: forward and back
//      substitution in fp64 (the columns in shared memory, the threads
//      split over the columns and the rows of each right-looking update),
//      b = ybar - xbar W; W and b stored as fp32.  A non-positive
//      pivot leaves W and b NaN and sets KVX_FLAG_NOT_SPD.
// A single tf32 or bf16 operand would keep 11 or 8 significant bits of the
// centred features, and the solve amplifies Gram errors by the condition
// number of G + lam I; the two-term split keeps about 22.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>

#include "../../include/kvx.h"
#include "kvx_chol.cuh"
#include "kvx_moments.cuh"

namespace {

constexpr int64_t kShiftRows = 256;  // observations behind each column's shift
constexpr int kSplitObs = 128;       // observations per CTA of the split pass

template <typename T>
__device__ __forceinline__ float ldv(const T *p);
template <>
__device__ __forceinline__ float ldv<float>(const float *p) { return __ldg(p); }
template <>
__device__ __forceinline__ float ldv<__nv_bfloat16>(const __nv_bfloat16 *p) {
  return __bfloat162float(*p);
}

__global__ void clear_kernel(double *x, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    x[i] = 0.0;
}

// shift[b][c] = the mean of min(n, kShiftRows) observations of column c of
// [X | Y] spread evenly over all n (rows k n / m), rounded to fp32 (the split
// subtracts it in fp32); a sample spread over the whole set keeps the shift
// near the mean even when the observations drift in order.  A CTA covers 32
// columns (one per lane, so a warp's loads are consecutive columns of a row)
// and 8 groups of the sample, summed in fp64 and combined in shared memory.
template <typename T>
__global__ void __launch_bounds__(256) shift_kernel(const T *__restrict__ x, const T *__restrict__ y,
                                                    double *__restrict__ shift, int64_t n, int p,
                                                    int q) {
  __shared__ double red[8][32];
  const int b = blockIdx.y, pq = p + q;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int c = blockIdx.x * 32 + tx;
  const int64_t m = n < kShiftRows ? n : kShiftRows;
  double acc = 0.0;
  if (c < pq) {
    const T *col = c < p ? x + (int64_t)b * n * p + c : y + (int64_t)b * n * q + (c - p);
    const int64_t ld = c < p ? p : q;
#pragma unroll 4
    for (int64_t k = ty; k < m; k += 8) acc += (double)ldv<T>(col + (k * n / m) * ld);
  }
  red[ty][tx] = acc;
  __syncthreads();
  if (ty == 0 && c < pq) {
    double t = 0.0;
#pragma unroll
    for (int g = 0; g < 8; ++g) t += red[g][tx];
    shift[(int64_t)b * pq + c] = (double)(float)(t / (double)m);
  }
}

// Per chunk [n0, n0 + np): the shifted values v of [X | Y] of fit b as tf32
// hi and lo planes, plane row b (p + q) + f, column t - n0 (observations
// beyond n are zero), and sums[b][f] += the column sums of v.  A CTA
// transposes 32 features x 128 observations through shared memory: loads run
// along the features (16 per thread in flight), stores along the
// observations; the sums go fp32 per thread, fp64 across the CTA, one atomic
// per feature.
template <typename T>
__global__ void __launch_bounds__(256) split_kernel(const T *__restrict__ x, const T *__restrict__ y,
                                                    const double *__restrict__ shift,
                                                    double *__restrict__ sums, int64_t n, int p,
                                                    int q, int64_t n0, int64_t np, int64_t R,
                                                    float *__restrict__ planes) {
  __shared__ float blk[kSplitObs][33];
  __shared__ double part[8][32];
  const int b = blockIdx.z, pq = p + q;
  const int f0 = blockIdx.y * 32;
  const int64_t c0 = (int64_t)blockIdx.x * kSplitObs;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int f = f0 + tx;
  const float sh = f < pq ? (float)shift[(int64_t)b * pq + f] : 0.f;
  const T *base = f < p ? x + (int64_t)b * n * p + f : y + (int64_t)b * n * q + (f - p);
  const int64_t ld = f < p ? p : q;
  float v[kSplitObs / 8];
#pragma unroll
  for (int i = 0; i < kSplitObs / 8; ++i) {
    const int64_t t = n0 + c0 + ty + 8 * i;
    v[i] = f < pq && t < n ? ldv<T>(base + t * ld) - sh : 0.f;
  }
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < kSplitObs / 8; ++i) {
    blk[ty + 8 * i][tx] = v[i];
    acc += v[i];
  }
  part[ty][tx] = (double)acc;
  __syncthreads();
  if (ty == 0 && f < pq) {
    double t = 0.0;
#pragma unroll
    for (int g = 0; g < 8; ++g) t += part[g][tx];
    atomicAdd(sums + (int64_t)b * pq + f, t);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int fr = f0 + ty + 8 * i;
    if (fr >= pq) continue;
#pragma unroll
    for (int j = 0; j < kSplitObs / 32; ++j) {
      const int64_t col = c0 + tx + 32 * j;
      if (col < np) mom_put(planes, R, np, (int64_t)b * pq + fr, col, blk[tx + 32 * j][ty + 8 * i]);
    }
  }
}

// The centring, as a rank-one correction of the shifted moments: for fit b,
// row i (CTA blockIdx.x) of G (its upper triangle, the part the
// factorisation reads) and of C, subtract s_i s_j / n, s = sums (the column
// sums of the shifted values); thread 0 also turns columns i, i + p, ... of
// the shift into column sums of [X | Y], n shift + s, in `shift`.
__global__ void __launch_bounds__(256) centre_kernel(double *__restrict__ G, double *__restrict__ C,
                                                     const double *__restrict__ sums,
                                                     double *__restrict__ shift, int64_t n, int p,
                                                     int q) {
  const int b = blockIdx.y, i = blockIdx.x, pq = p + q;
  const double *sb = sums + (int64_t)b * pq;
  const double si = sb[i] / (double)n;
  double *g = G + ((int64_t)b * p + i) * p;
  for (int j = i + threadIdx.x; j < p; j += blockDim.x) g[j] = fma(-si, sb[j], g[j]);
  double *c = C + ((int64_t)b * p + i) * q;
  for (int j = threadIdx.x; j < q; j += blockDim.x) c[j] = fma(-si, sb[p + j], c[j]);
  if (threadIdx.x == 0)
    for (int k = i; k < pq; k += p) {
      double *sh = shift + (int64_t)b * pq + k;
      *sh = fma((double)n, *sh, sb[k]);
    }
}

// Tiles of one chunk: fit b, row block mi of G, column block nj >= mi of
// [G | C] (128 x 128 each, the upper triangle of G and all of C).
struct RidgeTiles {
  int p, q, nb, per_fit;
  double *G, *C;
  __device__ MomTile tile(int t) const {
    const int b = t / per_fit;
    int r = t - b * per_fit, mi = 0;
    while (r >= nb - mi) {
      r -= nb - mi;
      ++mi;
    }
    const int nj = mi + r;
    const int base = b * (p + q), col0 = nj * kMomRows, row0 = mi * kMomRows;
    MomTile m;
    m.a_row = base + row0;
    m.b_row = base + col0;
    m.m_valid = min(kMomRows, p - row0);
    m.n_split = max(0, min(kMomRows, p - col0));
    m.n_valid = min(kMomRows, p + q - col0);
    m.out0 = G + (int64_t)b * p * p + (int64_t)row0 * p + (col0 < p ? col0 : 0);
    m.ld0 = p;
    m.out1 = C + (int64_t)b * p * q + (int64_t)row0 * q + (col0 > p ? col0 - p : 0);
    m.ld1 = q;
    return m;
  }
};

// Per (fit, nc output columns): forward L Z = C and back L^T W = Z in fp64
// (chol_solve_cols: the columns in shared memory, right-looking updates with
// the threads split over columns and rows), then b = ybar - xbar W.  W and b
// are stored as fp32 (NaN for a failed fit).
__global__ void __launch_bounds__(kSolveThreads) trsm_kernel(
    const double *__restrict__ G, const double *__restrict__ C, const double *__restrict__ sums,
    int64_t n, int p, int q, int nc, float *__restrict__ W, float *__restrict__ bias) {
  extern __shared__ double cols[];   // [p][nc], then p reciprocals
  const int b = blockIdx.x;
  const double *A = G + (int64_t)b * p * p;
  const double *Z = C + (int64_t)b * p * q;
  const double *mx = sums + (int64_t)b * (p + q);
  const double inv_n = 1.0 / (double)n;
  const int t = threadIdx.x, c0 = blockIdx.y * nc;
  if (isnan(A[0])) {
    for (int e = t; e < p * nc; e += kSolveThreads)
      if (c0 + e % nc < q) W[((int64_t)b * p + e / nc) * q + c0 + e % nc] = nanf("");
    if (t < nc && c0 + t < q) bias[(int64_t)b * q + c0 + t] = nanf("");
    return;
  }
  for (int e = t; e < p * nc; e += kSolveThreads) {
    const int i = e / nc, j = e % nc;
    cols[e] = c0 + j < q ? Z[(int64_t)i * q + c0 + j] : 0.0;
  }
  double zn, wn;
  chol_solve_cols(A, p, cols, cols + (size_t)p * nc, nc, zn, wn);
  for (int e = t; e < p * nc; e += kSolveThreads)
    if (c0 + e % nc < q) W[((int64_t)b * p + e / nc) * q + c0 + e % nc] = (float)cols[e];
  if (t < nc && c0 + t < q) {
    double s = 0.0;
    for (int i = 0; i < p; ++i) s = fma(mx[i] * inv_n, cols[i * nc + t], s);
    bias[(int64_t)b * q + c0 + t] = (float)(mx[p + c0 + t] * inv_n - s);
  }
}

// Epilogue of the blocked solves: W (fp32) and b = ybar - xbar W of the
// CTA's columns.
struct RidgeEpi {
  const double *sums;
  int64_t n;
  int p, q;
  float *W, *bias;
  __device__ void operator()(int b, int c0, const double *col, double, double) const {
    for (int e = threadIdx.x; e < p * kBlkCols; e += blockDim.x) {
      const int i = e / kBlkCols, c = e % kBlkCols;
      if (c0 + c < q) W[((int64_t)b * p + i) * q + c0 + c] = (float)col[e];
    }
    if (threadIdx.x < kBlkCols && c0 + (int)threadIdx.x < q) {
      const double *mx = sums + (int64_t)b * (p + q);
      const double inv_n = 1.0 / (double)n;
      double s = 0.0;
      for (int i = 0; i < p; ++i) s = fma(mx[i] * inv_n, col[i * kBlkCols + threadIdx.x], s);
      bias[(int64_t)b * q + c0 + threadIdx.x] = (float)(mx[p + c0 + threadIdx.x] * inv_n - s);
    }
  }
  __device__ void failed(int b, int c0) const {
    for (int e = threadIdx.x; e < p * kBlkCols; e += blockDim.x) {
      const int i = e / kBlkCols, c = e % kBlkCols;
      if (c0 + c < q) W[((int64_t)b * p + i) * q + c0 + c] = nanf("");
    }
    if (threadIdx.x < kBlkCols && c0 + (int)threadIdx.x < q)
      bias[(int64_t)b * q + c0 + threadIdx.x] = nanf("");
  }
};

constexpr int kMaxDim = 4096;

size_t ws_sums(int batch, int p, int q) { return (size_t)batch * (p + q) * sizeof(double); }
size_t ws_gram(int batch, int p) { return (size_t)batch * p * p * sizeof(double); }
size_t ws_cross(int batch, int p, int q) { return (size_t)batch * p * q * sizeof(double); }
size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }
size_t ws_dinv(int batch, int p) { return (size_t)batch * ((p + 63) / 64) * 64 * 64 * 8; }
size_t ws_planes(int batch, int p, int q) {
  return (size_t)2 * batch * (p + q) * kMomChunk * sizeof(float);
}

}  // namespace

extern "C" size_t kvx_ridge_workspace_bytes(int32_t batch, int32_t p, int32_t q) {
  if (batch < 1 || p < 1 || q < 1 || p > kMaxDim || q > kMaxDim) return 0;
  return round256(ws_sums(batch, p, q)) + round256(ws_gram(batch, p)) +
         round256(ws_cross(batch, p, q)) + round256(ws_planes(batch, p, q)) +
         round256(ws_dinv(batch, p)) + ws_sums(batch, p, q);
}

extern "C" kvx_status kvx_ridge_fit(const kvx_ridge_args *a, void *stream) {
  if (!a) return KVX_ERR_INVALID_ARG;
  if (a->batch < 1 || a->batch > 65535 || a->n < 1 || a->p < 1 || a->q < 1 ||
      a->p > kMaxDim || a->q > kMaxDim || !std::isfinite(a->lambda) || !a->x || !a->y ||
      !a->w || !a->b || !a->workspace ||
      (a->x_dtype != KVX_F32 && a->x_dtype != KVX_BF16))
    return KVX_ERR_INVALID_ARG;
  if (a->workspace_bytes < kvx_ridge_workspace_bytes(a->batch, a->p, a->q) ||
      (reinterpret_cast<uintptr_t>(a->workspace) & 15u) != 0)
    return KVX_ERR_INVALID_ARG;
  const int64_t n = a->n;
  if (n > 65535LL * 16384) return KVX_ERR_INVALID_ARG;   // the documented limit
  cudaStream_t s = (cudaStream_t)stream;
  const int batch = a->batch, p = a->p, q = a->q;
  unsigned char *ws = reinterpret_cast<unsigned char *>(a->workspace);
  double *sums = reinterpret_cast<double *>(ws);
  double *G = reinterpret_cast<double *>(ws + round256(ws_sums(batch, p, q)));
  double *C = reinterpret_cast<double *>(ws + round256(ws_sums(batch, p, q)) +
                                         round256(ws_gram(batch, p)));
  float *planes = reinterpret_cast<float *>(ws + round256(ws_sums(batch, p, q)) +
                                            round256(ws_gram(batch, p)) +
                                            round256(ws_cross(batch, p, q)));
  double *dinv = reinterpret_cast<double *>(reinterpret_cast<unsigned char *>(planes) +
                                            round256(ws_planes(batch, p, q)));
  double *shift = reinterpret_cast<double *>(reinterpret_cast<unsigned char *>(dinv) +
                                             round256(ws_dinv(batch, p)));
  const int64_t words = (int64_t)(round256(ws_sums(batch, p, q)) + round256(ws_gram(batch, p)) +
                                  ws_cross(batch, p, q)) / 8;
  clear_kernel<<<1024, 256, 0, s>>>(sums, words);
  if (cudaGetLastError() != cudaSuccess) return KVX_ERR_CUDA;

  dim3 hgrid((unsigned)((p + q + 31) / 32), (unsigned)batch);
  if (a->x_dtype == KVX_F32)
    shift_kernel<float><<<hgrid, 256, 0, s>>>(reinterpret_cast<const float *>(a->x),
                                              reinterpret_cast<const float *>(a->y), shift, n, p,
                                              q);
  else
    shift_kernel<__nv_bfloat16><<<hgrid, 256, 0, s>>>(
        reinterpret_cast<const __nv_bfloat16 *>(a->x),
        reinterpret_cast<const __nv_bfloat16 *>(a->y), shift, n, p, q);
  if (cudaGetLastError() != cudaSuccess) return KVX_ERR_CUDA;
  // centred moments on the tensor cores, one chunk of observations at a time
  const int64_t R = (int64_t)batch * (p + q);
  const int nb = (p + q + kMomRows - 1) / kMomRows, mb = (p + kMomRows - 1) / kMomRows;
  const RidgeTiles tiles{p, q, nb, mb * nb - mb * (mb - 1) / 2, G, C};
  for (int64_t n0 = 0; n0 < n; n0 += kMomChunk) {
    const int64_t len = n - n0 < kMomChunk ? n - n0 : kMomChunk;
    const int64_t np = (len + kMomKB - 1) / kMomKB * kMomKB;
    dim3 sgrid((unsigned)((np + kSplitObs - 1) / kSplitObs), (unsigned)((p + q + 31) / 32),
               (unsigned)batch);
    if (a->x_dtype == KVX_F32)
      split_kernel<float><<<sgrid, 256, 0, s>>>(reinterpret_cast<const float *>(a->x),
                                                reinterpret_cast<const float *>(a->y), shift, sums,
                                                n, p, q, n0, np, R, planes);
    else
      split_kernel<__nv_bfloat16><<<sgrid, 256, 0, s>>>(
          reinterpret_cast<const __nv_bfloat16 *>(a->x),
          reinterpret_cast<const __nv_bfloat16 *>(a->y), shift, sums, n, p, q, n0, np, R,
          planes);
    if (cudaGetLastError() != cudaSuccess) return KVX_ERR_CUDA;
    if (mom_launch(planes, R, np, tiles, batch * tiles.per_fit, a->status, s) != cudaSuccess)
      return KVX_ERR_CUDA;
  }
  // centring: G and C corrected, `shift` now holds the column sums
  centre_kernel<<<dim3((unsigned)p, (unsigned)batch), 256, 0, s>>>(G, C, sums, shift, n, p, q);
  if (cudaGetLastError() != cudaSuccess) return KVX_ERR_CUDA;
  // blocked fp64 Cholesky
  if (chol_factor(G, batch, p, a->lambda, a->status, s) != cudaSuccess) return KVX_ERR_CUDA;
  // triangular solves: by 64-row blocks (p <= 1024), else right-looking
  // with nc output columns per CTA in shared memory
  if (p <= kBlkMaxP) {
    chol_block_inverse_kernel<<<dim3((unsigned)batch, (unsigned)((p + 63) / 64)), 64, 0, s>>>(
        G, p, dinv);
    if (cudaFuncSetAttribute(chol_solve_blocked_kernel<RidgeEpi>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)blk_solve_smem_bytes(p)) != cudaSuccess)
      return KVX_ERR_CUDA;
    chol_solve_blocked_kernel<RidgeEpi>
        <<<dim3((unsigned)batch, (unsigned)((q + kBlkCols - 1) / kBlkCols)), kBlkThreads,
           blk_solve_smem_bytes(p), s>>>(G, dinv, C, p, q, RidgeEpi{shift, n, p, q, a->w, a->b});
  } else {
    const int nc = solve_cols_per_cta(p, batch, q);
    if (solve_smem_bytes(p, nc) > 48 * 1024 &&
        cudaFuncSetAttribute(trsm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)solve_smem_bytes(p, nc)) != cudaSuccess)
      return KVX_ERR_CUDA;
    dim3 tgrid((unsigned)batch, (unsigned)((q + nc - 1) / nc));
    trsm_kernel<<<tgrid, kSolveThreads, solve_smem_bytes(p, nc), s>>>(G, C, shift, n, p, q, nc,
                                                                      a->w, a->b);
  }
  return cudaGetLastError() == cudaSuccess ? KVX_OK : KVX_ERR_CUDA;
}
