// kvx_ridge.cu -- the ridge fit of the maps (kvx_ridge_fit), on the GPU.
//
// The Qwen3 14B -> 32B article, section "Линейного моста, как ни странно,
// хватает", fits one ridge regression per target (layer, head), one for
// keys and one for values, on paired source / target cache observations; its
// ridge demo centres X and Y on their column means, solves
// (XcT Xc + lam I) W = XcT Yc and sets b = ybar - xbar W.  For a batch of
// independent fits (X [n][p], Y [n][q] each) this runs as 4 + 3 ceil(p / 64) - 1
// launches:
//   1. clear the fp64 workspace;
//   2. column means of X and Y (fp32 partial sums over 256 rows, fp64 across
//      them, chunks of rows in parallel with fp64 atomics);
//   3. the centred Gram blocks G = XcT Xc (upper triangle of 64 x 64 tiles)
//      and C = XcT Yc: a register-tiled fp32 FMA contraction over the
//      observations (each thread 4 x 4 outputs; fp32 observations with p
//      and q multiples of 4 are staged through a 4-stage cp.async ring),
//      fp32 partial sums over 256 observations summed in fp32 over a slice
//      of 16,384, slices in parallel and added in fp64 with atomics;
//   4. G + lam I mirrored to full, then a Cholesky factorisation in fp64
//      blocked by 64 (per diagonal block: factor it, solve the panel below,
//      update the trailing blocks, each step spread over CTAs);
//   5. per (fit, nc output columns), one CTA: forward and back
//      substitution in fp64 (the columns in shared memory, the threads
//      split over the columns and the rows of each right-looking update),
//      b = ybar - xbar W; W and b stored as fp32.  A non-positive
//      pivot leaves W and b NaN and sets KVX_FLAG_NOT_SPD.
// The contraction is a dense Gram product, but it runs on the CUDA cores in
// fp32: bf16 or tf32 tensor-core operands would round the centred features
// to 8 or 11 significant bits, and the solve amplifies Gram errors by the
// condition number of G + lam I.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>

#include "../../include/kvx.h"
#include "kvx_async.cuh"
#include "kvx_chol.cuh"

namespace {

constexpr int kTile = 64;           // Gram tile (features x features or outputs)
constexpr int kChunkObs = 32;       // observations staged in shared memory per step
constexpr int kFlushObs = 256;      // fp32 partial sums are added into fp64 this often
constexpr int64_t kRowsPerSlice = 16384;   // observations per CTA of the Gram / means

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

// sums[b][c] += column c of [X | Y] over this CTA's slice of observations
template <typename T>
__global__ void __launch_bounds__(256) mean_kernel(const T *__restrict__ x, const T *__restrict__ y,
                                                   double *__restrict__ sums, int64_t n, int p,
                                                   int q) {
  const int b = blockIdx.z;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= p + q) return;
  const int64_t t0 = (int64_t)blockIdx.y * kRowsPerSlice;
  const int64_t t1 = t0 + kRowsPerSlice < n ? t0 + kRowsPerSlice : n;
  const T *col = c < p ? x + (int64_t)b * n * p + c : y + (int64_t)b * n * q + (c - p);
  const int ld = c < p ? p : q;
  double acc = 0.0;
  for (int64_t t = t0; t < t1; t += kFlushObs) {
    float part = 0.f;
    const int64_t te = t + kFlushObs < t1 ? t + kFlushObs : t1;
    for (int64_t u = t; u < te; ++u) part += ldv<T>(col + u * ld);
    acc += (double)part;
  }
  atomicAdd(sums + (int64_t)b * (p + q) + c, acc);
}

// One 64 x 64 tile of Z = Xc^T [Xc | Yc] over a slice of observations.
// Tile (ti, tj): rows are features 64 ti.., columns are features (tj <
// tiles_p, upper triangle only) or outputs 64 (tj - tiles_p)...
template <typename T>
__global__ void __launch_bounds__(256) gram_kernel(const T *__restrict__ x, const T *__restrict__ y,
                                                   const double *__restrict__ sums,
                                                   double *__restrict__ G, double *__restrict__ C,
                                                   int64_t n, int p, int q, int tiles_p,
                                                   int tiles_q) {
  __shared__ float sa[kChunkObs][kTile];
  __shared__ float sb[kChunkObs][kTile];
  __shared__ float mean_a[kTile], mean_b[kTile];
  const int b = blockIdx.z;
  // decode the tile: upper-triangle G tiles first, then the C tiles
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
  const T *xa = x + (int64_t)b * n * p;
  const T *xb = is_c ? y + (int64_t)b * n * q : xa;
  const double inv_n = 1.0 / (double)n;
  const int tid = threadIdx.x;
  if (tid < kTile) {
    const int i = i0 + tid;
    mean_a[tid] = i < p ? (float)(sums[(int64_t)b * (p + q) + i] * inv_n) : 0.f;
  } else if (tid < 2 * kTile) {
    const int j = j0 + tid - kTile;
    mean_b[tid - kTile] =
        j < ncols ? (float)(sums[(int64_t)b * (p + q) + (is_c ? p : 0) + j] * inv_n) : 0.f;
  }
  const int tx = tid & 15, ty = tid >> 4;   // thread's 4 x 4 block: rows 4 ty.., cols 4 tx..
  const int64_t t0 = (int64_t)blockIdx.y * kRowsPerSlice;
  const int64_t t1 = t0 + kRowsPerSlice < n ? t0 + kRowsPerSlice : n;
  // two fp32 levels: 256-observation partial sums, summed over the slice
  // (at most 64 of them); slices meet in fp64 (FP64 adds are ~64x slower
  // than FP32 FMAs here, so none sit in the inner loops)
  float acc[4][4];
  float part[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[r][c] = 0.f, part[r][c] = 0.f;
  __syncthreads();
  int since_flush = 0;
  for (int64_t t = t0; t < t1; t += kChunkObs) {
    // stage 32 observations x 64 columns of each operand, centred, fp32
    for (int e = tid; e < kChunkObs * kTile; e += blockDim.x) {
      const int o = e / kTile, c = e % kTile;
      const int64_t u = t + o;
      const int i = i0 + c, j = j0 + c;
      sa[o][c] = (u < t1 && i < p) ? ldv<T>(xa + u * p + i) - mean_a[c] : 0.f;
      sb[o][c] = (u < t1 && j < ncols) ? ldv<T>(xb + u * ncols + j) - mean_b[c] : 0.f;
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

// The same tile with the observations staged asynchronously (fp32 inputs, p
// and q multiples of 4, 16-byte aligned bases): every thread copies its own
// 16-byte words of the next kGramStages - 1 chunks into a ring with
// cp.async, so global latency overlaps the FMAs; once a chunk has landed the
// thread centres the words it copied in place (padding stays zero) and the
// CTA computes on it.
constexpr int kGramStages = 4;
constexpr size_t kGramRingBytes = (size_t)kGramStages * 2 * kChunkObs * kTile * sizeof(float);

__global__ void __launch_bounds__(256) gram_async_kernel(const float *__restrict__ x,
                                                         const float *__restrict__ y,
                                                         const double *__restrict__ sums,
                                                         double *__restrict__ G,
                                                         double *__restrict__ C, int64_t n, int p,
                                                         int q, int tiles_p, int tiles_q) {
  extern __shared__ __align__(16) float ring_s[];   // [stage][operand a|b][32][64]
  __shared__ __align__(16) float mean_a[kTile], mean_b[kTile];
  const int b = blockIdx.z;
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
  const float *xa = x + (int64_t)b * n * p;
  const float *xb = is_c ? y + (int64_t)b * n * q : xa;
  const double inv_n = 1.0 / (double)n;
  const int tid = threadIdx.x;
  if (tid < kTile) {
    const int i = i0 + tid;
    mean_a[tid] = i < p ? (float)(sums[(int64_t)b * (p + q) + i] * inv_n) : 0.f;
  } else if (tid < 2 * kTile) {
    const int j = j0 + tid - kTile;
    mean_b[tid - kTile] =
        j < ncols ? (float)(sums[(int64_t)b * (p + q) + (is_c ? p : 0) + j] * inv_n) : 0.f;
  }
  const int64_t t0 = (int64_t)blockIdx.y * kRowsPerSlice;
  const int64_t t1 = t0 + kRowsPerSlice < n ? t0 + kRowsPerSlice : n;
  const int chunks = (int)((t1 - t0 + kChunkObs - 1) / kChunkObs);
  constexpr int kStage = 2 * kChunkObs * kTile;      // floats per stage
  constexpr int kWords = kChunkObs * kTile / 4;      // 16-byte words per operand per chunk
  // this thread's words: w = tid + 256 k, k = 0, 1 -> row w / 16, columns 4 (w % 16)..
  auto issue = [&](int c) {
    float *st = ring_s + (c % kGramStages) * kStage;
#pragma unroll
    for (int k = 0; k < kWords / 256; ++k) {
      const int w = tid + 256 * k, o = w / (kTile / 4), c4 = 4 * (w % (kTile / 4));
      const int64_t u = t0 + (int64_t)c * kChunkObs + o;
      const bool ra = c < chunks && u < t1 && i0 + c4 < p;
      const bool rb = c < chunks && u < t1 && j0 + c4 < ncols;
      cp_async16(st + o * kTile + c4, ra ? xa + u * p + i0 + c4 : xa, ra ? 16u : 0u);
      cp_async16(st + kChunkObs * kTile + o * kTile + c4, rb ? xb + u * ncols + j0 + c4 : xb,
                 rb ? 16u : 0u);
    }
    cp_async_commit();
  };
  const int tx = tid & 15, ty = tid >> 4;
  float acc[4][4], part[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[r][c] = 0.f, part[r][c] = 0.f;
  for (int c = 0; c < kGramStages - 1; ++c) issue(c);
  __syncthreads();   // the means are in place
  int since_flush = 0;
  for (int c = 0; c < chunks; ++c) {
    issue(c + kGramStages - 1);
    cp_async_wait<kGramStages - 1>();
    float *st = ring_s + (c % kGramStages) * kStage;
    // centre the words this thread copied (rows and columns past the data
    // stay zero)
#pragma unroll
    for (int k = 0; k < kWords / 256; ++k) {
      const int w = tid + 256 * k, o = w / (kTile / 4), c4 = 4 * (w % (kTile / 4));
      const int64_t u = t0 + (int64_t)c * kChunkObs + o;
      if (u < t1 && i0 + c4 < p) {
        float4 *v = reinterpret_cast<float4 *>(st + o * kTile + c4);
        const float4 m = *reinterpret_cast<const float4 *>(mean_a + c4);
        float4 a = *v;
        a.x -= m.x, a.y -= m.y, a.z -= m.z, a.w -= m.w;
        *v = a;
      }
      if (u < t1 && j0 + c4 < ncols) {
        float4 *v = reinterpret_cast<float4 *>(st + kChunkObs * kTile + o * kTile + c4);
        const float4 m = *reinterpret_cast<const float4 *>(mean_b + c4);
        float4 a = *v;
        a.x -= m.x, a.y -= m.y, a.z -= m.z, a.w -= m.w;
        *v = a;
      }
    }
    __syncthreads();
    const float *sa = st, *sb = st + kChunkObs * kTile;
#pragma unroll 8
    for (int o = 0; o < kChunkObs; ++o) {
      const float4 a4 = *reinterpret_cast<const float4 *>(sa + o * kTile + 4 * ty);
      const float4 b4 = *reinterpret_cast<const float4 *>(sb + o * kTile + 4 * tx);
      const float av[4] = {a4.x, a4.y, a4.z, a4.w};
      const float bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) part[r][cc] = fmaf(av[r], bv[cc], part[r][cc]);
    }
    __syncthreads();   // the stage is free for the copy issued next
    since_flush += kChunkObs;
    if (since_flush >= kFlushObs) {
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) acc[r][cc] += part[r][cc], part[r][cc] = 0.f;
      since_flush = 0;
    }
  }
  cp_async_wait<0>();
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      const int i = i0 + 4 * ty + r, j = j0 + 4 * tx + cc;
      if (i >= p || j >= ncols) continue;
      const double v = (double)acc[r][cc] + (double)part[r][cc];
      if (is_c)
        atomicAdd(C + ((int64_t)b * p + i) * q + j, v);
      else
        atomicAdd(G + ((int64_t)b * p + i) * p + j, v);
    }
}

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

constexpr int kMaxDim = 4096;

size_t ws_sums(int batch, int p, int q) { return (size_t)batch * (p + q) * sizeof(double); }
size_t ws_gram(int batch, int p) { return (size_t)batch * p * p * sizeof(double); }
size_t ws_cross(int batch, int p, int q) { return (size_t)batch * p * q * sizeof(double); }
size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

extern "C" size_t kvx_ridge_workspace_bytes(int32_t batch, int32_t p, int32_t q) {
  if (batch < 1 || p < 1 || q < 1 || p > kMaxDim || q > kMaxDim) return 0;
  return round256(ws_sums(batch, p, q)) + round256(ws_gram(batch, p)) + ws_cross(batch, p, q);
}

extern "C" kvx_status kvx_ridge_fit(const kvx_ridge_args *a, void *stream) {
  if (!a) return KVX_ERR_INVALID_ARG;
  if (a->batch < 1 || a->batch > 65535 || a->n < 1 || a->p < 1 || a->q < 1 ||
      a->p > kMaxDim || a->q > kMaxDim || !std::isfinite(a->lambda) || !a->x || !a->y ||
      !a->w || !a->b || !a->workspace ||
      (a->x_dtype != KVX_F32 && a->x_dtype != KVX_BF16))
    return KVX_ERR_INVALID_ARG;
  if (a->workspace_bytes < kvx_ridge_workspace_bytes(a->batch, a->p, a->q))
    return KVX_ERR_INVALID_ARG;
  const int64_t n = a->n;
  const int64_t slices64 = (n + kRowsPerSlice - 1) / kRowsPerSlice;
  if (slices64 > 65535) return KVX_ERR_INVALID_ARG;  // grid y; checked before any launch
  const int slices = (int)slices64;
  cudaStream_t s = (cudaStream_t)stream;
  const int batch = a->batch, p = a->p, q = a->q;
  unsigned char *ws = reinterpret_cast<unsigned char *>(a->workspace);
  double *sums = reinterpret_cast<double *>(ws);
  double *G = reinterpret_cast<double *>(ws + round256(ws_sums(batch, p, q)));
  double *C = reinterpret_cast<double *>(ws + round256(ws_sums(batch, p, q)) +
                                         round256(ws_gram(batch, p)));
  const int64_t words = (int64_t)(round256(ws_sums(batch, p, q)) + round256(ws_gram(batch, p)) +
                                  ws_cross(batch, p, q)) / 8;
  clear_kernel<<<1024, 256, 0, s>>>(sums, words);
  if (cudaGetLastError() != cudaSuccess) return KVX_ERR_CUDA;

  dim3 mgrid((unsigned)((p + q + 255) / 256), (unsigned)slices, (unsigned)batch);
  const int tiles_p = (p + kTile - 1) / kTile, tiles_q = (q + kTile - 1) / kTile;
  dim3 ggrid((unsigned)(tiles_p * (tiles_p + 1) / 2 + tiles_p * tiles_q), (unsigned)slices,
             (unsigned)batch);
  if (a->x_dtype == KVX_F32) {
    const float *x = reinterpret_cast<const float *>(a->x);
    const float *y = reinterpret_cast<const float *>(a->y);
    mean_kernel<float><<<mgrid, 256, 0, s>>>(x, y, sums, n, p, q);
    const bool async_ok = p % 4 == 0 && q % 4 == 0 &&
                          ((((uintptr_t)x) | ((uintptr_t)y)) & 15u) == 0;
    if (async_ok) {
      if (cudaFuncSetAttribute(gram_async_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kGramRingBytes) != cudaSuccess)
        return KVX_ERR_CUDA;
      gram_async_kernel<<<ggrid, 256, kGramRingBytes, s>>>(x, y, sums, G, C, n, p, q, tiles_p,
                                                           tiles_q);
    } else {
      gram_kernel<float><<<ggrid, 256, 0, s>>>(x, y, sums, G, C, n, p, q, tiles_p, tiles_q);
    }
  } else {
    const __nv_bfloat16 *x = reinterpret_cast<const __nv_bfloat16 *>(a->x);
    const __nv_bfloat16 *y = reinterpret_cast<const __nv_bfloat16 *>(a->y);
    mean_kernel<__nv_bfloat16><<<mgrid, 256, 0, s>>>(x, y, sums, n, p, q);
    gram_kernel<__nv_bfloat16><<<ggrid, 256, 0, s>>>(x, y, sums, G, C, n, p, q, tiles_p, tiles_q);
  }
  if (cudaGetLastError() != cudaSuccess) return KVX_ERR_CUDA;
  // blocked fp64 Cholesky
  if (chol_factor(G, batch, p, a->lambda, a->status, s) != cudaSuccess) return KVX_ERR_CUDA;
  // triangular solves: nc output columns per CTA, in shared memory
  const int nc = solve_cols_per_cta(p);
  if (solve_smem_bytes(p, nc) > 48 * 1024 &&
      cudaFuncSetAttribute(trsm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)solve_smem_bytes(p, nc)) != cudaSuccess)
    return KVX_ERR_CUDA;
  dim3 tgrid((unsigned)batch, (unsigned)((q + nc - 1) / nc));
  trsm_kernel<<<tgrid, kSolveThreads, solve_smem_bytes(p, nc), s>>>(G, C, sums, n, p, q, nc,
                                                                    a->w, a->b);
  return cudaGetLastError() == cudaSuccess ? KVX_OK : KVX_ERR_CUDA;
}
