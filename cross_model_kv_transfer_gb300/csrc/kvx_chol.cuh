// kvx_chol.cuh -- batched fp64 Cholesky factorisation of G + lam I, blocked
// by 64, shared by the ridge fit (kvx_ridge.cu) and the layer-selection
// scores (kvx_scores.cu).  G is [batch][p][p] fp64 in global memory holding
// the upper triangle of a symmetric matrix; after chol_factor it holds L in
// its lower triangle and L^T in its upper one.  Right-looking: per diagonal
// block, factor it (one CTA per fit), solve the panel below it (two CTAs of
// four warps per block row) and update the trailing lower triangle (one CTA
// per 64 x 64 block), so that the update, most of the work, is spread over
// the GPU.  GB300 retires about two fp64 lanes per clock per SM, so the
// diagonal and panel steps, a few CTAs each, are bound by latency: both keep
// one barrier per column and independent multiply-adds within a step.  A
// fit whose pivot is not positive gets G[0] = NaN (later steps skip it) and
// KVX_FLAG_NOT_SPD in *status.  chol_solve_cols then solves columns against
// the factor.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvx.h"

namespace {

constexpr int kB = 64;   // block of the factorisation

// G + lam I mirrored to full: row block blockIdx.y of fit blockIdx.x.
__global__ void __launch_bounds__(256) chol_prep_kernel(double *__restrict__ G, int p, double lam) {
  double *A = G + (int64_t)blockIdx.x * p * p;
  const int r0 = blockIdx.y * kB;
  for (int e = threadIdx.x; e < kB * p; e += blockDim.x) {
    const int i = r0 + e / p, j = e % p;
    if (i >= p) break;
    if (i > j) A[(int64_t)i * p + j] = A[(int64_t)j * p + i];
    else if (i == j) A[(int64_t)i * p + j] += lam;
  }
}

__device__ __forceinline__ int blk_len(int p, int kb) { return p - kb * kB < kB ? p - kb * kB : kB; }

// Factor the diagonal block kb of each fit in shared memory, right-looking
// over all threads, one barrier per column: step j updates the trailing lower
// triangle with L[i][m] -= (L[i][j] / d_j) L[m][j] from the unscaled column
// (a 16 x 16 thread grid walking rows and columns), scales column j - 1 by
// 1 / sqrt(d_{j-1}) (no one reads it any more), and thread 0, which alone
// owns element (j + 1, j + 1), updates it first and takes the next pivot's
// reciprocal square root while the others update.  The update of earlier
// blocks is already applied.  (Holding the rows in registers instead issues
// every thread's predicated multiply-adds on the narrow fp64 pipe and ran
// 1.4x slower.)
__device__ __forceinline__ bool chol_pivot(double d, double &diag, double &rp, double &rd) {
  if (!(d > 0.0)) return false;
  const double r = rsqrt(d);
  diag = d * r;
  rp = r;
  rd = r * r;
  return true;
}

__global__ void __launch_bounds__(256) chol_diag_kernel(double *__restrict__ G, int p, int kb,
                                                        uint32_t *status) {
  __shared__ double L[kB][kB + 1];
  __shared__ double rp[kB], rd[kB];   // 1 / sqrt(d_j) and 1 / d_j
  // pivot failures by step parity: step j reads fail[j & 1] and thread 0
  // writes fail[(j + 1) & 1] in the same step, so no read races a write
  __shared__ int fail[2];
  double *A = G + (int64_t)blockIdx.x * p * p;
  if (isnan(A[0])) return;
  const int o = kb * kB, nb = blk_len(p, kb);
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  for (int i = ty; i < nb; i += 16)
    for (int j = tx; j < nb; j += 16) L[i][j] = A[(int64_t)(o + i) * p + o + j];
  __syncthreads();
  if (tid == 0) fail[0] = chol_pivot(L[0][0], L[0][0], rp[0], rd[0]) ? 0 : 1;
  __syncthreads();
  bool failed = false;
  for (int j = 0; j < nb; ++j) {
    if (fail[j & 1]) {
      failed = true;
      break;
    }
    if (j > 0 && tid >= j && tid < nb) L[tid][j - 1] *= rp[j - 1];
    const double inv = rd[j];
    int i0 = j + 1 + ty;
    if (tid == 0 && j + 1 < nb) {
      const double d = fma(-L[j + 1][j] * inv, L[j + 1][j], L[j + 1][j + 1]);
      fail[(j + 1) & 1] = chol_pivot(d, L[j + 1][j + 1], rp[j + 1], rd[j + 1]) ? 0 : 1;
      i0 += 16;
    }
    for (int i = i0; i < nb; i += 16) {
      const double a = L[i][j] * inv;
      for (int m = j + 1 + tx; m <= i; m += 16) L[i][m] = fma(-a, L[m][j], L[i][m]);
    }
    __syncthreads();
  }
  if (failed) {
    if (tid == 0) {
      A[0] = nan("");
      if (status) atomicOr(status, KVX_FLAG_NOT_SPD);
    }
    return;
  }
  // L in the lower triangle, L^T in the upper (rows of L^T are what the
  // back substitution reads)
  for (int i = ty; i < nb; i += 16)
    for (int j = tx; j < nb; j += 16)
      A[(int64_t)(o + i) * p + o + j] = i >= j ? L[i][j] : L[j][i];
}

// Panel: rows r0 .. r0 + 31 of block row ib = kb + 1 + blockIdx.y / 2 of fit
// blockIdx.x solve X L_kb^T = A[ib][kb].  Lane l of every warp holds row
// r0 + l; warp w holds its columns 16 w .. 16 w + 15 in registers, so a block
// row spreads over two CTAs of four warps.  Right-looking: at step j the warp
// owning column j finishes x_j (times the pivot's reciprocal, taken once in
// shared memory) and publishes it; every warp with columns beyond j then
// takes its terms, L[m][j] x_j, all independent of one another.  The
// published values alternate between two buffers, one barrier per step.
constexpr int kPanelRows = 32;
constexpr int kPanelThreads = kB / 16 * 32;
__global__ void __launch_bounds__(kPanelThreads) chol_panel_kernel(double *__restrict__ G, int p,
                                                                  int kb) {
  __shared__ double L[kB][kB + 1];
  __shared__ double rd[kB];
  __shared__ double xs[2][kPanelRows];
  double *A = G + (int64_t)blockIdx.x * p * p;
  if (isnan(A[0])) return;
  const int o = kb * kB, nb = blk_len(p, kb);
  const int ib = kb + 1 + blockIdx.y / (kB / kPanelRows);
  const int r0 = ib * kB + (blockIdx.y % (kB / kPanelRows)) * kPanelRows;
  const int nr = p - r0 < kPanelRows ? p - r0 : kPanelRows;
  // the factor's lower triangle, zero elsewhere
#pragma unroll 8
  for (int e = threadIdx.x; e < kB * kB; e += kPanelThreads) {
    const int i = e / kB, j = e % kB;
    L[i][j] = (i < nb && j <= i) ? A[(int64_t)(o + i) * p + o + j] : 0.0;
  }
  __syncthreads();
  for (int j = threadIdx.x; j < nb; j += kPanelThreads) rd[j] = 1.0 / L[j][j];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const bool live = lane < nr;
  double *row = A + (int64_t)(r0 + lane) * p + o + 16 * w;
  double x[16];
#pragma unroll
  for (int v = 0; v < 16; ++v) x[v] = (live && 16 * w + v < nb) ? row[v] : 0.0;
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kB; ++j) {
    if (j >= nb) break;
    if (w == (j >> 4)) {
      x[j & 15] *= rd[j];
      xs[j & 1][lane] = x[j & 15];
    }
    __syncthreads();
    if (16 * w + 15 > j) {
      const double xj = xs[j & 1][lane];
#pragma unroll
      for (int v = 0; v < 16; ++v)
        if (16 * w + v > j) x[v] = fma(-xj, L[16 * w + v][j], x[v]);
    }
  }
  if (!live) return;
#pragma unroll
  for (int v = 0; v < 16; ++v) {
    const int c = 16 * w + v;
    if (c < nb) {
      row[v] = x[v];                                   // L[r0 + lane][o + c]
      A[(int64_t)(o + c) * p + r0 + lane] = x[v];      // and L^T
    }
  }
}

// Trailing update: lower-triangle block (ib, jb), ib >= jb > kb, of fit
// blockIdx.x: A[ib][jb] -= A[ib][kb] A[jb][kb]^T; 256 threads, 4 x 4 each.
__global__ void __launch_bounds__(256) chol_update_kernel(double *__restrict__ G, int p, int kb) {
  __shared__ double Pa[kB][kB / 2 + 1];
  __shared__ double Pb[kB][kB / 2 + 1];
  double *A = G + (int64_t)blockIdx.x * p * p;
  if (isnan(A[0])) return;
  // decode (ib, jb) from the lower triangle of the trailing blocks
  int t = blockIdx.y, ib = kb + 1, jb = kb + 1;
  while (t > ib - (kb + 1)) {
    t -= ib - kb;
    ++ib;
  }
  jb = kb + 1 + t;
  const int o = kb * kB, nk = blk_len(p, kb);
  const int ri = ib * kB, rj = jb * kB, ni = blk_len(p, ib), nj = blk_len(p, jb);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  double acc[4][4];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[a][c] = 0.0;
  for (int k0 = 0; k0 < nk; k0 += kB / 2) {
    for (int e = threadIdx.x; e < kB * (kB / 2); e += blockDim.x) {
      const int r = e / (kB / 2), k = e % (kB / 2);
      const bool kin = k0 + k < nk;
      Pa[r][k] = (r < ni && kin) ? A[(int64_t)(ri + r) * p + o + k0 + k] : 0.0;
      Pb[r][k] = (r < nj && kin) ? A[(int64_t)(rj + r) * p + o + k0 + k] : 0.0;
    }
    __syncthreads();
#pragma unroll 4
    for (int k = 0; k < kB / 2; ++k) {
      double av[4], bv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) av[a] = Pa[4 * ty + a][k];
#pragma unroll
      for (int c = 0; c < 4; ++c) bv[c] = Pb[4 * tx + c][k];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[a][c] = fma(av[a], bv[c], acc[a][c]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = 4 * ty + a, j = 4 * tx + c;
      if (i < ni && j < nj && (ib != jb || i >= j))
        A[(int64_t)(ri + i) * p + rj + j] -= acc[a][c];
    }
}

// Launch the whole factorisation (4 + 3 (p / 64 rounded up) - 1 launches).
// ---------------------------------------------------------------------------
// Blocked column solves (p <= kBlkMaxP): forward L Z = C and back L^T W = Z
// by 64-row blocks.  Per block, the right-hand side minus the product of the
// factor's panel with the rows already solved (a GEMM from shared memory),
// then the block's inverse diagonal block (chol_block_inverse_kernel); so
// nearly all of the fp64 work is GEMM-shaped and the fp64 pipe stays busy.
// ---------------------------------------------------------------------------
constexpr int kBlkCols = 16;      // columns per CTA
constexpr int kBlkThreads = 256;  // 16 row groups of 4 rows x 16 columns
constexpr int kBlkMaxP = 1024;

// Shared memory of a blocked solve: the columns [p][kBlkCols], T [64][kBlkCols]
// and one buffer that holds either a [64][33] panel tile or a [64][65]
// inverse diagonal block (rows padded against bank conflicts).
inline size_t blk_solve_smem_bytes(int p) {
  return ((size_t)p * kBlkCols + (size_t)kB * kBlkCols + (size_t)kB * (kB + 1)) * sizeof(double);
}

// Inverse of each 64 x 64 diagonal block of L: Dinv[fit][blk] (row-major,
// lower triangular; rows beyond p read as the identity).  One thread per
// column j of the inverse X, in fp64: X[j][j] = 1 / L[j][j] and, for i > j,
// X[i][j] = -(sum_{j <= k < i} L[i][k] X[k][j]) / L[i][i].  S holds L's
// strictly lower part and X's strictly lower part transposed (X[i][j] at
// S[j][i]); r holds the reciprocals of L's diagonal.
__global__ void __launch_bounds__(kB) chol_block_inverse_kernel(const double *__restrict__ G,
                                                                int p,
                                                                double *__restrict__ Dinv) {
  __shared__ double S[kB][kB + 1];
  __shared__ double r[kB];
  const int b = blockIdx.x, blk = blockIdx.y, nblk = (p + kB - 1) / kB;
  const double *A = G + (int64_t)b * p * p;
  if (isnan(A[0])) return;
  const int o = blk * kB, nb = blk_len(p, blk), j = threadIdx.x;
  for (int i = j + 1; i < kB; ++i)
    S[i][j] = i < nb ? A[(int64_t)(o + i) * p + o + j] : 0.0;
  r[j] = j < nb ? 1.0 / A[(int64_t)(o + j) * p + o + j] : 1.0;
  __syncthreads();
  for (int i = j + 1; i < kB; ++i) {
    double acc = S[i][j] * r[j];                  // k = j: L[i][j] X[j][j]
    for (int k = j + 1; k < i; ++k) acc = fma(S[i][k], S[j][k], acc);
    S[j][i] = -acc * r[i];
  }
  __syncthreads();
  double *D = Dinv + ((int64_t)b * nblk + blk) * kB * kB;
  for (int i = 0; i < kB; ++i) D[i * kB + j] = i > j ? S[j][i] : (i == j ? r[i] : 0.0);
}

// Per (fit b, kBlkCols columns of C [p][q]): Z and W in shared memory, then
// epi(b, c0, col, zn, wn): col holds W ([p][kBlkCols]); zn and wn are the
// column's |z|^2 and |w|^2 in threads t < kBlkCols.  A fit whose factor
// failed gets epi.failed(b, c0).
template <typename Epi>
__global__ void __launch_bounds__(kBlkThreads) chol_solve_blocked_kernel(
    const double *__restrict__ G, const double *__restrict__ Dinv, const double *__restrict__ C,
    int p, int q, Epi epi) {
  extern __shared__ double sm[];
  double *Z = sm;                                   // [p][kBlkCols]
  double *T = Z + (size_t)p * kBlkCols;             // [64][kBlkCols]
  double *Lp = T + (size_t)kB * kBlkCols;           // [64][33] panel tile, or
  double *Ds = Lp;                                  // [64][65] inverse diagonal block
  __shared__ double red[16][kBlkCols + 1];
  const int b = blockIdx.x, c0 = blockIdx.y * kBlkCols, nblk = (p + kB - 1) / kB;
  const double *A = G + (int64_t)b * p * p;
  if (isnan(A[0])) {
    epi.failed(b, c0);
    return;
  }
  const double *Cb = C + (int64_t)b * p * q;
  const int t = threadIdx.x, j = t & (kBlkCols - 1), g = t >> 4;
  for (int e = t; e < p * kBlkCols; e += kBlkThreads) {
    const int i = e / kBlkCols, c = e % kBlkCols;
    Z[e] = c0 + c < q ? Cb[(int64_t)i * q + c0 + c] : 0.0;
  }
  __syncthreads();
  double zsq = 0.0, wsq = 0.0;
  // forward: Z_blk = Dinv_blk (C_blk - L[blk][< blk] Z[< blk])
  for (int blk = 0; blk < nblk; ++blk) {
    const int r0 = blk * kB, nr = blk_len(p, blk);
    double acc[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) acc[a] = 4 * g + a < nr ? Z[(r0 + 4 * g + a) * kBlkCols + j] : 0.0;
    for (int k0 = 0; k0 < r0; k0 += 32) {
      for (int e = t; e < kB * 32; e += kBlkThreads) {
        const int i = e >> 5, kk = e & 31;
        Lp[i * 33 + kk] = i < nr ? A[(int64_t)(r0 + i) * p + k0 + kk] : 0.0;
      }
      __syncthreads();
#pragma unroll 8
      for (int kk = 0; kk < 32; ++kk) {
        const double z = Z[(k0 + kk) * kBlkCols + j];
#pragma unroll
        for (int a = 0; a < 4; ++a) acc[a] = fma(-Lp[(4 * g + a) * 33 + kk], z, acc[a]);
      }
      __syncthreads();
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) T[(4 * g + a) * kBlkCols + j] = acc[a];
    __syncthreads();
    const double *D = Dinv + ((int64_t)b * nblk + blk) * kB * kB;
    for (int e = t; e < kB * kB; e += kBlkThreads) Ds[(e >> 6) * (kB + 1) + (e & 63)] = D[e];
    __syncthreads();
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int i = 4 * g + a;
      double v = 0.0;
      for (int k = 0; k <= i; ++k) v = fma(Ds[i * (kB + 1) + k], T[k * kBlkCols + j], v);
      if (i < nr) {
        Z[(r0 + i) * kBlkCols + j] = v;
        zsq = fma(v, v, zsq);
      }
    }
    __syncthreads();
  }
  // back: W_blk = Dinv_blk^T (Z_blk - L[> blk][blk]^T W[> blk]); row r0 + i of
  // L^T is row r0 + i of the factor's upper triangle
  for (int blk = nblk - 1; blk >= 0; --blk) {
    const int r0 = blk * kB, nr = blk_len(p, blk);
    double acc[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) acc[a] = 4 * g + a < nr ? Z[(r0 + 4 * g + a) * kBlkCols + j] : 0.0;
    for (int k0 = r0 + kB; k0 < p; k0 += 32) {
      for (int e = t; e < kB * 32; e += kBlkThreads) {
        const int i = e >> 5, kk = e & 31;
        Lp[i * 33 + kk] = i < nr && k0 + kk < p ? A[(int64_t)(r0 + i) * p + k0 + kk] : 0.0;
      }
      __syncthreads();
#pragma unroll 8
      for (int kk = 0; kk < 32; ++kk) {
        const double w = k0 + kk < p ? Z[(k0 + kk) * kBlkCols + j] : 0.0;
#pragma unroll
        for (int a = 0; a < 4; ++a) acc[a] = fma(-Lp[(4 * g + a) * 33 + kk], w, acc[a]);
      }
      __syncthreads();
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) T[(4 * g + a) * kBlkCols + j] = acc[a];
    __syncthreads();
    const double *D = Dinv + ((int64_t)b * nblk + blk) * kB * kB;
    for (int e = t; e < kB * kB; e += kBlkThreads) Ds[(e >> 6) * (kB + 1) + (e & 63)] = D[e];
    __syncthreads();
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int i = 4 * g + a;
      double v = 0.0;
      for (int k = i; k < nr; ++k) v = fma(Ds[k * (kB + 1) + i], T[k * kBlkCols + j], v);
      if (i < nr) {
        Z[(r0 + i) * kBlkCols + j] = v;
        wsq = fma(v, v, wsq);
      }
    }
    __syncthreads();
  }
  red[g][j] = zsq;
  __syncthreads();
  double zn = 0.0, wn = 0.0;
  if (t < kBlkCols) {
    for (int r = 0; r < 16; ++r) zn += red[r][t];
  }
  __syncthreads();
  red[g][j] = wsq;
  __syncthreads();
  if (t < kBlkCols) {
    for (int r = 0; r < 16; ++r) wn += red[r][t];
  }
  epi(b, c0, Z, zn, wn);
}

constexpr int kSolveThreads = 128;   // threads per CTA of the column solves

// Columns one CTA of a triangular solve holds in shared memory: the largest
// power of two <= 32 with p x nc <= 4096 doubles (32 KB), halved while the
// `batch` fits of q columns would give fewer than four CTAs per SM (the
// steps of one CTA are a chain of latencies; more CTAs hide them).
inline int solve_cols_per_cta(int p, int batch, int q) {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      sms = 1;
  }
  int nc = 32;
  while (nc > 1 && (int64_t)p * nc > 4096) nc >>= 1;
  while (nc > 1 && (int64_t)batch * ((q + nc - 1) / nc) < 4LL * sms) nc >>= 1;
  return nc;
}
inline size_t solve_smem_bytes(int p, int nc) { return ((size_t)p * nc + p) * sizeof(double); }

// Forward L z = c, then back L^T w = z, in fp64, for the nc columns a CTA of
// kSolveThreads threads holds in shared memory (col[i * nc + j] is row i of
// column j; rd is p doubles of scratch), where A is a factor left by
// chol_factor.  Right-looking: once z_k = c_k / L_kk is known every later
// row takes c_i -= L_ik z_k (L_ik = A[k][i], row k of the upper triangle,
// contiguous), and the back solve does the same from the bottom with row i
// of the lower triangle.  Thread t works on column t % nc and, in each
// update, on the rows congruent to t / nc modulo kSolveThreads / nc, so that
// the fp64 pipe sees many independent multiply-adds per step; one barrier
// ends each step.  The pivots' reciprocals are taken once, so a step costs a
// multiply, not a division.  On return col holds w, and the threads t < nc
// hold |z|^2 and |w|^2 of column t (0 in the other threads).
__device__ inline void chol_solve_cols(const double *__restrict__ A, int p, double *col,
                                       double *rd, int nc, double &zn, double &wn) {
  const int t = threadIdx.x, rpc = kSolveThreads / nc, cl = t % nc, r0 = t / nc;
  for (int i = t; i < p; i += kSolveThreads) rd[i] = 1.0 / A[(int64_t)i * p + i];
  zn = 0.0;
  wn = 0.0;
  __syncthreads();
  // row k is final once step k - 1 has ended and is not written in step k
  for (int k = 0; k < p; ++k) {
    const double *lk = A + (int64_t)k * p;
    const double zk = col[k * nc + cl] * rd[k];
    if (r0 == 0) zn = fma(zk, zk, zn);
#pragma unroll 4
    for (int i = k + 1 + r0; i < p; i += rpc)
      col[i * nc + cl] = fma(-__ldg(lk + i), zk, col[i * nc + cl]);
    __syncthreads();
  }
  for (int e = t; e < p * nc; e += kSolveThreads) col[e] *= rd[e / nc];   // col = z
  __syncthreads();
  for (int i = p - 1; i >= 0; --i) {
    const double *li = A + (int64_t)i * p;
    const double wi = col[i * nc + cl] * rd[i];
    if (r0 == 0) wn = fma(wi, wi, wn);
#pragma unroll 4
    for (int m = r0; m < i; m += rpc) col[m * nc + cl] = fma(-__ldg(li + m), wi, col[m * nc + cl]);
    __syncthreads();
  }
  for (int e = t; e < p * nc; e += kSolveThreads) col[e] *= rd[e / nc];   // col = w
  __syncthreads();
}

inline cudaError_t chol_factor(double *G, int batch, int p, double lam, uint32_t *status,
                               cudaStream_t s) {
  const int nblk = (p + kB - 1) / kB;
  chol_prep_kernel<<<dim3((unsigned)batch, (unsigned)nblk), 256, 0, s>>>(G, p, lam);
  for (int kb = 0; kb < nblk; ++kb) {
    chol_diag_kernel<<<batch, 256, 0, s>>>(G, p, kb, status);
    const int rest = nblk - 1 - kb;
    if (rest > 0) {
      chol_panel_kernel<<<dim3((unsigned)batch, (unsigned)(rest * (kB / kPanelRows))),
                          kPanelThreads, 0, s>>>(G, p, kb);
      chol_update_kernel<<<dim3((unsigned)batch, (unsigned)(rest * (rest + 1) / 2)), 256, 0, s>>>(
          G, p, kb);
    }
  }
  return cudaGetLastError();
}

}  // namespace
