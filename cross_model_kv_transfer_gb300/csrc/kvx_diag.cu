// kvx_diag.cu -- fidelity diagnostics of a transfer (kvx_kv_diagnostics).
//
// How close is the mapped cache to the target model's own cache for the same
// tokens?  "Helm Intelligent Routing", section "Reading the retention score",
// reads the KV cosine between the two beside retention as a diagnostic; the
// Qwen3 14B -> 32B article, section "Линейного моста, как ни странно,
// хватает", measures how much of the target keys' and values' variance the
// selected source layers explain.  Per (target layer lt, head h, K|V) this
// computes, over the tokens a transfer writes: n, the sum of the per-token
// cosines, the residual energy sum |ref - mapped|^2, the reference energy
// sum |ref|^2 and the content-space sum of the reference (keys un-rotated at
// p' with the target RoPE base), from which mean cosine and centred R^2
// follow.
//
// The work is a streaming reduction over two caches of the target's size
// (HBM-bound).  One CTA takes a chunk of packed source tokens of one target
// layer; the chunk's rows are resolved once into shared memory (request,
// positions, contiguous or paged row, range checks -- the same rules as the
// transfer).  Each (head, K|V) row of a token is read by a group of G lanes,
// lane q holding RL consecutive RoPE pairs (i, i + d/2) of each of its runs,
// so the key un-rotation stays in registers; the per-token dot products are
// reduced across the group with shuffles.  Sums are kept in fp32 per thread
// over the chunk and added into the fp64 output with atomics.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "kvx_device.cuh"
#include "kvx_internal.h"
#include "kvx_async.cuh"
#include "kvx_ptx.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kMaxChunk = 1024;

struct DiagParams {
  KvxParams p;                   // request table, positions, rows, status
  const void *mk, *mv, *rk, *rv; // mapped / reference caches [Lt][rows][H][d]
  double *stats;                 // [Lt][H][2][d + 4]
  int32_t chunk;                 // tokens per CTA
  int32_t G;                     // lanes per (head, K|V) row, power of two
  int32_t NR;                    // runs of RL pairs per half row (half / RL)
  int32_t lanes_per_token;       // 2 * H * G
  int32_t tok_par;               // tokens a CTA works on at once
  int32_t slot_groups;           // CTAs per (layer, chunk) along the lanes
  unsigned long long turns[128]; // target RoPE frequencies, 2^-64 turns
};

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

// RL consecutive elements starting at `src` into fp32 registers.  With VEC
// the run is read in 16-byte loads (RL * sizeof(T) a multiple of 16, base
// 16-byte aligned), streaming (each byte is read once).
template <typename T, int RL, bool VEC>
__device__ __forceinline__ void load_run(const T *src, float *out) {
  if constexpr (VEC) {
    constexpr int kPer = 16 / (int)sizeof(T);
#pragma unroll
    for (int v = 0; v < RL / kPer; ++v) {
      const uint4 u = __ldcs(reinterpret_cast<const uint4 *>(src) + v);
      const T *e = reinterpret_cast<const T *>(&u);
#pragma unroll
      for (int j = 0; j < kPer; ++j) out[v * kPer + j] = to_f<T>(e[j]);
    }
  } else {
#pragma unroll
    for (int j = 0; j < RL; ++j) out[j] = to_f<T>(src[j]);
  }
}

// Stages of the cp.async ring: 3 (48 KB of shared memory at 256 threads for
// bf16, so that 3 CTAs fit on an SM; 96 KB for fp32, 2 CTAs).  At the
// 14B -> 32B shape 3 stages at 3 CTAs per SM ran 3.04 ms per call against
// 3.44 ms for 6 stages at 2 CTAs per SM: more warps per SM hide the
// shuffles and RoPE angles better than deeper rings per thread.
template <typename T>
constexpr int kStages = 3;
// CTAs per SM the register budget is sized for (3 for the bf16 ring, whose
// shared memory allows them)
template <typename T, bool RING>
constexpr int kMinCtas = (sizeof(T) == 2 && RING) ? 3 : 2;

template <typename T>
constexpr size_t ring_bytes(int nthreads) {
  return (size_t)kStages<T> * 4 * (8 * sizeof(T) / 16) * nthreads * 16;
}

// The 16 / sizeof(T) elements of one 16-byte word as fp32.
template <typename T>
__device__ __forceinline__ void unpack16(const uint4 &u, float *out) {
  const T *e = reinterpret_cast<const T *>(&u);
#pragma unroll
  for (int j = 0; j < 16 / (int)sizeof(T); ++j) out[j] = to_f<T>(e[j]);
}

template <typename T, int RL, int EMAX, bool VEC>
__global__ void __launch_bounds__(kThreads, kMinCtas<T, VEC && EMAX == 1>) kv_diag_kernel(
    const __grid_constant__ DiagParams P) {
  __shared__ int64_t s_row[kMaxChunk];
  __shared__ int32_t s_pt[kMaxChunk];
  __shared__ uint32_t s_bits;
  __shared__ int s_count;

  const KvxParams &p = P.p;
  const int tid = threadIdx.x;
  const int lt = blockIdx.y / P.slot_groups;
  const int sg = blockIdx.y % P.slot_groups;
  if (!kvx::seqlens_ok(p, tid, blockDim.x)) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && tid == 0) kvx::report(p, KVX_FLAG_BAD_SEQLENS);
    return;
  }

  // ---- the chunk's rows (the transfer's position and row rules) ----------
  const int64_t t0 = (int64_t)blockIdx.x * P.chunk;
  const int n = (int)min((int64_t)P.chunk, p.ntok - t0);
  if (tid == 0) {
    s_bits = 0;
    s_count = 0;
  }
  __syncthreads();
  int valid = 0;
  uint32_t bad = 0;
  for (int i = tid; i < n; i += blockDim.x) {
    int32_t ps = 0, pt = 0;
    int64_t row = -1;
    bad |= kvx::token_meta(p, t0 + i, ps, pt, row);
    s_row[i] = row;
    s_pt[i] = pt;
    valid += row >= 0;
  }
  if (bad) atomicOr(&s_bits, bad);
  if (valid) atomicAdd(&s_count, valid);
  __syncthreads();
  if (tid == 0 && lt == 0 && sg == 0) kvx::report(p, s_bits);

  // ---- this thread's (head, K|V, lane) -----------------------------------
  int tl, u;
  if (P.slot_groups == 1) {
    tl = tid / P.lanes_per_token;
    u = tid % P.lanes_per_token;
  } else {
    tl = 0;
    u = sg * kThreads + tid;
  }
  const bool lane_on = u < P.lanes_per_token && tl < P.tok_par;
  const int slot = lane_on ? u / P.G : 0;     // m * H + h
  const int q = u % P.G;
  const int m = slot / p.H, h = slot % p.H;
  const int half = p.d >> 1;
  const T *mapped = reinterpret_cast<const T *>(m == 0 ? P.mk : P.mv);
  const T *ref = reinterpret_cast<const T *>(m == 0 ? P.rk : P.rv);

  // frequencies of this lane's pairs (keys only)
  unsigned long long F[EMAX][RL];
#pragma unroll
  for (int e = 0; e < EMAX; ++e)
#pragma unroll
    for (int j = 0; j < RL; ++j) {
      const int i = (q + e * P.G) * RL + j;
      F[e][j] = (m == 0 && i < half) ? P.turns[i] : 0ull;
    }

  float acc_cos = 0.f, acc_res = 0.f, acc_yy = 0.f;
  float csum[EMAX][2 * RL];
#pragma unroll
  for (int e = 0; e < EMAX; ++e)
#pragma unroll
    for (int j = 0; j < 2 * RL; ++j) csum[e][j] = 0.f;

  // One token's row: fold the lane's runs into the per-token sums and the
  // content-space sums.  a = mapped, y = reference, both [EMAX][2 RL] fp32.
  auto fold = [&](const float (&a)[EMAX][2 * RL], const float (&y)[EMAX][2 * RL], bool on,
                  uint32_t pt) {
    float dot = 0.f, aa = 0.f, yy = 0.f, res = 0.f;
#pragma unroll
    for (int e = 0; e < EMAX; ++e)
#pragma unroll
      for (int j = 0; j < 2 * RL; ++j) {
        dot = fmaf(a[e][j], y[e][j], dot);
        aa = fmaf(a[e][j], a[e][j], aa);
        yy = fmaf(y[e][j], y[e][j], yy);
        const float df = y[e][j] - a[e][j];
        res = fmaf(df, df, res);
      }
    // content space: keys un-rotated at p' (multiply by exp(-j p' w_i))
    if (m == 0) {
#pragma unroll
      for (int e = 0; e < EMAX; ++e)
#pragma unroll
        for (int j = 0; j < RL; ++j) {
          float c, s;
          rope_cs(pt, F[e][j], c, s);   // exact fixed-point phase
          const float y0 = y[e][j], y1 = y[e][RL + j];
          csum[e][j] += fmaf(y0, c, y1 * s);
          csum[e][RL + j] += fmaf(y1, c, -y0 * s);
        }
    } else {
#pragma unroll
      for (int e = 0; e < EMAX; ++e)
#pragma unroll
        for (int j = 0; j < 2 * RL; ++j) csum[e][j] += y[e][j];
    }
    // per-token sums over the row's G lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      if (o >= P.G) break;
      dot += __shfl_xor_sync(0xffffffffu, dot, o);
      aa += __shfl_xor_sync(0xffffffffu, aa, o);
      yy += __shfl_xor_sync(0xffffffffu, yy, o);
      res += __shfl_xor_sync(0xffffffffu, res, o);
    }
    if (on) {
      if (aa > 0.f && yy > 0.f) acc_cos += dot * rsqrtf(aa) * rsqrtf(yy);
      acc_res += res;
      acc_yy += yy;
    }
  };

  // Every lane runs every iteration (the shuffles need the whole warp);
  // lanes without a token or a row contribute zeros.
  if constexpr (VEC && EMAX == 1) {
    // Each thread streams its own 16-byte words into a ring of kStages
    // shared-memory stages with cp.async (kStages - 1 tokens in flight per
    // thread, no registers held by loads in flight), reading back the
    // oldest stage; no barrier is needed, every thread reads only what it
    // copied.  Tokens past the chunk and rows that are skipped copy zeros.
    constexpr int kNV = RL * (int)sizeof(T) / 16;   // 16-byte words per half run
    constexpr int kW = 4 * kNV;                      // words per token: a lo, a hi, y lo, y hi
    constexpr int kS = kStages<T>;
    extern __shared__ uint4 ring[];                  // [kS][kW][blockDim.x]
    const int nt = blockDim.x;
    const int iters = (n + P.tok_par - 1) / P.tok_par;
    auto issue = [&](int it) {
      const int i = it * P.tok_par + tl;
      const int64_t row = (lane_on && i < n) ? s_row[i] : -1;
      const bool run_on = row >= 0 && q < P.NR;
      const int64_t off =
          run_on ? (((int64_t)lt * p.dst_rows + row) * p.H + h) * p.d + (int64_t)q * RL : 0;
      const uint4 *src[4] = {reinterpret_cast<const uint4 *>(mapped + off),
                             reinterpret_cast<const uint4 *>(mapped + off + half),
                             reinterpret_cast<const uint4 *>(ref + off),
                             reinterpret_cast<const uint4 *>(ref + off + half)};
      uint4 *dst = ring + (size_t)(it % kS) * kW * nt + tid;
#pragma unroll
      for (int w = 0; w < 4; ++w)
#pragma unroll
        for (int v = 0; v < kNV; ++v)
          cp_async16(dst + (size_t)(w * kNV + v) * nt, src[w] + v, run_on ? 16u : 0u);
      cp_async_commit();
    };
#pragma unroll 1
    for (int it = 0; it < kS - 1; ++it) issue(it);
#pragma unroll 1
    for (int it = 0; it < iters; ++it) {
      issue(it + kS - 1);
      cp_async_wait<kS - 1>();
      const uint4 *src = ring + (size_t)(it % kS) * kW * nt + tid;
      float a[1][2 * RL], y[1][2 * RL];
#pragma unroll
      for (int v = 0; v < kNV; ++v) {
        constexpr int kPer = 16 / (int)sizeof(T);
        unpack16<T>(src[(size_t)(0 * kNV + v) * nt], &a[0][v * kPer]);
        unpack16<T>(src[(size_t)(1 * kNV + v) * nt], &a[0][RL + v * kPer]);
        unpack16<T>(src[(size_t)(2 * kNV + v) * nt], &y[0][v * kPer]);
        unpack16<T>(src[(size_t)(3 * kNV + v) * nt], &y[0][RL + v * kPer]);
      }
      const int i = it * P.tok_par + tl;
      const int64_t row = (lane_on && i < n) ? s_row[i] : -1;
      fold(a, y, row >= 0, row >= 0 ? (uint32_t)s_pt[i] : 0u);
    }
    cp_async_wait<0>();
  } else {
    for (int base = 0; base < n; base += P.tok_par) {
      const int i = base + tl;
      const int64_t row = (lane_on && i < n) ? s_row[i] : -1;
      const bool on = row >= 0;
      const uint32_t pt = on ? (uint32_t)s_pt[i] : 0u;
      float a[EMAX][2 * RL], y[EMAX][2 * RL];
#pragma unroll
      for (int e = 0; e < EMAX; ++e) {
        const int r = q + e * P.G;
        if (on && r < P.NR) {
          const int64_t off = (((int64_t)lt * p.dst_rows + row) * p.H + h) * p.d + (int64_t)r * RL;
          load_run<T, RL, VEC>(mapped + off, a[e]);
          load_run<T, RL, VEC>(mapped + off + half, a[e] + RL);
          load_run<T, RL, VEC>(ref + off, y[e]);
          load_run<T, RL, VEC>(ref + off + half, y[e] + RL);
        } else {
#pragma unroll
          for (int j = 0; j < 2 * RL; ++j) a[e][j] = y[e][j] = 0.f;
        }
      }
      fold(a, y, on, pt);
    }
  }

  // ---- add into the fp64 output ------------------------------------------
  if (!lane_on) return;
  double *st = P.stats + (((int64_t)lt * p.H + h) * 2 + m) * (p.d + 4);
  if (q == 0) {
    if (tl == 0 && s_count) atomicAdd(st, (double)s_count);
    atomicAdd(st + 1, (double)acc_cos);
    atomicAdd(st + 2, (double)acc_res);
    atomicAdd(st + 3, (double)acc_yy);
  }
#pragma unroll
  for (int e = 0; e < EMAX; ++e) {
    const int r = q + e * P.G;
    if (r >= P.NR) continue;
#pragma unroll
    for (int j = 0; j < RL; ++j) {
      atomicAdd(st + 4 + r * RL + j, (double)csum[e][j]);
      atomicAdd(st + 4 + half + r * RL + j, (double)csum[e][RL + j]);
    }
  }
}

__global__ void zero_kernel(double *x, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    x[i] = 0.0;
}

int next_pow2(int x) {
  int g = 1;
  while (g < x) g <<= 1;
  return g;
}

}  // namespace

extern "C" kvx_status kvx_kv_diagnostics(const kvx_plan *plan, const kvx_diag_args *a,
                                         void *stream) {
  if (!plan || !a) return KVX_ERR_INVALID_ARG;
  const kvx_plan_desc &d = plan->desc;
  if (a->ntok < 0 || a->ntok > INT32_MAX || a->num_requests < 1 ||
      (!a->cu_seqlens && a->num_requests != 1) || !a->mapped_k || !a->mapped_v || !a->ref_k ||
      !a->ref_v || !a->stats)
    return KVX_ERR_INVALID_ARG;
  if (d.dst_layout == KVX_CONTIGUOUS ? a->dst_capacity < 1
                                     : (a->num_blocks < 1 || !a->block_table ||
                                        a->max_blocks_per_req < 1))
    return KVX_ERR_INVALID_ARG;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return KVX_ERR_CUDA;
  if (cur != plan->device) return KVX_ERR_INVALID_ARG;

  DiagParams P;
  std::memset(&P, 0, sizeof(P));
  KvxParams &p = P.p;
  p.cu_seqlens = a->cu_seqlens;
  p.src_pos = a->src_pos;
  p.tgt_pos = a->tgt_pos;
  p.tgt_offset = a->tgt_offset;
  p.block_table = a->block_table;
  p.status = a->status;
  p.ntok = a->ntok;
  p.dst_capacity = a->dst_capacity;
  p.num_blocks = a->num_blocks;
  p.dst_rows = d.dst_layout == KVX_CONTIGUOUS ? (int64_t)a->num_requests * a->dst_capacity
                                              : a->num_blocks * (int64_t)d.block_size;
  p.R = a->num_requests;
  p.max_blocks = a->max_blocks_per_req;
  p.Ls = d.src_layers;
  p.Lt = d.tgt_layers;
  p.H = d.tgt_kv_heads;
  p.d = d.tgt_head_dim;
  p.k = d.k;
  p.layout = d.dst_layout;
  p.block_size = d.block_size;
  p.max_position = d.max_position;
  p.src_layout = KVX_CONTIGUOUS;   // the source is not read: target-side rules only
  p.src_rows = a->ntok;
  P.mk = a->mapped_k;
  P.mv = a->mapped_v;
  P.rk = a->ref_k;
  P.rv = a->ref_v;
  P.stats = a->stats;
  std::memcpy(P.turns, plan->turns_tgt, sizeof(P.turns));

  cudaStream_t s = (cudaStream_t)stream;
  const int half = p.d / 2;
  const int64_t nstats = (int64_t)p.Lt * p.H * 2 * (p.d + 4);
  const int zb = (int)((nstats + 255) / 256 < 1024 ? (nstats + 255) / 256 : 1024);

  // lanes: runs of 8 pairs when half is a multiple of 8 (16- or 32-byte
  // loads), else single pairs, up to 32 lanes per row and EMAX runs a lane
  const bool bf = d.kv_dtype == KVX_BF16;
  const bool aligned = ((((uintptr_t)a->mapped_k | (uintptr_t)a->mapped_v |
                          (uintptr_t)a->ref_k | (uintptr_t)a->ref_v) & 15u) == 0);
  const bool runs8 = half % 8 == 0;
  const int RL = runs8 ? 8 : 1;
  P.NR = half / RL;
  P.G = next_pow2(P.NR < 32 ? P.NR : 32);
  const int lanes = 2 * p.H * P.G;
  P.lanes_per_token = lanes;
  if (lanes <= kThreads) {
    P.tok_par = kThreads / lanes;
    P.slot_groups = 1;
  } else {
    P.tok_par = 1;
    P.slot_groups = (lanes + kThreads - 1) / kThreads;
  }
  // whole warps: lanes past tok_par * lanes are idle but join the shuffles
  const int nthreads = lanes <= kThreads ? (P.tok_par * lanes + 31) / 32 * 32 : kThreads;

  // chunk: the largest of 1024..64 tokens that still gives ~8 CTAs per SM
  const int64_t want = (int64_t)plan->num_sms * 8;
  int chunk = kMaxChunk;
  while (chunk > 64 &&
         ((p.ntok + chunk - 1) / chunk) * (int64_t)p.Lt * P.slot_groups < want)
    chunk >>= 1;
  P.chunk = chunk;
  const int64_t gy = (int64_t)p.Lt * P.slot_groups;
  const int64_t gx = (p.ntok + chunk - 1) / chunk;
  if (gy > 65535 || gx > INT32_MAX) return KVX_ERR_UNSUPPORTED;  // before any launch
  dim3 grid((unsigned)gx, (unsigned)gy);

  zero_kernel<<<zb, 256, 0, s>>>(a->stats, nstats);
  if (cudaGetLastError() != cudaSuccess) return KVX_ERR_CUDA;
  if (a->ntok == 0) return KVX_OK;

  void *fn;
  using bf16 = __nv_bfloat16;
  if (runs8) {
    if (bf) fn = aligned ? (void *)&kv_diag_kernel<bf16, 8, 1, true>
                         : (void *)&kv_diag_kernel<bf16, 8, 1, false>;
    else fn = aligned ? (void *)&kv_diag_kernel<float, 8, 1, true>
                      : (void *)&kv_diag_kernel<float, 8, 1, false>;
  } else {
    // half <= 128 single pairs over at most 32 lanes: 4 runs a lane
    fn = bf ? (void *)&kv_diag_kernel<bf16, 1, 4, false>
            : (void *)&kv_diag_kernel<float, 1, 4, false>;
  }
  // the 16-byte-word instances stream through a cp.async ring in dynamic
  // shared memory
  size_t dyn = 0;
  if (runs8 && aligned) {
    dyn = bf ? ring_bytes<bf16>(nthreads) : ring_bytes<float>(nthreads);
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn) !=
        cudaSuccess)
      return KVX_ERR_CUDA;
  }
  void *args[] = {&P};
  return cudaLaunchKernel(fn, grid, dim3(nthreads), args, dyn, s) == cudaSuccess ? KVX_OK
                                                                                 : KVX_ERR_CUDA;
}
