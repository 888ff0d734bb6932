// kvx_moments.cuh -- centred second moments (Gram and cross blocks) on the
// 5th-generation tensor cores with split-precision operands, shared by the
// ridge fit (kvx_ridge.cu) and the layer-selection scores (kvx_scores.cu).
//
// The ridge demo of the Qwen3 14B -> 32B article (section "Линейного моста,
// как ни странно, хватает") solves (XcT Xc + lam I) W = XcT Yc: the Gram and
// cross blocks are dense contractions over the observations.  A tf32 operand
// keeps 11 significant bits, too few for a matrix that the solve multiplies by
// its condition number, so every centred fp32 value v is split into two tf32
// values, hi = tf32(v) and lo = tf32(v - hi) (v = hi + lo to 2^-22 of |v|),
// and each product is formed as hi*hi + hi*lo + lo*hi (the lo*lo term,
// 2^-22 of the product, is dropped): the "3xTF32" method of Ootomo and
// Yokota, "Recovering single precision accuracy from Tensor Cores while
// surpassing the FP32 theoretical peak performance" (2022).
//
// Data path:
//   * a split pass (one per user) writes the centred values as two planes,
//     hi and lo, K-major: plane row r holds one feature (or output) over the
//     observations of a chunk, [2][R][np] fp32, np a multiple of 32; padded
//     observations are zero;
//   * moments_kernel: persistent, one CTA per SM, 10 warps.  Work item =
//     (128 x 128 output tile, slice of 4,096 observations).  A producer
//     thread brings, per block of 32 observations, the tile's A rows (hi,
//     lo) and B rows (hi, lo) with 2-D TMA boxes [128 rows][32 obs] (128-byte
//     swizzle = the UMMA K-major layout) into a 3-stage ring; one thread of
//     the MMA warp issues 4 K steps x 3 tcgen05.mma.kind::tf32 (M = N = 128,
//     K = 8, fp32 accumulation in tensor memory) per block; every 8 blocks
//     (256 observations) the accumulator (one of two, 128 columns each) goes
//     to 8 epilogue warps, which add it into fp32 registers (each thread one
//     row, 64 columns); at the end of the item the sums go to the fp64
//     output with atomics.  The fp32 accumulation thus mirrors the CUDA-core
//     path it replaces: fp32 partial sums over 256 observations, summed in
//     fp32 over a slice, slices added in fp64.
// Every mbarrier wait is bounded (2 s without progress sets
// KVX_FLAG_TIMEOUT, the roles leave their loops, in-flight copies and MMAs
// are drained, tensor memory is freed).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvx.h"
#include "kvx_internal.h"
#include "kvx_ptx.cuh"

namespace {

constexpr int kMomRows = 128;                         // M = N of a tile
constexpr int kMomKB = 32;                            // observations per block (128 B of fp32)
constexpr int kMomFlushKB = 8;                        // blocks per tensor-memory partial sum
constexpr int kMomSliceKB = 128;                      // blocks per work item
constexpr int kMomChunk = 16384;                      // observations per plane buffer
constexpr int kMomStages = 3;
constexpr int kMomOpBytes = kMomRows * kMomKB * 4;    // one operand box: 16 KB
constexpr int kMomStageBytes = 4 * kMomOpBytes;       // A hi, A lo, B hi, B lo
constexpr int kMomEpiWarps = 8;
constexpr int kMomThreads = (2 + kMomEpiWarps) * 32;  // producer, MMA, epilogue
constexpr int kMomTmemCols = 2 * kMomRows;
constexpr uint64_t kMomWaitNs = 2000000000ull;        // 2 s without progress

// Instruction descriptor, kind::tf32: D fp32, A and B tf32, both K-major,
// N = 128, M = 128.
constexpr uint32_t kMomIdesc = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(kMomRows >> 3) << 17) |
                               ((uint32_t)(kMomRows >> 4) << 24);

// One output tile: rows a_row.. of the planes against rows b_row.. .
struct MomTile {
  int a_row, b_row;      // first plane row of the A block and of the B block
  int m_valid;           // tile rows that are outputs
  int n_split, n_valid;  // columns [0, n_split) go to out0, [n_split, n_valid) to out1
  double *out0;          // element (r, c) at out0[r * ld0 + c]
  double *out1;          // element (r, c) at out1[r * ld1 + c - n_split]
  int64_t ld0, ld1;
};

struct MomShared {
  uint64_t full[kMomStages], empty[kMomStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  volatile int abort;
};

__host__ __device__ constexpr size_t mom_smem_bytes() {
  return (size_t)kMomStages * kMomStageBytes + 1024 + sizeof(MomShared);
}

struct MomWaiter {
  MomShared *sh;
  uint32_t *status;
  // Bounded wait; false means the pipeline is being abandoned.
  __device__ __forceinline__ bool wait(uint64_t *bar, uint32_t parity) const {
    const uint32_t a = smem_addr(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
      if (mbar_try_wait(a, parity)) return true;
      if (sh->abort) return false;
      if (globaltimer() - t0 > kMomWaitNs) {
        sh->abort = 1;
        if (status) atomicOr(status, KVX_FLAG_TIMEOUT);
        return false;
      }
    }
  }
  __device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity) const {
    const bool ok = wait(bar, parity);
    return __all_sync(0xffffffffu, ok) != 0;
  }
};

// Bounded wait used while draining: ignores the abort flag.
__device__ __forceinline__ void mom_drain_wait(uint64_t *bar, uint32_t parity) {
  const uint32_t a = smem_addr(bar);
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(a, parity) && globaltimer() - t0 < kMomWaitNs) {
  }
}

__device__ __forceinline__ void mom_mma(uint32_t d_tmem, uint64_t a, uint64_t b,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %3, 0;\n"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %4, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(accumulate), "r"(kMomIdesc)
      : "memory");
}
// Arrival on `bar` once every MMA this thread issued so far is complete.
__device__ __forceinline__ void mom_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
// 32 lanes x 32 bits, 32 repetitions: register j holds column (col + j) of
// the thread's lane.
__device__ __forceinline__ void tc_ld32x32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}

// v as a tf32 value (round to nearest, ties away) in an fp32 register.
__device__ __forceinline__ float to_tf32(float v) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(v));
  return __uint_as_float(r);
}
// Write centred value v of plane row `row`, observation column `col`, as its
// hi and lo parts.
__device__ __forceinline__ void mom_put(float *planes, int64_t R, int64_t np, int64_t row,
                                        int64_t col, float v) {
  const float hi = to_tf32(v);
  const float lo = to_tf32(v - hi);
  planes[row * np + col] = hi;
  planes[(R + row) * np + col] = lo;
}

// Work items: slice-major, then tile, so that the CTAs running at the same
// time stream the same blocks of observations of neighbouring tiles (the
// operands they share stay in L2).
template <typename Tiles>
__global__ void __launch_bounds__(kMomThreads, 1)
    moments_kernel(const __grid_constant__ CUtensorMap map, int R, int kb_total, int slices,
                   int num_tiles, const Tiles tiles, uint32_t *status) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *sbuf = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  MomShared *sh = reinterpret_cast<MomShared *>(sbuf + (size_t)kMomStages * kMomStageBytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long items = (long long)num_tiles * slices;

  if (tid == 0) {
    for (int s = 0; s < kMomStages; ++s) {
      mbar_init(smem_addr(&sh->full[s]), 1);
      mbar_init(smem_addr(&sh->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_addr(&sh->acc_full[b]), 1);
      mbar_init(smem_addr(&sh->acc_empty[b]), kMomEpiWarps);
    }
    mbar_init(smem_addr(&sh->drain), 1);
    sh->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&sh->tmem_base)),
                 "r"(kMomTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;
  const MomWaiter W{sh, status};

  if (warp == 0) {
    // ------------------------------------------------------------------
    // producer (one thread): A hi, A lo, B hi, B lo boxes per block
    // ------------------------------------------------------------------
    if (lane == 0) {
      uint32_t x_seq = 0;
      for (long long it = blockIdx.x; it < items; it += gridDim.x) {
        const int s = (int)(it / num_tiles);
        const MomTile t = tiles.tile((int)(it % num_tiles));
        const int kb0 = s * kMomSliceKB;
        const int kb1 = min(kb0 + kMomSliceKB, kb_total);
        for (int kb = kb0; kb < kb1; ++kb) {
          const int stage = (int)(x_seq % kMomStages);
          if (!W.wait(&sh->empty[stage], ((x_seq / kMomStages) & 1) ^ 1)) goto producer_done;
          const uint32_t bar = smem_addr(&sh->full[stage]);
          const uint32_t dst = smem_addr(sbuf + (size_t)stage * kMomStageBytes);
          mbar_expect_tx(bar, kMomStageBytes);
          const int x = kb * kMomKB;
          tma_load_2d(dst, &map, x, t.a_row, bar);
          tma_load_2d(dst + kMomOpBytes, &map, x, R + t.a_row, bar);
          tma_load_2d(dst + 2 * kMomOpBytes, &map, x, t.b_row, bar);
          tma_load_2d(dst + 3 * kMomOpBytes, &map, x, R + t.b_row, bar);
          ++x_seq;
        }
      }
    producer_done:
      // the last stages may still be in flight
      for (uint32_t n = (x_seq > (uint32_t)kMomStages ? x_seq - kMomStages : 0); n < x_seq; ++n)
        mom_drain_wait(&sh->full[n % kMomStages], (n / kMomStages) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------
    // MMA issuer: the warp waits, lane 0 issues and commits
    // ------------------------------------------------------------------
    uint32_t x_seq = 0, a_seq = 0;
    bool issued = false;
    const uint64_t d0 = sw128_desc(smem_addr(sbuf));
    for (long long it = blockIdx.x; it < items; it += gridDim.x) {
      const int s = (int)(it / num_tiles);
      const int kb0 = s * kMomSliceKB;
      const int kb1 = min(kb0 + kMomSliceKB, kb_total);
      for (int g0 = kb0; g0 < kb1; g0 += kMomFlushKB) {
        const int buf = (int)(a_seq & 1);
        if (!W.warp_wait(&sh->acc_empty[buf], ((a_seq >> 1) & 1) ^ 1)) goto mma_done;
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(buf * kMomRows);
        const int g1 = min(g0 + kMomFlushKB, kb1);
        for (int kb = g0; kb < g1; ++kb) {
          const int stage = (int)(x_seq % kMomStages);
          if (!W.warp_wait(&sh->full[stage], (x_seq / kMomStages) & 1)) goto mma_done;
          tc_fence_after();
          if (lane == 0) {
            const uint64_t a_hi = d0 + (uint64_t)(((size_t)stage * kMomStageBytes) >> 4);
            const uint64_t a_lo = a_hi + (uint64_t)(kMomOpBytes >> 4);
            const uint64_t b_hi = a_hi + (uint64_t)((2 * kMomOpBytes) >> 4);
            const uint64_t b_lo = a_hi + (uint64_t)((3 * kMomOpBytes) >> 4);
#pragma unroll
            for (int ks = 0; ks < kMomKB / 8; ++ks) {   // K = 8 tf32 = 32 bytes per step
              const uint64_t o = (uint64_t)(2 * ks);
              mom_mma(d_tmem, a_hi + o, b_hi + o, (kb > g0 || ks > 0) ? 1u : 0u);
              mom_mma(d_tmem, a_hi + o, b_lo + o, 1u);
              mom_mma(d_tmem, a_lo + o, b_hi + o, 1u);
            }
            mom_commit(smem_addr(&sh->empty[stage]));
          }
          __syncwarp();
          issued = true;
          ++x_seq;
        }
        if (lane == 0) mom_commit(smem_addr(&sh->acc_full[buf]));
        __syncwarp();
        ++a_seq;
      }
    }
  mma_done:
    if (issued) {
      if (lane == 0) {
        mom_commit(smem_addr(&sh->drain));
        mom_drain_wait(&sh->drain, 0);
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------------
    // epilogue: per 256 observations, accumulator -> fp32 registers; per
    // item, registers -> fp64 output
    // ------------------------------------------------------------------
    const int ew = warp - 2;                   // 0..7
    const int quad = warp & 3;                 // tensor-memory lane quadrant of this warp
    const int half = ew >> 2;                  // columns [64 half, 64 half + 64)
    const int row = quad * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    uint32_t a_seq = 0;
    float acc[64];
#pragma unroll
    for (int c = 0; c < 64; ++c) acc[c] = 0.f;
    for (long long it = blockIdx.x; it < items; it += gridDim.x) {
      const int s = (int)(it / num_tiles);
      const int kb0 = s * kMomSliceKB;
      const int kb1 = min(kb0 + kMomSliceKB, kb_total);
      bool ok = true;
      for (int g0 = kb0; g0 < kb1; g0 += kMomFlushKB) {
        const int buf = (int)(a_seq & 1);
        if (!W.warp_wait(&sh->acc_full[buf], (a_seq >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t col = tmem + lane_base + (uint32_t)(buf * kMomRows + 64 * half);
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          uint32_t v[32];
          tc_ld32x32(col + 32 * h2, v);
          tc_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) acc[32 * h2 + j] += __uint_as_float(v[j]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&sh->acc_empty[buf]));
        ++a_seq;
      }
      if (!ok) break;
      const MomTile t = tiles.tile((int)(it % num_tiles));
      if (row < t.m_valid) {
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const int cc = 64 * half + c;
          if (cc < t.n_split)
            atomicAdd(t.out0 + (int64_t)row * t.ld0 + cc, (double)acc[c]);
          else if (cc < t.n_valid)
            atomicAdd(t.out1 + (int64_t)row * t.ld1 + (cc - t.n_split), (double)acc[c]);
        }
      }
#pragma unroll
      for (int c = 0; c < 64; ++c) acc[c] = 0.f;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kMomTmemCols)
                 : "memory");
}

// 2-D TMA map over the planes [2 R][np] fp32: box [128 rows][32 obs], 128-byte
// swizzle, rows beyond 2 R read as zero.
inline bool mom_encode_map(CUtensorMap *map, const float *planes, int64_t R, int64_t np) {
  typedef CUresult (*EncodeFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                               const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                               const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                               CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static EncodeFn fn = reinterpret_cast<EncodeFn>(kvx_tc_encoder());
  if (!fn || np % kMomKB != 0 || (reinterpret_cast<uintptr_t>(planes) & 15u) != 0) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)np, (cuuint64_t)(2 * R)};
  const cuuint64_t strides[1] = {(cuuint64_t)np * 4};
  const cuuint32_t box[2] = {(cuuint32_t)kMomKB, (cuuint32_t)kMomRows};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(planes), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Adds the moments of the chunk held in `planes` ([2][R][np], np a multiple
// of 32) to the fp64 outputs named by `tiles` (num_tiles tiles).
template <typename Tiles>
cudaError_t mom_launch(const float *planes, int64_t R, int64_t np, const Tiles &tiles,
                       int num_tiles, uint32_t *status, cudaStream_t s) {
  CUtensorMap map;
  if (!mom_encode_map(&map, planes, R, np)) return cudaErrorInvalidValue;
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return cudaErrorUnknown;
  }
  const int kb_total = (int)(np / kMomKB);
  const int slices = (kb_total + kMomSliceKB - 1) / kMomSliceKB;
  const long long items = (long long)num_tiles * slices;
  if (items <= 0) return cudaSuccess;
  const int grid = (int)(items < sms ? items : sms);
  cudaError_t e = cudaFuncSetAttribute(moments_kernel<Tiles>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)mom_smem_bytes());
  if (e != cudaSuccess) return e;
  moments_kernel<Tiles><<<grid, kMomThreads, mom_smem_bytes(), s>>>(map, (int)R, kb_total, slices,
                                                                    num_tiles, tiles, status);
  return cudaGetLastError();
}

}  // namespace
