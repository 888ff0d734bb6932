// kvx_wide.cu -- the wide-feature mapper on the 5th-generation tensor cores.
//
// The Qwen3 14B -> 32B article ("Перенос KV-кэша между моделями Qwen3 вместо
// повторного префилла", section "Ограничения, важные в продакшене") sizes its
// mapper at about 1.07e9 parameters, 4 GB per direction: 2^30 = 64 target
// layers x 8192 features x 2048 outputs, i.e. one dense map per target layer
// over all heads' keys and values of the k = 4 selected source layers
// (4 x 2 x 8 x 128 = 8192) to all heads' keys and values of the target layer
// (8 x 2 x 128 = 2048).  The steps are those of the per-head transfer
// ("Helm Intelligent Routing", "Why carrying the cache across is the hard
// part", steps 1-3: un-rotate, map, re-rotate; install into the cache), with
// Y[T x N] = X[T x F] . W[lt][F x N] + b[lt] as the map.  That is a large
// dense contraction per target layer (2 T F N flops), so it runs as a
// persistent tcgen05 GEMM on CTA pairs:
//
//  1. wide_unrotate_kernel: the keys of every source layer, un-rotated out of
//     the source RoPE at their source positions (fp32, angles from the exact
//     fixed-point phase), rounded once to bf16 into the plan's buffer
//     [Ls][max_tokens][H][d].  Values need no transform.
//  2. wide_w_image_kernel: W [Lt][F][N] -> bf16 chunks [256 n][64 k] in the
//     128-byte-swizzled K-major layout of the MMA's B operand, chunk
//     (lt, head, 64-feature step); b -> fp32.
//  3. wide_map_kernel: tile = (target layer lt, 256 tokens, output head h):
//     M = 256 tokens (128 per CTA of the pair), N = 256 (head h's key and
//     value columns: CTA rank 0 holds the key rows of B, rank 1 the value
//     rows), K = F in steps of 64 features.  Per step each CTA's producer
//     thread brings A (TMA box [128 tokens][64 dims] of the un-rotated key or
//     value cache of source layer idx[lt][j], head h', half) and its half of
//     B (16 KB bulk copy) into a ring of shared-memory stages; rank 0's MMA
//     warp issues four tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16,
//     both operands from shared memory) into one of two 256-column fp32
//     accumulators in tensor memory.  Eight epilogue warps per CTA read their
//     token rows back (tcgen05.ld), add b, re-rotate the key half into the
//     target RoPE at p' (step 3), cast to bf16 and store 32-byte sectors into
//     the contiguous or paged cache.
// Every mbarrier wait is bounded (2 s without progress): the CTA then sets
// KVX_FLAG_TIMEOUT, leaves its loops, drains in-flight copies and MMAs with
// bounded waits and frees tensor memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvx_device.cuh"
#include "kvx_internal.h"
#include "kvx_ptx.cuh"

namespace {

constexpr int kWD = 128;                       // head_dim of this path
constexpr int kWHalf = kWD / 2;
constexpr int kWRows = 128;                    // tokens per CTA per tile
constexpr int kWN = 256;                       // outputs per tile (one head's K and V)
constexpr int kWKStep = 64;                    // features per stage
constexpr int kWHalfBytes = kWRows * kWKStep * 2;   // 16 KB: A of one CTA, or its half of B
constexpr int kWStageBytes = 2 * kWHalfBytes;       // A + B half
constexpr int kWChunkBytes = 2 * kWHalfBytes;       // B image chunk [256 n][64 k]
constexpr int kWMaxStages = 7;
constexpr int kWSmemLimit = 232448;            // 227 KB opt-in per CTA
constexpr int kWTmemCols = 512;                // two 256-column accumulators
constexpr int kWProducerWarp = 0;
constexpr int kWMmaWarp = 1;                   // rank 0: MMA issuer; rank 1: forwarder
constexpr int kWEpiWarp0 = 2;
constexpr int kWEpiWarps = 8;
constexpr int kWThreads = (kWEpiWarp0 + kWEpiWarps) * 32;   // 320
constexpr uint64_t kWWaitNs = 2000000000ull;   // 2 s without progress
constexpr int kWSyncSteps = 16;                // feature steps per lockstep epoch
constexpr int kWSyncLag = 2;                   // epochs a producer may run ahead of the mean
constexpr uint64_t kWPaceGiveUpNs = 1000000ull; // 1 ms: pacing gives way to progress

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major,
// N = 256, M = 256 (CTA pair).
constexpr uint32_t kWIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                             ((uint32_t)(kWN >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);

struct WideTurns {
  unsigned long long f[kWHalf];   // RoPE frequencies, 2^-64 turns per position
};

struct WideGeom {
  int mt_count;          // 256-token tiles
  int nt_count;          // output heads (one tile column each)
  int kc_count;          // 64-feature steps: F / 64 = 4 k H
  int stages;
  long long num_tiles;   // Lt * mt_count * nt_count
  long long stride;      // CTA pairs
  // Loose lockstep of the producers (see wide_map_kernel): a counter of the
  // epochs (kWSyncSteps feature steps each) every producer has issued,
  // cleared by the W-image kernel; a producer issues epoch e only once the
  // producers together have issued (e - kWSyncLag) epochs each on average.
  unsigned int *sync;
  int epochs_per_tile;
  int max_epochs;        // epochs of a producer with the most tiles
};

struct WShared {
  uint64_t full[kWMaxStages], empty[kWMaxStages], peer_full[kWMaxStages];
  uint64_t d_full[2], d_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  volatile int abort;
};

struct WWaiter {
  WShared *sh;
  uint32_t *status;
  // Bounded wait; false means the pipeline is being abandoned.
  __device__ __forceinline__ bool wait(uint64_t *bar, uint32_t parity) const {
    const uint32_t a = smem_addr(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
      if (mbar_try_wait(a, parity)) return true;
      if (sh->abort) return false;
      if (globaltimer() - t0 > kWWaitNs) {
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
__device__ __forceinline__ void wdrain_wait(uint64_t *bar, uint32_t parity) {
  const uint32_t a = smem_addr(bar);
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(a, parity) && globaltimer() - t0 < kWWaitNs) {
  }
}

// The lockstep counter: relaxed loads and reductions at GPU scope (it paces
// the producers and orders no data).
__device__ __forceinline__ unsigned long long ld_relaxed_gpu(const unsigned int *p) {
  unsigned int v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_add_gpu(unsigned int *p, unsigned int v) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// The four MMAs of one 64-feature stage: A and B descriptors advance by
// 32 bytes (16 features) inside the 128-byte swizzle rows.  One elected lane
// of the converged warp issues; the CTA pair runs each as one M = 256 MMA.
__device__ __forceinline__ void wide_mma4_elect(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred e, p, t;\n.reg .b32 r;\n.reg .b64 a1, a2, a3, b1, b2, b3;\n"
      "elect.sync r|e, 0xffffffff;\n"
      "setp.ne.b32 p, %3, 0;\n"
      "setp.eq.u32 t, 0, 0;\n"
      "add.u64 a1, %1, 2; add.u64 a2, %1, 4; add.u64 a3, %1, 6;\n"
      "add.u64 b1, %2, 2; add.u64 b2, %2, 4; add.u64 b3, %2, 6;\n"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %4, p;\n"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a1, b1, %4, t;\n"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a2, b2, %4, t;\n"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a3, b3, %4, t;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(accumulate), "r"(kWIdesc)
      : "memory");
}

__device__ __forceinline__ void decode_tile(const WideGeom &g, long long t, int &lt, int &mt,
                                            int &nt) {
  nt = (int)(t % g.nt_count);
  const long long q = t / g.nt_count;
  mt = (int)(q % g.mt_count);
  lt = (int)(q / g.mt_count);
}

// ---------------------------------------------------------------------------
// The map kernel (CTA pairs, persistent)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kWThreads, 1)
    wide_map_kernel(const __grid_constant__ KvxParams p,
                    const __grid_constant__ CUtensorMap map_key,   // un-rotated keys
                    const __grid_constant__ CUtensorMap map_val,   // values as stored
                    const __grid_constant__ WideTurns rope_tgt,
                    const float *__restrict__ bias_f32, const unsigned char *__restrict__ w_img,
                    const WideGeom geo) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *sbuf = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  WShared *sh = reinterpret_cast<WShared *>(sbuf + (size_t)geo.stages * kWStageBytes);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const long long pair = blockIdx.x >> 1;

  if (tid == 0) {
    for (int s = 0; s < geo.stages; ++s) {
      mbar_init(smem_addr(&sh->full[s]), 1);
      mbar_init(smem_addr(&sh->empty[s]), 1);
      mbar_init(smem_addr(&sh->peer_full[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_addr(&sh->d_full[b]), 1);
      mbar_init(smem_addr(&sh->d_empty[b]), kWEpiWarps * 2);
    }
    mbar_init(smem_addr(&sh->drain), 1);
    sh->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kWMmaWarp) {
    // one warp in each CTA of the pair allocates (the same columns)
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&sh->tmem_base)),
                 "r"(kWTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  const bool seq_ok = kvx::seqlens_ok(p, tid, kWThreads);
  cluster_sync();   // the peer's barriers are initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;
  const WWaiter W{sh, p.status};

  if (!seq_ok) {
    if (blockIdx.x == 0 && tid == 0) kvx::report(p, KVX_FLAG_BAD_SEQLENS);
  } else if (warp == kWProducerWarp) {
    // ------------------------------------------------------------------
    // producer (one thread per CTA): A box + this CTA's half of B per stage
    // ------------------------------------------------------------------
    if (lane == 0) {
      uint32_t x_seq = 0;
      // Loose lockstep: every producer streams K in the same order, so the
      // 76 pairs together touch only the current feature slices of ~10 token
      // blocks and 8 W blocks when they stay close; left alone they drift
      // apart by whole tiles and the distinct operands of a wave (~70 MB)
      // no longer stay in L2.  Epochs already counted for this producer:
      uint32_t epochs = 0;
      const unsigned long long producers = 2ull * (unsigned long long)geo.stride;
      // Pacing is an optimisation only: a producer that has waited
      // kWPaceGiveUpNs for the others (say some pairs are not resident
      // because other work holds SMs) stops pacing for the rest of the
      // launch and runs free, so correctness never depends on co-residency.
      // Returns false only if the pipeline is being abandoned.
      bool pacing = true;
      auto pace = [&]() -> bool {
        const long long ahead = (long long)epochs - kWSyncLag;
        if (!pacing || geo.sync == nullptr || ahead <= 0) return true;
        const unsigned long long need = producers * (unsigned long long)ahead;
        if (ld_relaxed_gpu(geo.sync) >= need) return true;
        const uint64_t t0 = globaltimer();
        while (ld_relaxed_gpu(geo.sync) < need) {
          if (sh->abort) return false;
          if (globaltimer() - t0 > kWPaceGiveUpNs) {
            pacing = false;
            return true;
          }
          __nanosleep(100);
        }
        return true;
      };
      for (long long t = pair; t < geo.num_tiles; t += geo.stride) {
        int lt, mt, nt;
        decode_tile(geo, t, lt, mt, nt);
        if (!kvx::layer_row_ok(p, lt)) {
          if (geo.sync) red_add_gpu(geo.sync, (unsigned)geo.epochs_per_tile);
          epochs += geo.epochs_per_tile;
          continue;
        }
        const int tok0 = mt * 2 * kWRows + (int)rank * kWRows;
        const unsigned char *img = w_img +
                                   ((int64_t)lt * geo.nt_count + nt) * geo.kc_count * kWChunkBytes +
                                   (int64_t)rank * kWHalfBytes;
        int kc = 0;
        // features in (j, m, h, i) order, 64 at a time
        for (int j = 0; j < p.k; ++j) {
          const int sl = __ldg(p.layer_idx + lt * p.k + j);
          for (int m = 0; m < 2; ++m) {
            const CUtensorMap *map = m == 0 ? &map_key : &map_val;
            for (int h = 0; h < p.H; ++h) {
              for (int hf = 0; hf < 2; ++hf, ++kc) {
                if (kc % kWSyncSteps == 0 && !pace()) goto producer_done;
                const int stage = (int)(x_seq % (uint32_t)geo.stages);
                if (!W.wait(&sh->empty[stage], ((x_seq / geo.stages) & 1) ^ 1)) goto producer_done;
                const uint32_t bar = smem_addr(&sh->full[stage]);
                const uint32_t dst = smem_addr(sbuf + (size_t)stage * kWStageBytes);
                mbar_expect_tx(bar, kWStageBytes);
                tma_load_4d(dst, map, hf * kWHalf, h, tok0, sl, bar);
                bulk_g2s(dst + kWHalfBytes, img + (int64_t)kc * kWChunkBytes, kWHalfBytes, bar);
                ++x_seq;
                if (kc % kWSyncSteps == kWSyncSteps - 1 || kc == geo.kc_count - 1) {
                  if (geo.sync) red_add_gpu(geo.sync, 1u);
                  ++epochs;
                }
              }
            }
          }
        }
      }
    producer_done:
      // retire: count the epochs this producer will not issue, so that no
      // other producer waits for them
      if (geo.sync && epochs < (uint32_t)geo.max_epochs)
        red_add_gpu(geo.sync, (uint32_t)geo.max_epochs - epochs);
      // drain: the last `stages` loads (at most) may still be in flight
      for (uint32_t n = (x_seq > (uint32_t)geo.stages ? x_seq - geo.stages : 0); n < x_seq; ++n)
        wdrain_wait(&sh->full[n % geo.stages], (n / geo.stages) & 1);
    }
  } else if (warp == kWMmaWarp) {
    if (rank == 0) {
      // ----------------------------------------------------------------
      // MMA issuer (rank 0, converged warp, one elected lane issues)
      // ----------------------------------------------------------------
      uint32_t x_seq = 0, d_seq = 0;
      bool issued = false;
      const uint64_t a0 = sw128_desc(smem_addr(sbuf));
      for (long long t = pair; t < geo.num_tiles; t += geo.stride) {
        int lt, mt, nt;
        decode_tile(geo, t, lt, mt, nt);
        if (!kvx::layer_row_ok(p, lt)) continue;
        const int buf = d_seq & 1;
        if (!W.warp_wait(&sh->d_empty[buf], ((d_seq >> 1) & 1) ^ 1)) goto mma_done;
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(buf * kWN);
        for (int kc = 0; kc < geo.kc_count; ++kc) {
          const int stage = (int)(x_seq % (uint32_t)geo.stages);
          const uint32_t par = (x_seq / geo.stages) & 1;
          if (!W.warp_wait(&sh->full[stage], par)) goto mma_done;
          if (!W.warp_wait(&sh->peer_full[stage], par)) goto mma_done;
          tc_fence_after();
          const uint64_t ad = a0 + (uint64_t)(((size_t)stage * kWStageBytes) >> 4);
          wide_mma4_elect(d_tmem, ad, ad + (uint64_t)(kWHalfBytes >> 4), kc > 0 ? 1u : 0u);
          issued = true;
          tc_commit_elect<2>(smem_addr(&sh->empty[stage]));   // both CTAs' stage is free
          ++x_seq;
        }
        tc_commit_elect<2>(smem_addr(&sh->d_full[buf]));      // both CTAs' rows are done
        ++d_seq;
      }
    mma_done:
      if (issued) {
        tc_commit_elect<2>(smem_addr(&sh->drain), (uint16_t)1);
        if (lane == 0) wdrain_wait(&sh->drain, 0);
        __syncwarp();
      }
    } else if (lane == 0) {
      // ----------------------------------------------------------------
      // forwarder (rank 1): tells rank 0 each time a stage of this CTA is full
      // ----------------------------------------------------------------
      uint32_t x_seq = 0;
      for (long long t = pair; t < geo.num_tiles; t += geo.stride) {
        int lt, mt, nt;
        decode_tile(geo, t, lt, mt, nt);
        if (!kvx::layer_row_ok(p, lt)) continue;
        for (int kc = 0; kc < geo.kc_count; ++kc) {
          const int stage = (int)(x_seq % (uint32_t)geo.stages);
          if (!W.wait(&sh->full[stage], (x_seq / geo.stages) & 1)) goto forward_done;
          mbar_arrive_cluster(smem_addr(&sh->peer_full[stage]), 0);
          ++x_seq;
        }
      }
    forward_done:;
    }
  } else {
    // ------------------------------------------------------------------
    // epilogue: accumulator rows -> + b -> re-rotate keys -> bf16 -> cache
    // ------------------------------------------------------------------
    const int ew = warp - kWEpiWarp0;           // 0..7
    const int quad = warp & 3;                  // tensor-memory lane quadrant of this warp
    const int e = ew >> 2;                      // 0: key columns, 1: value columns
    const int row_in_tile = quad * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    uint32_t d_seq = 0;
    for (long long t = pair; t < geo.num_tiles; t += geo.stride) {
      int lt, mt, nt;
      decode_tile(geo, t, lt, mt, nt);
      const int64_t g = (int64_t)mt * 2 * kWRows + rank * kWRows + row_in_tile;
      int32_t ps = 0, pt = 0;
      int64_t row = -1;
      uint32_t bad = 0;
      if (g < p.ntok) bad = kvx::token_meta(p, g, ps, pt, row);
      // every token's row errors once (the tiles of target layer 0, head 0)
      if (lt == 0 && nt == 0 && e == 0) {
        const uint32_t any = __reduce_or_sync(0xffffffffu, bad);
        if (lane == 0) kvx::report(p, any);
      }
      if (!kvx::layer_row_ok(p, lt)) {
        if (mt == 0 && nt == 0 && rank == 0 && ew == 0 && lane == 0)
          kvx::report(p, KVX_FLAG_BAD_LAYER_INDEX);
        continue;
      }
      const int buf = d_seq & 1;
      if (!W.warp_wait(&sh->d_full[buf], (d_seq >> 1) & 1)) break;
      tc_fence_after();
      const uint32_t dcol = tmem + lane_base + (uint32_t)(buf * kWN + e * kWD);
      const float *bias = bias_f32 + (((int64_t)lt * p.H + nt) * 2 + e) * kWD;
      __nv_bfloat16 *orow = reinterpret_cast<__nv_bfloat16 *>(e == 0 ? p.dst_k : p.dst_v) +
                            (((int64_t)lt * p.dst_rows + (row < 0 ? 0 : row)) * p.H + nt) * kWD;
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        // pairs [16 cc, 16 cc + 16): one 32-byte sector of each half row
        uint32_t olo[8], ohi[8];
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          const int c = 2 * cc + c2;            // pairs [8 c, 8 c + 8)
          uint32_t vlo[8], vhi[8];
          tc_ld8(dcol + 8 * c, vlo);
          tc_ld8(dcol + kWHalf + 8 * c, vhi);
          tc_wait_ld();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int i = 8 * c + 2 * q;
            const float2 bl = __ldg(reinterpret_cast<const float2 *>(bias + i));
            const float2 bh = __ldg(reinterpret_cast<const float2 *>(bias + kWHalf + i));
            float2 y0 = __fadd2_rn(
                make_float2(__uint_as_float(vlo[2 * q]), __uint_as_float(vlo[2 * q + 1])), bl);
            float2 y1 = __fadd2_rn(
                make_float2(__uint_as_float(vhi[2 * q]), __uint_as_float(vhi[2 * q + 1])), bh);
            if (e == 0) {
              // (y0 + j y1) exp(+j p' w_i) for pairs i, i + 1
              float c0, s0, c1, s1;
              rope_cs((uint32_t)pt, rope_tgt.f[i], c0, s0);
              rope_cs((uint32_t)pt, rope_tgt.f[i + 1], c1, s1);
              const float2 cs = make_float2(c0, c1), sn = make_float2(s0, s1);
              const float2 r0 = __ffma2_rn(y0, cs, __fmul2_rn(y1, make_float2(-s0, -s1)));
              const float2 r1 = __ffma2_rn(y0, sn, __fmul2_rn(y1, cs));
              y0 = r0;
              y1 = r1;
            }
            olo[4 * c2 + q] = pack_bf16(y0.x, y0.y);
            ohi[4 * c2 + q] = pack_bf16(y1.x, y1.y);
          }
        }
        if (row >= 0) {
          st_global_v8(orow + 16 * cc, olo);
          st_global_v8(orow + kWHalf + 16 * cc, ohi);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0) mbar_arrive(smem_addr(&sh->d_empty[buf]));
        else mbar_arrive_cluster(smem_addr(&sh->d_empty[buf]), 0);
      }
      ++d_seq;
    }
  }

  tc_fence_before();
  // neither CTA leaves while the other may still arrive on its barriers or
  // (rank 0's MMAs, drained above) read its shared memory
  cluster_sync();
  tc_fence_after();
  if (warp == kWMmaWarp)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kWTmemCols)
                 : "memory");
}

// ---------------------------------------------------------------------------
// 1. Source keys of every layer, un-rotated at their source positions:
//    thread = (token, head, run of 8 pairs); content = x * exp(-j p w_i).
//    Rows with a position outside the table are written as zeros (the map
//    skips them).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) wide_unrotate_kernel(const __grid_constant__ KvxParams p,
                                                            const __grid_constant__ WideTurns rope_src,
                                                            __nv_bfloat16 *__restrict__ out,
                                                            int64_t out_tokens) {
  __shared__ unsigned long long s_turns[kWHalf];
  if (threadIdx.x < kWHalf) s_turns[threadIdx.x] = rope_src.f[threadIdx.x];
  __syncthreads();
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int per_tok = p.H * 8;
  const int64_t g = e / per_tok;
  if (g >= p.ntok) return;
  const int rem = (int)(e - g * per_tok);
  const int h = rem >> 3, q = rem & 7;
  const int s = blockIdx.y;
  int32_t ps = 0, pt = 0;
  int64_t row = -1, srow = -1;
  kvx::token_meta(p, g, ps, pt, row, srow);
  const bool pos_ok = srow >= 0;   // a valid position and, if paged, source block
  const __nv_bfloat16 *src = reinterpret_cast<const __nv_bfloat16 *>(p.src_k) +
                             (((int64_t)s * p.src_rows + (pos_ok ? srow : 0)) * p.H + h) * kWD;
  __nv_bfloat16 *dst = out + (((int64_t)s * out_tokens + g) * p.H + h) * kWD;
  uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
  if (pos_ok) {
    const uint4 a = __ldcs(reinterpret_cast<const uint4 *>(src + 8 * q));
    const uint4 b = __ldcs(reinterpret_cast<const uint4 *>(src + kWHalf + 8 * q));
    const __nv_bfloat162 *a2 = reinterpret_cast<const __nv_bfloat162 *>(&a);
    const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&b);
    uint32_t ol[4], oh[4];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const float2 x0 = __bfloat1622float2(a2[v]), x1 = __bfloat1622float2(b2[v]);
      float c0, s0, c1, s1;
      rope_cs((uint32_t)ps, s_turns[8 * q + 2 * v], c0, s0);
      rope_cs((uint32_t)ps, s_turns[8 * q + 2 * v + 1], c1, s1);
      // (x0 + j x1) exp(-j p w_i)
      ol[v] = pack_bf16(fmaf(x0.x, c0, x1.x * s0), fmaf(x0.y, c1, x1.y * s1));
      oh[v] = pack_bf16(fmaf(x1.x, c0, -x0.x * s0), fmaf(x1.y, c1, -x0.y * s1));
    }
    lo = make_uint4(ol[0], ol[1], ol[2], ol[3]);
    hi = make_uint4(oh[0], oh[1], oh[2], oh[3]);
  }
  *reinterpret_cast<uint4 *>(dst + 8 * q) = lo;
  *reinterpret_cast<uint4 *>(dst + kWHalf + 8 * q) = hi;
}

// ---------------------------------------------------------------------------
// 2. W [Lt][F][N] -> bf16 image: chunk (lt, head nt, step kc) is [256 n][64 k]
//    (n = the head's 128 key then 128 value outputs), two 16 KB halves in the
//    128-byte-swizzled K-major layout: byte (n, kk) of a half =
//    (n % 128) * 128 + ((kk / 8) ^ (n % 8)) * 16 + (kk % 8) * 2.  The kc = 0
//    CTA of each (lt, nt) also writes that head's 256 biases as fp32.
// ---------------------------------------------------------------------------
template <typename WT, typename BT>
__global__ void __launch_bounds__(256) wide_w_image_kernel(const WT *__restrict__ w,
                                                           uint4 *__restrict__ img,
                                                           const BT *__restrict__ b,
                                                           float *__restrict__ b_img, int64_t F,
                                                           int64_t N, int KC, int NT,
                                                           unsigned int *__restrict__ sync) {
  __shared__ float tile[kWKStep][kWRows + 1];
  const int kc = blockIdx.x, nt = blockIdx.y, lt = blockIdx.z;
  // the map kernel's lockstep counter starts every transfer at zero
  if (kc == 0 && nt == 0 && lt == 0 && threadIdx.x == 0) *sync = 0u;
  const WT *src = w + ((int64_t)lt * F + (int64_t)kc * kWKStep) * N + (int64_t)nt * kWN;
  uint4 *out = img + (((int64_t)lt * NT + nt) * KC + kc) * (kWChunkBytes / 16);
  for (int half = 0; half < 2; ++half) {
    for (int e = threadIdx.x; e < kWKStep * kWRows; e += blockDim.x) {
      const int kr = e / kWRows, n = e % kWRows;
      tile[kr][n] = (float)src[(int64_t)kr * N + half * kWRows + n];
    }
    __syncthreads();
    for (int q = threadIdx.x; q < kWHalfBytes / 16; q += blockDim.x) {
      const int n = q >> 3, k8 = (q & 7) ^ (n & 7);
      uint32_t v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        v[u] = pack_bf16(tile[k8 * 8 + 2 * u][n], tile[k8 * 8 + 2 * u + 1][n]);
      out[half * (kWHalfBytes / 16) + q] = make_uint4(v[0], v[1], v[2], v[3]);
    }
    __syncthreads();
  }
  if (kc == 0)
    for (int i = threadIdx.x; i < kWN; i += blockDim.x) {
      const int64_t o = (int64_t)lt * N + (int64_t)nt * kWN + i;
      b_img[o] = (float)b[o];
    }
}

size_t wide_smem_bytes(int stages) {
  return 1024 + (size_t)stages * kWStageBytes + sizeof(WShared) + 64;
}

int wide_stages() {
  int s = kWMaxStages;
  while (s > 2 && wide_smem_bytes(s) > (size_t)kWSmemLimit) --s;
  return s;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t wide_img_bytes(const kvx_plan_desc &d) {
  const size_t F = (size_t)d.k * 2 * d.src_kv_heads * kWD, N = (size_t)d.src_kv_heads * 2 * kWD;
  return (size_t)d.tgt_layers * F * N * 2;
}
size_t wide_bias_bytes(const kvx_plan_desc &d) {
  return (size_t)d.tgt_layers * d.src_kv_heads * 2 * kWD * sizeof(float);
}

// 4-D TMA map over a [Ls][tokens][H][128] bf16 cache whose layers are
// `layer_rows` token rows apart: box [1][128][1][64], 128-byte swizzle,
// rows at or past `tokens` read as zero.
bool encode_wide_map(const kvx_plan *plan, CUtensorMap *map, const void *base, int64_t tokens,
                     int64_t layer_rows, int H, int Ls) {
  typedef CUresult (*EncodeFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                               const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                               const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                               CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  EncodeFn fn = reinterpret_cast<EncodeFn>(plan->encode_tiled);
  if (!fn) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)kWD, (cuuint64_t)H, (cuuint64_t)tokens, (cuuint64_t)Ls};
  const cuuint64_t strides[3] = {(cuuint64_t)kWD * 2, (cuuint64_t)H * kWD * 2,
                                 (cuuint64_t)layer_rows * H * kWD * 2};
  const cuuint32_t box[4] = {(cuuint32_t)kWHalf, 1u, (cuuint32_t)kWRows, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool kvx_wide_supports(const kvx_plan_desc &d) {
  // grid limits of the pre-passes: y = heads or source layers, z = target layers
  return d.kv_dtype == KVX_BF16 && d.src_head_dim == kWD && d.k >= 1 && d.src_kv_heads >= 1 &&
         d.src_kv_heads <= 65535 && d.src_layers <= 65535 && d.tgt_layers <= 65535;
}

size_t kvx_wide_workspace_bytes(const kvx_plan_desc &d, int64_t max_tokens) {
  return align256(wide_img_bytes(d)) + align256(wide_bias_bytes(d)) + 256 +
         (size_t)d.src_layers * (size_t)max_tokens * d.src_kv_heads * kWD * 2;
}

cudaError_t kvx_wide_prepare(kvx_plan *plan) {
  if (!plan->encode_tiled) return cudaErrorNotSupported;
  const size_t smem = wide_smem_bytes(wide_stages());
  cudaError_t e = cudaFuncSetAttribute(wide_map_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * plan->num_sms, 1, 1);
  cfg.blockDim = dim3(kWThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, wide_map_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  plan->tc_pairs = n;
  return n > 0 ? cudaSuccess : cudaErrorNotSupported;   // the wide map needs CTA pairs
}

cudaError_t kvx_wide_launch(const kvx_plan *plan, const KvxParams &p, cudaStream_t s) {
  const kvx_plan_desc &d = plan->desc;
  const int64_t F = (int64_t)p.k * 2 * p.H * kWD, N = (int64_t)p.H * 2 * kWD;
  unsigned char *ws = reinterpret_cast<unsigned char *>(plan->workspace);
  uint4 *img = reinterpret_cast<uint4 *>(ws);
  float *bimg = reinterpret_cast<float *>(ws + align256(wide_img_bytes(d)));
  unsigned int *sync = reinterpret_cast<unsigned int *>(ws + align256(wide_img_bytes(d)) +
                                                        align256(wide_bias_bytes(d)));
  __nv_bfloat16 *content = reinterpret_cast<__nv_bfloat16 *>(
      ws + align256(wide_img_bytes(d)) + align256(wide_bias_bytes(d)) + 256);

  // values: read in place, or (paged source) packed first into the plan's
  // buffer; the keys' pre-pass below reads a paged source directly
  const void *vals = p.src_layout == KVX_PAGED ? plan->packed_v : p.src_v;
  const int64_t val_rows = p.src_layout == KVX_PAGED ? plan->max_tokens : p.src_rows;
  // the tensor maps before any launch: a map the driver refuses is reported
  // with nothing enqueued
  CUtensorMap mk, mv;
  if (!encode_wide_map(plan, &mk, content, p.ntok, plan->max_tokens, p.H, p.Ls) ||
      !encode_wide_map(plan, &mv, vals, p.ntok, val_rows, p.H, p.Ls))
    return cudaErrorInvalidValue;

  // 1. un-rotated source keys
  WideTurns src_turns, tgt_turns;
  for (int i = 0; i < kWHalf; ++i) {
    src_turns.f[i] = plan->turns_src[i];
    tgt_turns.f[i] = plan->turns_tgt[i];
  }
  const int64_t threads = p.ntok * p.H * 8;
  dim3 ugrid((unsigned)((threads + 255) / 256), (unsigned)p.Ls);
  wide_unrotate_kernel<<<ugrid, 256, 0, s>>>(p, src_turns, content, plan->max_tokens);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  // 2. W -> bf16 image, b -> fp32
  const int KC = (int)(F / kWKStep), NT = p.H;
  dim3 wgrid((unsigned)KC, (unsigned)NT, (unsigned)p.Lt);
  using bf = __nv_bfloat16;
  const bool wf = d.w_dtype == KVX_F32, bfp = d.b_dtype == KVX_F32;
  if (wf && bfp)
    wide_w_image_kernel<float, float><<<wgrid, 256, 0, s>>>((const float *)p.w, img,
                                                           (const float *)p.b, bimg, F, N, KC, NT, sync);
  else if (wf)
    wide_w_image_kernel<float, bf><<<wgrid, 256, 0, s>>>((const float *)p.w, img, (const bf *)p.b,
                                                        bimg, F, N, KC, NT, sync);
  else if (bfp)
    wide_w_image_kernel<bf, float><<<wgrid, 256, 0, s>>>((const bf *)p.w, img, (const float *)p.b,
                                                        bimg, F, N, KC, NT, sync);
  else
    wide_w_image_kernel<bf, bf><<<wgrid, 256, 0, s>>>((const bf *)p.w, img, (const bf *)p.b, bimg,
                                                     F, N, KC, NT, sync);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  // 3. the map on CTA pairs
  WideGeom geo;
  geo.mt_count = (int)((p.ntok + 2 * kWRows - 1) / (2 * kWRows));
  geo.nt_count = NT;
  geo.kc_count = KC;
  geo.stages = wide_stages();
  geo.num_tiles = (long long)p.Lt * geo.mt_count * geo.nt_count;
  geo.stride = geo.num_tiles < plan->tc_pairs ? geo.num_tiles : plan->tc_pairs;
  geo.epochs_per_tile = (KC + kWSyncSteps - 1) / kWSyncSteps;
  const long long max_epochs =
      (geo.num_tiles + geo.stride - 1) / geo.stride * (long long)geo.epochs_per_tile;
  // the 32-bit counter must hold every producer's epochs; past that the
  // kernel runs unpaced
  const bool paced = 2 * geo.stride * max_epochs < (1ll << 31);
  geo.sync = paced ? sync : nullptr;
  geo.max_epochs = paced ? (int)max_epochs : 0;
  if (p.src_layout == KVX_PAGED) {
    e = kvx_pack_source(p, nullptr, plan->packed_v, plan->max_tokens, 2, s);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * geo.stride), 1, 1);
  cfg.blockDim = dim3(kWThreads, 1, 1);
  cfg.dynamicSmemBytes = wide_smem_bytes(geo.stages);
  cfg.stream = s;
  // The producers pace each other (loose lockstep) when all pairs are
  // resident together, as the grid (the cluster occupancy of the device)
  // allows; if other work keeps some pairs off the device, the waiting
  // producers stop pacing after 1 ms and the kernel runs unpaced.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const unsigned char *wimg = reinterpret_cast<const unsigned char *>(img);
  return cudaLaunchKernelEx(&cfg, wide_map_kernel, p, mk, mv, tgt_turns, (const float *)bimg,
                            wimg, geo);
}
