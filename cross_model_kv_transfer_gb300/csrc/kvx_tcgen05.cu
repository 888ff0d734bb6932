// kvx_tcgen05.cu -- the transfer on the 5th-generation tensor cores (sm_103a).
//
// The map ("Helm Intelligent Routing", "Why carrying the cache across is the
// hard part", step 2; Qwen3 article, linear-bridge section: one ridge map per
// target (layer, head), separately for K and V, applied to the concatenated
// features of the selected source layers) is a dense contraction per
// (target layer lt, head h, K|V):  Y[T x d] = X[T x k*d] . W[k*d x d] + b.
// It runs as tcgen05.mma (kind::f16, bf16 operands, fp32 accumulation in
// tensor memory), M = 128 tokens per CTA (256 per CTA pair), N = d = 128,
// K = 16 per instruction.
//
// Data path of one CTA (persistent, one per SM; by default CTA pairs share
// each M = 256 MMA), per work item (h, lt, K|V, chunk of 128-token tiles):
//   * W producer (one thread): copies the item's bf16 W image (prepared by
//     w_image_kernel: 2k chunks of 16 KB in the UMMA 128-byte-swizzled
//     K-major layout, output channels in the epilogue's column order) into
//     shared memory with cp.async.bulk; W stays resident for all tiles of
//     the item and is the MMA's B operand.
//   * X loader (one thread): TMA (cp.async.bulk.tensor, 4-D map over
//     [Ls][T][H][d], 128-byte swizzle) brings the 128 rows x d of one
//     selected source layer for one tile into a ring of shared-memory stages,
//     two boxes of 64 dims; for key tiles of one request it also stages the
//     source-RoPE cos/sin couples of the tile's positions.
//   * 8 transform warps (two per tensor-memory lane quadrant): every thread
//     owns one token row and half of the RoPE pairs.  It reads its row from
//     the stage (16-byte shared loads, conflict-free thanks to the swizzle),
//     un-rotates keys out of the source RoPE (step 1, "strip source RoPE")
//     with bf16x2 FMAs, and writes the row with tcgen05.st into tensor
//     memory, operand A (a ring of four 64-column slots).  Values are copied
//     as stored.
//   * MMA warp: 8 tcgen05.mma per selection (one elected lane issues), A from
//     tensor memory, B = W from shared memory, into one of two 128-column
//     fp32 accumulators; tcgen05.commit frees A slots and W chunks and hands
//     finished accumulators to the epilogue.
//   * 8 epilogue warps (two per lane quadrant, 16 rows each): tcgen05.ld of
//     the 16x256b shape, one 64-column half at a time, gives each thread two
//     rows and, thanks to the W image's column order, 8 whole RoPE pairs per
//     half (channels 32H + 8q .. 32H + 8q + 7 and their partners at +64,
//     q = lane % 4); the accumulator is released as soon as the second half
//     is in registers.  Then + b, re-rotation of keys into the target RoPE at
//     p' (step 3), bf16 cast, and 16-byte stores: per half, the four threads
//     of a row write 64 consecutive bytes of the row's first 64 channels and
//     64 of its last 64.
// Every mbarrier wait is bounded: after 2 s without progress the CTA sets
// KVX_FLAG_TIMEOUT, all roles leave their loops, in-flight copies and MMAs
// are drained (again with bounded waits) and tensor memory is freed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "kvx_device.cuh"
#include "kvx_internal.h"
#include "kvx_ptx.cuh"

namespace {

constexpr int kD = 128;               // head_dim handled by this kernel
constexpr int kHalf = kD / 2;
constexpr int kTileM = 128;           // tokens per tile (MMA M)
constexpr int kMaxK = 6;              // selected layers: W = k * 32 KB of smem
constexpr int kSlots = 4;             // A ring slots (64 TMEM columns each)
constexpr int kSlotCols = kD / 2;     // bf16 pairs per selection row
constexpr int kDCol = kSlots * kSlotCols;  // first accumulator column (256)
constexpr int kTmemCols = 512;
constexpr int kChunkBytes = 16384;    // W chunk: 128 rows x 64 k x bf16
constexpr int kStageBytes = 2 * kChunkBytes;  // one selection of one tile
constexpr int kMaxStages = 6;
constexpr int kSmemLimit = 232448;            // 227 KB opt-in per CTA
constexpr int kCplBytes = 16 * kTileM * 16;   // one tile's source-RoPE quads: [16][128 rows][16 B]
constexpr int kTransformWarps = 8;
constexpr int kEpilogueWarps = 8;
constexpr int kMmaWarp = kTransformWarps + kEpilogueWarps;   // 16
constexpr int kProducerWarp = kMmaWarp + 1;                  // 17
constexpr int kLoaderWarp = kProducerWarp + 1;               // 18
constexpr int kThreads = (kLoaderWarp + 1) * 32;             // 608
constexpr uint64_t kWaitNs = 2000000000ull;                  // 2 s without progress
constexpr uint64_t kStallTestWaitNs = 20000000ull;           // 20 ms (stall test hook)

// PTX wrappers, the shared-memory descriptor, bf16 packing and the
// fixed-point RoPE angle helper live in kvx_ptx.cuh.

// The 8 MMAs of one selection (K = 128): A columns +8 per K step, B
// descriptor +2 (32 bytes) per step inside a W chunk, then the next chunk
// (this CTA's 16 KB / P of it).
// P = 2: the CTA pair runs one M = 256 MMA (each CTA's 128 rows of A from its
// own tensor memory, each CTA's half of B's N rows from its own shared memory
// at the same offset, D in both CTAs' tensor memory); only rank 0 issues.
template <int P>
__device__ __forceinline__ void tc_mma8_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
#define KVX_MMA8(G)                                                                            \
  asm volatile(                                                                                \
      "{\n.reg .pred e, p, t;\n.reg .b32 r, a1, a2, a3, a4, a5, a6, a7;\n"                     \
      ".reg .b64 b1, b2, b3, b4, b5, b6, b7;\n"                                                \
      "elect.sync r|e, 0xffffffff;\n"                                                          \
      "setp.ne.b32 p, %4, 0;\n"                                                                \
      "setp.eq.u32 t, 0, 0;\n"                                                                 \
      "add.u32 a1, %1, 8; add.u32 a2, %1, 16; add.u32 a3, %1, 24; add.u32 a4, %1, 32;\n"       \
      "add.u32 a5, %1, 40; add.u32 a6, %1, 48; add.u32 a7, %1, 56;\n"                          \
      "add.u64 b1, %2, 2; add.u64 b2, %2, 4; add.u64 b3, %2, 6; add.u64 b4, %2, %5;\n"        \
      "add.u64 b5, b4, 2; add.u64 b6, b4, 4; add.u64 b7, b4, 6;\n"                              \
      "@e tcgen05.mma.cta_group::" G ".kind::f16 [%0], [%1], %2, %3, p;\n"                     \
      "@e tcgen05.mma.cta_group::" G ".kind::f16 [%0], [a1], b1, %3, t;\n"                     \
      "@e tcgen05.mma.cta_group::" G ".kind::f16 [%0], [a2], b2, %3, t;\n"                     \
      "@e tcgen05.mma.cta_group::" G ".kind::f16 [%0], [a3], b3, %3, t;\n"                     \
      "@e tcgen05.mma.cta_group::" G ".kind::f16 [%0], [a4], b4, %3, t;\n"                     \
      "@e tcgen05.mma.cta_group::" G ".kind::f16 [%0], [a5], b5, %3, t;\n"                     \
      "@e tcgen05.mma.cta_group::" G ".kind::f16 [%0], [a6], b6, %3, t;\n"                     \
      "@e tcgen05.mma.cta_group::" G ".kind::f16 [%0], [a7], b7, %3, t;\n}\n" ::"r"(d_tmem),   \
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate),                                    \
      "l"((uint64_t)((kChunkBytes / P) >> 4))                                                   \
      : "memory")
  if constexpr (P == 1) KVX_MMA8("1");
  else KVX_MMA8("2");
#undef KVX_MMA8
}
// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major,
// N = 128, M = 128.
template <int P>
__host__ __device__ constexpr uint32_t idesc_for() {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kD >> 3) << 17) |
         ((uint32_t)((kTileM * P) >> 4) << 24);
}

struct RopeTurns {
  unsigned long long tgt[kHalf];
};

// Output channel held by accumulator column c of a per-head map.  The W
// image puts channel chan_of_col(c) in B's row c, so that a 16x256b
// tensor-memory load of the 64-column half H (thread t: columns 8i +
// 2(t%4) + e, i < 8) hands thread q = t%4 the channels 32H + 8q + v (v =
// 2i + e < 8) and their RoPE partners 64 + 32H + 8q + (v - 8) (v >= 8):
// the four threads of a row hold 32 consecutive channels and their partners.
__host__ __device__ constexpr int chan_of_col(int c) {
  return ((((c & 63) >> 3) << 1) | (c & 1)) < 8
             ? 32 * (c >> 6) + 8 * ((c >> 1) & 3) + ((((c & 63) >> 3) << 1) | (c & 1))
             : 64 + 32 * (c >> 6) + 8 * ((c >> 1) & 3) + ((((c & 63) >> 3) << 1) | (c & 1)) - 8;
}

// Padded shared-memory slots of the target-RoPE frequencies: the epilogue's
// four q groups read their runs of 8 from distinct banks.
__device__ __forceinline__ int pad_turn(int i) { return i + 2 * (i >> 4); }
constexpr int kTurnSlots = kHalf + 2 * 4;     // 64-bit entries


// bf16x2 helpers: un-rotation of two RoPE pairs at once in bf16x2 FMA
// arithmetic.  a = (x_i, x_{i+1}) of the first half, b = (x_{i+d/2},
// x_{i+1+d/2}), c/s the bf16 cos/sin couples, ns = -s.  Returns
// a*c + b*s and b*c - a*s, each rounded to bf16 (the operand precision of
// the MMA that consumes them).
__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t v) {
  return *reinterpret_cast<__nv_bfloat162 *>(&v);
}
__device__ __forceinline__ uint32_t as_u32(__nv_bfloat162 v) {
  return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ void unrotate2(uint32_t a, uint32_t b, uint32_t c, uint32_t s,
                                          uint32_t ns, uint32_t &x0, uint32_t &x1) {
  x0 = as_u32(__hfma2(as_bf2(a), as_bf2(c), __hmul2(as_bf2(b), as_bf2(s))));
  x1 = as_u32(__hfma2(as_bf2(b), as_bf2(c), __hmul2(as_bf2(a), as_bf2(ns))));
}

// ---------------------------------------------------------------------------
// Shared state of one CTA
// ---------------------------------------------------------------------------
struct Shared {
  uint64_t x_full[kMaxStages], x_empty[kMaxStages];
  uint64_t a_full[kSlots], a_empty[kSlots];
  uint64_t d_full[2], d_empty[2];
  uint64_t w_full[2 * kMaxK], w_empty[2 * kMaxK];
  uint64_t w_peer[2 * kMaxK];   // CTA pair: the peer's W half has landed (rank 0 only)
  uint64_t drain;
  uint64_t c_full, c_empty;   // CTA pairs: one K tile's source-RoPE quads in shared memory
  uint32_t tmem_base;
  volatile int c_mode;        // 1: the quads of positions p0 .. p0 + 127 are staged; 2: use global
  volatile int abort;
  __align__(16) unsigned long long turns[kTurnSlots];   // target-RoPE frequencies (padded)
};

struct Waiter {
  Shared *sh;
  uint32_t *status;
  uint64_t limit_ns;
  // Bounded wait; false means the pipeline is being abandoned.
  __device__ __forceinline__ bool wait(uint64_t *bar, uint32_t parity) const {
    const uint32_t a = smem_addr(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
      if (mbar_try_wait(a, parity)) return true;
      if (sh->abort) return false;
      if (globaltimer() - t0 > limit_ns) {
        sh->abort = 1;
        if (status) atomicOr(status, KVX_FLAG_TIMEOUT);
        return false;
      }
    }
  }
  // Every lane waits; the warp leaves together, with false if any lane gave up.
  __device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity) const {
    const bool ok = wait(bar, parity);
    return __all_sync(0xffffffffu, ok) != 0;
  }
};

// Bounded wait used while draining: ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
  const uint32_t a = smem_addr(bar);
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(a, parity) && globaltimer() - t0 < kWaitNs) {
  }
}

struct ItemGeom {
  int num_tiles, num_chunks, tiles_per_item, stages;
  long long num_items;
  long long stride;   // CTA groups (CTAs, or CTA pairs) running items concurrently
};

// Source-RoPE couples of row `row_in_tile` of a tile starting at packed row
// `row0`, for pairs [32 th, 32 th + 32): couple u holds (cos, cos) and (sin,
// sin) in bf16x2 for pairs 32 th + 2u and +1, read from the position-major
// quad table (a warp's 32 consecutive rows read contiguous memory).  Rows
// outside the transfer or with an invalid position get the identity rotation.
__device__ __forceinline__ void load_couples(const KvxParams &p, const uint4 *__restrict__ rope_src4,
                                             int64_t row0, int row_in_tile, int th,
                                             uint32_t (&c2)[16], uint32_t (&s2)[16]) {
#pragma unroll
  for (int u = 0; u < 16; ++u) {
    c2[u] = 0x3F803F80u;   // (1, 1)
    s2[u] = 0u;
  }
  const int64_t g = row0 + row_in_tile;
  int32_t ps = 0, pt = 0;
  int64_t row = -1;
  if (g < p.ntok) kvx::token_meta(p, g, ps, pt, row);
  if (row < 0) return;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint4 v = __ldg(rope_src4 + (int64_t)(8 * th + i) * p.max_position + ps);
    c2[2 * i] = v.x;
    s2[2 * i] = v.y;
    c2[2 * i + 1] = v.z;
    s2[2 * i + 1] = v.w;
  }
}

// Work items are (h, chunk, lt, m): Q = H * chunks * Lt groups (h, chunk,
// lt), lt fastest, each with a key item (m = 0) and a value item (m = 1).
// CTA group b of G runs items b, b + G, b + 2G, ...; round r = item / G holds the
// keys (r even) or the values (r odd) of groups [(r/2) G, (r/2) G + G), so
// every CTA alternates keys and values (keys cost more: two RoPE passes).
// Groups past the last whole pair of rounds alternate m item by item.
__device__ __forceinline__ void decode_item(const KvxParams &p, const ItemGeom &g, long long item,
                                            int &h, int &chunk, int &lt, int &m) {
  const long long G = g.stride;
  const long long full = (g.num_items >> 1) / G * G;   // groups in whole round pairs
  long long q;
  if (item < 2 * full) {
    const long long r = item / G;
    m = (int)(r & 1);
    q = (r >> 1) * G + (item - r * G);
  } else {
    const long long t = item - 2 * full;
    m = (int)(t & 1);
    q = full + (t >> 1);
  }
  lt = (int)(q % p.Lt);
  q /= p.Lt;
  chunk = (int)(q % g.num_chunks);
  h = (int)(q / g.num_chunks);
}

// ---------------------------------------------------------------------------
// The transfer kernel
// ---------------------------------------------------------------------------
template <int P>
__global__ void __launch_bounds__(kThreads, 1)
    tc_transfer_kernel(const __grid_constant__ KvxParams p,
                       const __grid_constant__ CUtensorMap tmap_k,
                       const __grid_constant__ CUtensorMap tmap_v,
                       const __grid_constant__ CUtensorMap tmap_cpl,
                       const uint4 *__restrict__ rope_src4,
                       const __grid_constant__ RopeTurns rope,
                       const float *__restrict__ bias_f32,
                       const __nv_bfloat16 *__restrict__ w_img, const ItemGeom geo,
                       const int stall_test) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // W chunks and X stages need 1024-byte alignment (128-byte swizzle atoms).
  unsigned char *wbuf = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int kWChunk = kChunkBytes / P;   // a CTA holds 128 / P rows n of each W chunk
  unsigned char *xbuf = wbuf + (size_t)2 * p.k * kWChunk;
  // CTA pairs have room to stage each K tile's source-RoPE quads by TMA
  constexpr bool kStageCpl = P == 2;
  unsigned char *cbuf = xbuf + (size_t)geo.stages * kStageBytes;
  Shared *sh = reinterpret_cast<Shared *>(cbuf + (kStageCpl ? kCplBytes : 0));

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int nchunks_w = 2 * p.k;
  // CTA pair: rank 0 issues the MMAs and owns the barriers the pair shares
  const uint32_t rank = P == 2 ? cluster_rank() : 0u;
  const long long group = blockIdx.x / P;
  const int tile_rows = kTileM * P;          // packed rows per tile of the group

  if (tid == 0) {
    for (int s = 0; s < geo.stages; ++s) {
      mbar_init(smem_addr(&sh->x_full[s]), 1);
      mbar_init(smem_addr(&sh->x_empty[s]), kTransformWarps);
    }
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(smem_addr(&sh->a_full[s]), kTransformWarps * P);
      mbar_init(smem_addr(&sh->a_empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_addr(&sh->d_full[b]), 1);
      mbar_init(smem_addr(&sh->d_empty[b]), kEpilogueWarps * P);
    }
    for (int c = 0; c < nchunks_w; ++c) {
      mbar_init(smem_addr(&sh->w_full[c]), 1);
      mbar_init(smem_addr(&sh->w_empty[c]), 1);
      mbar_init(smem_addr(&sh->w_peer[c]), 1);
    }
    mbar_init(smem_addr(&sh->drain), 1);
    mbar_init(smem_addr(&sh->c_full), 1);
    mbar_init(smem_addr(&sh->c_empty), kTransformWarps);
    sh->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // the target-RoPE frequencies for the epilogue (visible after the barrier
  // inside seqlens_ok below)
  if (tid < kHalf) sh->turns[pad_turn(tid)] = rope.tgt[tid];
  if (warp == kMmaWarp) {
    // CTA pair: one warp in each CTA allocates collectively (same columns)
    if constexpr (P == 1) {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_addr(&sh->tmem_base)),
                   "r"(kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    } else {
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_addr(&sh->tmem_base)),
                   "r"(kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
  }
  tc_fence_before();
  // The request table is validated by every CTA; a malformed one stops the
  // whole transfer before any write.
  const bool seq_ok = kvx::seqlens_ok(p, tid, kThreads);
  // CTA pair: the peer's barriers are initialised before any remote arrival
  if constexpr (P == 2) cluster_sync();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;
  const Waiter W{sh, p.status, stall_test ? kStallTestWaitNs : kWaitNs};

  if (!seq_ok) {
    if (blockIdx.x == 0 && tid == 0) kvx::report(p, KVX_FLAG_BAD_SEQLENS);
  } else if (warp < kTransformWarps) {
    // ------------------------------------------------------------------
    // transform warps: X rows -> tensor memory (operand A)
    // ------------------------------------------------------------------
    const int quad = warp & 3;                // TMEM lane quadrant
    const int th = warp >> 2;                 // RoPE pair half: pairs [32 th, 32 th + 32)
    const int row_in_tile = quad * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    uint32_t a_seq = 0;
    int x_stage = 0;                          // X ring position, tracked incrementally
    uint32_t x_par = 0;
    uint32_t c_par = 0;                       // staged-quads phase (K tiles, CTA pairs)
    // byte offsets in a swizzled 128-byte row of the thread's four 16-byte
    // chunks (dims 32 th .. 32 th + 31 of each 64-dim box)
    uint32_t choff[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) choff[q] = (uint32_t)(((4 * th + q) ^ (row_in_tile & 7)) * 16);
    // The tiles of one item; keys (un-rotated out of the source RoPE) and
    // values (copied as stored) are compiled as separate loops.  Returns
    // false when the pipeline is being abandoned.
    auto tiles = [&](auto key_c, int t_beg, int t_end) -> bool {
      constexpr bool kKey = decltype(key_c)::value;
      for (int tile = t_beg; tile < t_end; ++tile) {
        // bf16x2 cos/sin couples of the source RoPE at this row's position
        // for the thread's 32 pairs (couple u = pairs 32 th + 2u, +1)
        uint32_t c2[16], s2[16];
        if constexpr (kKey) {
          bool from_global = true;
          if constexpr (kStageCpl) {
            // the loader staged this tile's quads (positions p0 + row) or
            // left them to be read from the global table
            if (!W.wait(&sh->c_full, c_par)) return false;
            c_par ^= 1;
            if (sh->c_mode == 1) {
              from_global = false;
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const uint4 v = *reinterpret_cast<const uint4 *>(
                    cbuf + (8 * th + i) * (kTileM * 16) + row_in_tile * 16);
                c2[2 * i] = v.x;
                s2[2 * i] = v.y;
                c2[2 * i + 1] = v.z;
                s2[2 * i + 1] = v.w;
              }
            }
          }
          if (from_global)
            load_couples(p, rope_src4, (int64_t)tile * tile_rows + rank * kTileM, row_in_tile, th,
                         c2, s2);
        }
        for (int j = 0; j < p.k; ++j) {
          const int stage = x_stage;
          if (!W.wait(&sh->x_full[stage], x_par)) return false;
          // this row's dims [32 th, 32 th + 32) (box 0) and [64 + 32 th, ...)
          // (box 1)
          const unsigned char *rb = xbuf + stage * kStageBytes + row_in_tile * 128;
          uint32_t plo[16], phi[16];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 lo = *reinterpret_cast<const uint4 *>(rb + choff[q]);
            const uint4 hi = *reinterpret_cast<const uint4 *>(rb + kChunkBytes + choff[q]);
            plo[4 * q] = lo.x; plo[4 * q + 1] = lo.y; plo[4 * q + 2] = lo.z; plo[4 * q + 3] = lo.w;
            phi[4 * q] = hi.x; phi[4 * q + 1] = hi.y; phi[4 * q + 2] = hi.z; phi[4 * q + 3] = hi.w;
          }
          if (++x_stage == geo.stages) {
            x_stage = 0;
            x_par ^= 1;
          }
          const int slot = a_seq % kSlots;
          const uint32_t round = a_seq / kSlots;
          if constexpr (kKey) {
            // un-rotate: (x0 + j x1) * exp(-j p w_i), pairs i = 32 th + 2u (+1)
#pragma unroll
            for (int u = 0; u < 16; ++u)
              unrotate2(plo[u], phi[u], c2[u], s2[u], s2[u] ^ 0x80008000u, plo[u], phi[u]);
          }
          if (!W.wait(&sh->a_empty[slot], (round & 1) ^ 1)) return false;
          tc_fence_after();
          {
            // A column slot * 64 + f / 2 holds features (f, f + 1)
            const uint32_t col = (uint32_t)(slot * kSlotCols + 16 * th);
            tc_st16(tmem + lane_base + col, plo);
            tc_st16(tmem + lane_base + col + 32, phi);
          }
          tc_wait_st();
          // release the X stage only now: its words went through registers
          // into tensor memory (wait::st returned for the whole warp), so
          // every read of the stage is complete before the loader's next TMA
          // write lands there
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(smem_addr(&sh->x_empty[stage]));
            // likewise the staged quads, consumed by the first selection
            if (kKey && kStageCpl && j == 0) mbar_arrive(smem_addr(&sh->c_empty));
            if (!stall_test) {
              if (P == 1 || rank == 0) mbar_arrive(smem_addr(&sh->a_full[slot]));
              else mbar_arrive_cluster(smem_addr(&sh->a_full[slot]), 0);
            }
          }
          ++a_seq;
        }
      }
      return true;
    };
    for (long long item = group; item < geo.num_items; item += geo.stride) {
      int h, chunk, lt, m;
      decode_item(p, geo, item, h, chunk, lt, m);
      if (!kvx::layer_row_ok(p, lt)) continue;
      const int t_beg = chunk * geo.tiles_per_item;
      const int t_end = min(t_beg + geo.tiles_per_item, geo.num_tiles);
      const bool go = m == 0 ? tiles(std::true_type{}, t_beg, t_end)
                             : tiles(std::false_type{}, t_beg, t_end);
      if (!go) break;
    }
  } else if (warp < kMmaWarp) {
    // ------------------------------------------------------------------
    // epilogue warps: accumulator -> + b -> re-rotate (K) -> bf16 -> cache
    // ------------------------------------------------------------------
    const int ew = warp - kTransformWarps;
    const int quad = warp & 3;
    const int eh = ew >> 2;                          // rows 32 quad + 16 eh .. + 16
    const int q = lane & 3;                          // channels 16q.. and 64 + 16q..
    const uint32_t lane_base = (uint32_t)(quad * 32 + 16 * eh) << 16;
    const int meta_row = quad * 32 + 16 * eh + (lane & 15);   // resolved by lanes 0..15
    uint32_t d_seq = 0;
    // The tiles of one item (keys re-rotated into the target RoPE, values
    // not), compiled as separate loops.  Returns false when the pipeline is
    // being abandoned.
    auto tiles = [&](auto key_c, int lt, int h, int t_beg, int t_end, bool layer_ok,
                     bool reporter) -> bool {
      constexpr bool kKey = decltype(key_c)::value;
      // the item's bias (fp32 image, natural channel order; L1-resident)
      const float2 *bias2 = reinterpret_cast<const float2 *>(
          bias_f32 + (((int64_t)lt * p.H + h) * 2 + (kKey ? 0 : 1)) * kD);
      __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(kKey ? p.dst_k : p.dst_v);
      for (int tile = t_beg; tile < t_end; ++tile) {
        // lanes 0..15 resolve the positions and cache rows of the warp's 16
        // rows; every thread then takes its rows t/4 and t/4 + 8
        int32_t pt_l = 0;
        long long row_l = -1;
        uint32_t bad = 0;
        if (lane < 16) {
          const int64_t g = (int64_t)tile * tile_rows + rank * kTileM + meta_row;
          int32_t ps = 0, pt = 0;
          int64_t row = -1;
          if (g < p.ntok) bad = kvx::token_meta(p, g, ps, pt, row);
          pt_l = pt;
          row_l = row;
        }
        if (kKey && reporter) {
          const uint32_t any = __reduce_or_sync(0xffffffffu, bad);
          if (lane == 0) kvx::report(p, any);
        }
        if (!layer_ok) continue;
        const int32_t pt0 = __shfl_sync(0xffffffffu, pt_l, lane >> 2);
        const int32_t pt1 = __shfl_sync(0xffffffffu, pt_l, (lane >> 2) + 8);
        const long long row0 = __shfl_sync(0xffffffffu, row_l, lane >> 2);
        const long long row1 = __shfl_sync(0xffffffffu, row_l, (lane >> 2) + 8);
        const int buf = d_seq & 1;
        if (!W.wait(&sh->d_full[buf], (d_seq >> 1) & 1)) return false;
        tc_fence_after();
        const uint32_t dcol = tmem + lane_base + (uint32_t)(kDCol + buf * kD);
        __nv_bfloat16 *o0 = row0 >= 0 ? dst + (((int64_t)lt * p.dst_rows + row0) * p.H + h) * kD
                                      : nullptr;
        __nv_bfloat16 *o1 = row1 >= 0 ? dst + (((int64_t)lt * p.dst_rows + row1) * p.H + h) * kD
                                      : nullptr;
        // register 4i + 2rs + e of half H holds (row rs, channel 32H + 8q +
        // 2i + e) for i < 4 and its RoPE partner (+64) for i = 4..7; the two
        // 64-column halves are loaded, processed and stored one after the other
#pragma unroll
        for (int H = 0; H < 2; ++H) {
          uint32_t v[32];
          tc_ld16x256_x8(dcol + 64 * H, v);
          tc_wait_ld();
          if (H == 1) {
            // the accumulator is in registers: hand it back to the MMA warp
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              if (P == 1 || rank == 0) mbar_arrive(smem_addr(&sh->d_empty[buf]));
              else mbar_arrive_cluster(smem_addr(&sh->d_empty[buf]), 0);
            }
          }
          uint32_t olo[2][4], ohi[2][4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int n = 32 * H + 8 * q + 2 * i;    // channels n, n + 1 and n + 64, n + 65
            const float2 bl = __ldg(bias2 + (n >> 1));
            const float2 bh = __ldg(bias2 + ((64 + n) >> 1));
            float c0 = 1.f, s0 = 0.f, c1 = 1.f, s1 = 0.f, c2 = 1.f, s2 = 0.f, c3 = 1.f, s3 = 0.f;
            if constexpr (kKey) {
              const ulonglong2 f = *reinterpret_cast<const ulonglong2 *>(sh->turns + pad_turn(n));
              rope_cs((uint32_t)pt0, f.x, c0, s0);
              rope_cs((uint32_t)pt0, f.y, c1, s1);
              rope_cs((uint32_t)pt1, f.x, c2, s2);
              rope_cs((uint32_t)pt1, f.y, c3, s3);
            }
#pragma unroll
            for (int rs = 0; rs < 2; ++rs) {
              float2 y0 = __fadd2_rn(make_float2(__uint_as_float(v[4 * i + 2 * rs]),
                                                 __uint_as_float(v[4 * i + 2 * rs + 1])), bl);
              float2 y1 = __fadd2_rn(make_float2(__uint_as_float(v[4 * (i + 4) + 2 * rs]),
                                                 __uint_as_float(v[4 * (i + 4) + 2 * rs + 1])), bh);
              if constexpr (kKey) {
                // (y0 + j y1) exp(+j p' w_i), pairs i = n, n + 1
                const float2 cc = rs ? make_float2(c2, c3) : make_float2(c0, c1);
                const float2 ss = rs ? make_float2(s2, s3) : make_float2(s0, s1);
                const float2 nss = make_float2(-ss.x, -ss.y);
                const float2 r0 = __ffma2_rn(y0, cc, __fmul2_rn(y1, nss));
                const float2 r1 = __ffma2_rn(y0, ss, __fmul2_rn(y1, cc));
                y0 = r0;
                y1 = r1;
              }
              olo[rs][i] = pack_bf16(y0.x, y0.y);
              ohi[rs][i] = pack_bf16(y1.x, y1.y);
            }
          }
          // the four threads of a row write 64 consecutive bytes of each half
          const int c0 = 32 * H + 8 * q;
          if (o0) {
            st_global_v4(o0 + c0, olo[0]);
            st_global_v4(o0 + kHalf + c0, ohi[0]);
          }
          if (o1) {
            st_global_v4(o1 + c0, olo[1]);
            st_global_v4(o1 + kHalf + c0, ohi[1]);
          }
        }
        ++d_seq;
      }
      return true;
    };
    for (long long item = group; item < geo.num_items; item += geo.stride) {
      int h, chunk, lt, m;
      decode_item(p, geo, item, h, chunk, lt, m);
      const bool layer_ok = kvx::layer_row_ok(p, lt);
      const bool reporter = h == 0 && m == 0;
      if (!layer_ok && reporter && chunk == 0 && tid == kTransformWarps * 32)
        kvx::report(p, KVX_FLAG_BAD_LAYER_INDEX);
      const int t_beg = chunk * geo.tiles_per_item;
      const int t_end = min(t_beg + geo.tiles_per_item, geo.num_tiles);
      const bool go = m == 0 ? tiles(std::true_type{}, lt, h, t_beg, t_end, layer_ok, reporter)
                             : tiles(std::false_type{}, lt, h, t_beg, t_end, layer_ok, reporter);
      if (!go) break;
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------
    // MMA issuer: the whole warp runs the loop (its descriptors stay
    // warp-uniform) and one elected lane issues each tcgen05 instruction.
    // ------------------------------------------------------------------
    uint32_t a_seq = 0, d_seq = 0, w_seq = 0;
    bool issued = false;
    const uint64_t b0 = sw128_desc(smem_addr(wbuf));
    constexpr uint32_t kIdesc = idesc_for<P>();
    const long long first_item = (P == 1 || rank == 0) ? group : geo.num_items;   // the peer issues nothing
    for (long long item = first_item; item < geo.num_items; item += geo.stride) {
      int h, chunk, lt, m;
      decode_item(p, geo, item, h, chunk, lt, m);
      if (!kvx::layer_row_ok(p, lt)) continue;
      const int t_beg = chunk * geo.tiles_per_item;
      const int t_end = min(t_beg + geo.tiles_per_item, geo.num_tiles);
      for (int tile = t_beg; tile < t_end; ++tile) {
        const int buf = d_seq & 1;
        if (!W.warp_wait(&sh->d_empty[buf], ((d_seq >> 1) & 1) ^ 1)) goto mma_done;
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(kDCol + buf * kD);
        for (int j = 0; j < p.k; ++j) {
          const int slot = a_seq % kSlots;
          if (!W.warp_wait(&sh->a_full[slot], (a_seq / kSlots) & 1)) goto mma_done;
          if (tile == t_beg) {
            if (!W.warp_wait(&sh->w_full[2 * j], w_seq & 1)) goto mma_done;
            if (!W.warp_wait(&sh->w_full[2 * j + 1], w_seq & 1)) goto mma_done;
            if constexpr (P == 2) {   // the peer's halves of the same chunks
              if (!W.warp_wait(&sh->w_peer[2 * j], w_seq & 1)) goto mma_done;
              if (!W.warp_wait(&sh->w_peer[2 * j + 1], w_seq & 1)) goto mma_done;
            }
          }
          tc_fence_after();
          tc_mma8_elect<P>(d_tmem, tmem + (uint32_t)(slot * kSlotCols),
                           b0 + (uint64_t)((2 * j * kWChunk) >> 4), kIdesc, j > 0 ? 1u : 0u);
          issued = true;
          tc_commit_elect<P>(smem_addr(&sh->a_empty[slot]));
          if (tile == t_end - 1) {
            tc_commit_elect<P>(smem_addr(&sh->w_empty[2 * j]));
            tc_commit_elect<P>(smem_addr(&sh->w_empty[2 * j + 1]));
          }
          ++a_seq;
        }
        tc_commit_elect<P>(smem_addr(&sh->d_full[buf]));
        ++d_seq;
      }
      ++w_seq;
    }
  mma_done:
    // drain: every MMA issued so far has completed once `drain` flips
    if (issued) {
      tc_commit_elect<P>(smem_addr(&sh->drain), (uint16_t)1);
      if (lane == 0) drain_wait(&sh->drain, 0);
      __syncwarp();
    }
  } else if (warp == kProducerWarp) {
    // ------------------------------------------------------------------
    // W producer (one thread): bf16 W image -> shared memory
    // ------------------------------------------------------------------
    if (lane == 0) {
      // chunks [0, n_last) were last issued in round w_seq, chunks
      // [n_last, nchunks_w) in round w_seq - 1 (rounds count from 1)
      uint32_t w_seq = 0;
      int n_last = nchunks_w;
      for (long long item = group; item < geo.num_items; item += geo.stride) {
        int h, chunk, lt, m;
        decode_item(p, geo, item, h, chunk, lt, m);
        if (!kvx::layer_row_ok(p, lt)) continue;
        const unsigned char *img = reinterpret_cast<const unsigned char *>(w_img) +
                                   (((int64_t)lt * p.H + h) * 2 + m) * (int64_t)nchunks_w * kChunkBytes;
        ++w_seq;
        for (n_last = 0; n_last < nchunks_w; ++n_last) {
          const int c = n_last;
          if (!W.wait(&sh->w_empty[c], (w_seq & 1) ^ 0)) goto producer_done;
          const uint32_t bar = smem_addr(&sh->w_full[c]);
          mbar_expect_tx(bar, kWChunk);
          // rows n of the chunk in [rank * 128 / P, ...): bytes [rank * kWChunk, +kWChunk)
          bulk_g2s(smem_addr(wbuf + c * kWChunk),
                   img + (int64_t)c * kChunkBytes + (int64_t)rank * kWChunk, kWChunk, bar);
        }
        if (P == 2 && rank != 0) {
          // tell rank 0 (which issues the MMAs) that this CTA's halves landed
          for (int c = 0; c < nchunks_w; ++c) {
            if (!W.wait(&sh->w_full[c], (w_seq - 1) & 1)) goto producer_done;
            mbar_arrive_cluster(smem_addr(&sh->w_peer[c]), 0);
          }
        }
      }
    producer_done:
      // drain: wait (bounded) until every issued copy has landed; the copy of
      // round r completes phase r - 1 of its chunk's w_full
      for (int c = 0; c < nchunks_w; ++c) {
        const uint32_t r = c < n_last ? w_seq : w_seq - 1;
        if (r >= 1) drain_wait(&sh->w_full[c], (r - 1) & 1);
      }
    }
  } else {
    // ------------------------------------------------------------------
    // X loader (one thread): TMA boxes [128 tokens][64 dims] x 2 per
    // (tile, selection) into the stage ring
    // ------------------------------------------------------------------
    if (lane == 0) {
      uint32_t x_seq = 0;
      uint32_t c_seq = 0;   // K tiles whose quads went through the staging buffer
      for (long long item = group; item < geo.num_items; item += geo.stride) {
        int h, chunk, lt, m;
        decode_item(p, geo, item, h, chunk, lt, m);
        if (!kvx::layer_row_ok(p, lt)) continue;
        const CUtensorMap *map = m == 0 ? &tmap_k : &tmap_v;
        const int t_beg = chunk * geo.tiles_per_item;
        const int t_end = min(t_beg + geo.tiles_per_item, geo.num_tiles);
        // the item's selected source layers, read once per item
        int sl_all[kMaxK];
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) sl_all[j] = j < p.k ? p.layer_idx[lt * p.k + j] : 0;
        for (int tile = t_beg; tile < t_end; ++tile) {
          if (kStageCpl && m == 0) {
            // a K tile: stage the source-RoPE quads of its positions when
            // they are p0, p0 + 1, ... (one request, implicit positions),
            // else let the transform warps read the global table
            if (!W.wait(&sh->c_empty, (c_seq & 1) ^ 1)) goto loader_done;
            const int64_t g0 = (int64_t)tile * tile_rows + rank * kTileM;
            int mode = 2;
            int64_t p0 = 0;
            if (p.src_pos == nullptr && g0 < p.ntok) {
              const int64_t g1 = g0 + kTileM - 1 < p.ntok ? g0 + kTileM - 1 : p.ntok - 1;
              const int r0 = kvx::request_of(p, g0);
              if (kvx::request_of(p, g1) == r0) {
                p0 = g0 - (p.cu_seqlens ? (int64_t)p.cu_seqlens[r0] : 0);
                mode = p0 < p.max_position ? 1 : 2;
              }
            }
            sh->c_mode = mode;
            const uint32_t cbar = smem_addr(&sh->c_full);
            if (mode == 1) {
              mbar_expect_tx(cbar, kCplBytes);
              tma_load_2d(smem_addr(cbuf), &tmap_cpl, (int)(2 * p0), 0, cbar);
            } else {
              mbar_arrive(cbar);
            }
            ++c_seq;
          }
#pragma unroll
          for (int j = 0; j < kMaxK; ++j) {
            if (j >= p.k) break;
            const int stage = x_seq % geo.stages;
            if (!W.wait(&sh->x_empty[stage], ((x_seq / geo.stages) & 1) ^ 1)) goto loader_done;
            const int sl = sl_all[j];
            const uint32_t bar = smem_addr(&sh->x_full[stage]);
            const uint32_t dst = smem_addr(xbuf + stage * kStageBytes);
            mbar_expect_tx(bar, kStageBytes);
            const int r0 = tile * tile_rows + (int)rank * kTileM;
            tma_load_4d(dst, map, 0, h, r0, sl, bar);
            tma_load_4d(dst + kChunkBytes, map, kHalf, h, r0, sl, bar);
            ++x_seq;
          }
        }
      }
    loader_done:
      // drain: the last staged quads and the last `stages` loads (at most)
      // may still be in flight
      if (c_seq > 0) drain_wait(&sh->c_full, (c_seq - 1) & 1);
      for (uint32_t n = (x_seq > (uint32_t)geo.stages ? x_seq - geo.stages : 0); n < x_seq; ++n)
        drain_wait(&sh->x_full[n % geo.stages], (n / geo.stages) & 1);
    }
  }

  tc_fence_before();
  // CTA pair: neither CTA leaves while the other may still arrive on its
  // barriers or (rank 0's MMAs, drained above) use its memory
  if constexpr (P == 2) cluster_sync();
  else __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) {
    if constexpr (P == 1)
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                   "r"(kTmemCols)
                   : "memory");
    else
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                   "r"(kTmemCols)
                   : "memory");
  }
}

// ---------------------------------------------------------------------------
// W ([Lt][H][2][k*d][d]) -> bf16 image, per (lt, h, m) 2k chunks of
// [128 rows n][64 k] in the 128-byte-swizzled K-major layout the MMA reads:
// byte (n, kk) of a chunk = n*128 + ((kk/8) ^ (n%8))*16 + (kk%8)*2; row n
// holds output channel chan_of_col(n) (the epilogue's column order).
// One CTA converts one chunk through a shared-memory transpose; the first
// chunk's CTA also writes b of its (lt, h, m) as fp32 (the epilogue's bias).
// ---------------------------------------------------------------------------
template <typename WT, typename BT>
__global__ void __launch_bounds__(256) w_image_kernel(const WT *__restrict__ w,
                                                      uint4 *__restrict__ img,
                                                      const BT *__restrict__ b,
                                                      float *__restrict__ b_img) {
  __shared__ float tile[64][kD + 1];
  const int64_t chunk = blockIdx.x;          // over (lt, h, m, c)
  const int nchunk = gridDim.y;              // chunks per (lt, h, m) = 2k
  const int64_t lhm = chunk;                 // index of (lt, h, m)
  const int c = blockIdx.y;
  const WT *src = w + (lhm * nchunk * 64 + (int64_t)c * 64) * kD;   // rows k = 64c.., [64][128]
  if (c == 0 && threadIdx.x < kD) b_img[lhm * kD + threadIdx.x] = (float)b[lhm * kD + threadIdx.x];
  for (int e = threadIdx.x; e < 64 * kD; e += blockDim.x) {
    const int kr = e / kD, n = e % kD;
    tile[kr][n] = (float)src[(int64_t)kr * kD + n];
  }
  __syncthreads();
  uint4 *out = img + (lhm * nchunk + c) * (kChunkBytes / 16);
  for (int q = threadIdx.x; q < kChunkBytes / 16; q += blockDim.x) {
    const int n = q >> 3, k8 = (q & 7) ^ (n & 7);
    const int ch = chan_of_col(n);   // the epilogue's column order
    uint32_t v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      v[e] = pack_bf16(tile[k8 * 8 + 2 * e][ch], tile[k8 * 8 + 2 * e + 1][ch]);
    out[q] = make_uint4(v[0], v[1], v[2], v[3]);
  }
}

size_t smem_bytes(int k, int stages, int pair) {
  return 1024 + (size_t)2 * k * (kChunkBytes / pair) + (size_t)stages * kStageBytes +
         (pair == 2 ? kCplBytes : 0) + sizeof(Shared) + 64;
}

int max_stages(int k, int pair) {
  int s = kMaxStages;
  while (s > 1 && smem_bytes(k, s, pair) > (size_t)kSmemLimit) --s;
  return s;
}

// 4-D TMA map over a [Ls][ntok][H][128] bf16 cache: box [1][128][1][64],
// 128-byte swizzle, out-of-range rows read as zero.
bool encode_map(const kvx_plan *plan, CUtensorMap *map, const void *base, const KvxParams &p) {
  typedef CUresult (*EncodeFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                               const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                               const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                               CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  EncodeFn fn = reinterpret_cast<EncodeFn>(plan->encode_tiled);
  if (!fn) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)p.H, (cuuint64_t)p.ntok,
                              (cuuint64_t)p.Ls};
  const cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)p.H * kD * 2,
                                 (cuuint64_t)p.src_rows * p.H * kD * 2};
  const cuuint32_t box[4] = {(cuuint32_t)kHalf, 1u, (cuuint32_t)kTileM, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D TMA map over the source-RoPE quad table [16][max_position] of 16-byte
// elements, seen as 8-byte elements: box [16 quads][128 positions].
bool encode_cpl_map(const kvx_plan *plan, CUtensorMap *map, const KvxParams &p) {
  typedef CUresult (*EncodeFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                               const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                               const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                               CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  EncodeFn fn = reinterpret_cast<EncodeFn>(plan->encode_tiled);
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)2 * p.max_position, (cuuint64_t)(kD / 8)};
  const cuuint64_t strides[1] = {(cuuint64_t)p.max_position * 16};
  const cuuint32_t box[2] = {(cuuint32_t)(2 * kTileM), (cuuint32_t)(kD / 8)};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, plan->tc_rope_src, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

static size_t w_image_bytes(const kvx_plan_desc &d) {
  return (size_t)d.tgt_layers * d.src_kv_heads * 2 * (size_t)d.k * kD * kD * 2;
}

bool kvx_tc_supports(const kvx_plan_desc &d) {
  return d.kv_dtype == KVX_BF16 && d.src_head_dim == kD && d.k >= 1 && d.k <= kMaxK;
}

size_t kvx_tc_workspace_bytes(const kvx_plan_desc &d) {
  return w_image_bytes(d) + (size_t)d.tgt_layers * d.src_kv_heads * 2 * kD * sizeof(float);
}

void *kvx_tc_encoder() {
  void *fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return fn;
}

cudaError_t kvx_tc_prepare(kvx_plan *plan) {
  if (!plan->encode_tiled) return cudaErrorNotSupported;
  const int k = plan->desc.k;
  cudaError_t e = cudaFuncSetAttribute(tc_transfer_kernel<1>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem_bytes(k, max_stages(k, 1), 1));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tc_transfer_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem_bytes(k, max_stages(k, 2), 2));
  if (e != cudaSuccess) return e;
  // CTA pairs that can be resident at once (0: run single CTAs)
  plan->tc_pairs = 0;
  if (!(plan->desc.flags & KVX_PLAN_TC_SINGLE_CTA)) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * plan->num_sms, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem_bytes(k, max_stages(k, 2), 2);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tc_transfer_kernel<2>, &cfg) == cudaSuccess)
      plan->tc_pairs = n;
    else
      cudaGetLastError();
  }
  return cudaSuccess;
}

cudaError_t kvx_tc_launch(const kvx_plan *plan, const KvxParams &p_in, cudaStream_t s) {
  const kvx_plan_desc &d = plan->desc;
  // 0. a paged source: its rows gathered into packed order first (the TMA
  // boxes read 128 consecutive rows); the kernel still applies the source
  // block checks to skip and flag the tokens it cannot read
  KvxParams p = p_in;
  const bool paged_src = p.src_layout == KVX_PAGED;
  if (paged_src) {
    p.src_k = plan->packed_k;
    p.src_v = plan->packed_v;
    p.src_rows = plan->max_tokens;
  }
  // the tensor maps before any launch: a map the driver refuses is reported
  // with nothing enqueued
  CUtensorMap mk, mv, mc;
  if (!encode_map(plan, &mk, p.src_k, p) || !encode_map(plan, &mv, p.src_v, p) ||
      !encode_cpl_map(plan, &mc, p))
    return cudaErrorInvalidValue;
  if (paged_src) {
    cudaError_t pe =
        kvx_pack_source(p_in, plan->packed_k, plan->packed_v, plan->max_tokens, 2, s);
    if (pe != cudaSuccess) return pe;
  }
  // 1. W -> bf16 image in the plan workspace
  dim3 wgrid((unsigned)((int64_t)p.Lt * p.H * 2), (unsigned)(2 * p.k));
  uint4 *img = reinterpret_cast<uint4 *>(plan->workspace);
  float *bimg = reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(plan->workspace) +
                                          w_image_bytes(d));
  using bf = __nv_bfloat16;
  const bool wf = d.w_dtype == KVX_F32, bfp = d.b_dtype == KVX_F32;
  if (wf && bfp)
    w_image_kernel<float, float><<<wgrid, 256, 0, s>>>((const float *)p.w, img, (const float *)p.b, bimg);
  else if (wf)
    w_image_kernel<float, bf><<<wgrid, 256, 0, s>>>((const float *)p.w, img, (const bf *)p.b, bimg);
  else if (bfp)
    w_image_kernel<bf, float><<<wgrid, 256, 0, s>>>((const bf *)p.w, img, (const float *)p.b, bimg);
  else
    w_image_kernel<bf, bf><<<wgrid, 256, 0, s>>>((const bf *)p.w, img, (const bf *)p.b, bimg);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // 2. the persistent transfer kernel: CTA pairs (one M = 256 MMA per K step
  // over both CTAs' rows) when the device can co-schedule them, else single CTAs
  const int P = plan->tc_pairs > 0 ? 2 : 1;
  ItemGeom geo;
  geo.num_tiles = (int)((p.ntok + kTileM * P - 1) / (kTileM * P));
  geo.tiles_per_item = plan->tiles_per_item;
  geo.num_chunks = (geo.num_tiles + geo.tiles_per_item - 1) / geo.tiles_per_item;
  geo.num_items = (long long)p.H * geo.num_chunks * p.Lt * 2;
  geo.stages = max_stages(p.k, P);
  const long long slots = P == 2 ? plan->tc_pairs : plan->num_sms;
  geo.stride = geo.num_items < slots ? geo.num_items : slots;
  RopeTurns rope;
  for (int i = 0; i < kHalf; ++i) rope.tgt[i] = plan->turns_tgt[i];
  const uint4 *rope_src4 = reinterpret_cast<const uint4 *>(plan->tc_rope_src);
  const __nv_bfloat16 *wimg = reinterpret_cast<const __nv_bfloat16 *>(plan->workspace);
  const size_t smem = smem_bytes(p.k, geo.stages, P);
  if (P == 1) {
    tc_transfer_kernel<1><<<(unsigned)geo.stride, kThreads, smem, s>>>(
        p, mk, mv, mc, rope_src4, rope, bimg, wimg, geo, plan->stall_test);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * geo.stride), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc_transfer_kernel<2>, p, mk, mv, mc, rope_src4, rope, bimg,
                            wimg, geo, plan->stall_test);
}
