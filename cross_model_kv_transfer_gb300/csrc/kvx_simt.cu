// kvx_simt.cu -- the transfer with an fp32 FMA contraction on the CUDA cores.
//
// Used for fp32 caches (where bf16 tensor-core operands would not meet an
// fp32 tolerance) and for head dimensions the tensor-core kernel does not
// take.  One CTA computes one (target layer lt, head h, K|V, tile of up to
// 8*G consecutive packed source rows, which may span requests):
//   1. gather the k selected source rows of each token into shared memory,
//      un-rotating keys out of the source RoPE ("Helm Intelligent Routing",
//      "Why carrying the cache across is the hard part", step 1; Qwen3
//      article, linear-bridge section: concatenate the selected layers'
//      features, strip source RoPE before mapping keys),
//   2. y = x W + b in fp32, thread (i, y) owning output channels i and
//      i + d/2 of 8 tokens, so the RoPE pair of step 3 stays in registers
//      (step 2: per-layer, per-head linear map),
//   3. re-rotate keys into the target RoPE at p' (step 3), store to the
//      contiguous or paged target cache.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "kvx_device.cuh"
#include "kvx_internal.h"

namespace {

constexpr int kRowsPerThread = 8;
constexpr int kThreads = 128;

__device__ __forceinline__ float ldf(const float *p) { return __ldg(p); }
__device__ __forceinline__ float ldf(const __nv_bfloat16 *p) {
  return __bfloat162float(__ldg(p));
}
__device__ __forceinline__ void stf(float *p, float v) { *p = v; }
__device__ __forceinline__ void stf(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

int row_groups(int half) { return half >= kThreads ? 1 : kThreads / half; }

size_t smem_bytes(int half, int kd) {
  const int tt = kRowsPerThread * row_groups(half);
  return (size_t)tt * (kd + 1) * sizeof(float) +
         (size_t)tt * (2 * sizeof(int64_t) + 2 * sizeof(int32_t));
}

template <typename KT, typename WT, typename BT>
__global__ void __launch_bounds__(kThreads) simt_transfer_kernel(KvxParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int half = p.d >> 1;
  const int G = blockDim.y;
  const int TT = kRowsPerThread * G;
  const int kd = p.k * p.d;
  const int ldx = kd + 1;
  float *X = reinterpret_cast<float *>(smem_raw);
  int64_t *s_row = reinterpret_cast<int64_t *>(X + (size_t)TT * ldx);
  int64_t *s_srow = s_row + TT;                  // row of the token in the source arrays
  int32_t *s_ps = reinterpret_cast<int32_t *>(s_srow + TT);
  int32_t *s_pt = s_ps + TT;
  __shared__ uint32_t s_bits;
  __shared__ int s_layer_ok;

  const int tx = threadIdx.x, ty = threadIdx.y;
  const int tid = ty * blockDim.x + tx;
  const int z = blockIdx.z;
  const int m = z & 1;  // 0: keys, 1: values
  const int h = (z >> 1) % p.H;
  const int lt = (z >> 1) / p.H;

  if (!kvx::seqlens_ok(p, tid, blockDim.x * blockDim.y)) {
    if (blockIdx.x == 0 && z == 0 && tid == 0) kvx::report(p, KVX_FLAG_BAD_SEQLENS);
    return;
  }
  const int64_t t0 = (int64_t)blockIdx.x * TT;

  if (tid == 0) {
    s_bits = 0;
    s_layer_ok = kvx::layer_row_ok(p, lt);
  }
  __syncthreads();
  // one entry per tile row; for head dims below 16 a tile has more rows
  // (8 G) than the CTA has threads (d/2 x G), so the threads stride over them
  for (int q = tid; q < TT; q += blockDim.x * blockDim.y) {
    const int64_t g = t0 + q;
    int32_t ps = 0, pt = 0;
    int64_t row = -1, srow = -1;
    if (g < p.ntok) {
      const uint32_t bad = kvx::token_meta(p, g, ps, pt, row, srow);
      if (bad) atomicOr(&s_bits, bad);
    }
    s_row[q] = row;
    s_srow[q] = srow;
    s_ps[q] = ps;
    s_pt[q] = pt;
  }
  __syncthreads();
  if (tid == 0) {
    // row errors are reported by the (lt 0, head 0, K) CTAs, layer errors by
    // the first token tile with head 0, K
    uint32_t bits = (lt == 0 && h == 0 && m == 0) ? s_bits : 0u;
    if (!s_layer_ok && blockIdx.x == 0 && h == 0 && m == 0) bits |= KVX_FLAG_BAD_LAYER_INDEX;
    kvx::report(p, bits);
  }
  if (!s_layer_ok) return;

  // ---- 1. gather + un-rotate (keys) into X[TT][k*d] -----------------------
  const KT *src = reinterpret_cast<const KT *>(m == 0 ? p.src_k : p.src_v);
  for (int q = ty; q < TT; q += G) {
    if (s_row[q] < 0) continue;
    const int64_t srow = s_srow[q];
    for (int i = tx; i < half; i += blockDim.x) {
      float c = 1.f, s = 0.f;
      if (m == 0) {
        const float2 cs = p.rope_src[(int64_t)s_ps[q] * half + i];
        c = cs.x;
        s = cs.y;
      }
      for (int j = 0; j < p.k; ++j) {
        const int sl = p.layer_idx[lt * p.k + j];
        const KT *v = src + (((int64_t)sl * p.src_rows + srow) * p.H + h) * p.d;
        const float x0 = ldf(v + i), x1 = ldf(v + i + half);
        // un-rotate: multiply (x0 + j x1) by exp(-j p w_i)
        X[q * ldx + j * p.d + i] = m == 0 ? fmaf(x0, c, x1 * s) : x0;
        X[q * ldx + j * p.d + i + half] = m == 0 ? fmaf(x1, c, -x0 * s) : x1;
      }
    }
  }
  __syncthreads();

  // ---- 2. y = x W + b (fp32) ----------------------------------------------
  const WT *W = reinterpret_cast<const WT *>(p.w) + (((int64_t)lt * p.H + h) * 2 + m) * kd * p.d;
  const BT *B = reinterpret_cast<const BT *>(p.b) + (((int64_t)lt * p.H + h) * 2 + m) * p.d;
  for (int i = tx; i < half; i += blockDim.x) {
    float acc0[kRowsPerThread], acc1[kRowsPerThread];
#pragma unroll
    for (int rr = 0; rr < kRowsPerThread; ++rr) acc0[rr] = acc1[rr] = 0.f;
    for (int qq = 0; qq < kd; ++qq) {
      const float w0 = ldf(W + (int64_t)qq * p.d + i);
      const float w1 = ldf(W + (int64_t)qq * p.d + i + half);
#pragma unroll
      for (int rr = 0; rr < kRowsPerThread; ++rr) {
        const float xv = X[(ty + rr * G) * ldx + qq];
        acc0[rr] = fmaf(xv, w0, acc0[rr]);
        acc1[rr] = fmaf(xv, w1, acc1[rr]);
      }
    }
    const float b0 = ldf(B + i), b1 = ldf(B + i + half);

    // ---- 3. bias, re-rotate keys at p', store -----------------------------
    KT *dst = reinterpret_cast<KT *>(m == 0 ? p.dst_k : p.dst_v);
#pragma unroll
    for (int rr = 0; rr < kRowsPerThread; ++rr) {
      const int q = ty + rr * G;
      const int64_t row = s_row[q];
      if (row < 0) continue;
      float y0 = acc0[rr] + b0, y1 = acc1[rr] + b1;
      if (m == 0) {
        const float2 cs = p.rope_tgt[(int64_t)s_pt[q] * half + i];
        const float r0 = fmaf(y0, cs.x, -y1 * cs.y);  // (y0 + j y1) exp(+j p' w_i)
        const float r1 = fmaf(y0, cs.y, y1 * cs.x);
        y0 = r0;
        y1 = r1;
      }
      KT *o = dst + (((int64_t)lt * p.dst_rows + row) * p.H + h) * p.d;
      stf(o + i, y0);
      stf(o + i + half, y1);
    }
  }
}

template <typename KT, typename WT, typename BT>
void *kernel_ptr() {
  return reinterpret_cast<void *>(&simt_transfer_kernel<KT, WT, BT>);
}

void *select_kernel(const kvx_plan_desc &d) {
  const bool kb = d.kv_dtype == KVX_BF16, wb = d.w_dtype == KVX_BF16, bb = d.b_dtype == KVX_BF16;
  using bf = __nv_bfloat16;
  if (kb) {
    if (wb) return bb ? kernel_ptr<bf, bf, bf>() : kernel_ptr<bf, bf, float>();
    return bb ? kernel_ptr<bf, float, bf>() : kernel_ptr<bf, float, float>();
  }
  if (wb) return bb ? kernel_ptr<float, bf, bf>() : kernel_ptr<float, bf, float>();
  return bb ? kernel_ptr<float, float, bf>() : kernel_ptr<float, float, float>();
}

constexpr size_t kMaxSmem = 227 * 1024;

}  // namespace

bool kvx_simt_supports(const kvx_plan_desc &d) {
  const int half = d.src_head_dim / 2;
  if ((int64_t)d.tgt_layers * d.src_kv_heads * 2 > 65535) return false;
  return smem_bytes(half, d.k * d.src_head_dim) + 64 <= kMaxSmem;
}

cudaError_t kvx_simt_prepare(const kvx_plan *plan) {
  const kvx_plan_desc &d = plan->desc;
  const size_t bytes = smem_bytes(plan->half, d.k * d.src_head_dim);
  return cudaFuncSetAttribute(select_kernel(d), cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)bytes);
}

cudaError_t kvx_simt_launch(const kvx_plan *plan, const KvxParams &p, cudaStream_t s) {
  const int half = plan->half;
  const int G = row_groups(half);
  const int tt = kRowsPerThread * G;
  dim3 block(half >= kThreads ? kThreads : half, G);
  dim3 grid((unsigned)((p.ntok + tt - 1) / tt), 1u, (unsigned)(p.Lt * p.H * 2));
  const size_t bytes = smem_bytes(half, p.k * p.d);
  void *fn = select_kernel(plan->desc);
  KvxParams pp = p;
  void *args[] = {&pp};
  return cudaLaunchKernel(fn, grid, block, args, bytes, s);
}

// ---------------------------------------------------------------------------
// Allocation-free entry point (kvx_transfer_static).
//
// Some callers cannot allocate device memory: serving engines that reserve
// nearly all of the GPU for their own paged KV-cache pool and forbid later
// cudaMalloc calls, and latency-critical paths where cudaMalloc/cudaFree
// (which may synchronise the device) are not acceptable.  This entry point
// runs the SIMT transfer kernel above without a plan: the RoPE tables it
// needs live in one fixed file-scope device array, filled on the device by
// every call.  The array holds kStaticRopeEntries (cos, sin) pairs, 8 MiB,
// and stays allocated on every GPU that loads the library until the process
// exits.  All calls share it, so calls whose kernels overlap on the GPU (for
// example on two streams) race on it; order them.  Nothing in it has to
// start at zero: each call rewrites the part it reads.
// ---------------------------------------------------------------------------
#include <mutex>

namespace {

constexpr size_t kStaticRopeEntries = (size_t)1 << 20;   // 8 MiB of float2
static __device__ __align__(256) float2 g_static_rope[kStaticRopeEntries];

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
float2 *g_static_ptr[kMaxDevices];    // device address of g_static_rope, per device
unsigned long long g_static_ctx[kMaxDevices];   // id of the context it was looked up in

// Unique id of the calling thread's current CUDA context (never reused within
// a process), 0 if there is none or the driver does not report it.  A device
// reset destroys the primary context and the module with it, so an address
// looked up in an earlier context is stale; the id tells the two apart.
unsigned long long current_context_id() {
  typedef int (*GetCurrentFn)(void **);
  typedef int (*GetIdFn)(void *, unsigned long long *);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    void *f = nullptr, *g = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q1) ==
            cudaSuccess &&
        q1 == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &g, 12000, cudaEnableDefault, &q2) ==
            cudaSuccess &&
        q2 == cudaDriverEntryPointSuccess) {
      get_current = reinterpret_cast<GetCurrentFn>(f);
      get_id = reinterpret_cast<GetIdFn>(g);
    } else {
      cudaGetLastError();
    }
    looked_up = true;
  }
  if (!get_current || !get_id) return 0;
  void *ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != 0 || !ctx || get_id(ctx, &id) != 0) return 0;
  return id;
}

// cos/sin(p * theta^(-2i/d)) for p in [0, max_position), i in [0, d/2), in
// double precision on the device, rounded once to fp32; same layout as the
// plan tables ([p][i]); the target table follows the source table.
__global__ void static_rope_fill_kernel(float2 *dst, int d, int max_position, double theta_src,
                                        double theta_tgt, int two_tables) {
  const int half = d / 2;
  const int64_t per = (int64_t)max_position * half;
  const int64_t n = per * (two_tables ? 2 : 1);
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(e / per);
    const int64_t r = e - t * per;
    const int p = (int)(r / half), i = (int)(r % half);
    const double w = pow(t ? theta_tgt : theta_src, -2.0 * (double)i / (double)d);
    double s, c;
    sincos((double)p * w, &s, &c);
    dst[e] = make_float2((float)c, (float)s);
  }
}

bool static_dtype_ok(int32_t t) { return t == KVX_F32 || t == KVX_BF16; }

}  // namespace

extern "C" kvx_status kvx_transfer_static(const kvx_plan_desc *desc,
                                          const kvx_transfer_args *a, void *stream) {
  // descriptor: the same rules as kvx_plan_create
  if (!desc || !a) return KVX_ERR_INVALID_ARG;
  const kvx_plan_desc &d = *desc;
  if (d.src_layers < 1 || d.tgt_layers < 1 || d.k < 1 || d.k > 64 || d.src_kv_heads < 1 ||
      d.tgt_kv_heads < 1 || d.src_head_dim < 2 || d.tgt_head_dim < 2 || d.src_head_dim > 256 ||
      d.tgt_head_dim > 256 || (d.src_head_dim & 1) || (d.tgt_head_dim & 1) ||
      !(d.rope_theta_src > 0.0 && d.rope_theta_src < 1e300) ||
      !(d.rope_theta_tgt > 0.0 && d.rope_theta_tgt < 1e300) || !static_dtype_ok(d.kv_dtype) ||
      !static_dtype_ok(d.w_dtype) || !static_dtype_ok(d.b_dtype) ||
      (d.dst_layout != KVX_CONTIGUOUS && d.dst_layout != KVX_PAGED) ||
      (d.dst_layout == KVX_PAGED && d.block_size < 1) || d.max_position < 1 ||
      (d.kernel != KVX_KERNEL_AUTO && d.kernel != KVX_KERNEL_SIMT) || d.flags != 0 ||
      d.mapper != KVX_MAPPER_PER_HEAD ||
      (d.src_layout != KVX_CONTIGUOUS && d.src_layout != KVX_PAGED) ||
      (d.src_layout == KVX_PAGED && d.src_block_size < 1))
    return KVX_ERR_INVALID_ARG;
  if (d.src_kv_heads != d.tgt_kv_heads || d.src_head_dim != d.tgt_head_dim)
    return KVX_ERR_PAIR_MISMATCH;
  if (!kvx_simt_supports(d)) return KVX_ERR_UNSUPPORTED;
  const int half = d.src_head_dim / 2;
  const bool two = d.rope_theta_tgt != d.rope_theta_src;
  if ((size_t)d.max_position * half * (two ? 2 : 1) > kStaticRopeEntries) return KVX_ERR_TOO_LARGE;

  // arguments: the same rules as kvx_transfer
  if (a->ntok < 0 || a->ntok > INT32_MAX || a->num_requests < 1 ||
      (!a->cu_seqlens && a->num_requests != 1) || !a->src_k || !a->src_v || !a->layer_idx ||
      !a->w || !a->b || !a->dst_k || !a->dst_v)
    return KVX_ERR_INVALID_ARG;
  if (d.dst_layout == KVX_CONTIGUOUS ? a->dst_capacity < 1
                                     : (a->num_blocks < 1 || !a->block_table ||
                                        a->max_blocks_per_req < 1))
    return KVX_ERR_INVALID_ARG;
  const bool src_paged = d.src_layout == KVX_PAGED;
  if (src_paged && (a->src_num_blocks < 1 || !a->src_block_table || a->max_src_blocks_per_req < 1))
    return KVX_ERR_INVALID_ARG;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVX_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KVX_ERR_UNSUPPORTED;
  {
    // once per device and context, with that device current: the device
    // address of the static array (its host-side name is only a stand-in for
    // it).  The lookup is repeated when the device's context has been
    // recreated (cudaDeviceReset), since the old address no longer holds.
    std::lock_guard<std::mutex> lock(g_static_mu);
    const unsigned long long ctx = current_context_id();
    if (!g_static_ptr[dev] || ctx == 0 || ctx != g_static_ctx[dev]) {
      cudaDeviceProp prop;
      if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return KVX_ERR_CUDA;
      if (prop.major != 10 || prop.minor != 3) return KVX_ERR_UNSUPPORTED;
      void *ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_static_rope) != cudaSuccess || !ptr) return KVX_ERR_CUDA;
      g_static_ptr[dev] = static_cast<float2 *>(ptr);
      g_static_ctx[dev] = current_context_id();   // the lookup made the context current
    }
  }
  if (a->ntok == 0) return KVX_OK;

  // the kernel's dynamic shared memory limit is raised, never lowered
  void *fn = select_kernel(d);
  const size_t bytes = smem_bytes(half, d.k * d.src_head_dim);
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) return KVX_ERR_CUDA;
  if ((size_t)fa.maxDynamicSharedSizeBytes < bytes &&
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) !=
          cudaSuccess)
    return KVX_ERR_CUDA;

  cudaStream_t s = (cudaStream_t)stream;
  float2 *rope = g_static_ptr[dev];
  const int64_t entries = (int64_t)d.max_position * half * (two ? 2 : 1);
  const int fill_blocks = (int)((entries + 255) / 256 < 4096 ? (entries + 255) / 256 : 4096);
  static_rope_fill_kernel<<<fill_blocks, 256, 0, s>>>(rope, d.src_head_dim, d.max_position,
                                                      d.rope_theta_src, d.rope_theta_tgt,
                                                      two ? 1 : 0);
  if (cudaGetLastError() != cudaSuccess) return KVX_ERR_CUDA;

  kvx_plan tmp;                     // launch description only; owns nothing
  std::memset(&tmp, 0, sizeof(tmp));
  tmp.desc = d;
  tmp.device = dev;
  tmp.kernel = KVX_KERNEL_SIMT;
  tmp.half = half;
  tmp.rope_src = rope;
  tmp.rope_tgt = two ? rope + (size_t)d.max_position * half : rope;

  KvxParams p;
  std::memset(&p, 0, sizeof(p));
  p.src_k = a->src_k;
  p.src_v = a->src_v;
  p.w = a->w;
  p.b = a->b;
  p.dst_k = a->dst_k;
  p.dst_v = a->dst_v;
  p.cu_seqlens = a->cu_seqlens;
  p.layer_idx = a->layer_idx;
  p.src_pos = a->src_pos;
  p.tgt_pos = a->tgt_pos;
  p.tgt_offset = a->tgt_offset;
  p.block_table = a->block_table;
  p.status = a->status;
  p.rope_src = tmp.rope_src;
  p.rope_tgt = tmp.rope_tgt;
  p.ntok = a->ntok;
  p.dst_capacity = a->dst_capacity;
  p.num_blocks = a->num_blocks;
  p.dst_rows = d.dst_layout == KVX_CONTIGUOUS ? (int64_t)a->num_requests * a->dst_capacity
                                              : a->num_blocks * (int64_t)d.block_size;
  p.R = a->num_requests;
  p.max_blocks = a->max_blocks_per_req;
  p.Ls = d.src_layers;
  p.Lt = d.tgt_layers;
  p.H = d.src_kv_heads;
  p.d = d.src_head_dim;
  p.k = d.k;
  p.layout = d.dst_layout;
  p.block_size = d.block_size;
  p.max_position = d.max_position;
  p.src_layout = d.src_layout;
  p.src_block_size = src_paged ? d.src_block_size : 1;
  p.src_max_blocks = src_paged ? a->max_src_blocks_per_req : 0;
  p.src_num_blocks = src_paged ? a->src_num_blocks : 0;
  p.src_block_table = src_paged ? a->src_block_table : nullptr;
  p.src_rows = src_paged ? a->src_num_blocks * (int64_t)d.src_block_size : a->ntok;
  return kvx_simt_launch(&tmp, p, s) == cudaSuccess ? KVX_OK : KVX_ERR_CUDA;
}
