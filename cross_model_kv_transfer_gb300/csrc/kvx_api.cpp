// kvx_api.cpp -- host side of the C ABI declared in include/kvx.h: argument
// validation, plan creation (RoPE tables), kernel selection and launch.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "kvx_internal.h"

namespace {

bool valid_dtype(int32_t t) { return t == KVX_F32 || t == KVX_BF16; }

kvx_status validate_desc(const kvx_plan_desc *d) {
  if (!d) return KVX_ERR_INVALID_ARG;
  if (d->src_layers < 1 || d->tgt_layers < 1 || d->k < 1 || d->k > 64)
    return KVX_ERR_INVALID_ARG;
  if (d->src_kv_heads < 1 || d->tgt_kv_heads < 1) return KVX_ERR_INVALID_ARG;
  if (d->src_head_dim < 2 || d->tgt_head_dim < 2 || d->src_head_dim > 256 ||
      d->tgt_head_dim > 256 || (d->src_head_dim & 1) || (d->tgt_head_dim & 1))
    return KVX_ERR_INVALID_ARG;
  if (!(std::isfinite(d->rope_theta_src) && d->rope_theta_src > 0.0) ||
      !(std::isfinite(d->rope_theta_tgt) && d->rope_theta_tgt > 0.0))
    return KVX_ERR_INVALID_ARG;
  if (!valid_dtype(d->kv_dtype) || !valid_dtype(d->w_dtype) || !valid_dtype(d->b_dtype))
    return KVX_ERR_INVALID_ARG;
  if (d->dst_layout != KVX_CONTIGUOUS && d->dst_layout != KVX_PAGED)
    return KVX_ERR_INVALID_ARG;
  if (d->dst_layout == KVX_PAGED && d->block_size < 1) return KVX_ERR_INVALID_ARG;
  if (d->max_position < 1) return KVX_ERR_INVALID_ARG;
  if (d->kernel != KVX_KERNEL_AUTO && d->kernel != KVX_KERNEL_SIMT &&
      d->kernel != KVX_KERNEL_TCGEN05)
    return KVX_ERR_INVALID_ARG;
  if (d->tiles_per_item < 0 || d->tiles_per_item > 4096) return KVX_ERR_INVALID_ARG;
  if (d->flags & ~(KVX_PLAN_TEST_STALL | KVX_PLAN_TC_SINGLE_CTA)) return KVX_ERR_INVALID_ARG;
  if (d->mapper != KVX_MAPPER_PER_HEAD && d->mapper != KVX_MAPPER_WIDE) return KVX_ERR_INVALID_ARG;
  if (d->max_tokens < 0) return KVX_ERR_INVALID_ARG;
  if (d->src_layout != KVX_CONTIGUOUS && d->src_layout != KVX_PAGED) return KVX_ERR_INVALID_ARG;
  if (d->src_layout == KVX_PAGED && d->src_block_size < 1) return KVX_ERR_INVALID_ARG;
  // "Requirements": same number of KV heads and the same per-head dimension.
  if (d->src_kv_heads != d->tgt_kv_heads || d->src_head_dim != d->tgt_head_dim)
    return KVX_ERR_PAIR_MISMATCH;
  return KVX_OK;
}

// cos/sin of p * theta^(-2i/d) for p in [0, max_position), i in [0, d/2):
// angles and trigonometry in double precision, rounded once to fp32.
std::vector<float2> rope_table(double theta, int d, int max_position) {
  const int half = d / 2;
  std::vector<float2> t((size_t)max_position * half);
  for (int i = 0; i < half; ++i) {
    const double w = std::pow(theta, -2.0 * (double)i / (double)d);
    for (int p = 0; p < max_position; ++p) {
      const double a = (double)p * w;
      t[(size_t)p * half + i] = make_float2((float)std::cos(a), (float)std::sin(a));
    }
  }
  return t;
}

// Round a double to the nearest bf16 (ties to even) in one step; returns
// the 16-bit pattern.  Used for |x| <= 1 (cos/sin), normal or zero.
uint16_t bf16_bits(double x) {
  if (x == 0.0) return std::signbit(x) ? 0x8000u : 0u;
  int e;
  const double m = std::frexp(x, &e);                  // |m| in [0.5, 1)
  const double r = std::nearbyint(std::ldexp(m, 8));   // 8 significant bits, ties to even
  const float f = (float)std::ldexp(r, e - 8);         // exact
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

// Tensor-core path source table, position-major per quad of pairs
// (4u .. 4u + 3): element [u][p] is 16 bytes, bf16x2 (cos_4u, cos_4u+1),
// (sin_4u, sin_4u+1), (cos_4u+2, cos_4u+3), (sin_4u+2, sin_4u+3) of p * w_i,
// so one tile's 128 consecutive positions of all quads are a 2-D TMA box.
void tc_rope_table(double theta, int d, int max_position, std::vector<uint32_t> &src) {
  const int quads = d / 8;
  src.assign((size_t)quads * max_position * 4, 0);
  for (int u = 0; u < quads; ++u) {
    double w[4];
    for (int e = 0; e < 4; ++e) w[e] = std::pow(theta, -2.0 * (4 * u + e) / d);
    for (int p = 0; p < max_position; ++p) {
      const size_t o = ((size_t)u * max_position + p) * 4;
      for (int h = 0; h < 2; ++h) {
        const double a0 = p * w[2 * h], a1 = p * w[2 * h + 1];
        src[o + 2 * h] =
            (uint32_t)bf16_bits(std::cos(a0)) | ((uint32_t)bf16_bits(std::cos(a1)) << 16);
        src[o + 2 * h + 1] =
            (uint32_t)bf16_bits(std::sin(a0)) | ((uint32_t)bf16_bits(std::sin(a1)) << 16);
      }
    }
  }
}

// w_i / (2 pi) as a 64-bit binary fraction of a turn, in extended precision.
void rope_turns(double theta, int d, unsigned long long *out) {
  const long double two_pi = 6.283185307179586476925286766559005768L;
  for (int i = 0; i < d / 2; ++i) {
    const long double w = powl((long double)theta, -2.0L * (long double)i / (long double)d);
    const long double f = w / two_pi;                  // turns per position
    const long double x = ldexpl(f - floorl(f), 32);   // [0, 2^32)
    const long double hi = floorl(x);
    const long double lo = roundl(ldexpl(x - hi, 32)); // [0, 2^32]
    unsigned long long v = (unsigned long long)hi << 32;
    v += (unsigned long long)lo;                       // a carry wraps mod 2^64 = mod 1 turn
    out[i] = v;
  }
}

kvx_status upload_bytes(const void *h, size_t bytes, void **dptr) {
  cudaError_t e = cudaMalloc(dptr, bytes);
  if (e == cudaErrorMemoryAllocation) {
    cudaGetLastError();
    *dptr = nullptr;
    return KVX_ERR_NO_MEMORY;
  }
  if (e != cudaSuccess) {
    *dptr = nullptr;
    return KVX_ERR_CUDA;
  }
  if (cudaMemcpy(*dptr, h, bytes, cudaMemcpyHostToDevice) != cudaSuccess) return KVX_ERR_CUDA;
  return KVX_OK;
}

kvx_status upload(const std::vector<float2> &h, float2 **dptr) {
  size_t bytes = h.size() * sizeof(float2);
  cudaError_t e = cudaMalloc((void **)dptr, bytes);
  if (e == cudaErrorMemoryAllocation) {
    cudaGetLastError();
    *dptr = nullptr;
    return KVX_ERR_NO_MEMORY;
  }
  if (e != cudaSuccess) {
    *dptr = nullptr;
    return KVX_ERR_CUDA;
  }
  if (cudaMemcpy(*dptr, h.data(), bytes, cudaMemcpyHostToDevice) != cudaSuccess)
    return KVX_ERR_CUDA;
  return KVX_OK;
}

void free_tables(kvx_plan *p) {
  if (p->rope_tgt && p->rope_tgt != p->rope_src) cudaFree(p->rope_tgt);
  if (p->rope_src) cudaFree(p->rope_src);
  if (p->workspace) cudaFree(p->workspace);
  if (p->tc_rope_src) cudaFree(p->tc_rope_src);
  if (p->packed_k) cudaFree(p->packed_k);
  if (p->packed_v) cudaFree(p->packed_v);
  p->rope_src = p->rope_tgt = nullptr;
  p->workspace = p->tc_rope_src = nullptr;
  p->packed_k = p->packed_v = nullptr;
}

kvx_status alloc_bytes(void **ptr, size_t bytes) {
  *ptr = nullptr;
  if (bytes == 0) return KVX_OK;
  cudaError_t e = cudaMalloc(ptr, bytes);
  if (e == cudaErrorMemoryAllocation) {
    cudaGetLastError();
    *ptr = nullptr;
    return KVX_ERR_NO_MEMORY;
  }
  if (e != cudaSuccess) {
    *ptr = nullptr;
    return KVX_ERR_CUDA;
  }
  return KVX_OK;
}

kvx_status alloc_workspace(kvx_plan *p, size_t bytes) {
  p->workspace_bytes = bytes;
  if (bytes == 0) return KVX_OK;
  cudaError_t e = cudaMalloc(&p->workspace, bytes);
  if (e == cudaErrorMemoryAllocation) {
    cudaGetLastError();
    p->workspace = nullptr;
    return KVX_ERR_NO_MEMORY;
  }
  if (e != cudaSuccess) {
    p->workspace = nullptr;
    return KVX_ERR_CUDA;
  }
  return KVX_OK;
}

}  // namespace

extern "C" {

const char *kvx_status_string(kvx_status s) {
  switch (s) {
    case KVX_OK: return "ok";
    case KVX_ERR_INVALID_ARG: return "invalid argument";
    case KVX_ERR_PAIR_MISMATCH:
      return "source and target differ in KV-head count or head dimension";
    case KVX_ERR_UNSUPPORTED: return "unsupported device or configuration";
    case KVX_ERR_CUDA: return "CUDA runtime error";
    case KVX_ERR_NO_MEMORY: return "out of device memory";
    case KVX_ERR_TOO_LARGE:
      return "RoPE tables exceed the fixed device array of the allocation-free entry point";
  }
  return "unknown status";
}

kvx_status kvx_plan_create(const kvx_plan_desc *desc, kvx_plan **out) {
  if (!out) return KVX_ERR_INVALID_ARG;
  *out = nullptr;
  kvx_status st = validate_desc(desc);
  if (st != KVX_OK) return st;

  const bool wide = desc->mapper == KVX_MAPPER_WIDE;
  int kernel = desc->kernel;
  if (wide) {
    // the wide map runs only as the tensor-core contraction
    if (kernel == KVX_KERNEL_SIMT || !kvx_wide_supports(*desc)) return KVX_ERR_UNSUPPORTED;
    kernel = KVX_KERNEL_TCGEN05;
  }
  if (kernel == KVX_KERNEL_AUTO)
    kernel = kvx_tc_supports(*desc) ? KVX_KERNEL_TCGEN05 : KVX_KERNEL_SIMT;
  if (!wide && kernel == KVX_KERNEL_TCGEN05 && !kvx_tc_supports(*desc)) return KVX_ERR_UNSUPPORTED;
  if (kernel == KVX_KERNEL_SIMT && !kvx_simt_supports(*desc)) return KVX_ERR_UNSUPPORTED;

  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) {
    cudaGetLastError();
    return KVX_ERR_UNSUPPORTED;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVX_ERR_CUDA;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return KVX_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return KVX_ERR_UNSUPPORTED;  // sm_103 only

  kvx_plan *p = new (std::nothrow) kvx_plan();
  if (!p) return KVX_ERR_NO_MEMORY;
  p->desc = *desc;
  p->device = dev;
  p->kernel = kernel;
  p->num_sms = prop.multiProcessorCount;
  p->half = desc->src_head_dim / 2;
  p->tiles_per_item = desc->tiles_per_item > 0 ? desc->tiles_per_item : 32;
  p->stall_test = (desc->flags & KVX_PLAN_TEST_STALL) ? 1 : 0;

  p->max_tokens = desc->max_tokens > 0 ? desc->max_tokens : desc->max_position;
  // RoPE tables: one device copy each, built on the host first.  Tables
  // larger than the device are refused before the host buffer is made, and
  // a failed host allocation is reported rather than thrown across the C ABI.
  const size_t positions = (size_t)desc->max_position;
  const size_t table_bytes =
      wide ? 0
      : kernel == KVX_KERNEL_SIMT
          ? positions * (size_t)p->half * sizeof(float2) *
                (desc->rope_theta_tgt == desc->rope_theta_src ? 1 : 2)
          : positions * (size_t)(desc->src_head_dim / 8) * 16;
  if (table_bytes > prop.totalGlobalMem) st = KVX_ERR_NO_MEMORY;
  try {
    if (st != KVX_OK || wide) {
      // wide: no RoPE tables, both bases are evaluated from fixed-point phases
    } else if (kernel == KVX_KERNEL_SIMT) {
      // fp32 tables from fp64 host trigonometry (the fp32 path's 1e-5 budget)
      st = upload(rope_table(desc->rope_theta_src, desc->src_head_dim, desc->max_position),
                  &p->rope_src);
      if (st == KVX_OK) {
        if (desc->rope_theta_tgt == desc->rope_theta_src)
          p->rope_tgt = p->rope_src;
        else
          st = upload(rope_table(desc->rope_theta_tgt, desc->tgt_head_dim, desc->max_position),
                      &p->rope_tgt);
      }
    } else {
      std::vector<uint32_t> ts;
      tc_rope_table(desc->rope_theta_src, desc->src_head_dim, desc->max_position, ts);
      st = upload_bytes(ts.data(), ts.size() * sizeof(uint32_t), &p->tc_rope_src);
    }
  } catch (...) {
    st = KVX_ERR_NO_MEMORY;
  }
  // target frequencies in turns: the tensor-core epilogue and the
  // diagnostics kernel (any plan) evaluate target RoPE angles from them
  rope_turns(desc->rope_theta_tgt, desc->tgt_head_dim, p->turns_tgt);
  rope_turns(desc->rope_theta_src, desc->src_head_dim, p->turns_src);
  if (st == KVX_OK && kernel == KVX_KERNEL_TCGEN05) {
    p->encode_tiled = kvx_tc_encoder();
    st = !p->encode_tiled ? KVX_ERR_UNSUPPORTED
         : alloc_workspace(p, wide ? kvx_wide_workspace_bytes(*desc, p->max_tokens)
                                   : kvx_tc_workspace_bytes(*desc));
  }
  if (st == KVX_OK && kernel == KVX_KERNEL_TCGEN05 && desc->src_layout == KVX_PAGED) {
    // packed rows of a paged source (values only for the wide map, whose
    // workspace holds the un-rotated keys)
    const size_t bytes = (size_t)desc->src_layers * (size_t)p->max_tokens *
                         desc->src_kv_heads * desc->src_head_dim * 2;
    st = alloc_bytes(&p->packed_v, bytes);
    if (st == KVX_OK && !wide) st = alloc_bytes(&p->packed_k, bytes);
  }
  if (st == KVX_OK) {
    cudaError_t e = wide ? kvx_wide_prepare(p)
                         : kernel == KVX_KERNEL_TCGEN05 ? kvx_tc_prepare(p) : kvx_simt_prepare(p);
    if (e == cudaErrorNotSupported) st = KVX_ERR_UNSUPPORTED;
    else if (e != cudaSuccess) st = KVX_ERR_CUDA;
  }
  if (st != KVX_OK) {
    free_tables(p);
    delete p;
    return st;
  }
  *out = p;
  return KVX_OK;
}

kvx_status kvx_plan_destroy(kvx_plan *plan) {
  if (!plan) return KVX_OK;
  int cur = 0;
  bool switched = false;
  if (cudaGetDevice(&cur) == cudaSuccess && cur != plan->device) {
    if (cudaSetDevice(plan->device) == cudaSuccess) switched = true;
  }
  cudaDeviceSynchronize();
  free_tables(plan);
  if (switched) cudaSetDevice(cur);
  delete plan;
  return KVX_OK;
}

int32_t kvx_plan_kernel(const kvx_plan *plan) { return plan ? plan->kernel : -1; }

int32_t kvx_plan_launches(const kvx_plan *plan) {
  if (!plan) return -1;
  // a paged source adds the packing launch on the tensor-core paths
  const int pack = plan->kernel == KVX_KERNEL_TCGEN05 && plan->desc.src_layout == KVX_PAGED;
  if (plan->desc.mapper == KVX_MAPPER_WIDE) return 3 + pack;  // un-rotated keys, W image, map
  return (plan->kernel == KVX_KERNEL_TCGEN05 ? 2 : 1) + pack;  // W image + transfer, or transfer
}

int32_t kvx_plan_cta_group(const kvx_plan *plan) {
  if (!plan) return -1;
  if (plan->kernel != KVX_KERNEL_TCGEN05) return 0;
  return plan->tc_pairs > 0 ? 2 : 1;
}

kvx_status kvx_transfer(const kvx_plan *plan, const kvx_transfer_args *a, void *stream) {
  if (!plan || !a) return KVX_ERR_INVALID_ARG;
  const kvx_plan_desc &d = plan->desc;
  if (a->ntok < 0 || a->ntok > INT32_MAX) return KVX_ERR_INVALID_ARG;
  if (a->num_requests < 1) return KVX_ERR_INVALID_ARG;
  if (!a->cu_seqlens && a->num_requests != 1) return KVX_ERR_INVALID_ARG;
  // with no tokens nothing is read from the source: its pointers may be NULL
  // (zero-row arrays have no storage)
  if ((a->ntok > 0 && (!a->src_k || !a->src_v)) || !a->layer_idx || !a->w || !a->b ||
      !a->dst_k || !a->dst_v)
    return KVX_ERR_INVALID_ARG;
  // the tensor-core path reads the source through TMA (16-byte aligned bases)
  // and writes the cache in whole 32-byte sectors (32-byte aligned bases)
  if (plan->kernel == KVX_KERNEL_TCGEN05 &&
      ((((uintptr_t)a->src_k | (uintptr_t)a->src_v) & 15u) ||
       (((uintptr_t)a->dst_k | (uintptr_t)a->dst_v) & 31u)))
    return KVX_ERR_INVALID_ARG;
  if (d.dst_layout == KVX_CONTIGUOUS) {
    if (a->dst_capacity < 1) return KVX_ERR_INVALID_ARG;
  } else {
    if (a->num_blocks < 1 || !a->block_table || a->max_blocks_per_req < 1)
      return KVX_ERR_INVALID_ARG;
  }
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return KVX_ERR_CUDA;
  if (cur != plan->device) return KVX_ERR_INVALID_ARG;
  const bool wide = d.mapper == KVX_MAPPER_WIDE;
  const bool src_paged = d.src_layout == KVX_PAGED;
  if (src_paged && (a->src_num_blocks < 1 || !a->src_block_table || a->max_src_blocks_per_req < 1))
    return KVX_ERR_INVALID_ARG;
  if ((wide || (src_paged && plan->kernel == KVX_KERNEL_TCGEN05)) && a->ntok > plan->max_tokens)
    return KVX_ERR_INVALID_ARG;
  if (a->ntok == 0) return KVX_OK;  // nothing to transfer; status untouched

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
  p.rope_src = plan->rope_src;
  p.rope_tgt = plan->rope_tgt;
  p.ntok = a->ntok;
  p.dst_capacity = a->dst_capacity;
  p.num_blocks = a->num_blocks;
  p.dst_rows = d.dst_layout == KVX_CONTIGUOUS
                   ? (int64_t)a->num_requests * a->dst_capacity
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

  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = wide ? kvx_wide_launch(plan, p, s)
                  : plan->kernel == KVX_KERNEL_TCGEN05 ? kvx_tc_launch(plan, p, s)
                                                       : kvx_simt_launch(plan, p, s);
  return e == cudaSuccess ? KVX_OK : KVX_ERR_CUDA;
}

}  // extern "C"
