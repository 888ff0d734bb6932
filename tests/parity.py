"""Helpers for the GPU-vs-oracle parity tests (test infrastructure).

The CUDA side runs through the C ABI (``cross_model_kv_transfer_gb300.kvx``);
the reference side is the fp64 oracle (``oracle``).  Both read the same
stored tensors drawn by ``cross_model_kv_transfer_gb300.workloads``.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from cross_model_kv_transfer_gb300 import kvx
from cross_model_kv_transfer_gb300.workloads import PAGED, Workload, make_inputs, sentinel_like

TOL = {torch.float32: 1e-5, torch.bfloat16: 1e-2}


# Kernel choices of the tests: a kvx.KVX_KERNEL_* code, or TC_SINGLE for the
# tensor-core kernel on single CTAs (the default runs it on CTA pairs).
TC_SINGLE = "tcgen05_single_cta"


def kernel_code(kernel) -> int:
    return kvx.KVX_KERNEL_TCGEN05 if kernel == TC_SINGLE else kernel


def make_plan(wl: Workload, kernel=kvx.KVX_KERNEL_AUTO, max_position=None):
    return kvx.Plan(src_layers=wl.src_layers, tgt_layers=wl.tgt_layers, kv_heads=wl.kv_heads,
                    head_dim=wl.head_dim, k=wl.k, rope_theta_src=wl.theta_src,
                    rope_theta_tgt=wl.theta_tgt,
                    max_position=wl.max_position if max_position is None else max_position,
                    kv_dtype=wl.kv_dtype, w_dtype=torch.float32, b_dtype=wl.b_dtype,
                    layout=wl.layout, block_size=wl.block_size if wl.layout == PAGED else 0,
                    kernel=kernel_code(kernel),
                    flags=kvx.KVX_PLAN_TC_SINGLE_CTA if kernel == TC_SINGLE else 0)


def gpu_args(wl: Workload, inp: dict, dst_k, dst_v, status, **over):
    args = dict(src_k=inp["src_k"], src_v=inp["src_v"], layer_idx=inp["layer_idx"],
                w=inp["w"], b=inp["b"], dst_k=dst_k, dst_v=dst_v, status=status)
    if wl.num_requests > 1 or wl.layout == PAGED:
        args["cu_seqlens"] = inp["cu_seqlens"]
    if any(wl.tgt_offsets):
        args["tgt_offset"] = inp["tgt_offset"]
    if wl.layout == PAGED:
        args["block_table"] = inp["block_table"]
        args["num_blocks"] = wl.num_blocks
    else:
        args["dst_capacity"] = wl.dst_capacity
    args.update(over)
    return args


def run_gpu(wl: Workload, inp: dict, kernel=kvx.KVX_KERNEL_AUTO, plan=None, **over):
    """One transfer on the GPU into sentinel-filled destinations."""
    plan = plan or make_plan(wl, kernel)
    shape = (wl.tgt_layers, wl.dst_rows, wl.kv_heads, wl.head_dim)
    dst_k = sentinel_like(shape, wl.kv_dtype, "cuda")
    dst_v = sentinel_like(shape, wl.kv_dtype, "cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    plan.transfer(**gpu_args(wl, inp, dst_k, dst_v, status, **over))
    torch.cuda.synchronize()
    return dst_k, dst_v, int(status.item()), plan


def run_oracle(wl: Workload, inp: dict, **over):
    f64 = lambda t: t.detach().cpu().to(torch.float64).numpy()
    i64 = lambda t: None if t is None else t.detach().cpu().to(torch.int64).numpy()
    kw = dict(src_k=f64(inp["src_k"]), src_v=f64(inp["src_v"]),
              layer_idx=inp["layer_idx"].cpu().numpy(), w=f64(inp["w"]), b=f64(inp["b"]),
              theta_src=wl.theta_src, theta_tgt=wl.theta_tgt, max_position=wl.max_position,
              cu_seqlens=i64(inp["cu_seqlens"]), tgt_offset=i64(inp["tgt_offset"]))
    if wl.layout == PAGED:
        kw.update(layout=oracle.PAGED, block_size=wl.block_size, num_blocks=wl.num_blocks,
                  block_table=inp["block_table"].cpu().numpy())
    else:
        kw.update(layout=oracle.CONTIGUOUS, dst_capacity=wl.dst_capacity)
    kw.update(over)
    return oracle.transfer(**kw)


def assert_parity(wl: Workload, gpu_k, gpu_v, ref_k, ref_v, tol=None):
    """Written rows: relative Frobenius error per (target layer, head, K|V)
    within ``tol``; unwritten rows: the sentinel bits, untouched."""
    tol = TOL[wl.kv_dtype] if tol is None else tol
    worst = 0.0
    for name, g, r in (("K", gpu_k, ref_k), ("V", gpu_v, ref_v)):
        written = ~np.isnan(r[..., 0])                         # [Lt][rows][H]
        gw = torch.from_numpy(written).to(g.device)
        bits = g.view(torch.int16 if g.dtype == torch.bfloat16 else torch.int32)
        untouched = bits[~gw]
        assert bool((untouched == -1).all()), f"{name}: rows outside the transfer were written"
        gd = g.to(torch.float64).cpu().numpy()
        for lt in range(wl.tgt_layers):
            for h in range(wl.kv_heads):
                m = written[lt, :, h]
                if not m.any():
                    continue
                ref = r[lt, m, h]
                err = np.linalg.norm(gd[lt, m, h] - ref) / max(np.linalg.norm(ref), 1e-300)
                worst = max(worst, err)
                assert err <= tol, f"{name} lt={lt} h={h}: rel Frobenius {err:.3e} > {tol:.0e}"
    return worst


def inputs(wl: Workload, device="cuda", seed=None):
    return make_inputs(wl, device=device, seed=seed)
