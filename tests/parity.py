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


# ---------------------------------------------------------------------------
# Full-size parity: the oracle on a chosen set of tokens
# ---------------------------------------------------------------------------
def token_positions(wl: Workload, inp: dict):
    """Per packed token g: request r, source position p (0 .. len - 1 within
    its request) and target position p' = p + tgt_offset[r], the ABI's
    implicit positions.  int64 numpy arrays."""
    cu = inp["cu_seqlens"].cpu().numpy().astype(np.int64)
    off = inp["tgt_offset"].cpu().numpy().astype(np.int64)
    r = np.repeat(np.arange(wl.num_requests), np.diff(cu))
    p = np.arange(wl.ntok, dtype=np.int64) - cu[r]
    return r, p, p + off[r]


def _runs(tokens, req):
    """Split sorted packed tokens into runs of consecutive tokens of one request."""
    out, start = [], 0
    for i in range(1, len(tokens) + 1):
        if i == len(tokens) or tokens[i] != tokens[i - 1] + 1 or req[tokens[i]] != req[tokens[start]]:
            out.append(tokens[start:i])
            start = i
    return out


def oracle_tokens(wl: Workload, inp: dict, tokens, threads: int = 0, wide: bool = False):
    """fp64 oracle outputs of the packed tokens ``tokens`` for every target
    layer and head: returns (ok, ov) of shape [Lt][n][H][d], in the order of
    ``sorted(set(tokens))``, and that sorted token array.

    Each share of the tokens is one oracle transfer of its own: its runs of
    consecutive tokens become the requests of a packed batch holding only
    those source rows, with the tokens' source and target positions given
    explicitly and a paged destination of one-row blocks whose table sends
    position p' of run r to the token's slot.  The shares run on ``threads``
    host threads (the oracle releases the interpreter lock)."""
    import concurrent.futures as cf
    import os

    tokens = np.unique(np.asarray(tokens, dtype=np.int64))
    req, p, pt = token_positions(wl, inp)
    threads = threads or min(16, os.cpu_count() or 1)
    shares = [s for s in np.array_split(tokens, min(threads, len(tokens))) if len(s)]
    f64 = lambda t: t.detach().cpu().to(torch.float64).numpy()
    w = f64(inp["w"])
    b = f64(inp["b"])
    idx = inp["layer_idx"].cpu().numpy()
    tok_dev = torch.from_numpy(tokens).to(inp["src_k"].device)
    sk_all = f64(inp["src_k"][:, tok_dev])
    sv_all = f64(inp["src_v"][:, tok_dev])
    maxp = int(pt.max()) + 1

    def one(share):
        at = np.searchsorted(tokens, share)
        runs = _runs(share, req)
        cu = np.zeros(len(runs) + 1, dtype=np.int64)
        cu[1:] = np.cumsum([len(x) for x in runs])
        table = np.full((len(runs), maxp), -1, dtype=np.int32)
        for i, run in enumerate(runs):
            table[i, pt[run]] = np.arange(cu[i], cu[i + 1], dtype=np.int32)
        dk, dv, st = oracle.transfer(
            src_k=sk_all[:, at], src_v=sv_all[:, at], layer_idx=idx, w=w, b=b,
            theta_src=wl.theta_src, theta_tgt=wl.theta_tgt, max_position=wl.max_position,
            cu_seqlens=cu, src_pos=p[share], tgt_pos=pt[share], layout=oracle.PAGED,
            block_size=1, num_blocks=len(share), block_table=table, wide=wide)
        assert st == 0, st
        return dk, dv

    with cf.ThreadPoolExecutor(max_workers=len(shares)) as ex:
        parts = list(ex.map(one, shares))
    ok = np.concatenate([x[0] for x in parts], axis=1)
    ov = np.concatenate([x[1] for x in parts], axis=1)
    return ok, ov, tokens


def dst_rows_of(wl: Workload, inp: dict, tokens):
    """Destination rows of the packed tokens under the workload's layout,
    from the oracle's row rule (every token must have one)."""
    req, _, pt = token_positions(wl, inp)
    table = inp["block_table"].cpu().numpy() if wl.layout == PAGED else None
    rows = np.empty(len(tokens), dtype=np.int64)
    for i, g in enumerate(tokens):
        if wl.layout == PAGED:
            row, bad = oracle.dst_row(oracle.PAGED, int(req[g]), int(pt[g]),
                                      block_size=wl.block_size, num_blocks=wl.num_blocks,
                                      block_table=table, max_blocks_per_req=table.shape[1])
        else:
            row, bad = oracle.dst_row(oracle.CONTIGUOUS, int(req[g]), int(pt[g]),
                                      dst_capacity=wl.dst_capacity)
        assert bad == 0 and row >= 0
        rows[i] = row
    return rows


def assert_token_parity(wl: Workload, gpu_k, gpu_v, ok, ov, rows, tol=None):
    """The GPU cache rows ``rows`` against the oracle outputs of those tokens
    ([Lt][n][H][d]): relative Frobenius error per (target layer, head, K|V)
    over the tokens within ``tol``.  Returns the worst error and where."""
    tol = TOL[wl.kv_dtype] if tol is None else tol
    rows_dev = torch.from_numpy(rows).to(gpu_k.device)
    worst = (0.0, None)
    Lt, H = ok.shape[0], ok.shape[2]
    for m, (g, r) in enumerate(((gpu_k, ok), (gpu_v, ov))):
        err = np.empty((Lt, H))
        for lt in range(Lt):
            got = g[lt, rows_dev].to(torch.float64).cpu().numpy()   # [n][H][d]
            assert bool(np.isfinite(got).all()), f"{'KV'[m]} lt={lt}: non-finite values"
            num = np.sqrt(((got - r[lt]) ** 2).sum(axis=(0, 2)))    # [H]
            den = np.sqrt((r[lt] ** 2).sum(axis=(0, 2)))
            err[lt] = num / np.maximum(den, 1e-300)
        lt, h = np.unravel_index(int(np.argmax(err)), err.shape)
        if err[lt, h] > worst[0]:
            worst = (float(err[lt, h]), ("KV"[m], int(lt), int(h)))
        bad = np.argwhere(err > tol)
        assert len(bad) == 0, (f"{'KV'[m]}: {len(bad)} (lt, h) maps above {tol:.0e}, worst "
                               f"{err.max():.3e} at lt={lt} h={h}")
    return worst
