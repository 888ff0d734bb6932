"""Benchmark of the cross-model KV-cache transfer on GB300.

One step = one ``kvx_transfer`` (gather, un-rotate, concatenate, map, re-rotate,
install) over every target layer, head and token of the workload.  With
``--op kv_diagnostics`` one step is instead one ``kvx_kv_diagnostics`` call
(KV cosine and explained variance of the mapped cache against the target's
own) over the same workload.  The default
workload is the Qwen3-14B -> 32B shape at 32,768 tokens (40 -> 64 layers, 8 KV
heads, head_dim 128, k = 4, bf16 caches, fp32 W, bf16 b, theta 1e6), with
synthetic inputs resident in HBM.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the fp64 CPU oracle
on a bounded sample of the same workload instead.

Multi-GPU: launched under torchrun each rank runs an independent replica of the
whole transfer on its own GPU (the transfer has no exchange step); the line
reports the tokens of all ranks over the slowest rank's time (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KV-transfer tokens/s at 14B→32B shape, 32K tokens; % of HBM/tensor roofline"
WIDE_METRIC = ("KV-transfer tokens/s at 14B→32B shape, 32K tokens, wide-feature mapper "
               "(one 8192x2048 map per target layer, 1.07e9 parameters); % of tensor roofline")
# Published context for this exact workload: the Qwen3 14B -> 32B mapper at
# 32,768 tokens took 277.6 ms on an 8xH100 node (Qwen3 KV-transfer article,
# section on what the headline number covers).
PUBLISHED_MS = {"qwen3_14b_32b": 277.6}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_FILES = {"tcgen05": "kvx_tcgen05.cu", "simt": "kvx_simt.cu", "diag": "kvx_diag.cu",
                "wide": "kvx_wide.cu", "ridge": "kvx_ridge.cu", "scores": "kvx_scores.cu",
                "features": "kvx_features.cu"}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["kvx", "reference"], default="kvx")
    ap.add_argument("--op", choices=["transfer", "kv_diagnostics", "ridge_fit", "layer_scores",
                                     "ridge_features"],
                    default="transfer",
                    help="transfer (the default step), the fidelity diagnostics of a "
                         "mapped cache against the target's own, a batch of ridge fits "
                         "of the per-head maps (calibration), the layer-selection "
                         "scores of paired calibration caches, or the content-space "
                         "observations of the maps' ridge fits")
    ap.add_argument("--score-tokens", type=int, default=4096,
                    help="calibration tokens of the layer-selection scores")
    ap.add_argument("--ridge-batch", type=int, default=16, help="ridge fits per step")
    ap.add_argument("--ridge-n", type=int, default=131072, help="observations per ridge fit")
    ap.add_argument("--workload", default="qwen3_14b_32b")
    ap.add_argument("--kernel", choices=["auto", "simt", "tcgen05"], default="auto")
    ap.add_argument("--mapper", choices=["per_head", "wide"], default="per_head",
                    help="per_head: one [k*d x d] map per (target layer, head, K|V); wide: one "
                         "[k*2*H*d x H*2*d] map per target layer (the 1.07e9-parameter "
                         "14B->32B mapper)")
    ap.add_argument("--src-block-size", type=int, default=0,
                    help="read the source from a paged pilot cache with this block size "
                         "(0: packed source rows)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the workload's token count (profiling of small cases)")
    ap.add_argument("--tgt-layers", type=int, default=0,
                    help="override the workload's target-layer count (profiling of small cases)")
    ap.add_argument("--tiles-per-item", type=int, default=0)
    ap.add_argument("--single-cta", action="store_true",
                    help="tensor-core kernel on single CTAs instead of CTA pairs")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle baseline sample")
    return ap.parse_args(argv)


# --------------------------------------------------------------------------
# distributed plumbing (barrier + max over ranks)
# --------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(backend: str):
    import torch.distributed as dist
    ws, rank, _ = dist_env()
    if ws > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=ws)
    return ws, rank


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(tokens_per_rank_step: int, ms_per_step_local: float, device=None):
    """Whole-job throughput: all ranks' tokens over the slowest rank's time."""
    import torch.distributed as dist
    ws = dist.get_world_size() if dist.is_available() and dist.is_initialized() else 1
    ms = max_over_ranks(ms_per_step_local, device)
    return ws * tokens_per_rank_step / (ms / 1e3), ms


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_index: int):
        self.proc = None
        self.lines = []
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            ident = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            ident = []
        self.cmd = ["nvidia-smi", *ident, "--query-gpu=" + ",".join(self.FIELDS),
                    "--format=csv,noheader,nounits", "-lms", "50"]

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) != len(self.FIELDS):
                continue
            try:
                sm.append(float(f[0]))
                smax = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[3:]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# roofline
# --------------------------------------------------------------------------

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_sha(kernel_name: str) -> str:
    """Hash of what decides a kernel's DRAM traffic: its source file, the
    library headers it includes (transitively), and the host code that sets
    its launch shape (tiles per item, CTA pairs)."""
    import re
    csrc = os.path.join(ROOT, "cross_model_kv_transfer_gb300", "csrc")
    seen, todo = [], [KERNEL_FILES.get(kernel_name), "kvx_api.cpp"]
    while todo:
        fn = todo.pop(0)
        if not fn or fn in seen or not os.path.exists(os.path.join(csrc, fn)):
            continue
        seen.append(fn)
        with open(os.path.join(csrc, fn), encoding="utf-8") as f:
            todo += re.findall(r'#include\s+"([^"/]+)"', f.read())
    h = hashlib.sha256()
    for fn in sorted(seen):
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def measured_traffic(workload: str, kernel_name: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(p) as f:
            rows = json.load(f)
    except Exception:
        return None
    sha = kernel_source_sha(kernel_name)
    for r in rows:
        if r.get("workload") == workload and r.get("kernel") == kernel_name \
                and r.get("source_sha") == sha:
            return r.get("dram_bytes_per_launch")
    return None


# Nominal figures, for context beside the measured ones: HBM3e 7.9 TB/s; dense
# bf16 tensor rate = SMs x 8192 flops per clock per SM x the SM clock.
NOMINAL_HBM_GBS = 7900.0
NOMINAL_SMS = 152
BF16_FLOPS_PER_CLK_PER_SM = 8192


def roofline(wl, layer_idx, ms_per_launch, kernel_name, peaks, peak_kind, wide=False,
             clocks=None):
    """Algorithmic bytes or flops per launch over the measured launch time,
    against the measured peaks.  A tensor-bound kernel whose timed region ran
    under the power cap (``sw_power_cap`` among the sampled clock reasons) is
    compared with the sustained cuBLAS figure, which was measured in the same
    power-capped regime; otherwise with the burst figure.  Both fractions and
    the nominal ones are always reported."""
    alg_bytes = wl.wide_algorithmic_bytes(layer_idx) if wide else wl.algorithmic_bytes(layer_idx)
    flops = wl.wide_algorithmic_flops() if wide else wl.algorithmic_flops()
    s = ms_per_launch / 1e3
    capped = bool(clocks) and "sw_power_cap" in (clocks.get("reasons") or [])
    tc_peak = peaks["bf16_tflops_sustained"] if capped else peaks["bf16_tflops"]
    t_hbm = alg_bytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (tc_peak * 1e12)
    traffic = measured_traffic(wl.name, kernel_name)
    if kernel_name in ("tcgen05", "wide") and t_tc >= t_hbm:
        r = {"bound": "tensor", "achieved": flops / s / 1e12, "peak": tc_peak,
             "unit": "TFLOP/s"}
    else:
        r = {"bound": "hbm", "achieved": alg_bytes / s / 1e9, "peak": peaks["hbm_gbs"],
             "unit": "GB/s"}
    r["frac"] = r["achieved"] / r["peak"]
    r["traffic"] = traffic
    if r["bound"] == "tensor":
        r["peak_source"] = (f"{peak_kind} sustained (timed region ran under the power cap)"
                            if capped else f"{peak_kind} burst")
        r["frac_of_burst"] = (flops / s / 1e12) / peaks["bf16_tflops"]
        r["frac_of_sustained"] = (flops / s / 1e12) / peaks["bf16_tflops_sustained"]
        mhz = (clocks or {}).get("sm_mhz") or (clocks or {}).get("sm_max_mhz") or 2070.0
        nominal = NOMINAL_SMS * BF16_FLOPS_PER_CLK_PER_SM * mhz * 1e6 / 1e12
        r["nominal_peak"] = nominal
        r["frac_of_nominal"] = (flops / s / 1e12) / nominal
    else:
        r["peak_source"] = f"{peak_kind} (copy bandwidth)"
    r["algorithmic_bytes"] = alg_bytes
    r["algorithmic_flops"] = flops
    r["hbm_frac"] = (alg_bytes / s / 1e9) / peaks["hbm_gbs"]
    r["hbm_frac_of_nominal"] = (alg_bytes / s / 1e9) / NOMINAL_HBM_GBS
    r["tensor_frac"] = (flops / s / 1e12) / tc_peak
    r["tighter_roofline_frac"] = max(t_hbm, t_tc) / s
    return r


# --------------------------------------------------------------------------
# CPU oracle on a bounded sample
# --------------------------------------------------------------------------

def oracle_sample_inputs(wl, inp, ntok_sample: int, layers=None, wide=False):
    """fp64 copies of the first ``ntok_sample`` source tokens (one request),
    for the first ``layers`` target layers (all by default)."""
    import torch
    f64 = lambda t: t.detach().cpu().to(torch.float64).numpy()
    L = wl.tgt_layers if layers is None else layers
    return dict(src_k=f64(inp["src_k"][:, :ntok_sample]), src_v=f64(inp["src_v"][:, :ntok_sample]),
                layer_idx=inp["layer_idx"][:L].cpu().numpy(), w=f64(inp["w"][:L]),
                b=f64(inp["b"][:L]), theta_src=wl.theta_src, theta_tgt=wl.theta_tgt,
                max_position=ntok_sample, dst_capacity=ntok_sample, wide=wide)


def time_oracle(wl, inp, target_seconds: float, wide=False):
    """Tokens/s of the fp64 oracle (one host thread) on a bounded sample:
    the first n tokens through the first L target layers, scaled to all Lt
    (the work is linear in the target layers).  Returns (tokens/s, n, L,
    seconds)."""
    import oracle
    L = min(wl.tgt_layers, 2) if wide else wl.tgt_layers
    probe = oracle_sample_inputs(wl, inp, 1, L, wide)
    t0 = time.perf_counter()
    oracle.transfer(**probe)
    per_tok = max(time.perf_counter() - t0, 1e-4)
    n = int(max(1, min(wl.ntok, target_seconds / per_tok)))
    sample = oracle_sample_inputs(wl, inp, n, L, wide)
    t0 = time.perf_counter()
    oracle.transfer(**sample)
    el = time.perf_counter() - t0
    return n / (el * wl.tgt_layers / L), n, L, el


# --------------------------------------------------------------------------
# arms
# --------------------------------------------------------------------------

def select_workload(args):
    """The transfer workload both arms run: the named one, with the
    profiling overrides of token count and target layers applied."""
    import dataclasses
    from cross_model_kv_transfer_gb300.workloads import WORKLOADS
    wl = WORKLOADS[args.workload]
    if args.tokens:
        wl = wl.with_tokens([args.tokens], [wl.tgt_offsets[0]], name=f"{wl.name}@{args.tokens}")
    if args.tgt_layers:
        wl = dataclasses.replace(wl, tgt_layers=args.tgt_layers,
                                 name=f"{wl.name}/Lt{args.tgt_layers}")
    return wl


def transfer_metric(wl, wide: bool) -> str:
    if wl.name == "qwen3_14b_32b":
        return WIDE_METRIC if wide else METRIC
    return (f"KV-transfer tokens/s, {wl.name} shape"
            f"{', wide-feature mapper' if wide else ''}; % of HBM/tensor roofline")


def transfer_config(wl, args) -> dict:
    """Workload keys of a transfer line, the same in both arms."""
    from cross_model_kv_transfer_gb300.workloads import PAGED
    return {"workload": wl.name, "src_layers": wl.src_layers, "tgt_layers": wl.tgt_layers,
            "kv_heads": wl.kv_heads, "head_dim": wl.head_dim, "k": wl.k, "tokens": wl.ntok,
            "requests": wl.num_requests,
            "layout": "paged" if wl.layout == PAGED else "contiguous",
            "mapper": args.mapper,
            "source": (f"paged, {args.src_block_size}-token blocks"
                       if args.src_block_size else "packed rows")}


def diag_config(wl) -> dict:
    """Workload keys of a diagnostics line, the same in both arms."""
    from cross_model_kv_transfer_gb300.workloads import PAGED
    return {"workload": wl.name, "tgt_layers": wl.tgt_layers, "kv_heads": wl.kv_heads,
            "head_dim": wl.head_dim, "tokens": wl.ntok, "requests": wl.num_requests,
            "layout": "paged" if wl.layout == PAGED else "contiguous"}


def ridge_config(wl, batch: int, n: int) -> dict:
    """Workload keys of a ridge-fit line, the same in both arms."""
    return {"workload": f"{wl.name} per-head maps", "fits": batch, "observations": n,
            "features": wl.k * wl.head_dim, "outputs": wl.head_dim, "lambda": 0.01}


def kernel_code(name):
    from cross_model_kv_transfer_gb300 import kvx
    return {"auto": kvx.KVX_KERNEL_AUTO, "simt": kvx.KVX_KERNEL_SIMT,
            "tcgen05": kvx.KVX_KERNEL_TCGEN05}[name]


def transfer_kwargs(wl, inp, dst_k, dst_v, status, paged_src=None):
    from cross_model_kv_transfer_gb300.workloads import PAGED
    kw = dict(src_k=inp["src_k"], src_v=inp["src_v"], layer_idx=inp["layer_idx"], w=inp["w"],
              b=inp["b"], dst_k=dst_k, dst_v=dst_v, status=status)
    if paged_src is not None:
        kw.update(src_k=paged_src[0], src_v=paged_src[1], src_block_table=paged_src[2],
                  ntok=wl.ntok)
    if wl.num_requests > 1 or wl.layout == PAGED:
        kw["cu_seqlens"] = inp["cu_seqlens"]
    if any(wl.tgt_offsets):
        kw["tgt_offset"] = inp["tgt_offset"]
    if wl.layout == PAGED:
        kw.update(block_table=inp["block_table"], num_blocks=wl.num_blocks)
    else:
        kw["dst_capacity"] = wl.dst_capacity
    return kw


RIDGE_METRIC = ("ridge fits/s of the 14B→32B per-head maps (512 features → 128 outputs, "
                "131,072 observations each); % of the roofline of the call's dominant phase")


# Nominal dense rates for the phases the measured peaks do not cover: tf32
# tensor 1.1 and fp64 1.25 PFLOP/s / TFLOP/s against bf16's 2.25 PFLOP/s.
TF32_PER_BF16 = 1.1 / 2.25
NOMINAL_FP64_TFLOPS = 1.25


def phase_roofline(call_ms, tensor_flops, fp64_flops, hbm_bytes, kernel_name, workload):
    """Roofline of a call made of phases that run one after another (the
    ridge fit, the layer scores): the ideal time of each phase at its own
    peak -- the split-precision products on the tensor cores (tf32 peak =
    measured bf16 burst x the nominal tf32/bf16 ratio), the fp64
    factorisations and solves (nominal fp64 rate), the algorithmic bytes at
    the measured HBM copy bandwidth -- and, as `bound`, the phase with the
    largest ideal time, its work over the whole call's time."""
    peaks, src = load_peaks()
    tf32 = peaks["bf16_tflops"] * TF32_PER_BF16
    ideal = {"tensor": tensor_flops / (tf32 * 1e12) * 1e3,
             "alu": fp64_flops / (NOMINAL_FP64_TFLOPS * 1e12) * 1e3,
             "hbm": hbm_bytes / (peaks["hbm_gbs"] * 1e9) * 1e3}
    bound = max(ideal, key=ideal.get)
    work = {"tensor": tensor_flops, "alu": fp64_flops, "hbm": hbm_bytes}[bound]
    peak = {"tensor": tf32, "alu": NOMINAL_FP64_TFLOPS, "hbm": peaks["hbm_gbs"]}[bound]
    scale = 1e12 if bound != "hbm" else 1e9
    achieved = work / (call_ms / 1e3) / scale
    return {"bound": bound, "achieved": achieved, "peak": peak,
            "unit": "GB/s" if bound == "hbm" else "TFLOP/s", "frac": achieved / peak,
            "traffic": measured_traffic(workload, kernel_name),
            "peak_source": {"tensor": f"tf32: {src} bf16 burst peak x 1.1/2.25 (nominal ratio)",
                            "alu": "nominal fp64 rate (1.25 TFLOP/s; no measured fp64 peak)",
                            "hbm": f"{src} HBM copy bandwidth"}[bound],
            "ideal_ms": {k: round(v, 4) for k, v in ideal.items()},
            "frac_of_ideal_sum": sum(ideal.values()) / call_ms,
            "tensor_flops": tensor_flops, "fp64_flops": fp64_flops, "algorithmic_bytes": hbm_bytes,
            "scope": "whole call; its phases run one after another"}


def run_ridge(args):
    """One step = one kvx_ridge_fit call: a batch of ridge fits of the
    per-head map shape from synthetic paired observations."""
    import ctypes
    import torch
    from cross_model_kv_transfer_gb300 import kvx
    from cross_model_kv_transfer_gb300.workloads import WORKLOADS, make_ridge_inputs
    ws, rank = init_dist("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = WORKLOADS[args.workload]
    B, n = args.ridge_batch, args.ridge_n
    x, y = make_ridge_inputs(wl, B, n, dev)
    p, q = x.shape[2], y.shape[2]
    w = torch.empty((B, p, q), dtype=torch.float32, device=dev)
    b = torch.empty((B, q), dtype=torch.float32, device=dev)
    scratch = torch.empty(kvx.kvx_ridge_workspace_bytes(B, p, q), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    a = kvx.RidgeArgs(B, n, p, q, 0.01, kvx.KVX_F32, x.data_ptr(), y.data_ptr(), w.data_ptr(),
                      b.data_ptr(), scratch.data_ptr(), scratch.numel(), status.data_ptr())
    sptr = ctypes.c_void_p(stream.cuda_stream)

    def step():
        e = kvx.kvx_ridge_fit(a, sptr)
        if e != kvx.KVX_OK:
            raise kvx.KvxError(e, "kvx_ridge_fit")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} during warm-up")
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
    ms_local = ev0.elapsed_time(ev1) / args.steps
    value, ms = aggregate(B, ms_local, dev)
    # useful flops: the symmetric Gram block once, the cross block, per fit;
    # each is three tf32 products on the tensor cores.  fp64: the Cholesky
    # (p^3 / 3 multiply-adds) and the two triangular solves (p^2 q) per fit.
    flops = B * 2.0 * n * (p * (p + 1) / 2 + p * q)
    fp64 = B * (2.0 * p ** 3 / 3 + 2.0 * p * p * q)
    roof = phase_roofline(ms_local, 3 * flops, fp64, (x.numel() + y.numel()) * 4, "ridge",
                          wl.name)
    roof["useful_gram_flops"] = flops

    e2e = None
    if not args.no_e2e:
        hx, hy = x.cpu().pin_memory(), y.cpu().pin_memory()
        hw = torch.empty(w.shape, dtype=w.dtype, pin_memory=True)
        hb = torch.empty(b.shape, dtype=b.dtype, pin_memory=True)

        def e2e_step():
            x.copy_(hx, non_blocking=True)
            y.copy_(hy, non_blocking=True)
            step()
            hw.copy_(w, non_blocking=True)
            hb.copy_(b, non_blocking=True)

        n_e = max(1, min(args.steps, 5))
        e2e_step()
        torch.cuda.synchronize(dev)
        barrier()
        ev0.record(stream)
        for _ in range(n_e):
            e2e_step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        e_val, e_ms = aggregate(B, ev0.elapsed_time(ev1) / n_e, dev)
        e2e = {"value": e_val, "unit": "fits/s", "ms_per_step": e_ms, "steps": n_e,
               "h2d_bytes_per_step": (hx.numel() + hy.numel()) * 4,
               "d2h_bytes_per_step": (hw.numel() + hb.numel()) * 4}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        import oracle
        xs, ys = x[0].double().cpu().numpy(), y[0].double().cpu().numpy()
        m = 256
        t0 = time.perf_counter()
        oracle.ridge_fit(xs[:m], ys[:m], 0.01)
        per_obs = max((time.perf_counter() - t0) / m, 1e-7)
        m = int(max(256, min(n, args.cpu_seconds / per_obs)))
        t0 = time.perf_counter()
        oracle.ridge_fit(xs[:m], ys[:m], 0.01)
        el = time.perf_counter() - t0
        cpu = {"value": 1.0 / (el * n / m), "unit": "fits/s", "cores": 1, "kind": "oracle",
               "sample": f"one fit on its first {m} of {n} observations ({el:.1f} s of fp64 "
                         f"CPU work, one thread), scaled to {n} observations"}
    line = {
        "metric": RIDGE_METRIC, "op": "ridge_fit", "value": value, "unit": "fits/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded paired observations with a planted map)",
        "config": {**ridge_config(wl, B, n),
                   "parallelism": f"replicas x{ws}",
                   "l2": f"inputs larger than L2 ({(x.numel() + y.numel()) * 4 / 1e9:.2f} GB "
                         "read per step, no flush needed)"},
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": (4 + 2 * ((n + 16383) // 16384) + 3 * ((p + 63) // 64) - 1) * args.steps,
        "clocks": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


SCORE_METRIC = ("layer-selection scores: calibration tokens/s through every (target layer, "
                "source layer, head, K|V) fit and every target layer's set fit at the 14B→32B "
                "shape, 4,096 tokens; % of the roofline of the call's dominant phase")


def score_config(wl, n: int) -> dict:
    """Workload keys of a layer-selection score line, the same in both arms."""
    return {"workload": f"{wl.name} layer-selection scores", "tokens": n,
            "src_layers": wl.src_layers, "tgt_layers": wl.tgt_layers, "kv_heads": wl.kv_heads,
            "head_dim": wl.head_dim, "k": wl.k, "lambda": 0.01}


def score_flops(Ls, Lt, H, d, k, n) -> float:
    """Useful flops of one scoring pass: per (head, K|V) the centred Gram
    (symmetric, counted once) and cross moments of every source layer
    against every target layer's d columns, and of every target layer's set
    of k source layers against its own d columns."""
    per = Ls * (d * (d + 1) / 2 + d * Lt * d) + Lt * (k * d * (k * d + 1) / 2 + k * d * d)
    return 2.0 * n * per * 2 * H


def score_fp64_flops(Ls, Lt, H, d, k) -> float:
    """fp64 flops of one scoring call: per (head, K|V) and source layer the
    Cholesky of G + lam I (d^3 / 3 multiply-adds), the inverse (d^3), N =
    M + lam M M (d^3), its Cholesky (d^3 / 3) and R^T C over the Lt d target
    columns (d^2 / 2 each); with a table, per set the Cholesky ((k d)^3 / 3)
    and the two solves of its d columns ((k d)^2 each)."""
    kd = k * d
    per = Ls * (d ** 3 * (2 / 3 + 2) + d * d / 2 * Lt * d) + Lt * (kd ** 3 / 3 + kd * kd * d)
    return 2.0 * per * 2 * H


def score_launches(Ls, Lt, H, d, k, n, sets=True) -> int:
    """Kernels one kvx_layer_scores call launches: the request-table check,
    with a table the clamped table and the row check, then per (head, K|V)
    clear, content, per chunk of 16,384 tokens the split and the tensor-core
    moments; for the per-layer fits the Cholesky of G + lam I (prep + per
    64-column block: diagonal, panel, update), the inverse, N, its Cholesky
    and the triangular norms; for the set fits the Cholesky and the solves;
    and the final ratios."""
    chol = lambda p: 1 + 3 * ((p + 63) // 64) - 2
    chunks = (n + 16383) // 16384
    per = 2 + 2 * chunks + 2 * chol(d) + 3 + (chol(k * d) + 1 if sets else 0) + 1
    return 1 + (2 if sets else 0) + H * 2 * per


def run_scores(args):
    """One step = one kvx_layer_scores call on seeded paired calibration
    caches (the pilot's and the target's caches of the same tokens)."""
    import torch
    from cross_model_kv_transfer_gb300 import kvx
    from cross_model_kv_transfer_gb300.workloads import WORKLOADS, make_score_inputs
    ws, rank = init_dist("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = WORKLOADS[args.workload].with_tokens([args.score_tokens], [0])
    n = wl.ntok
    inp = make_score_inputs(wl, dev)
    plan = kvx.Plan(src_layers=wl.src_layers, tgt_layers=wl.tgt_layers, kv_heads=wl.kv_heads,
                    head_dim=wl.head_dim, k=wl.k, rope_theta_src=wl.theta_src,
                    rope_theta_tgt=wl.theta_tgt, max_position=wl.max_position,
                    kv_dtype=wl.kv_dtype, w_dtype=torch.float32, b_dtype=wl.b_dtype,
                    kernel=kvx.KVX_KERNEL_SIMT)
    Ls, Lt, H, d, k = wl.src_layers, wl.tgt_layers, wl.kv_heads, wl.head_dim, wl.k
    r2 = torch.empty((Lt, Ls, H, 2), dtype=torch.float64, device=dev)
    r2s = torch.empty((Lt, H, 2), dtype=torch.float64, device=dev)
    scratch = torch.empty(kvx.kvx_layer_scores_workspace_bytes(plan.handle, n), dtype=torch.uint8,
                          device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    kw = dict(lam=0.01, layer_idx=inp["layer_idx"], r2=r2, r2_set=r2s, workspace=scratch,
              status=status, stream=stream)
    cache = ("src_k", "src_v", "tgt_k", "tgt_v")

    def step():
        plan.layer_scores(**{c: inp[c] for c in cache}, **kw)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} during warm-up")
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
    ms_local = ev0.elapsed_time(ev1) / args.steps
    value, ms = aggregate(n, ms_local, dev)
    flops = score_flops(Ls, Lt, H, d, k, n)
    in_bytes = sum(inp[c].numel() * inp[c].element_size() for c in cache)
    roof = phase_roofline(ms_local, 3 * flops, score_fp64_flops(Ls, Lt, H, d, k), in_bytes,
                          "scores", wl.name)
    roof["useful_gram_flops"] = flops

    e2e = None
    if not args.no_e2e:
        host = {c: inp[c].cpu().pin_memory() for c in cache}
        hr, hs = (torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (r2, r2s))

        def e2e_step():
            for c in cache:
                inp[c].copy_(host[c], non_blocking=True)
            step()
            hr.copy_(r2, non_blocking=True)
            hs.copy_(r2s, non_blocking=True)

        n_e = max(1, min(args.steps, 3))
        e2e_step()
        torch.cuda.synchronize(dev)
        barrier()
        ev0.record(stream)
        for _ in range(n_e):
            e2e_step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        e_val, e_ms = aggregate(n, ev0.elapsed_time(ev1) / n_e, dev)
        e2e = {"value": e_val, "unit": "tokens/s", "ms_per_step": e_ms, "steps": n_e,
               "h2d_bytes_per_step": in_bytes,
               "d2h_bytes_per_step": (hr.numel() + hs.numel()) * 8}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = time_oracle_scores(wl, args.cpu_seconds)
    line = {
        "metric": SCORE_METRIC, "op": "layer_scores", "value": value, "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if wl.kv_dtype == torch.bfloat16 else "f32",
        "data": "synthetic (seeded paired caches with planted source layers)",
        "config": {**score_config(wl, n), "parallelism": f"replicas x{ws}",
                   "l2": f"inputs larger than L2 ({in_bytes / 1e9:.2f} GB of caches read per "
                         "step, no flush needed)"},
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": score_launches(Ls, Lt, H, d, k, n) * args.steps,
        "clocks": clk.summary(),
        "mean_best_single_layer_r2": [float(x) for x in
                                      r2.max(dim=1).values.mean(dim=(0, 1)).cpu()],
        "mean_set_r2": [float(x) for x in r2s.mean(dim=(0, 1)).cpu()],
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def score_sample(wl, n: int, lt: int = 2, heads: int = 1):
    """A bounded slice of the scoring workload for the oracle: n tokens,
    every source layer, ``lt`` target layers, ``heads`` heads; returns
    (kwargs of oracle.layer_scores, the slice's useful flops)."""
    import dataclasses
    import torch
    from cross_model_kv_transfer_gb300.workloads import make_score_inputs
    small = dataclasses.replace(wl.with_tokens([n], [0]), tgt_layers=lt, kv_heads=heads)
    inp = make_score_inputs(small, "cpu")
    f64 = lambda t: t.to(torch.float64).numpy()
    kw = dict(src_k=f64(inp["src_k"]), src_v=f64(inp["src_v"]), tgt_k=f64(inp["tgt_k"]),
              tgt_v=f64(inp["tgt_v"]), theta_src=wl.theta_src, theta_tgt=wl.theta_tgt,
              max_position=n, lam=0.01, layer_idx=inp["layer_idx"].numpy())
    return kw, score_flops(wl.src_layers, lt, heads, wl.head_dim, wl.k, n)


def time_oracle_scores(wl, target_seconds: float):
    """The oracle on a growing slice until it takes about ``target_seconds``,
    scaled to the whole workload by useful flops."""
    import oracle
    full = score_flops(wl.src_layers, wl.tgt_layers, wl.kv_heads, wl.head_dim, wl.k, wl.ntok)
    n = 256
    while True:
        kw, f = score_sample(wl, n)
        t0 = time.perf_counter()
        oracle.layer_scores(**kw)
        el = time.perf_counter() - t0
        if el * 2 > target_seconds or n * 2 > wl.ntok:
            break
        n *= 2
    return {"value": wl.ntok / (el * full / f), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} tokens x all {wl.src_layers} source layers x 2 target layers x 1 "
                      f"head x K|V ({el:.1f} s of fp64 CPU work, one thread), scaled to the "
                      "whole workload by useful flops"}


FEATURE_METRIC = ("ridge-fit observations: calibration tokens/s of content-space features (each "
                  "target layer's k source layers side by side, keys un-rotated) and targets "
                  "for every (target layer, head, K|V) at the 14B→32B shape, 32K tokens, fp32 "
                  "out; % of HBM roofline")


def feature_config(wl) -> dict:
    """Workload keys of a ridge-features line, the same in both arms."""
    return {"workload": f"{wl.name} ridge-fit observations", "tokens": wl.ntok,
            "src_layers": wl.src_layers, "tgt_layers": wl.tgt_layers, "kv_heads": wl.kv_heads,
            "head_dim": wl.head_dim, "k": wl.k, "out_dtype": "f32"}


def feature_bytes(wl, layer_idx, elem_bytes: int, out_bytes: int = 4) -> int:
    """Algorithmic bytes of one kvx_ridge_features call: the source layers the
    table names and every target layer read once (K and V), x and y written."""
    used = len(set(int(v) for v in layer_idx.flatten().tolist()))
    row = wl.ntok * wl.kv_heads * wl.head_dim * 2 * elem_bytes
    B = wl.tgt_layers * wl.kv_heads * 2
    return (used + wl.tgt_layers) * row + B * wl.ntok * (wl.k + 1) * wl.head_dim * out_bytes


def run_features(args):
    """One step = one kvx_ridge_features call on seeded paired calibration
    caches: x [Lt H 2][ntok][k d] and y [Lt H 2][ntok][d] in fp32, the inputs
    of the per-head maps' ridge fits.  HBM-bound (writes dominate)."""
    import ctypes
    import torch
    from cross_model_kv_transfer_gb300 import kvx
    from cross_model_kv_transfer_gb300.workloads import WORKLOADS, make_score_inputs
    ws, rank = init_dist("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = WORKLOADS[args.workload]
    if args.tokens:
        wl = wl.with_tokens([args.tokens], [0])
    inp = make_score_inputs(wl, dev)
    Ls, Lt, H, d, k, n = wl.src_layers, wl.tgt_layers, wl.kv_heads, wl.head_dim, wl.k, wl.ntok
    plan = kvx.Plan(src_layers=Ls, tgt_layers=Lt, kv_heads=H, head_dim=d, k=k,
                    rope_theta_src=wl.theta_src, rope_theta_tgt=wl.theta_tgt,
                    max_position=wl.max_position, kv_dtype=wl.kv_dtype, w_dtype=torch.float32,
                    b_dtype=torch.float32, kernel=kvx.KVX_KERNEL_SIMT)
    B = Lt * H * 2
    x = torch.empty((B, n, k * d), dtype=torch.float32, device=dev)
    y = torch.empty((B, n, d), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    fa = kvx.FeatureArgs(inp["src_k"].data_ptr(), inp["src_v"].data_ptr(),
                         inp["tgt_k"].data_ptr(), inp["tgt_v"].data_ptr(), n, 1, None, None,
                         inp["layer_idx"].data_ptr(), kvx.KVX_F32, x.data_ptr(), y.data_ptr(),
                         status.data_ptr())
    sptr = ctypes.c_void_p(stream.cuda_stream)

    def step():
        e = kvx.kvx_ridge_features(plan.handle, fa, sptr)
        if e != kvx.KVX_OK:
            raise kvx.KvxError(e, "kvx_ridge_features")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} during warm-up")
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
    ms_local = ev0.elapsed_time(ev1) / args.steps
    value, ms = aggregate(n, ms_local, dev)
    alg = feature_bytes(wl, inp["layer_idx"], inp["src_k"].element_size())
    peaks, peak_kind = load_peaks()
    achieved = alg / (ms_local / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "traffic": measured_traffic(wl.name, "features"),
            "peak_source": f"{peak_kind} (burst)", "algorithmic_bytes": alg}
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = time_oracle_features(wl, args.cpu_seconds)
    in_bytes = sum(inp[c].numel() * inp[c].element_size()
                   for c in ("src_k", "src_v", "tgt_k", "tgt_v"))
    line = {
        "metric": FEATURE_METRIC, "op": "ridge_features", "value": value, "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if wl.kv_dtype == torch.bfloat16 else "f32",
        "data": "synthetic (seeded paired caches with planted source layers)",
        "config": {**feature_config(wl), "parallelism": f"replicas x{ws}",
                   "l2": f"inputs and outputs larger than L2 ({in_bytes / 1e9:.2f} GB read, "
                         f"{(x.numel() + y.numel()) * 4 / 1e9:.1f} GB written per step, no "
                         "flush needed)"},
        "roofline": roof, "cpu_baseline": cpu,
        "e2e": None,
        "e2e_note": "x and y are the device-side inputs of the ridge fit that follows; a read-"
                    "back of them to the host is not part of their use",
        "gpu_launches": args.steps, "clocks": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    plan.close()


def feature_sample(wl, n: int):
    """The first n tokens of the features workload for the oracle (all target
    layers, heads and K|V): kwargs of oracle.ridge_features."""
    import torch
    from cross_model_kv_transfer_gb300.workloads import make_score_inputs
    inp = make_score_inputs(wl.with_tokens([n], [0]), "cpu")
    f64 = lambda t: t.to(torch.float64).numpy()
    return dict(src_k=f64(inp["src_k"]), src_v=f64(inp["src_v"]), tgt_k=f64(inp["tgt_k"]),
                tgt_v=f64(inp["tgt_v"]), theta_src=wl.theta_src, theta_tgt=wl.theta_tgt,
                max_position=n, layer_idx=inp["layer_idx"].numpy())


def time_oracle_features(wl, target_seconds: float):
    """The oracle on a growing prefix of tokens until it takes about
    ``target_seconds``; tokens/s (the work is linear in the tokens)."""
    import oracle
    n = 16
    while True:
        kw = feature_sample(wl, n)
        t0 = time.perf_counter()
        oracle.ridge_features(**kw)
        el = time.perf_counter() - t0
        if el * 2 > target_seconds or n * 2 > wl.ntok:
            break
        n *= 2
    return {"value": n / el, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"first {n} tokens x all {wl.tgt_layers} target layers x "
                      f"{wl.kv_heads} heads x K|V ({el:.1f} s of fp64 CPU work, one thread)"}


def run_kvx(args):
    import torch
    from cross_model_kv_transfer_gb300 import kvx
    from cross_model_kv_transfer_gb300.workloads import PAGED, WORKLOADS, make_inputs

    ws, rank = init_dist("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = select_workload(args)
    inp = make_inputs(wl, dev)
    wide = args.mapper == "wide"
    if wide:
        from cross_model_kv_transfer_gb300.workloads import make_wide_weights
        inp["w"] = make_wide_weights(wl, dev)
    plan = kvx.Plan(src_layers=wl.src_layers, tgt_layers=wl.tgt_layers, kv_heads=wl.kv_heads,
                    head_dim=wl.head_dim, k=wl.k, rope_theta_src=wl.theta_src,
                    rope_theta_tgt=wl.theta_tgt, max_position=wl.max_position,
                    kv_dtype=wl.kv_dtype, w_dtype=torch.float32, b_dtype=wl.b_dtype,
                    layout=wl.layout, block_size=wl.block_size if wl.layout == PAGED else 0,
                    kernel=kernel_code(args.kernel), tiles_per_item=args.tiles_per_item,
                    flags=kvx.KVX_PLAN_TC_SINGLE_CTA if args.single_cta else 0,
                    mapper=kvx.KVX_MAPPER_WIDE if wide else kvx.KVX_MAPPER_PER_HEAD,
                    max_tokens=wl.ntok if (wide or args.src_block_size) else 0,
                    src_layout=kvx.KVX_PAGED if args.src_block_size else kvx.KVX_CONTIGUOUS,
                    src_block_size=args.src_block_size)
    kname = "wide" if wide else \
        {kvx.KVX_KERNEL_SIMT: "simt", kvx.KVX_KERNEL_TCGEN05: "tcgen05"}[plan.kernel]
    shape = (wl.tgt_layers, wl.dst_rows, wl.kv_heads, wl.head_dim)
    dst_k = torch.empty(shape, dtype=wl.kv_dtype, device=dev)
    dst_v = torch.empty(shape, dtype=wl.kv_dtype, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    paged_src = None
    if args.src_block_size:
        from cross_model_kv_transfer_gb300.workloads import make_paged_source
        paged_src = make_paged_source(wl, inp, args.src_block_size)
    targs = plan.make_args(**transfer_kwargs(wl, inp, dst_k, dst_v, status, paged_src))
    stream = torch.cuda.current_stream(dev)
    sptr = __import__("ctypes").c_void_p(stream.cuda_stream)
    if args.op == "kv_diagnostics":
        if wide or paged_src is not None:
            raise SystemExit("kv_diagnostics bench: per-head mapper, packed source only")
        if wl.layout != PAGED and any(wl.tgt_offsets):
            raise SystemExit("kv_diagnostics bench: contiguous workloads with offset 0 only")
        run_diag(args, wl, inp, plan, dev, stream, dst_k, dst_v, status, ws, rank)
        plan.close()
        return

    def step():
        st = kvx.kvx_transfer(plan.handle, targs, sptr)
        if st != kvx.KVX_OK:
            raise kvx.KvxError(st, "kvx_transfer")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} during warm-up")

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
    ms_local = ev0.elapsed_time(ev1) / args.steps
    value, ms = aggregate(wl.ntok, ms_local, dev)

    peaks, peak_kind = load_peaks()
    roof = roofline(wl, inp["layer_idx"], ms_local, kname, peaks, peak_kind, wide=wide,
                    clocks=clk.summary())

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, wl, inp, plan, dev, stream, dst_k, dst_v, status, paged_src)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        tps, n, L, el = time_oracle(wl, inp, args.cpu_seconds, wide=wide)
        scaled = "" if L == wl.tgt_layers else \
            f", timed on the first {L} target layers and scaled to all {wl.tgt_layers}"
        cpu = {"value": tps, "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": f"first {n} source tokens of the workload through "
                         f"{L} target layers x {wl.kv_heads} heads x K|V "
                         f"({el:.1f} s of fp64 CPU work, one thread{scaled})"}
    pub = PUBLISHED_MS.get(wl.name)
    line = {
        "metric": transfer_metric(wl, wide),
        "value": value, "unit": "tokens/s",
        "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": (value / (wl.ntok / (pub / 1e3))) if pub else None,
        "dtype": "bf16" if wl.kv_dtype == torch.bfloat16 else "f32",
        "data": "synthetic (seeded; shapes and value recipe of the pages' workloads)",
        "config": {**transfer_config(wl, args),
                   "kernel": kname, "cta_group": plan.cta_group,
                   "parallelism": f"replicas x{ws}",
                   "l2": "inputs larger than L2 (source "
                         f"{inp['src_k'].numel() * 2 * inp['src_k'].element_size() / 1e9:.2f} GB,"
                         " no flush needed)"},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * plan.launches_per_transfer,
        "clocks": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    plan.close()


DIAG_METRIC = ("KV-diagnostics tokens/s (KV cosine + explained variance of a mapped cache "
               "against the target's own) at 14B→32B shape, 32K tokens; % of HBM roofline")


def diag_kwargs(wl, inp):
    from cross_model_kv_transfer_gb300.workloads import PAGED
    kw = dict(ntok=wl.ntok)
    if wl.num_requests > 1 or wl.layout == PAGED:
        kw["cu_seqlens"] = inp["cu_seqlens"]
    if any(wl.tgt_offsets):
        kw["tgt_offset"] = inp["tgt_offset"]
    if wl.layout == PAGED:
        kw.update(block_table=inp["block_table"], num_blocks=wl.num_blocks)
    else:
        kw["dst_capacity"] = wl.dst_capacity
    return kw


def run_diag(args, wl, inp, plan, dev, stream, dst_k, dst_v, status, ws, rank):
    """One step = one kvx_kv_diagnostics call over the whole mapped cache (the
    output of one transfer) against a stand-in for the target's own cache.
    HBM-bound: the algorithmic bytes are the two caches read once."""
    import ctypes
    import torch
    from cross_model_kv_transfer_gb300 import kvx
    from cross_model_kv_transfer_gb300.workloads import PAGED, perturbed_like

    st = kvx.kvx_transfer(plan.handle, plan.make_args(**transfer_kwargs(wl, inp, dst_k, dst_v,
                                                                        status)),
                          ctypes.c_void_p(stream.cuda_stream))
    if st != kvx.KVX_OK:
        raise kvx.KvxError(st, "kvx_transfer")
    ref_k, ref_v = perturbed_like(dst_k, 101), perturbed_like(dst_v, 102)
    stats = torch.empty((wl.tgt_layers, wl.kv_heads, 2, wl.head_dim + 4), dtype=torch.float64,
                        device=dev)
    dargs = plan.make_diag_args(mapped_k=dst_k, mapped_v=dst_v, ref_k=ref_k, ref_v=ref_v,
                                stats=stats, status=status, **diag_kwargs(wl, inp))
    sptr = ctypes.c_void_p(stream.cuda_stream)

    def step():
        e = kvx.kvx_kv_diagnostics(plan.handle, dargs, sptr)
        if e != kvx.KVX_OK:
            raise kvx.KvxError(e, "kvx_kv_diagnostics")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} during warm-up")
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        barrier()
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
    ms_local = ev0.elapsed_time(ev1) / args.steps
    value, ms = aggregate(wl.ntok, ms_local, dev)

    eb = dst_k.element_size()
    alg_bytes = 4 * wl.tgt_layers * wl.ntok * wl.kv_heads * wl.head_dim * eb \
        + stats.numel() * 8
    peaks, peak_kind = load_peaks()
    achieved = alg_bytes / (ms_local / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"],
            "traffic": measured_traffic(wl.name, "diag"),
            "peak_source": f"{peak_kind} (burst)", "algorithmic_bytes": alg_bytes}

    e2e = None
    if not args.no_e2e:
        # host buffers: both caches copied in, the statistics read back, every step
        hk, hv = dst_k.cpu().pin_memory(), dst_v.cpu().pin_memory()
        hrk, hrv = ref_k.cpu().pin_memory(), ref_v.cpu().pin_memory()
        hs = torch.empty(stats.shape, dtype=stats.dtype, pin_memory=True)
        pairs = [(dst_k, hk), (dst_v, hv), (ref_k, hrk), (ref_v, hrv)]

        def e2e_step():
            for d_, h_ in pairs:
                d_.copy_(h_, non_blocking=True)
            step()
            hs.copy_(stats, non_blocking=True)

        n_e = max(1, min(args.steps, 3))
        e2e_step()
        torch.cuda.synchronize(dev)
        barrier()
        ev0.record(stream)
        for _ in range(n_e):
            e2e_step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        e_ms_local = ev0.elapsed_time(ev1) / n_e
        e_val, e_ms = aggregate(wl.ntok, e_ms_local, dev)
        e2e = {"value": e_val, "unit": "tokens/s", "ms_per_step": e_ms, "steps": n_e,
               "h2d_bytes_per_step": sum(h.numel() * h.element_size() for _, h in pairs),
               "d2h_bytes_per_step": hs.numel() * 8}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = time_oracle_diag(wl, dst_k, dst_v, ref_k, ref_v, args.cpu_seconds)
    line = {
        "metric": DIAG_METRIC, "op": "kv_diagnostics", "value": value, "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if wl.kv_dtype == torch.bfloat16 else "f32",
        "data": "synthetic (mapped cache from one transfer of the seeded workload; the "
                "target's own cache stood in by a seeded perturbation of it)",
        "config": {**diag_config(wl),
                   "parallelism": f"replicas x{ws}",
                   "l2": f"inputs larger than L2 ({4 * dst_k.numel() * eb / 1e9:.2f} GB of "
                         "caches read per step, no flush needed)"},
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": 2 * args.steps,
        "clocks": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def time_oracle_diag(wl, mk, mv, rk, rv, target_seconds: float):
    """Tokens/s of the fp64 oracle's diagnostics (one host thread) on the
    first n tokens of a contiguous, offset-0 cache."""
    import torch
    import oracle

    def sample(n):
        f64 = lambda t: t[:, :n].detach().cpu().to(torch.float64).numpy()
        return dict(mapped_k=f64(mk), mapped_v=f64(mv), ref_k=f64(rk), ref_v=f64(rv),
                    theta_tgt=wl.theta_tgt, max_position=n, ntok=n, dst_capacity=n)

    s1 = sample(16)
    t0 = time.perf_counter()
    oracle.kv_diagnostics(**s1)
    per_tok = max((time.perf_counter() - t0) / 16, 1e-6)
    n = int(max(16, min(wl.ntok, target_seconds / per_tok)))
    sn = sample(n)
    t0 = time.perf_counter()
    oracle.kv_diagnostics(**sn)
    el = time.perf_counter() - t0
    return {"value": n / el, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"first {n} tokens of the mapped and reference caches through all "
                      f"{wl.tgt_layers} target layers x {wl.kv_heads} heads x K|V "
                      f"({el:.1f} s of fp64 CPU work, one thread)"}


def run_e2e(args, wl, inp, plan, dev, stream, dst_k, dst_v, status, paged_src=None):
    """Same metric through the C ABI with HOST buffers: every step copies its
    inputs from pinned host memory, transfers, and reads the whole target
    cache back to pinned host memory.  Steps are pipelined the way a serving
    loop would run them: host-to-device copies on one stream, the transfer on
    another, device-to-host copies on a third, with two device buffer sets
    so that step i's input copy and step i-1's output copy overlap step i's
    neighbours (events order every reuse of a buffer).  The timed region runs
    from before the first step's input copy to after the last step's output
    copy."""
    import ctypes
    import torch
    from cross_model_kv_transfer_gb300 import kvx
    src = dict(inp)
    if paged_src is not None:
        src.update(src_k=paged_src[0], src_v=paged_src[1], src_block_table=paged_src[2])
    names = ["src_k", "src_v", "w", "b", "layer_idx", "cu_seqlens", "tgt_offset"]
    names += [n for n in ("block_table", "src_block_table") if n in src]
    # one pinned host set each way (the read-backs run in order on one
    # stream, so they can share the host buffer); the read-back buffer is
    # pinned first: on these hosts later large pinned allocations copied
    # slower (measured 194 GB/s against 119 GB/s device-to-host)
    hk = torch.empty(dst_k.shape, dtype=dst_k.dtype, pin_memory=True)
    hv = torch.empty(dst_v.shape, dtype=dst_v.dtype, pin_memory=True)
    host = {n: src[n].cpu().pin_memory() for n in names}
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = dst_k.numel() * dst_k.element_size() * 2
    nbuf = 2
    dev_in = [{n: torch.empty_like(src[n]) for n in names} for _ in range(nbuf)]
    dev_out = [(dst_k, dst_v)] + [(torch.empty_like(dst_k), torch.empty_like(dst_v))
                                  for _ in range(nbuf - 1)]
    host_out = [(hk, hv)] * nbuf
    targs = []
    for i in range(nbuf):
        dp = None
        if paged_src is not None:
            dp = (dev_in[i]["src_k"], dev_in[i]["src_v"], dev_in[i]["src_block_table"])
        targs.append(plan.make_args(**transfer_kwargs(wl, dev_in[i], dev_out[i][0],
                                                      dev_out[i][1], status, dp)))
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    cmp_ptr = ctypes.c_void_p(s_cmp.cuda_stream)
    ev_in = [torch.cuda.Event() for _ in range(nbuf)]
    ev_cmp = [torch.cuda.Event() for _ in range(nbuf)]
    ev_out = [torch.cuda.Event() for _ in range(nbuf)]
    issued = [0]

    def step():
        i = issued[0] % nbuf
        if issued[0] >= nbuf:
            s_in.wait_event(ev_cmp[i])         # the transfer that read these inputs is done
        with torch.cuda.stream(s_in):
            for n in names:
                dev_in[i][n].copy_(host[n], non_blocking=True)
        ev_in[i].record(s_in)
        s_cmp.wait_event(ev_in[i])
        if issued[0] >= nbuf:
            s_cmp.wait_event(ev_out[i])        # the read-back of this cache is done
        st = kvx.kvx_transfer(plan.handle, targs[i], cmp_ptr)
        if st != kvx.KVX_OK:
            raise kvx.KvxError(st, "kvx_transfer")
        ev_cmp[i].record(s_cmp)
        s_out.wait_event(ev_cmp[i])
        with torch.cuda.stream(s_out):
            host_out[i][0].copy_(dev_out[i][0], non_blocking=True)
            host_out[i][1].copy_(dev_out[i][1], non_blocking=True)
        ev_out[i].record(s_out)
        issued[0] += 1

    steps = max(1, min(args.steps, 20))
    for _ in range(min(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    t0.record(s_in)
    for _ in range(steps):
        step()
    t1.record(s_out)
    torch.cuda.synchronize(dev)
    barrier()
    ms_local = t0.elapsed_time(t1) / steps
    value, ms = aggregate(wl.ntok, ms_local, dev)
    return {"value": value, "unit": "tokens/s", "ms_per_step": ms, "steps": steps,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "pipelining": "input copy, transfer and read-back on three streams, two buffer sets"}


def run_reference(args):
    """The fp64 oracle, as it stands, on the machine's host cores (one thread),
    for the same op, workload, metric and config as the GPU arm.  Each step
    is a bounded sample of that workload, stated in ``cpu_baseline.sample``:
    a few source tokens through every target layer, head and K|V (through
    two target layers for the wide map, scaled to all: the work is linear in
    the target layers), a few tokens of the two caches for the diagnostics,
    one fit on its first observations for the ridge fit (scaled to all
    observations)."""
    import torch
    import oracle
    from cross_model_kv_transfer_gb300 import workloads as W
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    f64 = lambda t: t.detach().cpu().to(torch.float64).numpy()
    if args.op == "ridge_features":
        wl = W.WORKLOADS[args.workload]
        if args.tokens:
            wl = wl.with_tokens([args.tokens], [0])
        m = 64
        kw = feature_sample(wl, m)
        run = lambda: oracle.ridge_features(**kw)
        scale, units = 1.0, float(m)
        metric, unit, config = FEATURE_METRIC, "tokens/s", feature_config(wl)
        sample = (f"{m} tokens per step through all {wl.tgt_layers} target layers x "
                  f"{wl.kv_heads} heads x K|V")
    elif args.op == "layer_scores":
        wl = W.WORKLOADS[args.workload].with_tokens([args.score_tokens], [0])
        m = 512
        kw, f = score_sample(wl, m)
        run = lambda: oracle.layer_scores(**kw)
        full = score_flops(wl.src_layers, wl.tgt_layers, wl.kv_heads, wl.head_dim, wl.k, wl.ntok)
        scale, units = full / f, float(wl.ntok)
        metric, unit, config = SCORE_METRIC, "tokens/s", score_config(wl, wl.ntok)
        sample = (f"{m} tokens x all {wl.src_layers} source layers x 2 target layers x 1 head "
                  "x K|V per step, scaled to the whole workload by useful flops")
    elif args.op == "ridge_fit":
        wl = W.WORKLOADS[args.workload]
        m = 256
        x, y = W.make_ridge_inputs(wl, 1, m, "cpu")
        xs, ys = f64(x[0]), f64(y[0])
        run = lambda: oracle.ridge_fit(xs, ys, 0.01)
        scale = args.ridge_n / m                    # one fit = n / m samples
        metric, unit, config = RIDGE_METRIC, "fits/s", ridge_config(wl, args.ridge_batch,
                                                                    args.ridge_n)
        units = 1.0
        sample = (f"one fit on its first {m} of {args.ridge_n} observations per step, "
                  f"scaled to {args.ridge_n} observations")
    elif args.op == "kv_diagnostics":
        wl = select_workload(args)
        n = 16
        small = wl.with_tokens([n], [0])
        inp = W.make_inputs(small, "cpu")
        mk, mv, _ = oracle.transfer(**oracle_sample_inputs(small, inp, n))
        rk = f64(W.perturbed_like(torch.from_numpy(mk), 101))
        rv = f64(W.perturbed_like(torch.from_numpy(mv), 102))
        run = lambda: oracle.kv_diagnostics(mapped_k=mk, mapped_v=mv, ref_k=rk, ref_v=rv,
                                            theta_tgt=wl.theta_tgt, max_position=n, ntok=n,
                                            dst_capacity=n)
        scale, units = 1.0, float(n)
        metric, unit, config = DIAG_METRIC, "tokens/s", diag_config(wl)
        sample = (f"{n} tokens of a mapped cache and a perturbed copy per step through all "
                  f"{wl.tgt_layers} target layers x {wl.kv_heads} heads x K|V")
    else:
        import dataclasses
        wl = select_workload(args)
        wide = args.mapper == "wide"
        n = 1 if wide else 2
        L = min(wl.tgt_layers, 2) if wide else wl.tgt_layers
        small = dataclasses.replace(wl.with_tokens([n], [0]), tgt_layers=L)
        inp = W.make_inputs(small, "cpu")
        if wide:
            inp["w"] = W.make_wide_weights(small, "cpu")
        kw = oracle_sample_inputs(small, inp, n, wide=wide)
        if args.src_block_size:
            pk, pv, table = W.make_paged_source(small, inp, args.src_block_size)
            kw.update(src_k=f64(pk), src_v=f64(pv), src_layout=oracle.PAGED,
                      src_block_size=args.src_block_size,
                      src_block_table=table.numpy(), ntok=n)
        run = lambda: oracle.transfer(**kw)
        scale, units = wl.tgt_layers / L, float(n)
        metric, unit, config = transfer_metric(wl, wide), "tokens/s", transfer_config(wl, args)
        sample = (f"{n} source token{'s' if n > 1 else ''} per step through {L} target layers"
                  f" x {wl.kv_heads} heads x K|V"
                  + (f", scaled to all {wl.tgt_layers}" if L < wl.tgt_layers else "")
                  + (f", read through {args.src_block_size}-token source blocks"
                     if args.src_block_size else ""))
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    el = (time.perf_counter() - t0) * scale
    value = units * args.steps / el
    line = {
        "impl": "reference", "metric": metric, "value": value, "unit": unit,
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config,
        "cpu_baseline": {"value": value, "unit": unit, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    if args.op != "transfer":
        line["op"] = args.op                      # as the GPU arm's line for this op
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    elif args.op == "ridge_fit":
        run_ridge(args)
    elif args.op == "layer_scores":
        run_scores(args)
    elif args.op == "ridge_features":
        run_features(args)
    else:
        run_kvx(args)


if __name__ == "__main__":
    main()
