"""The allocation-free entry point, kvx_transfer_static.

It is meant for callers that may not allocate device memory: serving engines
that reserve nearly all of the GPU for their own KV-cache pool and forbid
later cudaMalloc calls, and latency-critical paths that cannot accept the
device synchronisation cudaMalloc/cudaFree may cause.  It runs the SIMT
transfer kernel with its RoPE tables in a fixed device array compiled into
the library instead of plan-owned memory.  The tables are filled on the device
(fp64 math, rounded once to fp32), a different source from the plan path's
host-built tables, so each call is checked on its own against the fp64 oracle,
per (target layer, head, K|V), for two calls in a row: on the tiny fp32
workload and on a ragged paged batch whose target RoPE base differs from the
source's (two tables in the array).  This file is collected last on purpose:
if it fails, a run that stops at the first failure has run every other test.
"""
import ctypes
import dataclasses

import pytest
import torch

from cross_model_kv_transfer_gb300 import kvx
from cross_model_kv_transfer_gb300.workloads import WORKLOADS, make_inputs, sentinel_like

from parity import assert_parity, gpu_args, make_plan, run_oracle


def _desc(**over):
    base = dict(src_layers=4, tgt_layers=6, src_kv_heads=2, tgt_kv_heads=2, src_head_dim=64,
                tgt_head_dim=64, k=2, rope_theta_src=1e4, rope_theta_tgt=1e4,
                kv_dtype=kvx.KVX_F32, w_dtype=kvx.KVX_F32, b_dtype=kvx.KVX_F32,
                dst_layout=kvx.KVX_CONTIGUOUS, block_size=0, max_position=128,
                kernel=kvx.KVX_KERNEL_SIMT, tiles_per_item=0, flags=0)
    base.update(over)
    return kvx.PlanDesc(**base)


def test_static_entry_point_refuses_tables_beyond_its_array():
    # 2^20 (cos, sin) entries: 32768 positions x 64 pairs fit once, not twice
    args = kvx.TransferArgs()
    d = _desc(src_head_dim=128, tgt_head_dim=128, max_position=32768, rope_theta_tgt=5e5)
    assert kvx.kvx_transfer_static(d, args, None) == kvx.KVX_ERR_TOO_LARGE
    d = _desc(src_head_dim=128, tgt_head_dim=128, max_position=16385)
    assert kvx.kvx_transfer_static(d, args, None) == kvx.KVX_ERR_TOO_LARGE
    assert kvx.kvx_transfer_static(_desc(kernel=kvx.KVX_KERNEL_TCGEN05), args, None) \
        == kvx.KVX_ERR_INVALID_ARG
    assert "fixed device array" in kvx.kvx_status_string(kvx.KVX_ERR_TOO_LARGE)


def _static_run(wl, inp, plan):
    """One kvx_transfer_static call into sentinel-filled destinations (the
    plan object only builds the descriptor and argument structures)."""
    shape = (wl.tgt_layers, wl.dst_rows, wl.kv_heads, wl.head_dim)
    dk = sentinel_like(shape, wl.kv_dtype, "cuda")
    dv = sentinel_like(shape, wl.kv_dtype, "cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    args = plan.make_args(**gpu_args(wl, inp, dk, dv, status))
    stream = torch.cuda.current_stream()
    st = kvx.kvx_transfer_static(plan.desc, args, ctypes.c_void_p(stream.cuda_stream))
    assert st == kvx.KVX_OK, kvx.kvx_status_string(st)
    torch.cuda.synchronize()
    return dk, dv, int(status.item())


@pytest.mark.gpu
def test_static_entry_point_matches_the_oracle_on_two_calls():
    tiny = WORKLOADS["tiny_fp32"]
    paged = dataclasses.replace(
        WORKLOADS["llama31_8b_70b_paged"].with_tokens([100, 37, 260], [5, 64, 0]), tgt_layers=6,
        theta_tgt=1e6)   # a target base unlike the source's: two tables in the array
    for wl in (tiny, paged):
        inp = make_inputs(wl, "cuda")
        rk, rv, rst = run_oracle(wl, inp)
        assert rst == 0
        plan = make_plan(wl, kvx.KVX_KERNEL_SIMT)
        for call in range(2):
            sk, sv, sst = _static_run(wl, inp, plan)
            assert sst == 0, f"{wl.name} call {call}: device status {sst}"
            err = assert_parity(wl, sk, sv, rk, rv)
            print(f"{wl.name} static call {call}: worst rel Frobenius {err:.2e}")
