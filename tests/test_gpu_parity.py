"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances (relative Frobenius error per target layer, head and K|V):
1e-5 for fp32 caches, 1e-2 for bf16 caches with fp32 accumulation.  Index
gathering, routing and paged scatter are checked bit for bit: rows outside
the transfer keep their sentinel bits, and planted values land exactly.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from cross_model_kv_transfer_gb300 import kvx
from cross_model_kv_transfer_gb300.workloads import WORKLOADS, make_inputs, sentinel_like

from parity import (TC_SINGLE, assert_parity, gpu_args, kernel_code, make_plan, run_gpu,
                    run_oracle)

pytestmark = pytest.mark.gpu

BF16_KERNELS = [pytest.param(kvx.KVX_KERNEL_SIMT, id="simt"),
                pytest.param(kvx.KVX_KERNEL_TCGEN05, id="tcgen05"),
                pytest.param(TC_SINGLE, id="tcgen05_single_cta")]


def test_tiny_fp32_workload_matches_oracle():
    wl = WORKLOADS["tiny_fp32"]
    inp = make_inputs(wl, "cuda")
    gk, gv, st, plan = run_gpu(wl, inp)
    assert st == 0 and plan.kernel == kvx.KVX_KERNEL_SIMT
    rk, rv, rst = run_oracle(wl, inp)
    assert rst == 0
    assert_parity(wl, gk, gv, rk, rv)


@pytest.mark.parametrize("kernel", BF16_KERNELS)
def test_qwen3_0p6b_1p7b_512_tokens_matches_oracle(kernel):
    wl = WORKLOADS["qwen3_0p6b_1p7b"]
    inp = make_inputs(wl, "cuda")
    gk, gv, st, plan = run_gpu(wl, inp, kernel)
    assert st == 0 and plan.kernel == kernel_code(kernel)
    if kernel == TC_SINGLE:
        assert plan.cta_group == 1
    elif kernel == kvx.KVX_KERNEL_TCGEN05:
        assert plan.cta_group in (1, 2)
    rk, rv, _ = run_oracle(wl, inp)
    assert_parity(wl, gk, gv, rk, rv)


@pytest.mark.parametrize("kernel", BF16_KERNELS)
def test_offset37_ragged_tail_matches_oracle(kernel):
    # the 0.6B -> 1.7B pair with the target shifted by +37, at 300 tokens:
    # two full 128-token tiles and a ragged tail of 44
    wl = WORKLOADS["qwen3_0p6b_1p7b_off37_2k"].with_tokens([300], [37])
    inp = make_inputs(wl, "cuda")
    gk, gv, st, _ = run_gpu(wl, inp, kernel)
    assert st == 0
    rk, rv, _ = run_oracle(wl, inp)
    assert_parity(wl, gk, gv, rk, rv)


@pytest.mark.parametrize("kernel", BF16_KERNELS)
def test_batched_paged_varlen_matches_oracle(kernel):
    # the 8B -> 70B paged recipe with three short requests, per-request
    # offsets and a permuted block pool
    base = WORKLOADS["llama31_8b_70b_paged"]
    wl = base.with_tokens([100, 37, 260], [5, 64, 0])
    wl = dataclasses.replace(wl, tgt_layers=12)
    inp = make_inputs(wl, "cuda")
    gk, gv, st, _ = run_gpu(wl, inp, kernel)
    assert st == 0
    rk, rv, _ = run_oracle(wl, inp)
    assert_parity(wl, gk, gv, rk, rv)


@pytest.mark.parametrize("kernel", [pytest.param(kvx.KVX_KERNEL_SIMT, id="simt")])
def test_explicit_positions_match_oracle(kernel):
    # explicit (non-contiguous) source and target positions
    wl = WORKLOADS["tiny_fp32"].with_tokens([96], [0])
    inp = make_inputs(wl, "cuda")
    g = torch.Generator().manual_seed(11)
    src_pos = torch.randperm(120, generator=g)[:96].to(torch.int32)
    tgt_pos = torch.randperm(128, generator=g)[:96].to(torch.int32)
    wl = dataclasses.replace(wl, seqlens=(96,), tgt_offsets=(32,))  # capacity 128
    gk, gv, st, _ = run_gpu(wl, inp, kernel, src_pos=src_pos.cuda(), tgt_pos=tgt_pos.cuda())
    assert st == 0
    rk, rv, _ = run_oracle(wl, inp, src_pos=src_pos.numpy(), tgt_pos=tgt_pos.numpy())
    assert_parity(wl, gk, gv, rk, rv)


def _planted(wl, inp):
    """Source values that are exact small integers in the cache dtype, and
    maps W that select one feature per output (so y is exact)."""
    Ls, T, H, d = inp["src_v"].shape
    k = wl.k
    s = torch.arange(Ls).view(Ls, 1, 1, 1)
    t = torch.arange(T).view(1, T, 1, 1)
    c = torch.arange(d).view(1, 1, 1, d)
    h = torch.arange(H).view(1, 1, H, 1)
    vals = ((s * 37 + t * 11 + h * 5 + c * 3) % 251 - 125).to(torch.float32)
    g = torch.Generator().manual_seed(7)
    w = torch.zeros(wl.tgt_layers, H, 2, k * d, d)
    perm = torch.stack([torch.randperm(k * d, generator=g)[:d]
                        for _ in range(wl.tgt_layers * H * 2)]).view(wl.tgt_layers, H, 2, d)
    w.scatter_(3, perm.unsqueeze(3), 1.0)
    return vals, w, perm


@pytest.mark.parametrize("kernel", BF16_KERNELS)
def test_paged_routing_is_bit_exact(kernel):
    # Values carry no RoPE: with planted integer values and selection maps
    # every written value must equal the oracle's bit for bit, and every slot
    # the block tables do not reach must keep its sentinel.
    base = WORKLOADS["llama31_8b_70b_paged"]
    wl = base.with_tokens([45, 130, 17], [3, 0, 60])
    wl = dataclasses.replace(wl, tgt_layers=5)
    inp = make_inputs(wl, "cuda")
    vals, w, perm = _planted(wl, inp)
    inp["src_v"] = vals.to(wl.kv_dtype).cuda()
    inp["w"] = w.cuda()
    inp["b"] = torch.zeros_like(inp["b"])
    gk, gv, st, _ = run_gpu(wl, inp, kernel)
    assert st == 0
    _, rv, _ = run_oracle(wl, inp)
    written = ~np.isnan(rv)
    gvd = gv.to(torch.float64).cpu().numpy()
    assert np.array_equal(gvd[written], rv[written])
    assert bool((gv.view(torch.int16)[torch.from_numpy(~written).cuda()] == -1).all())


@pytest.mark.parametrize("kernel", BF16_KERNELS)
def test_identity_map_reproduces_source(kernel):
    # k = 1, W = I, b = 0, equal thetas, offset 0: values exactly, keys within
    # one bf16 rounding of the source.
    base = WORKLOADS["qwen3_0p6b_1p7b"].with_tokens([200], [0])
    wl = dataclasses.replace(base, k=1, tgt_layers=3)
    inp = make_inputs(wl, "cuda")
    inp["w"] = torch.eye(wl.head_dim).expand(3, wl.kv_heads, 2, wl.head_dim,
                                             wl.head_dim).contiguous().cuda()
    inp["b"] = torch.zeros_like(inp["b"])
    gk, gv, st, _ = run_gpu(wl, inp, kernel)
    assert st == 0
    for lt in range(3):
        s = int(inp["layer_idx"][lt, 0])
        assert torch.equal(gv[lt, :200], inp["src_v"][s])
        err = (gk[lt, :200].float() - inp["src_k"][s].float()).norm() / inp["src_k"][s].float().norm()
        assert err < 4e-3


@pytest.mark.parametrize("kernel", BF16_KERNELS)
def test_device_detected_errors_match_oracle_flags(kernel):
    base = WORKLOADS["llama31_8b_70b_paged"]
    wl = base.with_tokens([40, 150, 9], [0, 20, 7])
    wl = dataclasses.replace(wl, tgt_layers=4)
    inp = make_inputs(wl, "cuda")
    # a selection index outside [0, Ls) in target layer 2
    idx = inp["layer_idx"].clone()
    idx[2, 1] = wl.src_layers + 3
    # a referenced block-table entry of -1 in request 1
    table = inp["block_table"].clone()
    table[1, 3] = -1
    inp2 = dict(inp, layer_idx=idx, block_table=table)
    gk, gv, st, _ = run_gpu(wl, inp2, kernel)
    rk, rv, rst = run_oracle(wl, inp2)
    assert st == rst == (oracle.BAD_LAYER_INDEX | oracle.BAD_BLOCK)
    assert_parity(wl, gk, gv, rk, rv)


@pytest.mark.parametrize("kernel", BF16_KERNELS)
def test_positions_beyond_the_table_are_skipped_and_flagged(kernel):
    wl = WORKLOADS["qwen3_0p6b_1p7b_off37_2k"].with_tokens([150], [37])
    inp = make_inputs(wl, "cuda")
    plan = make_plan(wl, kernel, max_position=160)     # p' = p + 37 >= 160 for p >= 123
    gk, gv, st, _ = run_gpu(wl, inp, kernel, plan=plan)
    rk, rv, rst = run_oracle(wl, inp, max_position=160)
    assert st == rst == oracle.BAD_POSITION
    assert_parity(wl, gk, gv, rk, rv)


def test_capacity_too_small_is_flagged():
    # p' = p + 5 runs past a 128-row contiguous capacity (the table is large
    # enough): those rows are skipped with KVX_FLAG_BAD_ROW
    wl = WORKLOADS["tiny_fp32"]
    inp = make_inputs(wl, "cuda")
    off = torch.tensor([5], dtype=torch.int32, device="cuda")
    plan = make_plan(wl, max_position=200)
    gk, gv, st, _ = run_gpu(wl, inp, plan=plan, tgt_offset=off)
    rk, rv, rst = run_oracle(wl, inp, max_position=200, tgt_offset=np.array([5]))
    assert st == rst == oracle.BAD_ROW
    assert_parity(wl, gk, gv, rk, rv)


@pytest.mark.parametrize("kernel", BF16_KERNELS)
def test_malformed_request_table_invalidates_the_transfer(kernel):
    base = WORKLOADS["llama31_8b_70b_paged"]
    wl = base.with_tokens([40, 30, 20], [0, 0, 0])
    wl = dataclasses.replace(wl, tgt_layers=2)
    inp = make_inputs(wl, "cuda")
    for cu in ([0, 40, 35, 90], [0, 40, 70, 89], [2, 40, 70, 90]):
        cu = torch.tensor(cu, dtype=torch.int32, device="cuda")
        gk, gv, st, _ = run_gpu(wl, inp, kernel, cu_seqlens=cu)
        rk, rv, rst = run_oracle(wl, inp, cu_seqlens=cu.cpu().numpy().astype(np.int64))
        assert st == rst == oracle.BAD_SEQLENS
        assert bool((gk.view(torch.int16) == -1).all()) and bool((gv.view(torch.int16) == -1).all())


def test_host_rejects_missing_pointers_before_launch():
    wl = WORKLOADS["tiny_fp32"]
    inp = make_inputs(wl, "cuda")
    plan = make_plan(wl)
    shape = (wl.tgt_layers, wl.dst_rows, wl.kv_heads, wl.head_dim)
    dk = torch.zeros(shape, device="cuda")
    dv = torch.zeros(shape, device="cuda")
    args = plan.make_args(**gpu_args(wl, inp, dk, dv, None))
    args.w = None
    st = kvx.kvx_transfer(plan.handle, args, None)
    assert st == kvx.KVX_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert bool((dk == 0).all())


@pytest.mark.parametrize("flags", [pytest.param(0, id="pairs"),
                                   pytest.param(kvx.KVX_PLAN_TC_SINGLE_CTA, id="single_cta")])
@pytest.mark.parametrize("k,tiles_per_item", [(1, 1), (3, 2), (5, 3), (6, 8)])
def test_tcgen05_selection_counts_and_item_sizes(k, tiles_per_item, flags):
    # other k (ring wrap-around of the four operand slots, 2k W chunks) and
    # other work-item sizes (W reloaded every 1, 2, 3 or 8 tiles)
    base = WORKLOADS["qwen3_0p6b_1p7b_off37_2k"].with_tokens([700], [37])
    wl = dataclasses.replace(base, k=k, tgt_layers=5)
    inp = make_inputs(wl, "cuda")
    plan = kvx.Plan(src_layers=wl.src_layers, tgt_layers=wl.tgt_layers, kv_heads=wl.kv_heads,
                    head_dim=wl.head_dim, k=k, rope_theta_src=wl.theta_src,
                    rope_theta_tgt=5e5, max_position=wl.max_position, kv_dtype=wl.kv_dtype,
                    w_dtype=torch.float32, b_dtype=wl.b_dtype,
                    kernel=kvx.KVX_KERNEL_TCGEN05, tiles_per_item=tiles_per_item, flags=flags)
    gk, gv, st, _ = run_gpu(wl, inp, plan=plan)
    assert st == 0
    rk, rv, _ = run_oracle(wl, inp, theta_tgt=5e5)
    assert_parity(wl, gk, gv, rk, rv)


@pytest.mark.parametrize("flags", [pytest.param(0, id="pairs"),
                                   pytest.param(kvx.KVX_PLAN_TC_SINGLE_CTA, id="single_cta")])
def test_tcgen05_schedules_agree_bit_for_bit(flags):
    # the pipeline's scheduling must not touch the arithmetic: work items of
    # 1, 3 and 32 tiles (W reloaded every tile, every 3 tiles, once; the
    # stage and operand rings wrap at different points) give the same bytes
    base = WORKLOADS["llama31_8b_70b_paged"].with_tokens([900, 130, 2200], [3, 64, 0])
    wl = dataclasses.replace(base, tgt_layers=6)
    inp = make_inputs(wl, "cuda")
    outs = []
    for tpi in (1, 3, 32):
        plan = kvx.Plan(src_layers=wl.src_layers, tgt_layers=wl.tgt_layers,
                        kv_heads=wl.kv_heads, head_dim=wl.head_dim, k=wl.k,
                        rope_theta_src=wl.theta_src, rope_theta_tgt=wl.theta_tgt,
                        max_position=wl.max_position, kv_dtype=wl.kv_dtype,
                        w_dtype=torch.float32, b_dtype=wl.b_dtype, layout=wl.layout,
                        block_size=wl.block_size, kernel=kvx.KVX_KERNEL_TCGEN05,
                        tiles_per_item=tpi, flags=flags)
        gk, gv, st, _ = run_gpu(wl, inp, plan=plan)
        assert st == 0
        outs.append((gk.view(torch.int16), gv.view(torch.int16)))
    for gk, gv in outs[1:]:
        assert torch.equal(gk, outs[0][0]) and torch.equal(gv, outs[0][1])


@pytest.mark.parametrize("flags", [pytest.param(0, id="pairs"),
                                   pytest.param(kvx.KVX_PLAN_TC_SINGLE_CTA, id="single_cta")])
def test_tcgen05_pipeline_wait_gives_up_and_reports_timeout(flags):
    # Failure detection without a GPU fault: the operand-filling warps never
    # signal, every pipeline wait gives up after its limit, the kernel drains,
    # frees tensor memory and reports KVX_FLAG_TIMEOUT; the context stays
    # usable for the next (normal) transfer.
    wl = WORKLOADS["qwen3_0p6b_1p7b"].with_tokens([256], [0])
    wl = dataclasses.replace(wl, tgt_layers=2)
    inp = make_inputs(wl, "cuda")
    stalled = kvx.Plan(src_layers=wl.src_layers, tgt_layers=wl.tgt_layers,
                       kv_heads=wl.kv_heads, head_dim=wl.head_dim, k=wl.k,
                       rope_theta_src=wl.theta_src, rope_theta_tgt=wl.theta_tgt,
                       max_position=wl.max_position, kv_dtype=wl.kv_dtype,
                       w_dtype=torch.float32, b_dtype=wl.b_dtype,
                       kernel=kvx.KVX_KERNEL_TCGEN05, flags=kvx.KVX_PLAN_TEST_STALL | flags)
    _, _, st, _ = run_gpu(wl, inp, plan=stalled)
    assert st & kvx.KVX_FLAG_TIMEOUT
    gk, gv, st, _ = run_gpu(wl, inp, kvx.KVX_KERNEL_TCGEN05)
    assert st == 0
    rk, rv, _ = run_oracle(wl, inp)
    assert_parity(wl, gk, gv, rk, rv)


@pytest.mark.parametrize("d,k", [(2, 1), (4, 3), (6, 2), (10, 2), (14, 1), (256, 3)])
def test_simt_head_dims_at_the_limits_match_oracle(d, k):
    # Below d = 16 a SIMT tile holds more rows (8 G) than its CTA has threads
    # (d/2 x G), so the row bookkeeping is strided; d = 2 is a single RoPE
    # pair, 256 the largest head dim.  Three requests with target offsets
    # leave ragged tails across several tiles.
    seqlens = (700, 3, 333) if d < 256 else (300, 3, 33)
    wl = dataclasses.replace(WORKLOADS["tiny_fp32"], name=f"tiny_fp32_d{d}_k{k}", head_dim=d,
                             k=k, seqlens=seqlens, tgt_offsets=(0, 5, 2))
    inp = make_inputs(wl, "cuda")
    gk, gv, st, plan = run_gpu(wl, inp, kvx.KVX_KERNEL_SIMT)
    assert st == 0 and plan.kernel == kvx.KVX_KERNEL_SIMT
    rk, rv, rst = run_oracle(wl, inp)
    assert rst == 0
    assert_parity(wl, gk, gv, rk, rv)


@pytest.mark.parametrize("kernel", BF16_KERNELS)
def test_empty_transfer_enqueues_nothing(kernel):
    # ntok = 0 through the C ABI (valid buffers, zero tokens): the call
    # succeeds, the status word and both caches keep their bits
    wl = WORKLOADS["qwen3_0p6b_1p7b"]
    inp = make_inputs(wl, "cuda")
    plan = make_plan(wl, kernel)
    shape = (wl.tgt_layers, wl.dst_rows, wl.kv_heads, wl.head_dim)
    dk = sentinel_like(shape, wl.kv_dtype, "cuda")
    dv = sentinel_like(shape, wl.kv_dtype, "cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    args = plan.make_args(**gpu_args(wl, inp, dk, dv, status))
    args.ntok = 0
    assert kvx.kvx_transfer(plan.handle, args, None) == kvx.KVX_OK
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert bool((dk.view(torch.int16) == -1).all()) and bool((dv.view(torch.int16) == -1).all())
    # the same through the Python binding with zero-row source tensors (no
    # storage: NULL data pointers)
    empty = torch.empty((wl.src_layers, 0, wl.kv_heads, wl.head_dim), dtype=wl.kv_dtype,
                        device="cuda")
    plan.transfer(**gpu_args(wl, dict(inp, src_k=empty, src_v=empty.clone()), dk, dv, status,
                             cu_seqlens=torch.zeros(2, dtype=torch.int32, device="cuda")))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert bool((dk.view(torch.int16) == -1).all()) and bool((dv.view(torch.int16) == -1).all())


def test_empty_diagnostics_clear_the_statistics():
    wl = WORKLOADS["qwen3_0p6b_1p7b"]
    plan = make_plan(wl, kvx.KVX_KERNEL_TCGEN05)
    shape = (wl.tgt_layers, wl.dst_rows, wl.kv_heads, wl.head_dim)
    cache = torch.ones(shape, dtype=wl.kv_dtype, device="cuda")
    stats = torch.full((wl.tgt_layers, wl.kv_heads, 2, wl.head_dim + 4), 7.0,
                       dtype=torch.float64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    plan.kv_diagnostics(mapped_k=cache, mapped_v=cache, ref_k=cache, ref_v=cache, stats=stats,
                        status=status, ntok=0, dst_capacity=wl.dst_capacity)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and bool((stats == 0).all())
