"""GPU parity with a paged SOURCE: the pilot's own paged cache read through a
source block table (the target install's block-table rule, knlp.io routing
page, inject step, applied to the pilot's side).  Every kernel (SIMT, the
tensor-core kernel on CTA pairs and on single CTAs, the wide map) against the
fp64 oracle reading the same paged arrays, and against the oracle reading
the packed source (the two must agree: the layout changes no value).
Tolerances as in the other parity tests; routing bit for bit through the
sentinel rows."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from cross_model_kv_transfer_gb300 import kvx
from cross_model_kv_transfer_gb300.workloads import (PAGED, WORKLOADS, make_inputs,
                                                     make_paged_source, make_wide_weights)

from parity import TC_SINGLE, assert_parity, kernel_code, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

KERNELS = [pytest.param(kvx.KVX_KERNEL_SIMT, id="simt"),
           pytest.param(kvx.KVX_KERNEL_TCGEN05, id="tcgen05"),
           pytest.param(TC_SINGLE, id="tcgen05_single_cta"),
           pytest.param("wide", id="wide")]
SRC_BS = 16


def paged_plan(wl, kernel, src_bs=SRC_BS, max_tokens=None, max_position=None):
    wide = kernel == "wide"
    return kvx.Plan(src_layers=wl.src_layers, tgt_layers=wl.tgt_layers, kv_heads=wl.kv_heads,
                    head_dim=wl.head_dim, k=wl.k, rope_theta_src=wl.theta_src,
                    rope_theta_tgt=wl.theta_tgt,
                    max_position=wl.max_position if max_position is None else max_position,
                    kv_dtype=wl.kv_dtype, w_dtype=torch.float32, b_dtype=wl.b_dtype,
                    layout=wl.layout, block_size=wl.block_size if wl.layout == PAGED else 0,
                    kernel=kvx.KVX_KERNEL_TCGEN05 if wide else kernel_code(kernel),
                    flags=kvx.KVX_PLAN_TC_SINGLE_CTA if kernel == TC_SINGLE else 0,
                    mapper=kvx.KVX_MAPPER_WIDE if wide else kvx.KVX_MAPPER_PER_HEAD,
                    max_tokens=wl.ntok if max_tokens is None else max_tokens,
                    src_layout=kvx.KVX_PAGED, src_block_size=src_bs)


def paged_inputs(wl, kernel, src_bs=SRC_BS):
    inp = make_inputs(wl, "cuda")
    if kernel == "wide":
        inp["w"] = make_wide_weights(wl, "cuda")
    pk, pv, table = make_paged_source(wl, inp, src_bs)
    return inp, pk, pv, table


def run_paged(wl, inp, pk, pv, table, plan, **over):
    return run_gpu(wl, inp, plan=plan, src_k=pk, src_v=pv, src_block_table=table, ntok=wl.ntok,
                   **over)


def oracle_paged(wl, inp, pk, pv, table, kernel, src_bs=SRC_BS, **over):
    f64 = lambda t: t.detach().cpu().to(torch.float64).numpy()
    return run_oracle(wl, inp, src_k=f64(pk), src_v=f64(pv), src_layout=oracle.PAGED,
                      src_block_size=src_bs, src_block_table=table.cpu().numpy(),
                      ntok=wl.ntok, wide=kernel == "wide", **over)


@pytest.mark.parametrize("kernel", KERNELS)
def test_paged_source_and_paged_target_match_oracle(kernel):
    # three requests whose packed rows straddle the source blocks and the
    # 128 / 256-row tiles, per-request target offsets, both caches paged
    base = WORKLOADS["llama31_8b_70b_paged"]
    wl = dataclasses.replace(base.with_tokens([100, 37, 260], [5, 64, 0]), tgt_layers=4)
    if kernel == "wide":
        wl = dataclasses.replace(wl, kv_heads=2, k=2)
    inp, pk, pv, table = paged_inputs(wl, kernel)
    plan = paged_plan(wl, kernel)
    gk, gv, st, _ = run_paged(wl, inp, pk, pv, table, plan)
    assert st == 0
    rk, rv, rst = oracle_paged(wl, inp, pk, pv, table, kernel)
    assert rst == 0
    assert_parity(wl, gk, gv, rk, rv)
    # the same values from the packed source
    ck, cv, _ = run_oracle(wl, inp, wide=kernel == "wide")
    m = ~np.isnan(rk)
    assert np.array_equal(np.isnan(ck), np.isnan(rk))
    assert np.array_equal(ck[m], rk[m]) and np.array_equal(cv[m], rv[m])


@pytest.mark.parametrize("kernel", KERNELS)
def test_bad_source_blocks_are_skipped_and_flagged(kernel):
    base = WORKLOADS["llama31_8b_70b_paged"]
    wl = dataclasses.replace(base.with_tokens([40, 150, 9], [0, 20, 7]), tgt_layers=3)
    if kernel == "wide":
        wl = dataclasses.replace(wl, kv_heads=2, k=1)
    inp, pk, pv, table = paged_inputs(wl, kernel)
    table = table.clone()
    table[1, 2] = -1                       # request 1, positions 32..47
    table[0, 1] = 10 ** 6                  # request 0, positions 16..31: outside the pool
    plan = paged_plan(wl, kernel)
    gk, gv, st, _ = run_paged(wl, inp, pk, pv, table, plan)
    rk, rv, rst = oracle_paged(wl, inp, pk, pv, table, kernel)
    assert st == rst == oracle.BAD_SRC_BLOCK
    assert_parity(wl, gk, gv, rk, rv)


@pytest.mark.parametrize("kernel", [pytest.param(kvx.KVX_KERNEL_SIMT, id="simt"),
                                    pytest.param(kvx.KVX_KERNEL_TCGEN05, id="tcgen05")])
def test_paged_source_with_explicit_source_positions(kernel):
    # explicit source positions choose the slots (and the un-rotation angles)
    wl = WORKLOADS["qwen3_0p6b_1p7b"].with_tokens([300], [0])
    wl = dataclasses.replace(wl, tgt_layers=3)
    inp = make_inputs(wl, "cuda")
    g = torch.Generator().manual_seed(5)
    src_pos = torch.randperm(300, generator=g).to(torch.int32)
    # the pilot cache holds token g at position src_pos[g]
    nb = (300 + SRC_BS - 1) // SRC_BS
    table = torch.randperm(nb + 2, generator=g)[:nb].to(torch.int32).view(1, nb)
    rows = table[0, src_pos.long() // SRC_BS].long() * SRC_BS + src_pos.long() % SRC_BS
    pk = torch.zeros((wl.src_layers, (nb + 2) * SRC_BS, wl.kv_heads, wl.head_dim),
                     dtype=wl.kv_dtype, device="cuda")
    pv = torch.zeros_like(pk)
    pk[:, rows.cuda()] = inp["src_k"]
    pv[:, rows.cuda()] = inp["src_v"]
    table = table.cuda()
    plan = paged_plan(wl, kernel)
    gk, gv, st, _ = run_paged(wl, inp, pk, pv, table, plan, src_pos=src_pos.cuda())
    assert st == 0
    rk, rv, rst = oracle_paged(wl, inp, pk, pv, table, kernel, src_pos=src_pos.numpy())
    assert rst == 0
    assert_parity(wl, gk, gv, rk, rv)


def test_tensor_core_plan_rejects_more_tokens_than_its_buffers():
    wl = dataclasses.replace(WORKLOADS["qwen3_0p6b_1p7b"].with_tokens([300], [0]), tgt_layers=2)
    inp, pk, pv, table = paged_inputs(wl, kvx.KVX_KERNEL_TCGEN05)
    plan = paged_plan(wl, kvx.KVX_KERNEL_TCGEN05, max_tokens=299)
    assert plan.launches_per_transfer == 3     # pack, W image, transfer
    shape = (wl.tgt_layers, wl.dst_rows, wl.kv_heads, wl.head_dim)
    dk = torch.zeros(shape, dtype=wl.kv_dtype, device="cuda")
    dv = torch.zeros(shape, dtype=wl.kv_dtype, device="cuda")
    args = plan.make_args(src_k=pk, src_v=pv, layer_idx=inp["layer_idx"], w=inp["w"],
                          b=inp["b"], dst_k=dk, dst_v=dv, dst_capacity=wl.dst_capacity,
                          ntok=wl.ntok, src_block_table=table)
    assert kvx.kvx_transfer(plan.handle, args, None) == kvx.KVX_ERR_INVALID_ARG
    args.src_block_table = None
    assert kvx.kvx_transfer(plan.handle, args, None) == kvx.KVX_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert bool((dk == 0).all())


def test_full_size_8b_70b_paged_source_stratified_tokens_match_oracle():
    # the 8B -> 70B batched recipe (16 requests, 1,024..16,384 tokens, paged
    # target) with the pilot's cache paged too, in 16-token blocks, through
    # the tensor-core kernel; the oracle recomputes windows of 64 tokens at
    # both ends of every request, around every 8,192-token boundary of the
    # batch and at seeded random places, for every (target layer, head, K|V)
    from parity import assert_token_parity, dst_rows_of, oracle_tokens
    from test_gpu_full_size import check_sentinels, stratified_tokens
    wl = WORKLOADS["llama31_8b_70b_paged"]
    inp, pk, pv, table = paged_inputs(wl, kvx.KVX_KERNEL_TCGEN05)
    plan = paged_plan(wl, kvx.KVX_KERNEL_TCGEN05)
    gk, gv, st, _ = run_paged(wl, inp, pk, pv, table, plan)
    assert st == 0
    del pk, pv
    check_sentinels(wl, inp, gk, gv)
    tokens = stratified_tokens(wl, inp, seed=29, window=64)
    ok, ov, toks = oracle_tokens(wl, inp, tokens)
    worst = assert_token_parity(wl, gk, gv, ok, ov, dst_rows_of(wl, inp, toks))
    print(f"paged source 8B->70B: {len(toks)} tokens, worst map {worst[0]:.3e} at {worst[1]}")
