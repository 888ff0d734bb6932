"""GPU parity of the fidelity diagnostics (kvx_kv_diagnostics) against the
fp64 oracle: KV cosine ("Helm Intelligent Routing", "Reading the retention
score") and explained variance (Qwen3 14B -> 32B article, linear-bridge
section) of a mapped cache against the target's own cache.

The mapped cache is the output of a real transfer on the GPU; the target's
own cache is a seeded perturbation of it (so cosines and R^2 are neither 0
nor 1).  Tolerances: the token counts exactly; the cosine sums to 1e-5 of
n; residual and reference energies to 1e-5 relative; each content-space sum
to 1e-5 of sqrt(n * sum |ref|^2) (Cauchy-Schwarz bound of its size); mean
cosine and R^2 to 1e-5 absolute.  The kernel sums in fp32 per thread over at
most 1024 tokens and in fp64 across threads.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from cross_model_kv_transfer_gb300 import kvx
from cross_model_kv_transfer_gb300.workloads import PAGED, WORKLOADS, make_inputs, perturbed_like

from parity import make_plan, run_gpu

pytestmark = pytest.mark.gpu


def _perturb(x, seed):
    """The target's own cache stand-in (NaN sentinel rows stay NaN)."""
    return perturbed_like(x, seed)


def _diag_kwargs(wl, inp, **over):
    kw = dict(ntok=wl.ntok)
    if wl.num_requests > 1 or wl.layout == PAGED:
        kw["cu_seqlens"] = inp["cu_seqlens"]
    if any(wl.tgt_offsets):
        kw["tgt_offset"] = inp["tgt_offset"]
    if wl.layout == PAGED:
        kw["block_table"] = inp["block_table"]
        kw["num_blocks"] = wl.num_blocks
    else:
        kw["dst_capacity"] = wl.dst_capacity
    kw.update(over)
    return kw


def run_gpu_diag(plan, mk, mv, rk, rv, **kw):
    Lt, _, H, d = rk.shape
    stats = torch.full((Lt, H, 2, d + 4), float("nan"), dtype=torch.float64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    plan.kv_diagnostics(mapped_k=mk, mapped_v=mv, ref_k=rk, ref_v=rv, stats=stats,
                        status=status, **kw)
    torch.cuda.synchronize()
    return stats.cpu().numpy(), int(status.item())


def run_oracle_diag(wl, mk, mv, rk, rv, max_position=None, theta_tgt=None, **kw):
    f64 = lambda t: t.detach().cpu().to(torch.float64).numpy()
    conv = {}
    for key, v in kw.items():
        if isinstance(v, torch.Tensor):
            v = v.cpu().numpy()
            if key != "block_table":
                v = v.astype(np.int64)
        conv[key] = v
    layout = oracle.PAGED if wl.layout == PAGED else oracle.CONTIGUOUS
    if layout == oracle.PAGED:
        conv.setdefault("block_size", wl.block_size)
    return oracle.kv_diagnostics(
        mapped_k=f64(mk), mapped_v=f64(mv), ref_k=f64(rk), ref_v=f64(rv),
        theta_tgt=wl.theta_tgt if theta_tgt is None else theta_tgt,
        max_position=wl.max_position if max_position is None else max_position,
        layout=layout, **conv)


def assert_stats_close(g, r, tol=1e-5):
    n = r[..., 0]
    assert np.array_equal(g[..., 0], n), "token counts differ"
    np.testing.assert_allclose(g[..., 1], r[..., 1], rtol=0, atol=tol * max(n.max(), 1))
    np.testing.assert_allclose(g[..., 2], r[..., 2], rtol=tol, atol=1e-30)
    np.testing.assert_allclose(g[..., 3], r[..., 3], rtol=tol, atol=1e-30)
    bound = np.sqrt(n * r[..., 3])[..., None]
    assert np.all(np.abs(g[..., 4:] - r[..., 4:]) <= tol * bound + 1e-30), \
        f"content sums: worst {np.max(np.abs(g[..., 4:] - r[..., 4:]) / (bound + 1e-300)):.2e}"
    has = n > 0
    np.testing.assert_allclose(oracle.mean_cosine(g)[has], oracle.mean_cosine(r)[has], atol=tol)
    np.testing.assert_allclose(oracle.explained_variance(g)[has],
                               oracle.explained_variance(r)[has], atol=tol)


def _mapped_and_ref(wl, kernel=kvx.KVX_KERNEL_AUTO, seed=21):
    inp = make_inputs(wl, "cuda")
    mk, mv, st, plan = run_gpu(wl, inp, kernel)
    assert st == 0
    return inp, plan, mk, mv, _perturb(mk, seed), _perturb(mv, seed + 1)


@pytest.mark.parametrize("kernel", [pytest.param(kvx.KVX_KERNEL_SIMT, id="simt_plan"),
                                    pytest.param(kvx.KVX_KERNEL_TCGEN05, id="tcgen05_plan")])
def test_offset37_ragged_contiguous_matches_oracle(kernel):
    # 1,300 tokens: a partial last chunk; target offset +37 (rows below it
    # hold sentinels and are never read)
    wl = WORKLOADS["qwen3_0p6b_1p7b_off37_2k"].with_tokens([1300], [37])
    wl = dataclasses.replace(wl, tgt_layers=6)
    inp, plan, mk, mv, rk, rv = _mapped_and_ref(wl, kernel)
    kw = _diag_kwargs(wl, inp)
    g, st = run_gpu_diag(plan, mk, mv, rk, rv, **kw)
    r, rst = run_oracle_diag(wl, mk, mv, rk, rv, **kw)
    assert st == rst == 0
    assert_stats_close(g, r)
    assert np.all(oracle.mean_cosine(g) > 0.5) and np.all(oracle.explained_variance(g) < 1)


def test_batched_paged_varlen_matches_oracle():
    wl = WORKLOADS["llama31_8b_70b_paged"].with_tokens([100, 37, 1260], [5, 64, 0])
    wl = dataclasses.replace(wl, tgt_layers=5)
    inp, plan, mk, mv, rk, rv = _mapped_and_ref(wl)
    kw = _diag_kwargs(wl, inp)
    g, st = run_gpu_diag(plan, mk, mv, rk, rv, **kw)
    r, rst = run_oracle_diag(wl, mk, mv, rk, rv, **kw)
    assert st == rst == 0
    assert_stats_close(g, r)


def test_fp32_cache_matches_oracle():
    wl = WORKLOADS["tiny_fp32"]
    inp, plan, mk, mv, rk, rv = _mapped_and_ref(wl)
    kw = _diag_kwargs(wl, inp)
    g, st = run_gpu_diag(plan, mk, mv, rk, rv, **kw)
    r, _ = run_oracle_diag(wl, mk, mv, rk, rv, **kw)
    assert st == 0
    assert_stats_close(g, r)


@pytest.mark.parametrize("d,dtype", [(20, torch.float32), (6, torch.bfloat16),
                                     (200, torch.bfloat16)])
def test_head_dims_without_8_pair_runs(d, dtype):
    # half = 10, 3 or 100: single-pair lanes (the general path), 5 heads
    Lt, H, T = 3, 5, 333
    g0 = torch.Generator(device="cuda").manual_seed(d)
    mk = torch.randn((Lt, T, H, d), generator=g0, device="cuda").to(dtype)
    mv = torch.randn((Lt, T, H, d), generator=g0, device="cuda").to(dtype)
    rk, rv = _perturb(mk, 3), _perturb(mv, 4)
    plan = kvx.Plan(src_layers=2, tgt_layers=Lt, kv_heads=H, head_dim=d, k=1,
                    rope_theta_src=1e4, rope_theta_tgt=5e5, max_position=T, kv_dtype=dtype,
                    w_dtype=torch.float32, b_dtype=torch.float32, kernel=kvx.KVX_KERNEL_SIMT)
    wl = dataclasses.replace(WORKLOADS["tiny_fp32"], seqlens=(T,), tgt_offsets=(0,),
                             theta_tgt=5e5)
    gs, st = run_gpu_diag(plan, mk, mv, rk, rv, ntok=T, dst_capacity=T)
    r, _ = run_oracle_diag(wl, mk, mv, rk, rv, ntok=T, dst_capacity=T)
    assert st == 0
    assert_stats_close(gs, r)


def test_unaligned_caches_take_the_scalar_loads():
    # caches that start 2 bytes past a 16-byte boundary: same results
    wl = WORKLOADS["qwen3_0p6b_1p7b"].with_tokens([300], [0])
    wl = dataclasses.replace(wl, tgt_layers=3)
    inp, plan, mk, mv, rk, rv = _mapped_and_ref(wl)

    def shifted(x):
        buf = torch.empty(x.numel() + 8, dtype=x.dtype, device=x.device)
        v = buf[1:1 + x.numel()].view(x.shape)
        v.copy_(x)
        assert v.data_ptr() % 16 == 2
        return v

    kw = _diag_kwargs(wl, inp)
    g, st = run_gpu_diag(plan, shifted(mk), shifted(mv), shifted(rk), shifted(rv), **kw)
    r, _ = run_oracle_diag(wl, mk, mv, rk, rv, **kw)
    assert st == 0
    assert_stats_close(g, r)


def test_skipped_rows_and_flags_match_oracle():
    # a referenced block-table entry of -1 and positions past the table:
    # those tokens are neither compared nor counted, with the transfer's bits
    wl = WORKLOADS["llama31_8b_70b_paged"].with_tokens([40, 150, 9], [0, 20, 7])
    wl = dataclasses.replace(wl, tgt_layers=3)
    inp, plan, mk, mv, rk, rv = _mapped_and_ref(wl)
    table = inp["block_table"].clone()
    table[1, 3] = -1
    kw = _diag_kwargs(wl, inp, block_table=table)
    small = make_plan(wl, max_position=160)           # p' = 20 + 149 >= 160 for some
    g, st = run_gpu_diag(small, mk, mv, rk, rv, **kw)
    r, rst = run_oracle_diag(wl, mk, mv, rk, rv, max_position=160, **kw)
    assert st == rst == (oracle.BAD_BLOCK | oracle.BAD_POSITION)
    assert_stats_close(g, r)
    # a malformed request table: nothing compared, every statistic 0
    bad = torch.tensor([0, 40, 30, 199], dtype=torch.int32, device="cuda")
    g, st = run_gpu_diag(plan, mk, mv, rk, rv, **_diag_kwargs(wl, inp, cu_seqlens=bad))
    assert st == oracle.BAD_SEQLENS and np.all(g == 0)


def test_identity_gives_cosine_one_and_full_explained_variance():
    wl = WORKLOADS["qwen3_0p6b_1p7b"].with_tokens([700], [0])
    wl = dataclasses.replace(wl, tgt_layers=2)
    inp, plan, mk, mv, _, _ = _mapped_and_ref(wl)
    g, st = run_gpu_diag(plan, mk, mv, mk, mv, **_diag_kwargs(wl, inp))
    assert st == 0 and np.all(g[..., 0] == 700) and np.all(g[..., 2] == 0)
    np.testing.assert_allclose(oracle.mean_cosine(g), 1.0, atol=1e-6)
    np.testing.assert_allclose(oracle.explained_variance(g), 1.0, atol=1e-12)


def test_host_rejects_missing_stats():
    wl = WORKLOADS["tiny_fp32"]
    inp, plan, mk, mv, rk, rv = _mapped_and_ref(wl)
    stats = torch.zeros((wl.tgt_layers, wl.kv_heads, 2, wl.head_dim + 4), dtype=torch.float64,
                        device="cuda")
    a = plan.make_diag_args(mapped_k=mk, mapped_v=mv, ref_k=rk, ref_v=rv, stats=stats,
                            **_diag_kwargs(wl, inp))
    a.stats = None
    assert kvx.kvx_kv_diagnostics(plan.handle, a, None) == kvx.KVX_ERR_INVALID_ARG
    assert kvx.kvx_kv_diagnostics(None, a, None) == kvx.KVX_ERR_INVALID_ARG
