"""GPU parity of the layer-selection scores (kvx_layer_scores) with the fp64
oracle (oracle.layer_scores): every (target layer, source layer, head, K|V)
score and every set score, on fp32 and bf16 caches, ragged request tables,
differing RoPE bases, a planted structure, and the error rules.

The scores are explained-variance fractions in [0, 1] for these inputs; the
GPU forms them from fp32 content features (fp32 products, fp64 sums, fp64
solves), so they are compared with an absolute tolerance of 2e-5."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from cross_model_kv_transfer_gb300 import kvx

pytestmark = pytest.mark.gpu

ATOL = 2e-5


@dataclasses.dataclass
class Case:
    Ls: int
    Lt: int
    H: int
    d: int
    k: int
    lens: tuple
    theta_src: float = 1e4
    theta_tgt: float = 1e6
    dtype: torch.dtype = torch.float32

    @property
    def ntok(self):
        return sum(self.lens)


def make_case(c: Case, seed: int, planted: bool = True):
    """Paired caches of the same tokens: target layer lt (head h, K|V) is a
    seeded linear function of source layer lt % Ls in content space plus
    noise; keys stored rotated by each model's RoPE at the token's position."""
    g = torch.Generator().manual_seed(seed)
    n, d, H = c.ntok, c.d, c.H
    pos = torch.cat([torch.arange(L) for L in c.lens]).double()

    def rotate(x, theta):
        half = d // 2
        w = theta ** (-2.0 * torch.arange(half, dtype=torch.float64) / d)
        a = pos[:, None] * w[None, :]
        cs, sn = torch.cos(a)[:, None, :], torch.sin(a)[:, None, :]
        x0, x1 = x[..., :half], x[..., half:]
        return torch.cat((x0 * cs - x1 * sn, x0 * sn + x1 * cs), dim=-1)

    scale = torch.exp(torch.randn((c.Ls, 1, H, d), generator=g, dtype=torch.float64))
    xk = torch.randn((c.Ls, n, H, d), generator=g, dtype=torch.float64) * scale
    xv = torch.randn((c.Ls, n, H, d), generator=g, dtype=torch.float64)
    yk = torch.randn((c.Lt, n, H, d), generator=g, dtype=torch.float64)
    yv = torch.randn((c.Lt, n, H, d), generator=g, dtype=torch.float64)
    if planted:
        for lt in range(c.Lt):
            s = lt % c.Ls
            A = torch.randn((H, d, d), generator=g, dtype=torch.float64) / d ** 0.5
            B = torch.randn((H, d, d), generator=g, dtype=torch.float64) / d ** 0.5
            yk[lt] = torch.einsum("nhi,hij->nhj", xk[s], A) + 0.5 * yk[lt]
            yv[lt] = torch.einsum("nhi,hij->nhj", xv[s], B) + 0.5 * yv[lt]
    sk = torch.stack([rotate(xk[s], c.theta_src) for s in range(c.Ls)])
    tk = torch.stack([rotate(yk[lt], c.theta_tgt) for lt in range(c.Lt)])
    out = dict(src_k=sk, src_v=xv, tgt_k=tk, tgt_v=yv)
    out = {k: v.to(c.dtype) for k, v in out.items()}   # the stored values
    gi = torch.Generator().manual_seed(seed + 1)
    out["layer_idx"] = torch.stack([torch.randperm(c.Ls, generator=gi)[:c.k]
                                    for _ in range(c.Lt)]).to(torch.int32)
    cu = torch.zeros(len(c.lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(c.lens), 0)
    out["cu_seqlens"] = cu
    return out


def plan_for(c: Case):
    return kvx.Plan(src_layers=c.Ls, tgt_layers=c.Lt, kv_heads=c.H, head_dim=c.d, k=c.k,
                    rope_theta_src=c.theta_src, rope_theta_tgt=c.theta_tgt,
                    max_position=max(c.lens), kv_dtype=c.dtype, w_dtype=torch.float32,
                    b_dtype=torch.float32, kernel=kvx.KVX_KERNEL_SIMT)


def run_both(c: Case, inp, lam=0.01, src_pos=None):
    plan = plan_for(c)
    dev = {k: v.cuda() for k, v in inp.items()}
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    r2, r2s = plan.layer_scores(src_k=dev["src_k"], src_v=dev["src_v"], tgt_k=dev["tgt_k"],
                                tgt_v=dev["tgt_v"], lam=lam,
                                cu_seqlens=dev["cu_seqlens"] if len(c.lens) > 1 else None,
                                src_pos=None if src_pos is None else src_pos.cuda(),
                                layer_idx=dev["layer_idx"], status=status)
    torch.cuda.synchronize()
    f64 = lambda t: t.to(torch.float64).numpy()
    ref, ref_s, st = oracle.layer_scores(
        src_k=f64(inp["src_k"]), src_v=f64(inp["src_v"]), tgt_k=f64(inp["tgt_k"]),
        tgt_v=f64(inp["tgt_v"]), theta_src=c.theta_src, theta_tgt=c.theta_tgt,
        max_position=max(c.lens), lam=lam,
        cu_seqlens=inp["cu_seqlens"].numpy() if len(c.lens) > 1 else None,
        src_pos=None if src_pos is None else src_pos.numpy(),
        layer_idx=inp["layer_idx"].numpy())
    return r2.cpu().numpy(), r2s.cpu().numpy(), int(status.item()), ref, ref_s, st


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_scores_match_oracle_ragged_batch(dtype):
    c = Case(Ls=4, Lt=3, H=2, d=32, k=2, lens=(70, 5, 133), dtype=dtype)
    g, gs, st, r, rs, rst = run_both(c, make_case(c, 11))
    assert st == 0 and rst == 0
    assert np.all(np.isfinite(g)) and np.all(np.isfinite(gs))
    assert np.abs(g - r).max() <= ATOL, np.abs(g - r).max()
    assert np.abs(gs - rs).max() <= ATOL, np.abs(gs - rs).max()
    # the planted source layer is the best single layer of every target
    assert np.all(g.argmax(axis=1) == np.arange(c.Lt)[:, None, None] % c.Ls)


def test_scores_match_oracle_head_dim_128_with_explicit_positions():
    c = Case(Ls=5, Lt=4, H=2, d=128, k=3, lens=(600,), theta_src=1e6, theta_tgt=5e5,
             dtype=torch.bfloat16)
    inp = make_case(c, 12, planted=False)
    # explicit positions (a permutation): the stored keys were rotated at
    # 0..599, so read them there
    pos = torch.arange(600, dtype=torch.int32)
    g, gs, st, r, rs, rst = run_both(c, inp, lam=0.5, src_pos=pos)
    assert st == 0 and rst == 0
    assert np.abs(g - r).max() <= ATOL, np.abs(g - r).max()
    assert np.abs(gs - rs).max() <= ATOL, np.abs(gs - rs).max()


def test_scores_over_several_token_chunks_match_oracle():
    # 20,000 + 13,001 tokens: the tensor-core moments run over three chunks
    # of up to 16,384 tokens (the last one ragged), summed in fp64
    c = Case(Ls=3, Lt=2, H=1, d=16, k=2, lens=(20000, 13001), dtype=torch.bfloat16)
    g, gs, st, r, rs, rst = run_both(c, make_case(c, 15))
    assert st == 0 and rst == 0
    assert np.abs(g - r).max() <= ATOL, np.abs(g - r).max()
    assert np.abs(gs - rs).max() <= ATOL, np.abs(gs - rs).max()


def test_scores_nan_and_flags_for_bad_inputs():
    c = Case(Ls=3, Lt=2, H=1, d=16, k=2, lens=(40, 24))
    inp = make_case(c, 13)
    inp["layer_idx"][1, 1] = 7                     # outside [0, Ls)
    g, gs, st, r, rs, rst = run_both(c, inp)
    assert st & kvx.KVX_FLAG_BAD_LAYER_INDEX and rst == oracle.BAD_LAYER_INDEX
    assert np.all(np.isnan(gs[1])) and np.all(np.isnan(rs[1]))
    assert np.abs(gs[0] - rs[0]).max() <= ATOL
    assert np.abs(g - r).max() <= ATOL
    # a position beyond the plan's table: nothing is scored
    pos = torch.cat([torch.arange(40), torch.arange(24)]).to(torch.int32)
    pos[3] = 10 ** 6
    inp = make_case(c, 13)
    g, gs, st, r, rs, rst = run_both(c, inp, src_pos=pos)
    assert st & kvx.KVX_FLAG_BAD_POSITION and rst == oracle.BAD_POSITION
    assert np.all(np.isnan(g)) and np.all(np.isnan(gs)) and np.all(np.isnan(r))
    # a request table that does not end at ntok: nothing is scored
    inp = make_case(c, 13)
    inp["cu_seqlens"][-1] = 63
    g, gs, st, r, rs, rst = run_both(c, inp)
    assert st & kvx.KVX_FLAG_BAD_SEQLENS and rst == oracle.BAD_SEQLENS
    assert np.all(np.isnan(g)) and np.all(np.isnan(gs)) and np.all(np.isnan(r))


def test_scores_refuse_bad_arguments_before_launch():
    c = Case(Ls=2, Lt=2, H=1, d=16, k=1, lens=(8,))
    plan = plan_for(c)
    assert kvx.kvx_layer_scores_workspace_bytes(plan.handle, 1) == 0
    need = kvx.kvx_layer_scores_workspace_bytes(plan.handle, 8)
    assert need > 0
    inp = {k: v.cuda() for k, v in make_case(c, 14).items()}
    r2 = torch.empty((2, 2, 1, 2), dtype=torch.float64, device="cuda")
    ws = torch.empty(need - 1, dtype=torch.uint8, device="cuda")
    a = kvx.ScoreArgs(inp["src_k"].data_ptr(), inp["src_v"].data_ptr(), inp["tgt_k"].data_ptr(),
                      inp["tgt_v"].data_ptr(), 8, 1, None, None, None, 0.01, r2.data_ptr(), None,
                      ws.data_ptr(), ws.numel(), None)
    assert kvx.kvx_layer_scores(plan.handle, a, None) == kvx.KVX_ERR_INVALID_ARG   # scratch
    a.workspace_bytes = need
    a.__setattr__("lambda", 0.0)
    assert kvx.kvx_layer_scores(plan.handle, a, None) == kvx.KVX_ERR_INVALID_ARG   # lambda
    a.__setattr__("lambda", 0.01)
    a.r2_set = r2.data_ptr()                       # a set output without a table
    assert kvx.kvx_layer_scores(plan.handle, a, None) == kvx.KVX_ERR_INVALID_ARG
    a.r2_set = None
    ws3 = torch.empty(need + 8, dtype=torch.uint8, device="cuda")
    a.workspace, a.workspace_bytes = ws3.data_ptr() + 8, need    # not 16-byte aligned
    assert kvx.kvx_layer_scores(plan.handle, a, None) == kvx.KVX_ERR_INVALID_ARG
    a.workspace_bytes = need
    ws2 = torch.empty(need, dtype=torch.uint8, device="cuda")
    a.workspace = ws2.data_ptr()
    assert kvx.kvx_layer_scores(plan.handle, a, None) == kvx.KVX_OK
    torch.cuda.synchronize()
    assert bool(torch.isfinite(r2).all())


def test_scores_full_size_sampled_entries_match_oracle():
    """The 14B -> 32B shape at 4,096 calibration tokens, in the launch
    configuration the benchmark times (every head, K|V and layer pair in one
    call).  Each score depends only on its own source layer(s), target layer
    and head, so the oracle recomputes sampled entries from those slices:
    single-layer scores at the first, last and seeded random (lt, s, h)
    and set scores of the first, last and random target layers.  Every
    score must lie in [0, 1] (ridge residual between 0 and SS_tot)."""
    from cross_model_kv_transfer_gb300.workloads import WORKLOADS, make_score_inputs
    wl = WORKLOADS["qwen3_14b_32b"].with_tokens([4096], [0])
    inp = make_score_inputs(wl, "cuda")
    Ls, Lt, H, d, k = wl.src_layers, wl.tgt_layers, wl.kv_heads, wl.head_dim, wl.k
    plan = kvx.Plan(src_layers=Ls, tgt_layers=Lt, kv_heads=H, head_dim=d, k=k,
                    rope_theta_src=wl.theta_src, rope_theta_tgt=wl.theta_tgt,
                    max_position=wl.max_position, kv_dtype=wl.kv_dtype, w_dtype=torch.float32,
                    b_dtype=wl.b_dtype, kernel=kvx.KVX_KERNEL_SIMT)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    r2, r2s = plan.layer_scores(src_k=inp["src_k"], src_v=inp["src_v"], tgt_k=inp["tgt_k"],
                                tgt_v=inp["tgt_v"], lam=0.01, layer_idx=inp["layer_idx"],
                                status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    g, gs = r2.cpu().numpy(), r2s.cpu().numpy()
    assert np.all((g >= 0) & (g <= 1)) and np.all((gs >= 0) & (gs <= 1))
    idx = inp["layer_idx"].cpu().numpy()
    rng = np.random.default_rng(5)
    picks = [(0, 0, 0), (Lt - 1, Ls - 1, H - 1), (0, int(idx[0, 0]), 1)]
    picks += [(int(rng.integers(Lt)), int(rng.integers(Ls)), int(rng.integers(H)))
              for _ in range(3)]
    f64 = lambda t: t.cpu().to(torch.float64).numpy()
    common = dict(theta_src=wl.theta_src, theta_tgt=wl.theta_tgt,
                  max_position=wl.max_position, lam=0.01)
    worst = 0.0
    for lt, s, h in picks:
        r, _, st = oracle.layer_scores(
            src_k=f64(inp["src_k"][s:s + 1, :, h:h + 1]), src_v=f64(inp["src_v"][s:s + 1, :, h:h + 1]),
            tgt_k=f64(inp["tgt_k"][lt:lt + 1, :, h:h + 1]),
            tgt_v=f64(inp["tgt_v"][lt:lt + 1, :, h:h + 1]), **common)
        assert st == 0
        err = np.abs(g[lt, s, h] - r[0, 0, 0]).max()
        worst = max(worst, err)
        assert err <= ATOL, (lt, s, h, err)
    for lt, h in ((0, 0), (Lt - 1, H - 1), (int(rng.integers(Lt)), int(rng.integers(H)))):
        sel = torch.from_numpy(idx[lt].astype(np.int64)).cuda()
        _, rs, st = oracle.layer_scores(
            src_k=f64(inp["src_k"][sel][:, :, h:h + 1]), src_v=f64(inp["src_v"][sel][:, :, h:h + 1]),
            tgt_k=f64(inp["tgt_k"][lt:lt + 1, :, h:h + 1]),
            tgt_v=f64(inp["tgt_v"][lt:lt + 1, :, h:h + 1]),
            layer_idx=np.arange(k, dtype=np.int32)[None, :], **common)
        assert st == 0
        err = np.abs(gs[lt, h] - rs[0, 0]).max()
        worst = max(worst, err)
        assert err <= ATOL, (lt, h, err)
    print(f"layer scores at 4,096 tokens: worst sampled |r2 - oracle| {worst:.2e}; "
          f"mean best single layer {g.max(axis=1).mean(axis=(0, 1))}, mean set {gs.mean(axis=(0, 1))}")


def test_scores_with_large_means_match_oracle():
    # caches whose content means are ~50x their spread (values only, keys
    # carry the same offsets before rotation): the totals and moments come
    # from centred values
    c = Case(Ls=3, Lt=2, H=2, d=32, k=2, lens=(900,), dtype=torch.float32)
    inp = make_case(c, 16)
    for name in ("src_v", "tgt_v"):
        inp[name] = inp[name] + 50.0
    g, gs, st, r, rs, rst = run_both(c, inp)
    assert st == 0 and rst == 0
    assert np.abs(g - r).max() <= ATOL, np.abs(g - r).max()
    assert np.abs(gs - rs).max() <= ATOL, np.abs(gs - rs).max()
