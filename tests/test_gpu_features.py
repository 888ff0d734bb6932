"""GPU parity of the ridge-fit observations (kvx_ridge_features) with the
fp64 oracle (oracle.ridge_features), element by element: x (the table row's
source layers side by side, keys un-rotated with the source base) and y (the
target layer, keys un-rotated with the target base) on fp32 and bf16 caches,
ragged request tables, explicit positions, the flag rules and the refusals.

Values are copied, so they must match exactly.  Keys are un-rotated in fp32
with angles from the plan's fixed-point phases: the angle carries at most
~4e-7 rad of error and __sincosf ~4e-7 more, so each output of a RoPE pair
(x0, x1) is within ~1e-6 (|x0| + |x1|) of the exact value; the tests allow
3e-6 (|o0| + |o1|) over the oracle's output pair (o0, o1), whose |o0| + |o1|
is at least (|x0| + |x1|) / sqrt 2.  A bf16 output adds its own rounding: half
an ulp of the result, allowed as 2^-8 |o|."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from cross_model_kv_transfer_gb300 import kvx

pytestmark = pytest.mark.gpu


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
    max_position: int = 4096

    @property
    def ntok(self):
        return sum(self.lens)


def make_inputs(c: Case, seed: int):
    """Seeded caches of the same tokens (stored values), a layer table with
    repeated and out-of-order layers, a request table and positions."""
    g = torch.Generator().manual_seed(seed)
    n, H, d = c.ntok, c.H, c.d
    scale = torch.exp(torch.randn((c.Ls, 1, H, d), generator=g))
    out = dict(src_k=torch.randn((c.Ls, n, H, d), generator=g) * scale,
               src_v=torch.randn((c.Ls, n, H, d), generator=g),
               tgt_k=torch.randn((c.Lt, n, H, d), generator=g) * 3.0,
               tgt_v=torch.randn((c.Lt, n, H, d), generator=g))
    out = {k: v.to(c.dtype) for k, v in out.items()}
    out["layer_idx"] = torch.randint(0, c.Ls, (c.Lt, c.k), generator=g, dtype=torch.int32)
    cu = torch.zeros(len(c.lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(c.lens), 0)
    out["cu_seqlens"] = cu
    out["src_pos"] = torch.randint(0, c.max_position, (n,), generator=g, dtype=torch.int32)
    return out


def plan_for(c: Case, **over):
    kw = dict(src_layers=c.Ls, tgt_layers=c.Lt, kv_heads=c.H, head_dim=c.d, k=c.k,
              rope_theta_src=c.theta_src, rope_theta_tgt=c.theta_tgt,
              max_position=c.max_position, kv_dtype=c.dtype, w_dtype=torch.float32,
              b_dtype=torch.float32, kernel=kvx.KVX_KERNEL_SIMT)
    kw.update(over)
    return kvx.Plan(**kw)


def run_gpu(c, inp, plan=None, with_y=True, out_dtype=torch.float32, positions=True,
            table=True, **over):
    plan = plan_for(c) if plan is None else plan
    dev = {k: v.cuda() for k, v in inp.items()}
    dev.update({k: v.cuda() for k, v in over.items()})
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    x, y = plan.ridge_features(src_k=dev["src_k"], src_v=dev["src_v"],
                               tgt_k=dev["tgt_k"] if with_y else None,
                               tgt_v=dev["tgt_v"] if with_y else None,
                               layer_idx=dev["layer_idx"],
                               cu_seqlens=dev["cu_seqlens"] if table else None,
                               src_pos=dev["src_pos"] if positions else None,
                               out_dtype=out_dtype, status=status)
    torch.cuda.synchronize()
    y = None if y is None else y.float().cpu().numpy()
    return x.float().cpu().numpy(), y, int(status.item())


def run_oracle(c, inp, positions=True, table=True, **over):
    f64 = lambda t: t.to(torch.float64).numpy()
    inp = dict(inp, **over)
    x, y, st = oracle.ridge_features(
        src_k=f64(inp["src_k"]), src_v=f64(inp["src_v"]), tgt_k=f64(inp["tgt_k"]),
        tgt_v=f64(inp["tgt_v"]), theta_src=c.theta_src, theta_tgt=c.theta_tgt,
        max_position=c.max_position, layer_idx=inp["layer_idx"].numpy(),
        cu_seqlens=inp["cu_seqlens"].numpy() if table else None,
        src_pos=inp["src_pos"].numpy() if positions else None)
    B = c.Lt * c.H * 2
    return x.reshape(B, c.ntok, c.k * c.d), y.reshape(B, c.ntok, c.d), st


def pair_tol(o, d, rel=3e-6):
    """3e-6 (|o0| + |o1|) for every element of the RoPE pair (i, i + d/2)
    within each d-wide piece of the last axis."""
    s = o.reshape(o.shape[:-1] + (o.shape[-1] // d, 2, d // 2))
    t = rel * (np.abs(s[..., 0, :]) + np.abs(s[..., 1, :]))
    return np.concatenate([t, t], axis=-1).reshape(o.shape)


def check(c, gx, gy, ox, oy, bf16_out=False):
    """Keys within the pair tolerance (+ bf16 rounding), values exact."""
    kd = c.k * c.d
    gx = gx.reshape(c.Lt, c.H, 2, c.ntok, kd)
    ox = ox.reshape(c.Lt, c.H, 2, c.ntok, kd)
    round_tol = (lambda o: np.abs(o) * 2.0 ** -8) if bf16_out else (lambda o: 0.0)
    for g, o, w in ((gx, ox, kd), (gy, oy, c.d)):
        if g is None:
            continue
        g = g.reshape(c.Lt, c.H, 2, c.ntok, w)
        o = o.reshape(c.Lt, c.H, 2, c.ntok, w)
        kk, ok = g[:, :, 0], o[:, :, 0]
        err = np.abs(kk - ok)
        assert np.all(err <= pair_tol(ok, c.d) + round_tol(ok)), err.max()
        want_v = o[:, :, 1].astype(np.float32)
        if bf16_out:
            want_v = torch.from_numpy(want_v).to(torch.bfloat16).float().numpy()
        np.testing.assert_array_equal(g[:, :, 1], want_v)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_features_match_oracle_ragged_with_positions(dtype):
    c = Case(Ls=5, Lt=3, H=2, d=64, k=3, lens=(70, 1, 133, 0, 37), dtype=dtype)
    inp = make_inputs(c, 21)
    gx, gy, st = run_gpu(c, inp)
    ox, oy, ost = run_oracle(c, inp)
    assert st == 0 and ost == 0
    check(c, gx, gy, ox, oy)


def test_features_request_offsets_without_positions_d128_bf16_out():
    # positions from each request's own offsets; head_dim 128, bf16 output
    c = Case(Ls=4, Lt=2, H=2, d=128, k=4, lens=(300, 45, 211), dtype=torch.bfloat16,
             max_position=300)
    inp = make_inputs(c, 22)
    gx, gy, st = run_gpu(c, inp, positions=False, out_dtype=torch.bfloat16)
    ox, oy, ost = run_oracle(c, inp, positions=False)
    assert st == 0 and ost == 0
    check(c, gx, gy, ox, oy, bf16_out=True)


def test_features_single_request_small_head_dim_without_target():
    # one request, no table; head_dim 8 (one thread per token); y omitted:
    # x is written alone and equals the x of a call with the target caches
    c = Case(Ls=3, Lt=4, H=3, d=8, k=2, lens=(517,), theta_src=5e5, theta_tgt=1e4,
             max_position=517)
    inp = make_inputs(c, 23)
    gx, gy, st = run_gpu(c, inp, with_y=False, positions=False, table=False)
    gx2, gy2, _ = run_gpu(c, inp, positions=False, table=False)
    ox, oy, ost = run_oracle(c, inp, positions=False, table=False)
    assert st == 0 and ost == 0 and gy is None
    np.testing.assert_array_equal(gx, gx2)
    check(c, gx, gy2, ox, oy)


def test_features_long_table_rows():
    # k = 10 selected layers per target layer (rows of 160 features)
    c = Case(Ls=12, Lt=2, H=1, d=16, k=10, lens=(97, 64))
    inp = make_inputs(c, 26)
    gx, gy, st = run_gpu(c, inp)
    ox, oy, ost = run_oracle(c, inp)
    assert st == 0 and ost == 0
    check(c, gx, gy, ox, oy)


def test_features_flags_zero_what_they_name():
    c = Case(Ls=3, Lt=2, H=2, d=32, k=2, lens=(50, 30), max_position=64)
    inp = make_inputs(c, 24)
    # a position past the limit: that token's rows are zero in x and y
    pos = inp["src_pos"].clone()
    pos[17] = 64
    pos[61] = -1
    gx, gy, st = run_gpu(c, inp, src_pos=pos)
    ox, oy, ost = run_oracle(c, inp, src_pos=pos)
    assert st == ost == kvx.KVX_FLAG_BAD_POSITION
    assert not gx[:, [17, 61]].any() and not gy[:, [17, 61]].any()
    check(c, gx, gy, ox, oy)
    # a table row naming a missing layer: that target layer's x is zero, y kept
    bad = inp["layer_idx"].clone()
    bad[1, 1] = 3
    gx, gy, st = run_gpu(c, inp, layer_idx=bad)
    ox, oy, ost = run_oracle(c, inp, layer_idx=bad)
    assert st == ost == kvx.KVX_FLAG_BAD_LAYER_INDEX
    assert not gx[c.H * 2:].any() and gx[:c.H * 2].any()
    check(c, gx, gy, ox, oy)
    # a request table that does not end at ntok: all zeros
    cu = inp["cu_seqlens"].clone()
    cu[-1] -= 1
    gx, gy, st = run_gpu(c, inp, cu_seqlens=cu)
    _, _, ost = run_oracle(c, inp, cu_seqlens=cu)
    assert st == ost == kvx.KVX_FLAG_BAD_SEQLENS
    assert not gx.any() and not gy.any()


def test_features_refusals():
    c = Case(Ls=2, Lt=2, H=1, d=16, k=1, lens=(40,))
    inp = {k: v.cuda() for k, v in make_inputs(c, 25).items()}
    plan = plan_for(c)
    x = torch.zeros((c.Lt * 2, c.ntok, c.d), device="cuda")
    y = torch.zeros_like(x)
    raw = torch.zeros(x.numel() + 4, device="cuda")

    def call(**over):
        a = dict(src_k=inp["src_k"].data_ptr(), src_v=inp["src_v"].data_ptr(),
                 tgt_k=inp["tgt_k"].data_ptr(), tgt_v=inp["tgt_v"].data_ptr(), ntok=c.ntok,
                 num_requests=1, cu_seqlens=None, src_pos=None,
                 layer_idx=inp["layer_idx"].data_ptr(), out_dtype=kvx.KVX_F32,
                 x=x.data_ptr(), y=y.data_ptr(), status=None)
        a.update(over)
        return kvx.kvx_ridge_features(plan.handle, kvx.FeatureArgs(**a), None)

    assert call() == kvx.KVX_OK
    assert call(x=raw.data_ptr() + 4) == kvx.KVX_ERR_INVALID_ARG        # misaligned
    assert call(tgt_v=None) == kvx.KVX_ERR_INVALID_ARG                  # y without target
    assert call(num_requests=2) == kvx.KVX_ERR_INVALID_ARG              # R > 1, no table
    assert call(out_dtype=5) == kvx.KVX_ERR_INVALID_ARG
    assert call(layer_idx=None) == kvx.KVX_ERR_INVALID_ARG
    assert call(ntok=-1) == kvx.KVX_ERR_INVALID_ARG
    # ntok = 0: nothing to write, nothing launched
    x.fill_(7.0)
    assert call(ntok=0) == kvx.KVX_OK
    torch.cuda.synchronize()
    assert bool((x == 7.0).all())
    # zero tokens through the binding: torch gives the empty caches NULL data
    e = torch.empty((c.Ls, 0, c.H, c.d), device="cuda")
    et = torch.empty((c.Lt, 0, c.H, c.d), device="cuda")
    xe, ye = plan.ridge_features(src_k=e, src_v=e, tgt_k=et, tgt_v=et,
                                 layer_idx=inp["layer_idx"])
    torch.cuda.synchronize()
    assert tuple(xe.shape) == (c.Lt * c.H * 2, 0, c.k * c.d) and ye.shape[1] == 0
    # a wide-mapper plan has no per-head fits
    wide = kvx.Plan(src_layers=2, tgt_layers=2, kv_heads=1, head_dim=128, k=1,
                    rope_theta_src=1e4, rope_theta_tgt=1e4, max_position=64,
                    kv_dtype=torch.bfloat16, w_dtype=torch.bfloat16, b_dtype=torch.float32,
                    kernel=kvx.KVX_KERNEL_TCGEN05, mapper=kvx.KVX_MAPPER_WIDE)
    a = kvx.FeatureArgs(inp["src_k"].data_ptr(), inp["src_v"].data_ptr(), None, None, 0, 1,
                        None, None, inp["layer_idx"].data_ptr(), kvx.KVX_F32, x.data_ptr(), None,
                        None)
    assert kvx.kvx_ridge_features(wide.handle, a, None) == kvx.KVX_ERR_UNSUPPORTED


def test_features_full_size_sampled_tokens():
    # the 14B -> 32B shape at 32,768 calibration tokens with fp32 output, as
    # the benchmark times it: 64 target layers x 8 heads x K|V, k = 4 (68.7 GB
    # of x, 17.2 GB of y); 40 sampled tokens checked against the oracle, which
    # computes each token on its own given its position
    from cross_model_kv_transfer_gb300.workloads import WORKLOADS, make_score_inputs
    wl = WORKLOADS["qwen3_14b_32b"]
    Ls, Lt, H, d, k, n = wl.src_layers, wl.tgt_layers, wl.kv_heads, wl.head_dim, wl.k, wl.ntok
    inp = make_score_inputs(wl, "cuda")
    plan = kvx.Plan(src_layers=Ls, tgt_layers=Lt, kv_heads=H, head_dim=d, k=k,
                    rope_theta_src=wl.theta_src, rope_theta_tgt=wl.theta_tgt,
                    max_position=wl.max_position, kv_dtype=wl.kv_dtype, w_dtype=torch.float32,
                    b_dtype=torch.float32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    x, y = plan.ridge_features(src_k=inp["src_k"], src_v=inp["src_v"], tgt_k=inp["tgt_k"],
                               tgt_v=inp["tgt_v"], layer_idx=inp["layer_idx"], status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    g = torch.Generator().manual_seed(31)
    idx = torch.cat([torch.tensor([0, 15, 16, n - 1]), torch.randint(0, n, (36,), generator=g)])
    idx_d = idx.cuda()
    gx = x[:, idx_d].cpu().numpy()
    gy = y[:, idx_d].cpu().numpy()
    del x, y
    sub = {c: inp[c][:, idx_d].cpu() for c in ("src_k", "src_v", "tgt_k", "tgt_v")}
    c = Case(Ls=Ls, Lt=Lt, H=H, d=d, k=k, lens=(len(idx),), theta_src=wl.theta_src,
             theta_tgt=wl.theta_tgt, dtype=wl.kv_dtype, max_position=wl.max_position)
    sub.update(layer_idx=inp["layer_idx"].cpu(), cu_seqlens=torch.tensor([0, len(idx)]),
               src_pos=idx.to(torch.int32))
    ox, oy, ost = run_oracle(c, sub, table=False)
    assert ost == 0
    check(c, gx, gy, ox, oy)
