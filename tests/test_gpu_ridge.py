"""GPU parity of the ridge fit (kvx_ridge_fit) against the fp64 oracle's
ridge demo restatement (``oracle.ridge_fit``: centred X and Y, (XcT Xc +
lam I) W = XcT Yc by Cholesky, b = ybar - xbar W; the Qwen3 article's
linear-bridge section).

Tolerances.  The GPU forms the centred Gram blocks from fp32 products (fp32
partial sums over 256 observations, summed in fp32 over slices of 16,384,
slices added in fp64) and solves in fp64, so its Gram blocks carry a relative
error of ~1e-6; the solve amplifies that by
at most the condition number kappa of XcT Xc + lam I.  The tests draw
features with moderate scale spread (kappa below ~1e3, computed and checked
in each test) and require, per fit, a relative Frobenius error of W and of
b within 1e-6 * kappa (at least 1e-5), and predictions X W + b within 1e-5
of the oracle's.  W and b are stored as fp32 (relative rounding 6e-8).
"""
import numpy as np
import pytest
import torch

import oracle
from cross_model_kv_transfer_gb300 import kvx

pytestmark = pytest.mark.gpu


def _data(batch, n, p, q, seed, dtype=torch.float32, spread=0.5, noise=0.1):
    g = torch.Generator(device="cuda").manual_seed(seed)
    scale = torch.exp(spread * torch.randn((batch, 1, p), generator=g, device="cuda"))
    x = torch.randn((batch, n, p), generator=g, device="cuda") * scale + \
        torch.randn((batch, 1, p), generator=g, device="cuda")
    w = torch.randn((batch, p, q), generator=g, device="cuda") / p ** 0.5
    y = x @ w + 0.3 * torch.randn((batch, 1, q), generator=g, device="cuda") + \
        noise * torch.randn((batch, n, q), generator=g, device="cuda")
    return x.to(dtype).contiguous(), y.to(dtype).contiguous()


def _check(x, y, w, b, lam):
    xs = x.double().cpu().numpy()
    ys = y.double().cpu().numpy()
    wg = w.double().cpu().numpy()
    bg = b.double().cpu().numpy()
    for i in range(xs.shape[0]):
        wr, br = oracle.ridge_fit(xs[i], ys[i], lam)
        xc = xs[i] - xs[i].mean(axis=0)
        kappa = np.linalg.cond(xc.T @ xc + lam * np.eye(xc.shape[1]))
        assert kappa < 1e4, kappa
        tol = max(1e-5, 1e-6 * kappa)
        ew = np.linalg.norm(wg[i] - wr) / np.linalg.norm(wr)
        eb = np.linalg.norm(bg[i] - br) / max(np.linalg.norm(br), 1e-12)
        assert ew <= tol, (i, ew, tol)
        assert eb <= tol, (i, eb, tol)
        pr = xs[i] @ wr + br
        pg = xs[i] @ wg[i] + bg[i]
        assert np.linalg.norm(pg - pr) / np.linalg.norm(pr) <= 1e-5


@pytest.mark.parametrize("n,p,q", [(2000, 96, 40), (300, 64, 64), (40000, 70, 33)])
def test_ridge_fit_matches_oracle(n, p, q):
    # ragged Gram tiles (96, 70, 33), one full tile, and several observation
    # slices added with atomics (40,000 > 16,384)
    x, y = _data(3, n, p, q, seed=n + p)
    w, b = kvx.ridge_fit(x, y, lam=0.01)
    torch.cuda.synchronize()
    _check(x, y, w, b, 0.01)


def test_ridge_fit_bf16_observations():
    # stored bf16: the oracle reads the same rounded values
    x, y = _data(2, 3000, 128, 64, seed=7, dtype=torch.bfloat16)
    w, b = kvx.ridge_fit(x, y, lam=0.5)
    torch.cuda.synchronize()
    _check(x, y, w, b, 0.5)


def test_ridge_fit_per_head_map_shape():
    # the 14B -> 32B per-head map: 4 selected layers x 128 dims -> 128 dims
    x, y = _data(2, 4096, 512, 128, seed=11, spread=0.3)
    w, b = kvx.ridge_fit(x, y, lam=0.01)
    torch.cuda.synchronize()
    _check(x, y, w, b, 0.01)


def test_ridge_fit_recovers_a_planted_map():
    # noiseless y = x W* + b*: as lam -> 0 the fit returns W*, b*
    g = torch.Generator(device="cuda").manual_seed(3)
    x = torch.randn((1, 5000, 48), generator=g, device="cuda")
    ws = torch.randn((1, 48, 20), generator=g, device="cuda")
    bs = torch.randn((1, 20), generator=g, device="cuda")
    y = (x.double() @ ws.double() + bs.double()[:, None, :]).float()
    w, b = kvx.ridge_fit(x, y, lam=1e-8)
    torch.cuda.synchronize()
    assert torch.allclose(w, ws, rtol=0, atol=2e-4)
    assert torch.allclose(b, bs, rtol=0, atol=2e-4)


def test_ridge_fit_flags_a_matrix_that_is_not_positive_definite():
    x, y = _data(2, 500, 32, 8, seed=5)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    w, b = kvx.ridge_fit(x, y, lam=-1e9, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == kvx.KVX_FLAG_NOT_SPD
    assert bool(torch.isnan(w).all()) and bool(torch.isnan(b).all())
    # the next (valid) fit on the same stream is unaffected
    w, b = kvx.ridge_fit(x, y, lam=0.01)
    torch.cuda.synchronize()
    _check(x, y, w, b, 0.01)


def test_ridge_fit_writes_the_transfer_layout():
    # a batch ordered (target layer, head, K|V) with p = k*d, q = d is the
    # [Lt][H][2][k*d][d] map and [Lt][H][2][d] bias a per-head plan reads
    Lt, H, k, d, n = 2, 2, 2, 16, 600
    x, y = _data(Lt * H * 2, n, k * d, d, seed=17)
    w, b = kvx.ridge_fit(x, y, lam=0.01)
    torch.cuda.synchronize()
    W = w.view(Lt, H, 2, k * d, d)
    B = b.view(Lt, H, 2, d)
    xs, ys = x.double().cpu().numpy(), y.double().cpu().numpy()
    wr, br = oracle.ridge_fit(xs[5], ys[5], 0.01)     # fit 5 = (lt 1, h 0, V)
    np.testing.assert_allclose(W[1, 0, 1].double().cpu().numpy(), wr, rtol=0, atol=1e-4)
    np.testing.assert_allclose(B[1, 0, 1].double().cpu().numpy(), br, rtol=0, atol=1e-4)


def test_host_rejects_a_small_workspace():
    x, y = _data(1, 100, 16, 4, seed=1)
    need = kvx.kvx_ridge_workspace_bytes(1, 16, 4)
    ws = torch.empty(need - 8, dtype=torch.uint8, device="cuda")
    with pytest.raises(kvx.KvxError):
        kvx.ridge_fit(x, y, workspace=ws)
    # large enough but not 16-byte aligned (the split-precision planes are
    # read by TMA)
    ws = torch.empty(need + 8, dtype=torch.uint8, device="cuda")[8:]
    with pytest.raises(kvx.KvxError):
        kvx.ridge_fit(x, y, workspace=ws)


def test_ridge_fit_wide_feature_block_solves_in_large_shared_memory():
    # p = 3,100 features: one output column per solve CTA, whose columns and
    # pivot reciprocals take more than 48 KB of shared memory.  The fp64
    # reference here is the normal equations solved by LAPACK on the same
    # observations (a plain library solve of the ridge problem).
    x, y = _data(1, 6500, 3100, 3, seed=23, spread=0.2)
    w, b = kvx.ridge_fit(x, y, lam=0.01)
    torch.cuda.synchronize()
    xs, ys = x[0].double().cpu().numpy(), y[0].double().cpu().numpy()
    xm, ym = xs.mean(axis=0), ys.mean(axis=0)
    xc, yc = xs - xm, ys - ym
    g = xc.T @ xc + 0.01 * np.eye(xs.shape[1])
    wr = np.linalg.solve(g, xc.T @ yc)
    br = ym - xm @ wr
    kappa = np.linalg.cond(g)
    wg, bg = w[0].double().cpu().numpy(), b[0].double().cpu().numpy()
    assert np.linalg.norm(wg - wr) / np.linalg.norm(wr) <= max(1e-5, 1e-6 * kappa)
    assert np.linalg.norm(bg - br) / np.linalg.norm(br) <= max(1e-5, 1e-6 * kappa)
    pg, pr = xs @ wg + bg, xs @ wr + br
    assert np.linalg.norm(pg - pr) / np.linalg.norm(pr) <= 1e-5


def test_ridge_fit_centres_before_the_products_large_offsets():
    # features and targets whose means are ~100x their spread: the Gram
    # blocks are formed from centred values, so no cancellation eats the
    # split-precision products (an uncentred XtX - n mu mu^T would lose ~4
    # digits here)
    g = torch.Generator(device="cuda").manual_seed(31)
    n, p, q = 6000, 64, 16
    x = torch.randn((1, n, p), generator=g, device="cuda") + \
        100.0 * (1.0 + torch.rand((1, 1, p), generator=g, device="cuda"))
    w = torch.randn((p, q), generator=g, device="cuda") / p ** 0.5
    y = (x - x.mean(dim=1, keepdim=True)) @ w + 300.0 + \
        0.1 * torch.randn((1, n, q), generator=g, device="cuda")
    wg, bg = kvx.ridge_fit(x.contiguous(), y.contiguous(), lam=0.01)
    torch.cuda.synchronize()
    _check(x, y, wg, bg, 0.01)


def test_ridge_fit_drifting_observations_and_fewer_than_the_shift_sample():
    # column means that drift along the observation order by several
    # spreads, on top of a large offset: the moments are formed about a
    # per-column shift taken from observations spread over the whole set and
    # centred exactly afterwards, so neither the offset nor the drift costs
    # digits; and a fit with fewer observations (120) than the shift's
    # sample of 256
    g = torch.Generator(device="cuda").manual_seed(37)
    n, p, q = 20000, 48, 24
    t = torch.linspace(0.0, 1.0, n, device="cuda")[None, :, None]
    x = torch.randn((1, n, p), generator=g, device="cuda") + \
        5.0 * t * torch.randn((1, 1, p), generator=g, device="cuda") + 50.0
    w = torch.randn((p, q), generator=g, device="cuda") / p ** 0.5
    y = x @ w - 20.0 + 0.1 * torch.randn((1, n, q), generator=g, device="cuda")
    wg, bg = kvx.ridge_fit(x.contiguous(), y.contiguous(), lam=0.01)
    torch.cuda.synchronize()
    _check(x, y, wg, bg, 0.01)
    x, y = _data(2, 120, 32, 8, seed=38)
    wg, bg = kvx.ridge_fit(x, y, lam=0.01)
    torch.cuda.synchronize()
    _check(x, y, wg, bg, 0.01)
