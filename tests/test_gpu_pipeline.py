"""The method end to end through the library, on one synthetic model pair:
choose each target layer's source layers by their scores (kvx_layer_scores),
fit the per-(target layer, head, K|V) maps on those layers' content features
(kvx_ridge_features, kvx_ridge_fit), transfer the pilot's cache with them (kvx_transfer), and
measure the mapped cache against the target's own (kvx_kv_diagnostics).

The pieces check one another: the scorer must find the planted source
layers, and the explained variance of the mapped cache (the diagnostics, on
the transfer's bf16 output) must equal the scorer's in-sample set score for
the chosen table (both are the R^2 of the same centred ridge fit on the same
tokens), up to the rounding of the transfer's bf16 output (measured 1.4e-5;
the test allows 1e-4)."""
import dataclasses

import numpy as np
import pytest
import torch

from cross_model_kv_transfer_gb300 import kvx
from cross_model_kv_transfer_gb300.workloads import WORKLOADS, make_score_inputs

pytestmark = pytest.mark.gpu


def test_scores_fit_transfer_and_diagnostics_agree():
    wl = dataclasses.replace(WORKLOADS["qwen3_14b_32b"].with_tokens([3000], [0]), src_layers=6,
                             tgt_layers=4, kv_heads=2, k=2, theta_tgt=5e5)
    Ls, Lt, H, d, k, n = wl.src_layers, wl.tgt_layers, wl.kv_heads, wl.head_dim, wl.k, wl.ntok
    inp = make_score_inputs(wl, "cuda")
    plan = kvx.Plan(src_layers=Ls, tgt_layers=Lt, kv_heads=H, head_dim=d, k=k,
                    rope_theta_src=wl.theta_src, rope_theta_tgt=wl.theta_tgt,
                    max_position=wl.max_position, kv_dtype=wl.kv_dtype, w_dtype=torch.float32,
                    b_dtype=torch.float32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    # 1. layer selection: the k best source layers of each target layer by
    #    their single-layer scores (mean over heads and K|V)
    r2, _ = plan.layer_scores(src_k=inp["src_k"], src_v=inp["src_v"], tgt_k=inp["tgt_k"],
                              tgt_v=inp["tgt_v"], lam=0.01, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    best = r2.mean(dim=(2, 3)).argsort(dim=1, descending=True)[:, :k]
    table = best.sort(dim=1).values.to(torch.int32).contiguous()
    planted = inp["layer_idx"].long().sort(dim=1).values
    assert torch.equal(table.long(), planted), (table, planted)
    _, r2_set = plan.layer_scores(src_k=inp["src_k"], src_v=inp["src_v"], tgt_k=inp["tgt_k"],
                                  tgt_v=inp["tgt_v"], lam=0.01, layer_idx=table, status=status)

    # 2. the maps: one ridge fit per (target layer, head, K|V) on the content
    #    features of the chosen layers (kvx_ridge_features writes them in the
    #    batch order the transfer reads W in)
    x, y = plan.ridge_features(src_k=inp["src_k"], src_v=inp["src_v"], tgt_k=inp["tgt_k"],
                               tgt_v=inp["tgt_v"], layer_idx=table, status=status)
    w, b = kvx.ridge_fit(x, y, lam=0.01)
    del x, y

    # 3. the transfer with the chosen table and the fitted maps
    mk = torch.empty((Lt, n, H, d), dtype=wl.kv_dtype, device="cuda")
    mv = torch.empty_like(mk)
    plan.transfer(src_k=inp["src_k"], src_v=inp["src_v"], layer_idx=table,
                  w=w.view(Lt, H, 2, k * d, d), b=b.view(Lt, H, 2, d), dst_k=mk, dst_v=mv,
                  dst_capacity=n, status=status)

    # 4. the mapped cache against the target's own
    stats = torch.empty((Lt, H, 2, d + 4), dtype=torch.float64, device="cuda")
    plan.kv_diagnostics(mapped_k=mk, mapped_v=mv, ref_k=inp["tgt_k"], ref_v=inp["tgt_v"],
                        stats=stats, ntok=n, dst_capacity=n, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    s = stats.cpu().numpy()
    cnt = s[..., 0]
    ss_tot = s[..., 3] - np.sum(s[..., 4:] ** 2, axis=-1) / cnt
    ev = 1.0 - s[..., 2] / ss_tot
    score = r2_set.cpu().numpy()
    assert np.all(cnt == n)
    assert np.all(score > 0.9), score
    err = np.abs(ev - score).max()
    print(f"pipeline: table {table.tolist()}, set scores {score.min():.4f}..{score.max():.4f}, "
          f"|diagnostics R^2 - set score| <= {err:.2e}")
    assert err <= 1e-4, err
