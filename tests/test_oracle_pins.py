"""Pins of the fp64 oracle against what the sources and mathematics fix.

Each test is chosen so that a plausible mistake in the oracle fails it:
a wrong RoPE pairing (interleaved instead of half-split), exponent or sign;
a transposed map or wrong concatenation order; a dropped bias; a wrong cache
row; a wrong ridge centring.  None of them re-types the oracle's loops: they
use closed forms (complex multiplication), invariants, planted values read
back from the destination side, and library routines for special cases.
"""
import cmath
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.linalg

import oracle

RNG = np.random.default_rng(1234)
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# RoPE ("Helm Intelligent Routing", "Why carrying the cache across is the
# hard part": the position is folded into a key as a rotation; steps 1, 3)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("p", [0, 1, 7, 1000, 32767])
def test_rope_d2_is_complex_multiplication(p):
    # d = 2: one pair, frequency theta^0 = 1, so the rotation is (a + jb) e^{jp}.
    a, b = 0.75, -1.25
    z = complex(a, b) * cmath.exp(1j * p)
    got = oracle.rope([a, b], p, 1e4, +1)
    assert got == pytest.approx([z.real, z.imag], abs=1e-12)
    z = complex(a, b) * cmath.exp(-1j * p)
    got = oracle.rope([a, b], p, 1e4, -1)
    assert got == pytest.approx([z.real, z.imag], abs=1e-12)


@pytest.mark.parametrize("theta", [1e4, 5e5, 1e6])
def test_rope_half_split_frequency_ladder(theta):
    # Basis vector e_i turns within the plane (i, i + d/2) at angle
    # p * theta^(-2i/d): catches interleaved pairing and a wrong exponent.
    d, p = 8, 123.0
    for i in range(d // 2):
        w = math.pow(theta, -2.0 * i / d)
        e = np.zeros(d)
        e[i] = 1.0
        want = np.zeros(d)
        want[i], want[i + d // 2] = math.cos(p * w), math.sin(p * w)
        np.testing.assert_allclose(oracle.rope(e, p, theta, +1), want, atol=1e-14)
        e = np.zeros(d)
        e[i + d // 2] = 1.0
        want = np.zeros(d)
        want[i], want[i + d // 2] = -math.sin(p * w), math.cos(p * w)
        np.testing.assert_allclose(oracle.rope(e, p, theta, +1), want, atol=1e-14)


def test_unrotate_inverts_rotate():
    for d in (2, 64, 128):
        x = RNG.standard_normal(d) * np.exp(RNG.standard_normal(d))
        for p in (0, 3, 511, 32767, 32831):
            y = oracle.rope(oracle.rope(x, p, 1e6, +1), p, 1e6, -1)
            np.testing.assert_allclose(y, x, rtol=0, atol=1e-12 * np.abs(x).max())


def test_rotate_after_unrotate_is_rotation_by_difference():
    d = 128
    x = RNG.standard_normal(d)
    for p, q in ((100, 37), (37, 100), (32768, 5), (0, 9)):
        lhs = oracle.rope(oracle.rope(x, q, 1e6, -1), p, 1e6, +1)
        rhs = oracle.rope(x, p - q, 1e6, +1)
        np.testing.assert_allclose(lhs, rhs, rtol=0, atol=1e-11)


def test_rotate_at_zero_is_exact_identity_and_norm_is_kept():
    d = 64
    x = RNG.standard_normal(d)
    assert np.array_equal(oracle.rope(x, 0, 1e4, +1), x)
    y = oracle.rope(x, 4321, 1e4, +1)
    pair_norm = lambda v: v[: d // 2] ** 2 + v[d // 2:] ** 2
    np.testing.assert_allclose(pair_norm(y), pair_norm(x), rtol=1e-13)


# --------------------------------------------------------------------------
# The map ("Helm Intelligent Routing" step 2; Qwen3 article, linear bridge:
# concatenated features of the selected layers, one fit per target
# (layer, head), separately for K and V, map x @ w + b)
# --------------------------------------------------------------------------

def _planted_source(Ls, T, H, d):
    """src[s][t][h][c] = a distinct exact integer encoding (s, t, h, c)."""
    s, t, h, c = np.meshgrid(np.arange(Ls), np.arange(T), np.arange(H), np.arange(d),
                             indexing="ij")
    return (((s * 1000 + t) * 100 + h) * 1000 + c + 1).astype(np.float64)


def test_identity_map_reproduces_source():
    # k = 1, W = I, b = 0, same theta both sides, offset 0: the target cache is
    # the selected source layer, keys included (un-rotate then re-rotate at
    # the same position cancels).
    Ls, Lt, H, d, T = 3, 4, 2, 16, 10
    src_k = RNG.standard_normal((Ls, T, H, d))
    src_v = RNG.standard_normal((Ls, T, H, d))
    idx = np.array([[2], [0], [1], [2]], dtype=np.int32)
    w = np.zeros((Lt, H, 2, d, d))
    w[..., :, :] = np.eye(d)
    b = np.zeros((Lt, H, 2, d))
    dk, dv, st = oracle.transfer(src_k=src_k, src_v=src_v, layer_idx=idx, w=w, b=b,
                                 theta_src=1e4, theta_tgt=1e4, max_position=T,
                                 dst_capacity=T)
    assert st == 0
    for lt in range(Lt):
        np.testing.assert_array_equal(dv[lt], src_v[idx[lt, 0]])
        np.testing.assert_allclose(dk[lt], src_k[idx[lt, 0]], rtol=0, atol=1e-13)


def test_selection_matrix_routes_concatenated_features():
    # W picks feature perm[n] of the concatenated vector into output n.  With
    # positions all zero RoPE is exactly the identity, so every output must be
    # exactly the planted source value of layer idx[lt][perm[n] // d],
    # channel perm[n] % d: checks concatenation order and W orientation.
    Ls, Lt, H, d, T, k = 5, 3, 2, 8, 4, 3
    src = _planted_source(Ls, T, H, d)
    idx = np.array([[4, 0, 2], [1, 3, 0], [2, 2, 4]], dtype=np.int32)
    perms = RNG.permuted(np.tile(np.arange(k * d), (Lt, H, 2, 1)), axis=-1)[..., :d]
    w = np.zeros((Lt, H, 2, k * d, d))
    for lt in range(Lt):
        for h in range(H):
            for m in range(2):
                w[lt, h, m, perms[lt, h, m], np.arange(d)] = 1.0
    b = np.zeros((Lt, H, 2, d))
    src_pos = np.zeros(T, dtype=np.int64)
    tgt_pos = np.zeros(T, dtype=np.int64)
    # all tokens land on row 0 with zero positions; use T = 1 per call instead
    for t in range(T):
        dk, dv, st = oracle.transfer(src_k=src[:, t:t + 1] * 2, src_v=src[:, t:t + 1],
                                     layer_idx=idx, w=w, b=b, theta_src=1e4,
                                     theta_tgt=1e6, max_position=1, dst_capacity=1,
                                     src_pos=src_pos[:1], tgt_pos=tgt_pos[:1])
        assert st == 0
        for lt in range(Lt):
            for h in range(H):
                for m, (dst, mult) in enumerate(((dk, 2), (dv, 1))):
                    q = perms[lt, h, m]
                    want = mult * src[idx[lt, q // d], t, h, q % d]
                    np.testing.assert_array_equal(dst[lt, 0, h], want)


def test_bias_only_and_key_bias_is_rotated():
    # W = 0: values equal b exactly; keys equal b turned by the target RoPE at
    # p' (complex multiplication per pair, frequency theta^(-2i/d)).
    Ls, Lt, H, d, T, k = 2, 2, 1, 4, 3, 2
    src = RNG.standard_normal((Ls, T, H, d))
    idx = np.array([[0, 1], [1, 0]], dtype=np.int32)
    w = np.zeros((Lt, H, 2, k * d, d))
    b = RNG.standard_normal((Lt, H, 2, d))
    theta_t, off = 5e5, 11
    dk, dv, st = oracle.transfer(src_k=src, src_v=src, layer_idx=idx, w=w, b=b,
                                 theta_src=1e4, theta_tgt=theta_t, max_position=T + off,
                                 dst_capacity=T + off, tgt_offset=[off])
    assert st == 0
    for lt in range(Lt):
        for t in range(T):
            np.testing.assert_array_equal(dv[lt, t + off, 0], b[lt, 0, 1])
            p = t + off
            for i in range(d // 2):
                z = complex(b[lt, 0, 0, i], b[lt, 0, 0, i + d // 2])
                z *= cmath.exp(1j * p * theta_t ** (-2.0 * i / d))
                assert dk[lt, p, 0, i] == pytest.approx(z.real, abs=1e-13)
                assert dk[lt, p, 0, i + d // 2] == pytest.approx(z.imag, abs=1e-13)


def test_key_path_closed_form_with_different_thetas():
    # A key stored as content c turned by the source RoPE at p, mapped with
    # W = I (k = 1), lands as c turned by the target RoPE at p' = p + off:
    # un-rotation really strips theta_src and re-rotation really applies
    # theta_tgt at the target position.
    d, T, off, ts, tt = 8, 6, 37, 1e4, 1e6
    c = RNG.standard_normal((T, d))
    zc = c[:, : d // 2] + 1j * c[:, d // 2:]
    i = np.arange(d // 2)
    p = np.arange(T)[:, None]
    zs = zc * np.exp(1j * p * ts ** (-2.0 * i / d))
    src_k = np.concatenate([zs.real, zs.imag], axis=1).reshape(1, T, 1, d)
    w = np.eye(d).reshape(1, 1, 1, d, d).repeat(2, axis=2)
    b = np.zeros((1, 1, 2, d))
    dk, dv, st = oracle.transfer(src_k=src_k, src_v=src_k, layer_idx=[[0]], w=w, b=b,
                                 theta_src=ts, theta_tgt=tt, max_position=T + off,
                                 dst_capacity=T + off, tgt_offset=[off])
    assert st == 0
    zt = zc * np.exp(1j * (p + off) * tt ** (-2.0 * i / d))
    want = np.concatenate([zt.real, zt.imag], axis=1)
    np.testing.assert_allclose(dk[0, off:, 0], want, rtol=0, atol=1e-12)
    assert np.isnan(dk[0, :off]).all()


def test_linear_in_features_sum_of_two_terms():
    # Two nonzeros per column: output = 0.5 * feature a + 3 * feature b + bias.
    Ls, H, d, T, k = 3, 1, 4, 1, 2
    src = _planted_source(Ls, T, H, d)
    idx = np.array([[2, 1]], dtype=np.int32)
    w = np.zeros((1, H, 2, k * d, d))
    b = np.full((1, H, 2, d), 0.25)
    for n in range(d):
        w[0, 0, 1, n, n] = 0.5          # layer idx[0] = 2, channel n
        w[0, 0, 1, d + (n + 1) % d, n] = 3.0   # layer idx[1] = 1, channel n+1
    _, dv, st = oracle.transfer(src_k=src, src_v=src, layer_idx=idx, w=w, b=b,
                                theta_src=1e4, theta_tgt=1e4, max_position=1,
                                dst_capacity=1)
    assert st == 0
    for n in range(d):
        want = 0.25 + 0.5 * src[2, 0, 0, n] + 3.0 * src[1, 0, 0, (n + 1) % d]
        assert dv[0, 0, 0, n] == want


# --------------------------------------------------------------------------
# Cache install: contiguous rows and paged blocks ("Helm Intelligent
# Routing", "Current limitation": installer into the engine's paged cache;
# knlp.io routing page: inject through the block table)
# --------------------------------------------------------------------------

def _varlen_problem(bs=4, seed=5):
    rng = np.random.default_rng(seed)
    lens = [5, 1, 9]
    offs = [0, 3, 6]
    R, H, d, Ls, Lt, k = 3, 2, 4, 3, 2, 1
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T = int(cu[-1])
    nb = [(n + o + bs - 1) // bs for n, o in zip(lens, offs)]
    pool = int(sum(nb)) + 2                     # two blocks nobody owns
    perm = rng.permutation(pool).astype(np.int32)
    table = np.full((R, max(nb) + 1), -1, dtype=np.int32)
    at = 0
    for r in range(R):
        table[r, :nb[r]] = perm[at:at + nb[r]]
        at += nb[r]
    src = _planted_source(Ls, T, H, d)
    idx = np.array([[2], [0]], dtype=np.int32)
    w = np.zeros((Lt, H, 2, d, d))
    w[...] = np.eye(d)
    b = np.zeros((Lt, H, 2, d))
    return dict(lens=lens, offs=offs, cu=cu, table=table, pool=pool, src=src, idx=idx,
                w=w, b=b, bs=bs, T=T, H=H, d=d, Lt=Lt)


def test_paged_scatter_routes_every_token_and_leaves_the_rest():
    P = _varlen_problem()
    bs = P["bs"]
    dk, dv, st = oracle.transfer(src_k=P["src"], src_v=P["src"], layer_idx=P["idx"],
                                 w=P["w"], b=P["b"], theta_src=1e4, theta_tgt=1e4,
                                 max_position=32, cu_seqlens=P["cu"],
                                 tgt_offset=P["offs"], layout=oracle.PAGED,
                                 block_size=bs, num_blocks=P["pool"],
                                 block_table=P["table"])
    assert st == 0
    # Read back from the destination side: physical block -> (request,
    # logical block) from the table, slot -> target position -> source token.
    owner = {}
    for r in range(len(P["lens"])):
        for lb, pb in enumerate(P["table"][r]):
            if pb >= 0:
                owner[int(pb)] = (r, lb)
    written = 0
    for pb in range(P["pool"]):
        for slot in range(bs):
            row = pb * bs + slot
            tok = None
            if pb in owner:
                r, lb = owner[pb]
                pt = lb * bs + slot
                pos = pt - P["offs"][r]
                if 0 <= pos < P["lens"][r]:
                    tok = int(P["cu"][r]) + pos
            for lt in range(P["Lt"]):
                s = P["idx"][lt, 0]
                if tok is None:
                    assert np.isnan(dv[lt, row]).all() and np.isnan(dk[lt, row]).all()
                else:
                    np.testing.assert_array_equal(dv[lt, row], P["src"][s, tok])
                    # keys: un-rotate at p, re-rotate at p' = p + off: differs
                    # from the source by the rotation through the offset
                    want = oracle.rope(P["src"][s, tok, 0], P["offs"][owner[pb][0]], 1e4, +1)
                    np.testing.assert_allclose(dk[lt, row, 0], want, rtol=1e-12)
                    written += 1
    assert written == P["Lt"] * P["T"]


def test_contiguous_offset_leaves_rows_below_offset():
    T, off, d = 5, 3, 4
    src = _planted_source(1, T, 1, d)
    w = np.eye(d).reshape(1, 1, 1, d, d).repeat(2, axis=2)
    b = np.zeros((1, 1, 2, d))
    dk, dv, st = oracle.transfer(src_k=src, src_v=src, layer_idx=[[0]], w=w, b=b,
                                 theta_src=1e4, theta_tgt=1e4, max_position=T + off,
                                 dst_capacity=T + off + 2, tgt_offset=[off])
    assert st == 0
    assert np.isnan(dv[0, :off]).all() and np.isnan(dv[0, off + T:]).all()
    np.testing.assert_array_equal(dv[0, off:off + T], src[0])


def test_out_of_range_rows_are_skipped_and_flagged():
    P = _varlen_problem()
    base = dict(src_k=P["src"], src_v=P["src"], w=P["w"], b=P["b"], theta_src=1e4,
                theta_tgt=1e4, cu_seqlens=P["cu"], tgt_offset=P["offs"],
                layout=oracle.PAGED, block_size=P["bs"], num_blocks=P["pool"])
    # a selection index outside [0, Ls): that target layer is left untouched
    dk, dv, st = oracle.transfer(layer_idx=[[2], [3]], max_position=32,
                                 block_table=P["table"], **base)
    assert st == oracle.BAD_LAYER_INDEX
    assert np.isnan(dv[1]).all() and not np.isnan(dv[0]).all()
    # a position beyond the table: only those tokens are skipped
    _, dv, st = oracle.transfer(layer_idx=P["idx"], max_position=12,
                                block_table=P["table"], **base)
    assert st == oracle.BAD_POSITION
    assert np.count_nonzero(~np.isnan(dv[0, :, 0, 0])) == 5 + 1 + (12 - 6)
    # a referenced table entry of -1
    table = P["table"].copy()
    table[2, 1] = -1
    _, dv, st = oracle.transfer(layer_idx=P["idx"], max_position=32,
                                block_table=table, **base)
    assert st == oracle.BAD_BLOCK
    # request 2 (offset 6) puts target positions 6 and 7 in logical block 1
    assert np.count_nonzero(~np.isnan(dv[0, :, 0, 0])) == P["T"] - 2
    # contiguous capacity too small
    _, dv, st = oracle.transfer(src_k=P["src"], src_v=P["src"], w=P["w"], b=P["b"],
                                theta_src=1e4, theta_tgt=1e4, cu_seqlens=P["cu"],
                                tgt_offset=P["offs"], layer_idx=P["idx"], max_position=32,
                                dst_capacity=8)
    assert st == oracle.BAD_ROW
    # a request table that runs backwards, or does not end at ntok, makes the
    # whole transfer invalid: nothing is written
    for cu in ([0, 5, 4, 15], [0, 5, 6, 14], [1, 5, 6, 15]):
        dk, dv, st = oracle.transfer(src_k=P["src"], src_v=P["src"], w=P["w"], b=P["b"],
                                     theta_src=1e4, theta_tgt=1e4, cu_seqlens=cu,
                                     layer_idx=[[2], [3]], max_position=32, dst_capacity=16)
        assert st == oracle.BAD_SEQLENS
        assert np.isnan(dv).all() and np.isnan(dk).all()


def test_dst_row_examples():
    table = np.array([[7, 2, 5]], dtype=np.int32)
    assert oracle.dst_row(oracle.PAGED, 0, 0, block_size=16, num_blocks=8,
                          block_table=table, max_blocks_per_req=3) == (7 * 16, 0)
    assert oracle.dst_row(oracle.PAGED, 0, 17, block_size=16, num_blocks=8,
                          block_table=table, max_blocks_per_req=3) == (2 * 16 + 1, 0)
    assert oracle.dst_row(oracle.PAGED, 0, 48, block_size=16, num_blocks=8,
                          block_table=table, max_blocks_per_req=3) == (-1, oracle.BAD_BLOCK)
    assert oracle.dst_row(oracle.CONTIGUOUS, 2, 5, dst_capacity=10) == (25, 0)
    assert oracle.dst_row(oracle.CONTIGUOUS, 0, 10, dst_capacity=10) == (-1, oracle.BAD_ROW)


# --------------------------------------------------------------------------
# Brute force: a second formulation of the whole transfer in numpy (complex
# phasors, einsum over the stacked selection, vectorised routing), on the
# tiny workload and on a varlen paged problem.
# --------------------------------------------------------------------------

def _numpy_transfer(src_k, src_v, idx, w, b, ts, tt, cu, offs, layout, cap, bs, table,
                    rows):
    Ls, T, H, d = src_k.shape
    half = d // 2
    i = np.arange(half)
    req = np.searchsorted(cu, np.arange(T), side="right") - 1
    p = np.arange(T) - cu[req]
    pt = p + np.asarray(offs)[req]
    zs = src_k[..., :half] + 1j * src_k[..., half:]
    zc = zs * np.exp(-1j * p[None, :, None, None] * ts ** (-2.0 * i / d))
    kc = np.concatenate([zc.real, zc.imag], -1)                  # [Ls][T][H][d]
    xk = np.moveaxis(kc[idx], 1, 3).reshape(idx.shape[0], T, H, -1)   # [Lt][T][H][k d]
    xv = np.moveaxis(src_v[idx], 1, 3).reshape(idx.shape[0], T, H, -1)
    yk = np.einsum("lthq,lhqn->lthn", xk, w[:, :, 0]) + b[:, None, :, 0]
    yv = np.einsum("lthq,lhqn->lthn", xv, w[:, :, 1]) + b[:, None, :, 1]
    zy = (yk[..., :half] + 1j * yk[..., half:]) * np.exp(
        1j * pt[None, :, None, None] * tt ** (-2.0 * i / d))
    yk = np.concatenate([zy.real, zy.imag], -1)
    if layout == oracle.PAGED:
        row = table[req, pt // bs] * bs + pt % bs
    else:
        row = req * cap + pt
    Lt = idx.shape[0]
    dk = np.full((Lt, rows, H, d), np.nan)
    dv = np.full((Lt, rows, H, d), np.nan)
    dk[:, row] = yk
    dv[:, row] = yv
    return dk, dv


def test_brute_force_tiny_workload():
    Ls, Lt, H, d, T, k = 4, 6, 2, 64, 128, 2
    src_k = RNG.standard_normal((Ls, T, H, d)) * np.exp(RNG.standard_normal((Ls, 1, H, d)))
    src_v = RNG.standard_normal((Ls, T, H, d)) * np.exp(RNG.standard_normal((Ls, 1, H, d)))
    idx = np.stack([RNG.permutation(Ls)[:k] for _ in range(Lt)]).astype(np.int32)
    w = RNG.standard_normal((Lt, H, 2, k * d, d)) / math.sqrt(k * d)
    b = RNG.standard_normal((Lt, H, 2, d)) * 0.01
    cu = np.array([0, T])
    dk, dv, st = oracle.transfer(src_k=src_k, src_v=src_v, layer_idx=idx, w=w, b=b,
                                 theta_src=1e4, theta_tgt=1e4, max_position=T,
                                 dst_capacity=T)
    assert st == 0
    nk, nv = _numpy_transfer(src_k, src_v, idx, w, b, 1e4, 1e4, cu, [0],
                             oracle.CONTIGUOUS, T, 1, None, T)
    np.testing.assert_allclose(dk, nk, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dv, nv, rtol=1e-12, atol=1e-12)


def test_brute_force_varlen_paged_different_thetas():
    rng = np.random.default_rng(99)
    lens, offs, bs = [7, 3, 12], [2, 0, 5], 4
    Ls, Lt, H, d, k = 5, 3, 2, 8, 3
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1])
    nb = [(n + o + bs - 1) // bs for n, o in zip(lens, offs)]
    pool = sum(nb)
    perm = rng.permutation(pool).astype(np.int32)
    table = np.full((3, max(nb)), -1, dtype=np.int32)
    at = 0
    for r in range(3):
        table[r, :nb[r]] = perm[at:at + nb[r]]
        at += nb[r]
    src_k = rng.standard_normal((Ls, T, H, d))
    src_v = rng.standard_normal((Ls, T, H, d))
    idx = np.stack([rng.permutation(Ls)[:k] for _ in range(Lt)]).astype(np.int32)
    w = rng.standard_normal((Lt, H, 2, k * d, d))
    b = rng.standard_normal((Lt, H, 2, d))
    dk, dv, st = oracle.transfer(src_k=src_k, src_v=src_v, layer_idx=idx, w=w, b=b,
                                 theta_src=1e4, theta_tgt=5e5, max_position=20,
                                 cu_seqlens=cu, tgt_offset=offs, layout=oracle.PAGED,
                                 block_size=bs, num_blocks=pool, block_table=table)
    assert st == 0
    nk, nv = _numpy_transfer(src_k, src_v, idx, w, b, 1e4, 5e5, cu, offs,
                             oracle.PAGED, 0, bs, table, pool * bs)
    np.testing.assert_allclose(dk, nk, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dv, nv, rtol=1e-12, atol=1e-12)


def test_map_token_matches_transfer_row():
    # The per-token entry point used for sampled checks at full size gives the
    # same bits as the whole transfer.
    rng = np.random.default_rng(3)
    Ls, Lt, H, d, T, k = 4, 2, 2, 8, 6, 2
    src_k = rng.standard_normal((Ls, T, H, d))
    src_v = rng.standard_normal((Ls, T, H, d))
    idx = np.array([[3, 1], [0, 3]], dtype=np.int32)
    w = rng.standard_normal((Lt, H, 2, k * d, d))
    b = rng.standard_normal((Lt, H, 2, d))
    dk, dv, _ = oracle.transfer(src_k=src_k, src_v=src_v, layer_idx=idx, w=w, b=b,
                                theta_src=1e4, theta_tgt=1e6, max_position=T + 4,
                                dst_capacity=T + 4, tgt_offset=[4])
    for lt in range(Lt):
        for h in range(H):
            for t in range(T):
                ok, ov = oracle.map_token(src_k[idx[lt], t, h], src_v[idx[lt], t, h],
                                          w[lt, h, 0], w[lt, h, 1], b[lt, h, 0], b[lt, h, 1],
                                          t, t + 4, 1e4, 1e6)
                assert np.array_equal(ok, dk[lt, t + 4, h])
                assert np.array_equal(ov, dv[lt, t + 4, h])


# --------------------------------------------------------------------------
# Ridge fit (Qwen3 article, linear bridge: the ridge demo)
# --------------------------------------------------------------------------

def test_ridge_worked_example_exact_fractions():
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "ridge_worked_example.txt"))
            if ln.strip() and not ln.startswith("#")]
    x = np.array([float(v) for v in rows[0][1:]])
    y = np.array([float(v) for v in rows[1][1:]])
    for r in rows[2:]:
        ln, ld, wn, wd, bn, bd = map(int, r[1:])
        W, b = oracle.ridge_fit(x[:, None], y[:, None], lam=ln / ld)
        assert W[0, 0] == pytest.approx(float(Fraction(wn, wd)), rel=1e-14)
        assert b[0] == pytest.approx(float(Fraction(bn, bd)), rel=1e-14)


def test_ridge_recovers_planted_map_as_lambda_vanishes():
    n, p, q = 400, 12, 5
    X = RNG.standard_normal((n, p)) * 3 + RNG.standard_normal(p)
    Wstar = RNG.standard_normal((p, q))
    bstar = RNG.standard_normal(q)
    Y = X @ Wstar + bstar
    W, b = oracle.ridge_fit(X, Y, lam=1e-10)
    assert np.linalg.norm(W - Wstar) / np.linalg.norm(Wstar) < 1e-8
    assert np.linalg.norm(b - bstar) / np.linalg.norm(bstar) < 1e-8


def test_ridge_shrinkage_closed_form():
    # Noiseless Y = X W* + b*: the centred fit is (XcT Xc + lam I)^-1 XcT Xc W*,
    # solved here with LAPACK's LU (not the oracle's Cholesky).
    n, p, q, lam = 300, 10, 4, 7.5
    X = RNG.standard_normal((n, p)) + 2.0
    Wstar = RNG.standard_normal((p, q))
    Y = X @ Wstar + 0.5
    Xc = X - X.mean(0)
    G = Xc.T @ Xc
    want = scipy.linalg.solve(G + lam * np.eye(p), G @ Wstar)
    W, b = oracle.ridge_fit(X, Y, lam=lam)
    np.testing.assert_allclose(W, want, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(b, Y.mean(0) - X.mean(0) @ want, rtol=1e-10, atol=1e-12)


def test_ridge_equals_augmented_least_squares():
    # Ridge on centred data = least squares on [Xc; sqrt(lam) I] vs [Yc; 0]
    # (numpy lstsq, an SVD solver).
    n, p, q, lam = 200, 8, 3, 0.01
    X = RNG.standard_normal((n, p)) * np.arange(1, p + 1)
    Y = RNG.standard_normal((n, q)) + X[:, :q] * 2
    Xc, Yc = X - X.mean(0), Y - Y.mean(0)
    A = np.vstack([Xc, math.sqrt(lam) * np.eye(p)])
    B = np.vstack([Yc, np.zeros((p, q))])
    want = np.linalg.lstsq(A, B, rcond=None)[0]
    W, b = oracle.ridge_fit(X, Y, lam=lam)
    np.testing.assert_allclose(W, want, rtol=1e-9, atol=1e-11)


# --------------------------------------------------------------------------
# Fidelity diagnostics: KV cosine ("Helm Intelligent Routing", "Reading the
# retention score") and explained variance (the Qwen3 article, section on
# the linear bridge: the share of target K / V variance the source explains)
# --------------------------------------------------------------------------

def _golden_rows(name):
    rows = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, *vals = line.split()
            rows[key] = vals
    return rows


def _diag(mk, mv, rk, rv, **kw):
    kw.setdefault("theta_tgt", 1e4)
    kw.setdefault("max_position", 64)
    return oracle.kv_diagnostics(mapped_k=mk, mapped_v=mv, ref_k=rk, ref_v=rv, **kw)


def test_kv_diagnostics_worked_example():
    g = _golden_rows("kv_diagnostics_worked_example.txt")
    cache = lambda key: np.array([float(x) for x in g[key]]).reshape(1, 2, 1, 2)
    stats, st = _diag(cache("mapped_k"), cache("mapped_v"), cache("ref_k"), cache("ref_v"),
                      ntok=2, dst_capacity=2)
    assert st == 0
    frac = lambda v: float(Fraction(v))
    k, v = stats[0, 0, 0], stats[0, 0, 1]
    np.testing.assert_allclose(k[:4], [frac(x) for x in g["stats_k"]], rtol=1e-15)
    # keys in content space: token 0 at p' = 0 as stored, token 1 at p' = 1
    # un-rotated: (0 + 2j) e^{-j} = 2 sin 1 + 2j cos 1
    ksum = [3 + 2 * math.sin(1.0), 4 + 2 * math.cos(1.0)]
    np.testing.assert_allclose(k[4:], ksum, rtol=1e-15)
    ss_tot = (29 - 12 * math.sin(1.0) - 16 * math.cos(1.0)) / 2
    assert oracle.explained_variance(stats)[0, 0, 0] == pytest.approx(1 - 2 / ss_tot, rel=1e-14)
    assert oracle.mean_cosine(stats)[0, 0, 0] == pytest.approx(49 / 50, rel=1e-15)
    assert v[0] == 2 and v[1] == pytest.approx(1 / math.sqrt(2), rel=1e-15)
    np.testing.assert_allclose(v[2:4], [frac(x) for x in g["stats_v"][2:]], rtol=1e-15)
    np.testing.assert_allclose(v[4:], [frac(x) for x in g["sum_v"]], atol=0)
    assert oracle.explained_variance(stats)[0, 0, 1] == pytest.approx(frac(g["r2_v"][0]), rel=1e-14)


def _paged_case(rng, Lt=2, H=3, d=8):
    # three requests, a permuted block pool, target offsets: every row a
    # transfer writes is filled, every other row is NaN (never to be read)
    cu = np.array([0, 5, 9, 16])
    off = np.array([0, 3, 1])
    bs, nblk, mbpr = 4, 12, 4
    table = rng.permutation(nblk)[:3 * mbpr].reshape(3, mbpr).astype(np.int32)
    rows = nblk * bs
    ref_k = np.full((Lt, rows, H, d), np.nan)
    ref_v = np.full((Lt, rows, H, d), np.nan)
    pts, used = [], []
    for r in range(3):
        for g in range(cu[r], cu[r + 1]):
            pt = g - cu[r] + off[r]
            row = table[r][pt // bs] * bs + pt % bs
            pts.append(pt)
            used.append(row)
    used = np.array(used)
    ref_k[:, used] = rng.standard_normal((Lt, len(used), H, d))
    ref_v[:, used] = rng.standard_normal((Lt, len(used), H, d))
    kw = dict(ntok=16, cu_seqlens=cu, tgt_offset=off, layout=oracle.PAGED, block_size=bs,
              num_blocks=nblk, block_table=table)
    return ref_k, ref_v, np.array(pts), used, kw


def test_kv_diagnostics_identity_negation_and_scale():
    ref_k, ref_v, _, used, kw = _paged_case(np.random.default_rng(7))
    s, st = _diag(ref_k, ref_v, ref_k, ref_v, **kw)
    assert st == 0
    assert np.all(s[..., 0] == 16)
    np.testing.assert_allclose(oracle.mean_cosine(s), 1.0, rtol=1e-14)
    assert np.all(s[..., 2] == 0)
    np.testing.assert_allclose(oracle.explained_variance(s), 1.0, rtol=1e-14)
    s, _ = _diag(-ref_k, 2.5 * ref_v, ref_k, ref_v, **kw)
    np.testing.assert_allclose(oracle.mean_cosine(s)[..., 0], -1.0, rtol=1e-14)
    np.testing.assert_allclose(oracle.mean_cosine(s)[..., 1], 1.0, rtol=1e-14)
    # |y - 2.5 y|^2 = 2.25 |y|^2, summed over the compared tokens
    np.testing.assert_allclose(s[..., 1, 2], 2.25 * s[..., 1, 3], rtol=1e-13)
    yy = np.einsum("lthd,lthd->lh", ref_v[:, used], ref_v[:, used])
    np.testing.assert_allclose(s[..., 1, 3], yy, rtol=1e-13)


def test_kv_diagnostics_keys_are_averaged_in_content_space():
    # every key is one content vector c rotated to its own p': un-rotating
    # at p' with the target base gives back n * c (a wrong sign, base or
    # pairing would not); the stored vectors themselves do not sum to n * c
    rng = np.random.default_rng(11)
    ref_k, ref_v, pts, used, kw = _paged_case(rng, Lt=1, H=2, d=8)
    theta = 5e5
    c = rng.standard_normal((2, 8))
    for i, row in enumerate(used):
        for h in range(2):
            ref_k[0, row, h] = oracle.rope(c[h], pts[i], theta, +1)
    s, st = _diag(ref_k, ref_v, ref_k, ref_v, theta_tgt=theta, **kw)
    assert st == 0
    np.testing.assert_allclose(s[0, :, 0, 4:], 16 * c, rtol=1e-12, atol=1e-12)
    stored = ref_k[0, used].sum(axis=0)
    assert np.max(np.abs(stored - 16 * c)) > 1.0


def test_kv_diagnostics_mean_predictor_explains_nothing():
    # predicting every token by the content-space mean (re-rotated to its p'
    # for keys) gives R^2 = 0 exactly: the residual is the centred spread
    rng = np.random.default_rng(5)
    ref_k, ref_v, pts, used, kw = _paged_case(rng, Lt=1, H=2, d=6)
    theta = 1e4
    cont = np.stack([np.stack([oracle.rope(ref_k[0, row, h], pts[i], theta, -1)
                               for h in range(2)]) for i, row in enumerate(used)])
    mean_c = cont.mean(axis=0)
    mk = np.full_like(ref_k, np.nan)
    mv = np.full_like(ref_v, np.nan)
    vmean = ref_v[0, used].mean(axis=0)
    for i, row in enumerate(used):
        for h in range(2):
            mk[0, row, h] = oracle.rope(mean_c[h], pts[i], theta, +1)
        mv[0, row] = vmean
    s, _ = _diag(mk, mv, ref_k, ref_v, theta_tgt=theta, **kw)
    np.testing.assert_allclose(oracle.explained_variance(s), 0.0, atol=1e-12)


def test_kv_diagnostics_zero_vector_cosine_is_zero():
    rk = np.ones((1, 1, 1, 4))
    s, _ = _diag(np.zeros_like(rk), rk, rk, rk, ntok=1, dst_capacity=1)
    assert s[0, 0, 0, 1] == 0.0 and s[0, 0, 0, 0] == 1
    assert s[0, 0, 1, 1] == pytest.approx(1.0, rel=1e-15)


def test_kv_diagnostics_skips_what_a_transfer_skips():
    # the token at p' = 4 >= max_position is neither compared nor counted;
    # a malformed request table compares nothing
    rk = np.arange(2 * 5 * 1 * 2, dtype=np.float64).reshape(2, 5, 1, 2) + 1
    s, st = _diag(rk, rk, rk, rk, ntok=5, dst_capacity=5, max_position=4)
    assert st == oracle.BAD_POSITION
    assert np.all(s[..., 0] == 4)
    rk3 = np.ones((2, 15, 1, 2))
    s, st = _diag(rk3, rk3, rk3, rk3, ntok=5, dst_capacity=5, cu_seqlens=[0, 3, 2, 5])
    assert st == oracle.BAD_SEQLENS
    assert np.all(s == 0)


# --------------------------------------------------------------------------
# Wide-feature mapper (Qwen3 article, production-limits section: a 14B ->
# 32B mapper of about 1.07e9 parameters = 64 target layers x 8192 features
# x 2048 outputs, i.e. all heads' keys and values of the selected layers
# feed every head's key and value map)
# --------------------------------------------------------------------------

def _wide_case(rng, Ls=4, Lt=3, H=3, d=8, k=2, lens=(5, 9), offs=(0, 3)):
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1])
    src_k = rng.standard_normal((Ls, T, H, d))
    src_v = rng.standard_normal((Ls, T, H, d))
    idx = np.stack([rng.permutation(Ls)[:k] for _ in range(Lt)]).astype(np.int32)
    cap = max(n + o for n, o in zip(lens, offs))
    kw = dict(theta_src=1e4, theta_tgt=5e5, max_position=cap, cu_seqlens=cu, tgt_offset=offs,
              dst_capacity=cap)
    return src_k, src_v, idx, kw


def _wide_from_per_head(w_head, k, H, d):
    """The wide map that is block-diagonal over (head, K|V): feature
    (j, m, h, i) feeds output (h, m, i') through w_head[h][m][j*d + i][i']."""
    Lt = w_head.shape[0]
    F, N = k * 2 * H * d, H * 2 * d
    W = np.zeros((Lt, F, N))
    for lt in range(Lt):
        for j in range(k):
            for m in range(2):
                for h in range(H):
                    q0 = ((j * 2 + m) * H + h) * d
                    n0 = (h * 2 + m) * d
                    W[lt, q0:q0 + d, n0:n0 + d] = w_head[lt, h, m, j * d:(j + 1) * d]
    return W


def test_wide_block_diagonal_map_is_the_per_head_transfer_bit_for_bit():
    # Zero weights add exact zeros and the non-zero terms are summed in the
    # same (j, i) order, so the two oracles give the same bits.
    rng = np.random.default_rng(31)
    src_k, src_v, idx, kw = _wide_case(rng)
    Lt, k = idx.shape
    H, d = src_k.shape[2], src_k.shape[3]
    w_head = rng.standard_normal((Lt, H, 2, k * d, d))
    b = rng.standard_normal((Lt, H, 2, d))
    hk, hv, hst = oracle.transfer(src_k=src_k, src_v=src_v, layer_idx=idx, w=w_head, b=b, **kw)
    wk, wv, wst = oracle.transfer(src_k=src_k, src_v=src_v, layer_idx=idx,
                                  w=_wide_from_per_head(w_head, k, H, d), b=b, wide=True, **kw)
    assert hst == wst == 0
    assert np.array_equal(np.isnan(hk), np.isnan(wk))
    written = ~np.isnan(hk)
    assert np.array_equal(hk[written], wk[written]) and np.array_equal(hv[written], wv[written])


def test_wide_selection_routes_across_heads_and_kinds():
    # Every output (h, m, i) copies one feature chosen at random from the
    # whole width (any selected layer, head, key or value).  Keys are stored
    # as integer content rotated at p, so the expected features are written
    # down here from the documented order without the oracle's gather:
    # feature (j, m, h, i) = content key (m = 0) or value (m = 1) of source
    # layer idx[lt][j], head h, dim i.  Key outputs come back re-rotated.
    rng = np.random.default_rng(41)
    Ls, Lt, H, d, k, T = 4, 2, 3, 6, 2, 5
    th_s, th_t = 1e4, 1e6
    content = rng.integers(-50, 50, size=(Ls, T, H, d)).astype(np.float64)
    vals = rng.integers(-50, 50, size=(Ls, T, H, d)).astype(np.float64)
    src_k = np.empty_like(content)
    for s in range(Ls):
        for t in range(T):
            for h in range(H):
                src_k[s, t, h] = oracle.rope(content[s, t, h], t, th_s, +1)
    idx = np.array([[2, 0], [1, 3]], dtype=np.int32)
    F, N = k * 2 * H * d, H * 2 * d
    pick = rng.integers(0, F, size=(Lt, N))
    W = np.zeros((Lt, F, N))
    for lt in range(Lt):
        W[lt, pick[lt], np.arange(N)] = 1.0
    b = np.zeros((Lt, H, 2, d))
    dk, dv, st = oracle.transfer(src_k=src_k, src_v=vals, layer_idx=idx, w=W, b=b,
                                 theta_src=th_s, theta_tgt=th_t, max_position=T,
                                 dst_capacity=T, wide=True)
    assert st == 0
    for lt in range(Lt):
        for t in range(T):
            feat = np.empty(F)
            for q in range(F):
                j, rest = divmod(q, 2 * H * d)
                m, rest = divmod(rest, H * d)
                h, i = divmod(rest, d)
                s = idx[lt, j]
                feat[q] = (content if m == 0 else vals)[s, t, h, i]
            y = feat[pick[lt]].reshape(H, 2, d)
            for h in range(H):
                np.testing.assert_allclose(dv[lt, t, h], y[h, 1], rtol=0, atol=1e-12)
                np.testing.assert_allclose(dk[lt, t, h], oracle.rope(y[h, 0], t, th_t, +1),
                                           rtol=0, atol=1e-11)


def test_wide_brute_force_numpy_phasors():
    # An independent formulation: RoPE as complex phasors on (x_i + j x_{i+d/2}),
    # the map as one matmul over the stacked features, the cache rows by a
    # vectorised paged lookup.
    rng = np.random.default_rng(53)
    lens, offs, bs = [6, 11], [3, 0], 4
    Ls, Lt, H, d, k = 5, 2, 2, 8, 3
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1])
    nb = [(n + o + bs - 1) // bs for n, o in zip(lens, offs)]
    pool = sum(nb)
    perm = rng.permutation(pool).astype(np.int32)
    table = np.full((2, max(nb)), -1, dtype=np.int32)
    table[0, :nb[0]], table[1, :nb[1]] = perm[:nb[0]], perm[nb[0]:]
    src_k = rng.standard_normal((Ls, T, H, d))
    src_v = rng.standard_normal((Ls, T, H, d))
    idx = np.stack([rng.permutation(Ls)[:k] for _ in range(Lt)]).astype(np.int32)
    F, N = k * 2 * H * d, H * 2 * d
    W = rng.standard_normal((Lt, F, N)) / math.sqrt(F)
    b = rng.standard_normal((Lt, H, 2, d))
    th_s, th_t = 1e4, 5e5
    dk, dv, st = oracle.transfer(src_k=src_k, src_v=src_v, layer_idx=idx, w=W, b=b,
                                 theta_src=th_s, theta_tgt=th_t, max_position=20,
                                 cu_seqlens=cu, tgt_offset=offs, layout=oracle.PAGED,
                                 block_size=bs, num_blocks=pool, block_table=table, wide=True)
    assert st == 0
    half = d // 2
    req = np.searchsorted(cu, np.arange(T), side="right") - 1
    p = np.arange(T) - cu[req]
    pt = p + np.asarray(offs)[req]
    row = table[req, pt // bs] * bs + pt % bs

    def phasor(theta, pos):
        w = theta ** (-2.0 * np.arange(half) / d)
        return np.exp(1j * np.outer(pos, w))                          # [T][half]

    ck = src_k[..., :half] + 1j * src_k[..., half:]                  # [Ls][T][H][half]
    ck = ck * np.conj(phasor(th_s, p))[None, :, None, :]
    content = np.concatenate([ck.real, ck.imag], axis=-1)             # [Ls][T][H][d]
    for lt in range(Lt):
        X = np.stack([np.stack([content[idx[lt, j]], src_v[idx[lt, j]]], axis=1)
                      for j in range(k)], axis=1)                     # [T][k][2][H][d]
        Y = X.reshape(T, F) @ W[lt] + b[lt].reshape(N)                # [T][N]
        Y = Y.reshape(T, H, 2, d)
        yk = Y[:, :, 0, :half] + 1j * Y[:, :, 0, half:]
        yk = yk * phasor(th_t, pt)[:, None, :]
        np.testing.assert_allclose(dk[lt, row], np.concatenate([yk.real, yk.imag], -1),
                                   rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dv[lt, row], Y[:, :, 1], rtol=1e-12, atol=1e-12)
    untouched = np.ones(pool * bs, dtype=bool)
    untouched[row] = False
    assert np.isnan(dk[:, untouched]).all() and np.isnan(dv[:, untouched]).all()


def test_wide_bias_only_and_skip_rules():
    # W = 0: values are b, keys are b rotated to p' (closed form); a bad
    # layer index skips its target layer, a position past the table its token
    rng = np.random.default_rng(61)
    src_k, src_v, idx, kw = _wide_case(rng, Lt=3)
    Lt, k = idx.shape
    H, d = src_k.shape[2], src_k.shape[3]
    b = rng.standard_normal((Lt, H, 2, d))
    W = np.zeros((Lt, k * 2 * H * d, H * 2 * d))
    idx = idx.copy()
    idx[1, 0] = 99
    kw = dict(kw, max_position=kw["max_position"] - 1)
    dk, dv, st = oracle.transfer(src_k=src_k, src_v=src_v, layer_idx=idx, w=W, b=b, wide=True,
                                 **kw)
    assert st == oracle.BAD_LAYER_INDEX | oracle.BAD_POSITION
    assert np.isnan(dk[1]).all() and np.isnan(dv[1]).all()
    # request 1 (9 tokens, offset 3): p' = 3 .. 11, the last one is past the table
    cap = kw["dst_capacity"]
    for lt in (0, 2):
        for pt in range(3, 11):
            row = cap + pt
            for h in range(H):
                assert np.array_equal(dv[lt, row, h], b[lt, h, 1])
                z = b[lt, h, 0, :d // 2] + 1j * b[lt, h, 0, d // 2:]
                z = z * np.exp(1j * pt * 5e5 ** (-2.0 * np.arange(d // 2) / d))
                np.testing.assert_allclose(dk[lt, row, h], np.concatenate([z.real, z.imag]),
                                           rtol=0, atol=1e-13)
        assert np.isnan(dk[lt, cap + 11]).all()


def test_map_token_wide_matches_transfer_row():
    rng = np.random.default_rng(71)
    src_k, src_v, idx, kw = _wide_case(rng, lens=(7,), offs=(2,))
    Lt, k = idx.shape
    H, d = src_k.shape[2], src_k.shape[3]
    W = rng.standard_normal((Lt, k * 2 * H * d, H * 2 * d))
    b = rng.standard_normal((Lt, H, 2, d))
    dk, dv, _ = oracle.transfer(src_k=src_k, src_v=src_v, layer_idx=idx, w=W, b=b, wide=True,
                                **kw)
    for lt in range(Lt):
        for t in range(7):
            ok, ov = oracle.map_token_wide(src_k[idx[lt], t], src_v[idx[lt], t], W[lt], b[lt],
                                           t, t + 2, kw["theta_src"], kw["theta_tgt"])
            assert np.array_equal(ok, dk[lt, t + 2]) and np.array_equal(ov, dv[lt, t + 2])


# --------------------------------------------------------------------------
# Paged source: the pilot's own cache read through its block table (the
# target install's block-table rule of the knlp.io inject step, applied to
# the source position)
# --------------------------------------------------------------------------

def _scatter_paged_source(rng, src, cu, pos, bs, spare=3):
    """Scatter the packed rows of ``src`` [Ls][ntok][H][d] into a permuted
    pool of ``bs``-row blocks: request r's token at source position p goes to
    slot table[r][p // bs] * bs + p % bs.  Written out here with numpy, apart
    from the oracle's own row rule.  Unused slots are NaN."""
    R = len(cu) - 1
    Ls, _, H, d = src.shape
    nblk = [int(pos[cu[r]:cu[r + 1]].max()) // bs + 1 for r in range(R)]
    pool = sum(nblk) + spare
    perm = rng.permutation(pool).astype(np.int32)
    table = np.full((R, max(nblk) + 1), -1, dtype=np.int32)
    at = 0
    for r in range(R):
        table[r, :nblk[r]] = perm[at:at + nblk[r]]
        at += nblk[r]
    paged = np.full((Ls, pool * bs, H, d), np.nan)
    for r in range(R):
        for g in range(cu[r], cu[r + 1]):
            p = int(pos[g])
            paged[:, table[r, p // bs] * bs + p % bs] = src[:, g]
    return paged, table


@pytest.mark.parametrize("wide", [False, True])
def test_paged_source_equals_contiguous_source_bit_for_bit(wide):
    rng = np.random.default_rng(81)
    lens, offs, bs = [7, 12, 5], [0, 3, 9], 4
    Ls, Lt, H, d, k = 4, 2, 2, 8, 2
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1])
    pos = np.concatenate([np.arange(n) for n in lens])
    src_k = rng.standard_normal((Ls, T, H, d))
    src_v = rng.standard_normal((Ls, T, H, d))
    idx = np.stack([rng.permutation(Ls)[:k] for _ in range(Lt)]).astype(np.int32)
    if wide:
        w = rng.standard_normal((Lt, k * 2 * H * d, H * 2 * d))
    else:
        w = rng.standard_normal((Lt, H, 2, k * d, d))
    b = rng.standard_normal((Lt, H, 2, d))
    kw = dict(layer_idx=idx, w=w, b=b, theta_src=1e4, theta_tgt=5e5, max_position=24,
              cu_seqlens=cu, tgt_offset=offs, dst_capacity=24, wide=wide)
    ck, cv, cst = oracle.transfer(src_k=src_k, src_v=src_v, **kw)
    pk, table = _scatter_paged_source(rng, src_k, cu, pos, bs)
    # values through the same table
    pv = np.full_like(pk, np.nan)
    for r in range(3):
        for g in range(cu[r], cu[r + 1]):
            p = int(pos[g])
            pv[:, table[r, p // bs] * bs + p % bs] = src_v[:, g]
    gk, gv, gst = oracle.transfer(src_k=pk, src_v=pv, src_layout=oracle.PAGED,
                                  src_block_size=bs, src_block_table=table, **kw)
    assert cst == gst == 0
    assert np.array_equal(np.isnan(ck), np.isnan(gk))
    m = ~np.isnan(ck)
    assert np.array_equal(ck[m], gk[m]) and np.array_equal(cv[m], gv[m])


def test_paged_source_follows_explicit_source_positions():
    # the slot is chosen by the token's source position, not its packed index
    rng = np.random.default_rng(83)
    Ls, Lt, H, d, k, T, bs = 3, 2, 1, 4, 1, 6, 2
    src_k = rng.standard_normal((Ls, T, H, d))
    src_v = rng.standard_normal((Ls, T, H, d))
    idx = np.array([[2], [0]], dtype=np.int32)
    w = rng.standard_normal((Lt, H, 2, k * d, d))
    b = np.zeros((Lt, H, 2, d))
    src_pos = np.array([5, 0, 3, 1, 4, 2])
    cu = np.array([0, T])
    kw = dict(layer_idx=idx, w=w, b=b, theta_src=1e4, theta_tgt=1e4, max_position=8,
              cu_seqlens=cu, src_pos=src_pos, dst_capacity=8)
    ck, cv, _ = oracle.transfer(src_k=src_k, src_v=src_v, **kw)
    pk, table = _scatter_paged_source(rng, src_k, cu, src_pos, bs)
    pv = np.full_like(pk, np.nan)
    for g in range(T):
        p = int(src_pos[g])
        pv[:, table[0, p // bs] * bs + p % bs] = src_v[:, g]
    gk, gv, st = oracle.transfer(src_k=pk, src_v=pv, src_layout=oracle.PAGED, src_block_size=bs,
                                 src_block_table=table, **kw)
    assert st == 0
    m = ~np.isnan(ck)
    assert np.array_equal(ck[m], gk[m]) and np.array_equal(cv[m], gv[m])


def test_paged_source_bad_blocks_skip_and_flag():
    # a -1 entry and a position past the table's width: those tokens are
    # skipped (destination rows keep their NaN) with BAD_SRC_BLOCK; the source
    # check comes before the destination check
    rng = np.random.default_rng(87)
    lens, bs = [6, 5], 2
    Ls, Lt, H, d, k = 2, 1, 1, 4, 1
    cu = np.array([0, 6, 11])
    pos = np.concatenate([np.arange(n) for n in lens])
    src = rng.standard_normal((Ls, 11, H, d))
    pk, table = _scatter_paged_source(rng, src, cu, pos, bs)
    table = table[:, :3].copy()            # request 0 needs blocks 0..2, request 1 0..2
    table[1, 1] = -1                       # request 1, positions 2 and 3
    narrow = table[:, :2].copy()           # request 0 positions 4, 5 past the width
    w = np.tile(np.eye(d), (Lt, H, 2, 1, 1))
    b = np.zeros((Lt, H, 2, d))
    kw = dict(layer_idx=np.array([[1]], dtype=np.int32), w=w, b=b, theta_src=1e4,
              theta_tgt=1e4, max_position=8, cu_seqlens=cu, dst_capacity=8,
              src_layout=oracle.PAGED, src_block_size=bs)
    dk, dv, st = oracle.transfer(src_k=pk, src_v=pk, src_block_table=table, **kw)
    assert st == oracle.BAD_SRC_BLOCK
    assert np.isnan(dv[0, 8 + 2]).all() and np.isnan(dv[0, 8 + 3]).all()
    assert np.array_equal(dv[0, 8 + 4], src[1, 6 + 4])
    assert np.array_equal(dv[0, 5], src[1, 5])
    dk, dv, st = oracle.transfer(src_k=pk, src_v=pk, src_block_table=narrow, **kw)
    assert st == oracle.BAD_SRC_BLOCK
    assert np.isnan(dv[0, 4]).all() and np.isnan(dv[0, 5]).all()
    assert np.array_equal(dv[0, 3], src[1, 3])
    # capacity 4: the tokens at p' = 4, 5 have a bad source block AND a bad
    # row; the source check comes first, so only BAD_SRC_BLOCK is reported
    kw2 = dict(kw, dst_capacity=4)
    _, _, st = oracle.transfer(src_k=pk, src_v=pk, src_block_table=narrow, **kw2)
    assert st == oracle.BAD_SRC_BLOCK
    # with the full table the same rows only fail the row check
    _, _, st = oracle.transfer(src_k=pk, src_v=pk, src_block_table=table[:, :3], **kw2)
    assert st == oracle.BAD_SRC_BLOCK | oracle.BAD_ROW


# ---------------------------------------------------------------------------
# Layer-selection scores (kvxo_layer_scores)
# ---------------------------------------------------------------------------
def _rotate_np(x, pos, theta):
    """Half-split RoPE written out here with numpy (test input preparation)."""
    d = x.shape[-1]
    half = d // 2
    w = theta ** (-2.0 * np.arange(half) / d)
    a = np.asarray(pos, dtype=np.float64)[:, None] * w[None, :]
    x0, x1 = x[..., :half], x[..., half:]
    c, s = np.cos(a), np.sin(a)
    if x.ndim == 3:        # [n][H][d]
        c, s = c[:, None, :], s[:, None, :]
    return np.concatenate((x0 * c - x1 * s, x0 * s + x1 * c), axis=-1)


def test_layer_scores_worked_example_exact_fractions():
    g = _golden_rows("layer_scores_worked_example.txt")
    a = np.array([float(v) for v in g["a"]])
    b = np.array([float(v) for v in g["b"]])
    lam = float(g["lam"][0]) / float(g["lam"][1])
    ts, tt = float(g["theta_src"][0]), float(g["theta_tgt"][0])
    n = len(a)
    xc = np.zeros((n, 4)); xc[:, 1] = a
    yc = np.zeros((n, 4)); yc[:, 1] = b
    pos = np.arange(n)
    src_v = xc[None, :, None, :]
    tgt_v = yc[None, :, None, :]
    src_k = _rotate_np(xc, pos, ts)[None, :, None, :]
    tgt_k = _rotate_np(yc, pos, tt)[None, :, None, :]
    r2, r2s, st = oracle.layer_scores(src_k=src_k, src_v=src_v, tgt_k=tgt_k, tgt_v=tgt_v,
                                      theta_src=ts, theta_tgt=tt, max_position=n, lam=lam,
                                      layer_idx=np.array([[0]]))
    assert st == 0
    frac = lambda key: float(g[key][0]) / float(g[key][1])
    assert r2[0, 0, 0, 1] == pytest.approx(frac("r2_values"), abs=1e-13)
    assert r2[0, 0, 0, 0] == pytest.approx(frac("r2_keys"), abs=1e-12)
    assert r2s[0, 0, 1] == pytest.approx(frac("r2_set"), abs=1e-13)
    assert r2s[0, 0, 0] == pytest.approx(frac("r2_set"), abs=1e-12)


def _score_case(seed, Ls=3, Lt=2, H=2, d=8, n=40, noise=0.3):
    rng = np.random.default_rng(seed)
    xs_k = rng.normal(size=(Ls, n, H, d)) * np.exp(rng.normal(size=(Ls, 1, H, d)))
    xs_v = rng.normal(size=(Ls, n, H, d))
    # target layer lt is a linear function of source layer lt (+ noise)
    yk = np.empty((Lt, n, H, d)); yv = np.empty((Lt, n, H, d))
    for lt in range(Lt):
        for h in range(H):
            A = rng.normal(size=(d, d)); B = rng.normal(size=(d, d))
            yk[lt, :, h] = xs_k[lt, :, h] @ A + 0.5 + noise * rng.normal(size=(n, d))
            yv[lt, :, h] = xs_v[lt, :, h] @ B - 0.2 + noise * rng.normal(size=(n, d))
    return xs_k, xs_v, yk, yv


def test_layer_scores_equal_least_squares_r2_as_lambda_vanishes():
    # lam -> 0: the ridge fit is the least-squares fit with intercept, whose
    # in-sample R^2 (summed over outputs) LAPACK's lstsq gives independently
    xk, xv, yk, yv = _score_case(3)
    Ls, n, H, d = xv.shape
    r2, _, st = oracle.layer_scores(src_k=xk, src_v=xv, tgt_k=yk, tgt_v=yv, theta_src=1.0,
                                    theta_tgt=1.0, max_position=n, lam=1e-10)
    assert st == 0
    pos = np.arange(n)
    for lt in range(yk.shape[0]):
        for s in range(Ls):
            for h in range(H):
                for m, (X, Y) in enumerate(((xk, yk), (xv, yv))):
                    x = X[s, :, h]; y = Y[lt, :, h]
                    if m == 0:   # content space: un-rotate at p with base 1
                        x = _rotate_np(x, -pos, 1.0); y = _rotate_np(y, -pos, 1.0)
                    A = np.hstack([x, np.ones((n, 1))])
                    coef, *_ = np.linalg.lstsq(A, y, rcond=None)
                    res = y - A @ coef
                    ref = 1 - (res ** 2).sum() / ((y - y.mean(0)) ** 2).sum()
                    assert r2[lt, s, h, m] == pytest.approx(ref, abs=1e-8)


def test_layer_scores_see_content_only_through_each_models_rope():
    # keys stored rotated, with different bases on the two sides, related
    # exactly (linear, noiseless) in content space: the matched layer scores
    # 1 - O(lam); un-rotating with the wrong base or skipping it would not
    xk, xv, yk, yv = _score_case(5, noise=0.0)
    Ls, n, H, d = xk.shape
    pos = np.arange(n)
    sk = np.stack([_rotate_np(xk[s], pos, 1e4) for s in range(Ls)])
    tk = np.stack([_rotate_np(yk[lt], pos, 5e5) for lt in range(yk.shape[0])])
    r2, _, st = oracle.layer_scores(src_k=sk, src_v=xv, tgt_k=tk, tgt_v=yv, theta_src=1e4,
                                    theta_tgt=5e5, max_position=n, lam=1e-9)
    assert st == 0
    for lt in range(yk.shape[0]):
        assert np.all(r2[lt, lt] > 1 - 1e-6)
    # the same stored keys read with swapped bases lose the linear relation
    r2w, _, _ = oracle.layer_scores(src_k=sk, src_v=xv, tgt_k=tk, tgt_v=yv, theta_src=5e5,
                                    theta_tgt=1e4, max_position=n, lam=1e-9)
    assert np.all(r2w[0, 0, :, 0] < 0.99)


def test_layer_scores_invariances_and_set_bounds():
    xk, xv, yk, yv = _score_case(7)
    Ls, n, H, d = xk.shape
    kw = dict(theta_src=1e4, theta_tgt=1e4, max_position=n, lam=0.01)
    r2, r2s, st = oracle.layer_scores(src_k=xk, src_v=xv, tgt_k=yk, tgt_v=yv,
                                      layer_idx=np.array([[0, 2], [1, 0]]), **kw)
    assert st == 0 and np.all(r2 <= 1) and np.all(r2s <= 1)
    # scaling the target changes nothing for values; for keys the scale
    # commutes with the rotation
    r2b, _, _ = oracle.layer_scores(src_k=xk, src_v=xv, tgt_k=3 * yk, tgt_v=3 * yv, **kw)
    # ridge with the same lam on a scaled target: identical fit up to scale
    assert np.allclose(r2b, r2, atol=1e-12)
    # a set of one layer is that layer's fit
    r21, r2s1, _ = oracle.layer_scores(src_k=xk, src_v=xv, tgt_k=yk, tgt_v=yv,
                                       layer_idx=np.array([[2], [1]]), **kw)
    assert np.allclose(r2s1[0], r21[0, 2]) and np.allclose(r2s1[1], r21[1, 1])
    # more features never fit worse in sample (tiny lam); the layer each
    # target was drawn from is listed second, so a set that read only its
    # first layer would fall short of it
    kw["lam"] = 1e-10
    r2t, r2st, _ = oracle.layer_scores(src_k=xk, src_v=xv, tgt_k=yk, tgt_v=yv,
                                       layer_idx=np.array([[2, 0], [0, 1]]), **kw)
    assert np.all(r2st[0] >= np.maximum(r2t[0, 0], r2t[0, 2]) - 1e-9)
    assert np.all(r2st[1] >= np.maximum(r2t[1, 1], r2t[1, 0]) - 1e-9)
    # the score of a set does not depend on the order of its layers
    _, r2sr, _ = oracle.layer_scores(src_k=xk, src_v=xv, tgt_k=yk, tgt_v=yv,
                                     layer_idx=np.array([[0, 2], [1, 0]]), **kw)
    assert np.allclose(r2sr, r2st, atol=1e-9)
    # a bad position scores nothing
    r2e, _, ste = oracle.layer_scores(src_k=xk, src_v=xv, tgt_k=yk, tgt_v=yv,
                                      theta_src=1e4, theta_tgt=1e4, max_position=n - 1)
    assert ste == oracle.BAD_POSITION and np.all(np.isnan(r2e))


# ---------------------------------------------------------------------------
# Ridge-fit inputs in content space (kvxo_ridge_features)
# ---------------------------------------------------------------------------
def test_ridge_features_recover_planted_content_in_table_order():
    # keys stored as content turned at each token's own position (ragged
    # requests, explicit positions), with different bases on the two sides;
    # the features must give the content back, the table's layers side by
    # side in the table's order, values as stored
    rng = np.random.default_rng(11)
    Ls, Lt, H, d, n = 4, 3, 2, 8, 23
    cs_k = rng.normal(size=(Ls, n, H, d)); cs_v = rng.normal(size=(Ls, n, H, d))
    ct_k = rng.normal(size=(Lt, n, H, d)); ct_v = rng.normal(size=(Lt, n, H, d))
    cu = np.array([0, 9, 9, 23])
    pos = rng.integers(0, 500, size=n)
    sk = np.stack([_rotate_np(cs_k[s], pos, 1e4) for s in range(Ls)])
    tk = np.stack([_rotate_np(ct_k[t], pos, 1e6) for t in range(Lt)])
    table = np.array([[3, 0], [1, 1], [2, 3]])
    x, y, st = oracle.ridge_features(src_k=sk, src_v=cs_v, tgt_k=tk, tgt_v=ct_v, theta_src=1e4,
                                     theta_tgt=1e6, max_position=500, layer_idx=table,
                                     cu_seqlens=cu, src_pos=pos)
    assert st == 0 and x.shape == (Lt, H, 2, n, 2 * d) and y.shape == (Lt, H, 2, n, d)
    for lt in range(Lt):
        for h in range(H):
            for j, s in enumerate(table[lt]):
                np.testing.assert_allclose(x[lt, h, 0, :, j * d:(j + 1) * d], cs_k[s, :, h],
                                           atol=1e-12)
                np.testing.assert_array_equal(x[lt, h, 1, :, j * d:(j + 1) * d], cs_v[s, :, h])
            np.testing.assert_allclose(y[lt, h, 0], ct_k[lt, :, h], atol=1e-12)
            np.testing.assert_array_equal(y[lt, h, 1], ct_v[lt, :, h])
    # without the target caches only x is produced, and it is the same
    x2, y2, st2 = oracle.ridge_features(src_k=sk, src_v=cs_v, theta_src=1e4, theta_tgt=1e6,
                                        max_position=500, layer_idx=table, cu_seqlens=cu,
                                        src_pos=pos)
    assert st2 == 0 and y2 is None and np.array_equal(x2, x)
    # positions restart at 0 in every request when none are given
    x3, _, _ = oracle.ridge_features(src_k=sk, src_v=cs_v, theta_src=1e4, theta_tgt=1e6,
                                     max_position=500, layer_idx=table, cu_seqlens=cu)
    own = np.concatenate([np.arange(9), np.arange(14)])
    want = _rotate_np(sk[table[0, 0]][:, 1], -own, 1e4)
    np.testing.assert_allclose(x3[0, 1, 0, :, :d], want, atol=1e-12)


def test_ridge_features_fit_reproduces_the_set_score():
    # the set score of a table is the in-sample R^2 of the centred ridge fit
    # on exactly these features; with lam -> 0 that is least squares with an
    # intercept, which LAPACK's lstsq gives independently of both functions
    xk, xv, yk, yv = _score_case(9)
    Ls, n, H, d = xk.shape
    table = np.array([[2, 0], [1, 2]])
    kw = dict(theta_src=1e4, theta_tgt=5e5, max_position=n)
    _, r2s, st = oracle.layer_scores(src_k=xk, src_v=xv, tgt_k=yk, tgt_v=yv, lam=1e-10,
                                     layer_idx=table, **kw)
    x, y, st2 = oracle.ridge_features(src_k=xk, src_v=xv, tgt_k=yk, tgt_v=yv, layer_idx=table,
                                      **kw)
    assert st == 0 and st2 == 0
    for lt in range(2):
        for h in range(H):
            for m in range(2):
                A = np.hstack([x[lt, h, m], np.ones((n, 1))])
                coef, *_ = np.linalg.lstsq(A, y[lt, h, m], rcond=None)
                res = y[lt, h, m] - A @ coef
                yy = y[lt, h, m]
                ref = 1 - (res ** 2).sum() / ((yy - yy.mean(0)) ** 2).sum()
                assert r2s[lt, h, m] == pytest.approx(ref, abs=1e-8)


def test_ridge_features_flag_bad_inputs_and_zero_their_rows():
    rng = np.random.default_rng(12)
    Ls, Lt, H, d, n = 3, 2, 1, 4, 6
    sk = rng.normal(size=(Ls, n, H, d)); sv = rng.normal(size=(Ls, n, H, d))
    tk = rng.normal(size=(Lt, n, H, d)); tv = rng.normal(size=(Lt, n, H, d))
    kw = dict(src_k=sk, src_v=sv, tgt_k=tk, tgt_v=tv, theta_src=1e4, theta_tgt=1e4)
    # a position past the limit: that token's rows are zero, the rest intact
    pos = np.arange(n); pos[4] = 50
    x, y, st = oracle.ridge_features(max_position=10, layer_idx=np.array([[0], [2]]),
                                     src_pos=pos, **kw)
    assert st == oracle.BAD_POSITION
    assert not x[:, :, :, 4].any() and not y[:, :, :, 4].any()
    np.testing.assert_array_equal(x[1, 0, 1, 5], sv[2, 5, 0])
    # a table row naming a missing layer: that target layer's x is zero, its
    # y and the other layer's rows are intact
    x, y, st = oracle.ridge_features(max_position=10, layer_idx=np.array([[0, 1], [2, 3]]), **kw)
    assert st == oracle.BAD_LAYER_INDEX
    assert not x[1].any() and x[0].all()
    np.testing.assert_array_equal(y[1, 0, 1], tv[1, :, 0])
    # a malformed request table: nothing is written but zeros
    x, y, st = oracle.ridge_features(max_position=10, layer_idx=np.array([[0, 1], [1, 2]]),
                                     cu_seqlens=np.array([0, 4, 3, 6]), **kw)
    assert st == oracle.BAD_SEQLENS and not x.any() and not y.any()


def test_ridge_features_are_what_the_transfer_maps():
    # the transfer applies each (target layer, head, K|V) map to exactly these
    # features: x W + b, with keys then turned into the target RoPE at the
    # token's target position (numpy here), equals the transfer's output row
    rng = np.random.default_rng(13)
    Ls, Lt, H, d, k, n, off = 4, 3, 2, 8, 2, 11, 5
    sk = rng.normal(size=(Ls, n, H, d)); sv = rng.normal(size=(Ls, n, H, d))
    table = np.array([[3, 1], [0, 0], [2, 3]])
    w = rng.normal(size=(Lt, H, 2, k * d, d)); b = rng.normal(size=(Lt, H, 2, d))
    kw = dict(theta_src=1e4, theta_tgt=5e5, max_position=n + off)
    x, _, st = oracle.ridge_features(src_k=sk, src_v=sv, layer_idx=table, **kw)
    dk, dv, st2 = oracle.transfer(src_k=sk, src_v=sv, layer_idx=table, w=w, b=b,
                                  tgt_offset=np.array([off]), dst_capacity=n + off, **kw)
    assert st == 0 and st2 == 0
    pos = np.arange(n) + off
    for lt in range(Lt):
        for h in range(H):
            yk = x[lt, h, 0] @ w[lt, h, 0] + b[lt, h, 0]
            yv = x[lt, h, 1] @ w[lt, h, 1] + b[lt, h, 1]
            np.testing.assert_allclose(_rotate_np(yk, pos, 5e5), dk[lt, off:, h], atol=1e-10)
            np.testing.assert_allclose(yv, dv[lt, off:, h], atol=1e-10)
