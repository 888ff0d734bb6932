"""fp64 CPU oracle of the cross-model KV-cache transfer (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package; the library under
``cross_model_kv_transfer_gb300`` never does.  The arithmetic lives in
``kvx_oracle.c`` (plain nested loops in double precision); this module only
compiles it with gcc, marshals numpy arrays and returns numpy arrays.

What each function computes, and the passages it follows, is documented in
``kvx_oracle.h``.  In short:

* ``rope``        half-split RoPE rotate / un-rotate of one head vector
                  ("Helm Intelligent Routing", "Why carrying the cache across
                  is the hard part", steps 1 and 3).
* ``map_token``   one token of one (target layer, head): gather, un-rotate,
                  concatenate, ``x @ W + b`` for K and V, re-rotate K
                  (same steps; the Qwen3 article's section on the linear
                  bridge for feature concatenation and the map).
* ``dst_row``     contiguous / paged cache row of one token.
* ``transfer``    the whole transfer over all requests, tokens, layers, heads;
                  ``wide=True`` for the wide-feature mapper (one dense map per
                  target layer over all heads' keys and values of the
                  selected layers: the Qwen3 article's mapper size, section
                  on production limits); ``map_token_wide`` for one token.
* ``ridge_fit``   centred ridge regression with intercept (the Qwen3
                  article's ridge demo).
* ``layer_scores`` explained variance of each target (layer, head, K|V) by
                  the ridge fit on one source layer, or on a set (the Qwen3
                  article's linear-bridge section: layer choice by predictive
                  power).
* ``ridge_features`` the inputs of those ridge fits in content space: the
                  table row's source layers side by side (keys un-rotated)
                  and the target layer's content, per (target layer, head,
                  K|V) (the same section).
* ``kv_diagnostics`` KV cosine ("Helm Intelligent Routing", "Reading the
                  retention score") and explained variance (the Qwen3
                  article's linear-structure analysis) of a mapped cache
                  against the target's own, per (target layer, head, K|V);
                  ``mean_cosine`` and ``explained_variance`` read them out.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvx_oracle.c")
_HDR = os.path.join(_HERE, "kvx_oracle.h")
_LIB = os.path.join(_HERE, "libkvx_oracle.so")
_lock = threading.Lock()
_lib = None

BAD_LAYER_INDEX = 1
BAD_POSITION = 2
BAD_BLOCK = 4
BAD_ROW = 8
BAD_SEQLENS = 32
BAD_SRC_BLOCK = 64

CONTIGUOUS = 0
PAGED = 1


def build(force: bool = False) -> str:
    """Compile ``kvx_oracle.c`` into ``libkvx_oracle.so`` with gcc.

    ``-ffp-contract=off`` keeps every multiply and add separately rounded, so
    the oracle gives the same bits on x86-64 and aarch64 hosts."""
    newest_src = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= newest_src:
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared",
           "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True, cwd=_HERE)
    os.replace(tmp, _LIB)
    return _LIB


class _Problem(ctypes.Structure):
    _fields_ = [
        ("src_layers", ctypes.c_int32), ("tgt_layers", ctypes.c_int32),
        ("kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("k", ctypes.c_int32),
        ("theta_src", ctypes.c_double), ("theta_tgt", ctypes.c_double),
        ("max_position", ctypes.c_int64),
        ("num_requests", ctypes.c_int32),
        ("ntok", ctypes.c_int64),
        ("cu_seqlens", ctypes.c_void_p),
        ("src_k", ctypes.c_void_p), ("src_v", ctypes.c_void_p),
        ("layer_idx", ctypes.c_void_p),
        ("w", ctypes.c_void_p), ("b", ctypes.c_void_p),
        ("src_pos", ctypes.c_void_p), ("tgt_pos", ctypes.c_void_p),
        ("tgt_offset", ctypes.c_void_p),
        ("layout", ctypes.c_int32),
        ("dst_capacity", ctypes.c_int64),
        ("block_size", ctypes.c_int64), ("num_blocks", ctypes.c_int64),
        ("max_blocks_per_req", ctypes.c_int64),
        ("block_table", ctypes.c_void_p),
        ("src_layout", ctypes.c_int32),
        ("src_block_size", ctypes.c_int64), ("src_num_blocks", ctypes.c_int64),
        ("src_max_blocks_per_req", ctypes.c_int64),
        ("src_block_table", ctypes.c_void_p),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            lib.kvxo_rope.argtypes = [dp, ctypes.c_int, ctypes.c_double,
                                      ctypes.c_double, ctypes.c_int, dp]
            lib.kvxo_rope.restype = None
            lib.kvxo_map_token.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_double,
                ctypes.POINTER(dp), ctypes.POINTER(dp), dp, dp, dp, dp,
                ctypes.c_double, ctypes.c_double, dp, dp]
            lib.kvxo_map_token.restype = None
            lib.kvxo_dst_row.argtypes = [
                ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                ctypes.POINTER(ctypes.c_int)]
            lib.kvxo_dst_row.restype = ctypes.c_int64
            lib.kvxo_transfer.argtypes = [ctypes.POINTER(_Problem), dp, dp]
            lib.kvxo_transfer.restype = ctypes.c_int
            lib.kvxo_ridge_fit.argtypes = [dp, dp, ctypes.c_int64, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_double, dp, dp]
            lib.kvxo_ridge_fit.restype = ctypes.c_int
            lib.kvxo_transfer_wide.argtypes = [ctypes.POINTER(_Problem), dp, dp]
            lib.kvxo_transfer_wide.restype = ctypes.c_int
            lib.kvxo_map_token_wide.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_double,
                ctypes.POINTER(dp), ctypes.POINTER(dp), dp, dp, ctypes.c_double,
                ctypes.c_double, dp, dp]
            lib.kvxo_map_token_wide.restype = None
            lib.kvxo_kv_diagnostics.argtypes = [ctypes.POINTER(_Problem), dp, dp, dp, dp, dp]
            lib.kvxo_kv_diagnostics.restype = ctypes.c_int
            lib.kvxo_layer_scores.argtypes = [ctypes.POINTER(_Problem), dp, dp, ctypes.c_double,
                                              dp, ctypes.c_void_p]
            lib.kvxo_layer_scores.restype = ctypes.c_int
            lib.kvxo_ridge_features.argtypes = [ctypes.POINTER(_Problem), dp, dp, dp, dp]
            lib.kvxo_ridge_features.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _dp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _vp(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def rope(x, pos: float, theta: float, sign: int) -> np.ndarray:
    """Rotate (sign=+1) or un-rotate (sign=-1) one head vector x[d]."""
    x = _f64(x)
    out = np.empty_like(x)
    _load().kvxo_rope(_dp(x), x.shape[0], float(pos), float(theta), int(sign), _dp(out))
    return out


def map_token(k_rows, v_rows, Wk, Wv, bk, bv, p_src, p_tgt, theta_src, theta_tgt):
    """One token of one (target layer, head).  k_rows / v_rows: [k][d] arrays
    of the selected source layers' head vectors, in index-table order."""
    k_rows, v_rows = _f64(k_rows), _f64(v_rows)
    k, d = k_rows.shape
    Wk, Wv, bk, bv = _f64(Wk), _f64(Wv), _f64(bk), _f64(bv)
    assert Wk.shape == (k * d, d) and Wv.shape == (k * d, d)
    dp = ctypes.POINTER(ctypes.c_double)
    kptr = (dp * k)(*[_dp(k_rows[j]) for j in range(k)])
    vptr = (dp * k)(*[_dp(v_rows[j]) for j in range(k)])
    out_k = np.empty(d)
    out_v = np.empty(d)
    _load().kvxo_map_token(d, k, float(theta_src), float(theta_tgt), kptr, vptr,
                           _dp(Wk), _dp(Wv), _dp(bk), _dp(bv),
                           float(p_src), float(p_tgt), _dp(out_k), _dp(out_v))
    return out_k, out_v


def dst_row(layout, r, p_tgt, dst_capacity=0, block_size=1, num_blocks=0,
            block_table=None, max_blocks_per_req=0):
    """Target-cache row of one token, or (-1, reason bits)."""
    bt = None if block_table is None else np.ascontiguousarray(block_table, dtype=np.int32)
    bad = ctypes.c_int(0)
    row = _load().kvxo_dst_row(int(layout), int(r), int(p_tgt), int(dst_capacity),
                               int(block_size), int(num_blocks), _vp(bt),
                               int(max_blocks_per_req), ctypes.byref(bad))
    return int(row), int(bad.value)


def transfer(*, src_k, src_v, layer_idx, w, b, theta_src, theta_tgt,
             max_position, cu_seqlens=None, src_pos=None, tgt_pos=None,
             tgt_offset=None, layout=CONTIGUOUS, dst_capacity=0,
             block_size=1, num_blocks=0, block_table=None, dst_k=None, dst_v=None,
             wide=False, src_layout=CONTIGUOUS, src_block_size=1, src_block_table=None,
             ntok=None):
    """The whole transfer in fp64.

    src_k / src_v: [Ls][ntok][H][d]; layer_idx: [Lt][k]; w: [Lt][H][2][k*d][d]
    (per-head maps) or, with ``wide``, [Lt][k*2*H*d][H*2*d] (one map per
    target layer over all heads' keys and values, ``kvxo_transfer_wide``);
    b: [Lt][H][2][d].  dst_k / dst_v (optional, fp64) are the initial target
    cache [Lt][rows][H][d]; rows not written keep their values (NaN if the
    caller gives none).  With ``src_layout=PAGED`` the source is the pilot's
    paged cache [Ls][src_num_blocks*src_block_size][H][d] read through
    ``src_block_table`` [R][max] (``kvxo_src_row``); ``ntok`` then defaults
    to cu_seqlens[-1].  Returns (dst_k, dst_v, status bits)."""
    src_k, src_v, w, b = _f64(src_k), _f64(src_v), _f64(w), _f64(b)
    Ls, src_rows, H, d = src_k.shape
    if src_layout == PAGED:
        if ntok is None:
            ntok = int(np.asarray(cu_seqlens)[-1]) if cu_seqlens is not None else None
        assert ntok is not None and src_rows % src_block_size == 0
        sbt = np.ascontiguousarray(src_block_table, dtype=np.int32)
        src_nb, src_mb = src_rows // src_block_size, sbt.shape[1]
    else:
        ntok = src_rows
        sbt, src_nb, src_mb = None, 0, 0
    idx = np.ascontiguousarray(layer_idx, dtype=np.int32)
    Lt, k = idx.shape
    if wide:
        assert w.shape == (Lt, k * 2 * H * d, H * 2 * d), w.shape
    else:
        assert w.shape == (Lt, H, 2, k * d, d), w.shape
    assert b.shape == (Lt, H, 2, d), b.shape
    cu = None if cu_seqlens is None else np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    R = 1 if cu is None else cu.shape[0] - 1
    sp = None if src_pos is None else np.ascontiguousarray(src_pos, dtype=np.int64)
    tp = None if tgt_pos is None else np.ascontiguousarray(tgt_pos, dtype=np.int64)
    to = None if tgt_offset is None else np.ascontiguousarray(tgt_offset, dtype=np.int64)
    bt = None
    mbpr = 0
    if layout == PAGED:
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        mbpr = bt.shape[1]
        rows = num_blocks * block_size
    else:
        rows = R * dst_capacity
    if dst_k is None:
        dst_k = np.full((Lt, rows, H, d), np.nan)
    else:
        dst_k = np.array(dst_k, dtype=np.float64, copy=True, order="C")
    if dst_v is None:
        dst_v = np.full((Lt, rows, H, d), np.nan)
    else:
        dst_v = np.array(dst_v, dtype=np.float64, copy=True, order="C")
    assert dst_k.shape == (Lt, rows, H, d) and dst_v.shape == (Lt, rows, H, d)
    P = _Problem(Ls, Lt, H, d, k, float(theta_src), float(theta_tgt),
                 int(max_position), R, ntok, _vp(cu), _vp(src_k), _vp(src_v),
                 _vp(idx), _vp(w), _vp(b), _vp(sp), _vp(tp), _vp(to), int(layout),
                 int(dst_capacity), int(block_size), int(num_blocks), int(mbpr), _vp(bt),
                 int(src_layout), int(src_block_size), int(src_nb), int(src_mb), _vp(sbt))
    fn = _load().kvxo_transfer_wide if wide else _load().kvxo_transfer
    st = fn(ctypes.byref(P), _dp(dst_k), _dp(dst_v))
    return dst_k, dst_v, int(st)


def map_token_wide(k_rows, v_rows, W, b, p_src, p_tgt, theta_src, theta_tgt):
    """One token of one target layer with the wide-feature map.  k_rows /
    v_rows: [k][H][d] (the selected source layers' head vectors, in
    index-table order); W: [k*2*H*d][H*2*d]; b: [H][2][d].  Returns the
    [H][d] key and value rows."""
    k_rows, v_rows, W, b = _f64(k_rows), _f64(v_rows), _f64(W), _f64(b)
    k, H, d = k_rows.shape
    assert v_rows.shape == (k, H, d)
    assert W.shape == (k * 2 * H * d, H * 2 * d) and b.shape == (H, 2, d)
    dp = ctypes.POINTER(ctypes.c_double)
    kptr = (dp * k)(*[_dp(k_rows[j]) for j in range(k)])
    vptr = (dp * k)(*[_dp(v_rows[j]) for j in range(k)])
    out_k = np.empty((H, d))
    out_v = np.empty((H, d))
    _load().kvxo_map_token_wide(H, d, k, float(theta_src), float(theta_tgt), kptr, vptr,
                                _dp(W), _dp(b), float(p_src), float(p_tgt), _dp(out_k),
                                _dp(out_v))
    return out_k, out_v


def ridge_fit(X, Y, lam: float = 0.01):
    """Centred ridge with intercept: returns (W [p][q], b [q])."""
    X, Y = _f64(X), _f64(Y)
    n, p = X.shape
    n2, q = Y.shape
    assert n == n2
    W = np.empty((p, q))
    b = np.empty(q)
    rc = _load().kvxo_ridge_fit(_dp(X), _dp(Y), n, p, q, float(lam), _dp(W), _dp(b))
    if rc != 0:
        raise np.linalg.LinAlgError("ridge normal matrix is not positive definite")
    return W, b


def kv_diagnostics(*, mapped_k, mapped_v, ref_k, ref_v, theta_tgt, max_position,
                   ntok, cu_seqlens=None, src_pos=None, tgt_pos=None, tgt_offset=None,
                   layout=CONTIGUOUS, dst_capacity=0, block_size=1, num_blocks=0,
                   block_table=None):
    """Per-(target layer, head, K|V) statistics [Lt][H][2][d + 4] of the
    mapped cache against the target's own cache (both [Lt][rows][H][d]),
    over the tokens a transfer with the same request table, positions and
    layout writes; see ``kvx_oracle.h``.  Returns (stats, status bits)."""
    mk, mv, rk, rv = _f64(mapped_k), _f64(mapped_v), _f64(ref_k), _f64(ref_v)
    Lt, rows, H, d = rk.shape
    assert mk.shape == mv.shape == rk.shape == rv.shape
    cu = None if cu_seqlens is None else np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    R = 1 if cu is None else cu.shape[0] - 1
    sp = None if src_pos is None else np.ascontiguousarray(src_pos, dtype=np.int64)
    tp = None if tgt_pos is None else np.ascontiguousarray(tgt_pos, dtype=np.int64)
    to = None if tgt_offset is None else np.ascontiguousarray(tgt_offset, dtype=np.int64)
    bt = None
    mbpr = 0
    if layout == PAGED:
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        mbpr = bt.shape[1]
        assert rows == num_blocks * block_size
    else:
        assert rows == R * dst_capacity
    P = _Problem(0, Lt, H, d, 0, 0.0, float(theta_tgt), int(max_position), R, int(ntok),
                 _vp(cu), None, None, None, None, None, _vp(sp), _vp(tp), _vp(to),
                 int(layout), int(dst_capacity), int(block_size), int(num_blocks), int(mbpr),
                 _vp(bt))
    stats = np.empty((Lt, H, 2, d + 4))
    st = _load().kvxo_kv_diagnostics(ctypes.byref(P), _dp(mk), _dp(mv), _dp(rk), _dp(rv),
                                     _dp(stats))
    return stats, int(st)


def layer_scores(*, src_k, src_v, tgt_k, tgt_v, theta_src, theta_tgt, max_position,
                 lam=0.01, cu_seqlens=None, src_pos=None, layer_idx=None):
    """Layer-selection scores (``kvxo_layer_scores``): in-sample explained
    variance of each target (layer, head, K|V) by the ridge fit on one source
    layer, r2 [Lt][Ls][H][2], and, with ``layer_idx`` [Lt][k], on the set of
    that table row, r2_set [Lt][H][2] (else None).  src_k / src_v
    [Ls][ntok][H][d] and tgt_k / tgt_v [Lt][ntok][H][d] hold the same tokens
    in the same order.  Returns (r2, r2_set, status bits)."""
    sk, sv, tk, tv = _f64(src_k), _f64(src_v), _f64(tgt_k), _f64(tgt_v)
    Ls, ntok, H, d = sk.shape
    Lt = tk.shape[0]
    assert sv.shape == sk.shape and tk.shape == tv.shape == (Lt, ntok, H, d)
    cu = None if cu_seqlens is None else np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    R = 1 if cu is None else cu.shape[0] - 1
    sp = None if src_pos is None else np.ascontiguousarray(src_pos, dtype=np.int64)
    idx = None if layer_idx is None else np.ascontiguousarray(layer_idx, dtype=np.int32)
    k = 0 if idx is None else idx.shape[1]
    P = _Problem(Ls, Lt, H, d, k, float(theta_src), float(theta_tgt), int(max_position), R,
                 int(ntok), _vp(cu), _vp(sk), _vp(sv), _vp(idx), None, None, _vp(sp), None,
                 None, CONTIGUOUS, 0, 1, 0, 0, None)
    r2 = np.empty((Lt, Ls, H, 2))
    r2_set = None if idx is None else np.empty((Lt, H, 2))
    st = _load().kvxo_layer_scores(ctypes.byref(P), _dp(tk), _dp(tv), float(lam), _dp(r2),
                                   None if r2_set is None else r2_set.ctypes.data)
    return r2, r2_set, int(st)


def ridge_features(*, src_k, src_v, theta_src, theta_tgt, max_position, layer_idx,
                   tgt_k=None, tgt_v=None, cu_seqlens=None, src_pos=None):
    """Content-space inputs of the ridge fits (``kvxo_ridge_features``):
    x [Lt][H][2][ntok][k d] (the table row's source layers concatenated,
    keys un-rotated with theta_src) and, with the target caches, y
    [Lt][H][2][ntok][d] (keys un-rotated with theta_tgt), at every token's
    position.  src_k / src_v [Ls][ntok][H][d], tgt_k / tgt_v [Lt][ntok][H][d].
    Returns (x, y or None, status bits)."""
    sk, sv = _f64(src_k), _f64(src_v)
    Ls, ntok, H, d = sk.shape
    idx = np.ascontiguousarray(layer_idx, dtype=np.int32)
    Lt, k = idx.shape
    tk = None if tgt_k is None else _f64(tgt_k)
    tv = None if tgt_v is None else _f64(tgt_v)
    cu = None if cu_seqlens is None else np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    R = 1 if cu is None else cu.shape[0] - 1
    sp = None if src_pos is None else np.ascontiguousarray(src_pos, dtype=np.int64)
    P = _Problem(Ls, Lt, H, d, k, float(theta_src), float(theta_tgt), int(max_position), R,
                 int(ntok), _vp(cu), _vp(sk), _vp(sv), _vp(idx), None, None, _vp(sp), None,
                 None, CONTIGUOUS, 0, 1, 0, 0, None)
    x = np.empty((Lt, H, 2, ntok, k * d))
    y = None if tk is None else np.empty((Lt, H, 2, ntok, d))
    st = _load().kvxo_ridge_features(ctypes.byref(P), None if tk is None else _dp(tk),
                                     None if tv is None else _dp(tv), _dp(x),
                                     None if y is None else _dp(y))
    return x, y, int(st)


def mean_cosine(stats):
    """Mean KV cosine per entry of ``stats[..., :]`` (NaN where n = 0)."""
    s = np.asarray(stats, dtype=np.float64)
    with np.errstate(invalid="ignore", divide="ignore"):
        return s[..., 1] / s[..., 0]


def explained_variance(stats):
    """Centred R^2 per entry of ``stats`` (content space, summed over d)."""
    s = np.asarray(stats, dtype=np.float64)
    n = s[..., 0]
    with np.errstate(invalid="ignore", divide="ignore"):
        ss_tot = s[..., 3] - np.sum(s[..., 4:] ** 2, axis=-1) / n
        return 1.0 - s[..., 2] / ss_tot
