"""Seeded synthetic inputs for the cross-model KV-cache transfer.

This module draws random inputs and nothing else: it holds none of the
transfer's arithmetic (no un-rotation, no map, no re-rotation, no cache
routing).  The one rotation here is the pilot model's own RoPE, applied once
when the synthetic pilot cache is drawn, as a real pilot cache stores its
keys.  The CUDA library and the fp64 oracle both consume what it returns;
neither is imported here.

Workloads (shapes of the pairs the pages measure; no model weights or
datasets are used -- every tensor is synthetic):

``tiny_fp32``     4 -> 6 layers, 2 KV heads, d=64, T=128, k=2, fp32, theta 1e4.
``qwen3_0p6b_1p7b`` 28 -> 28 layers, 8 KV heads, d=128, k=4, bf16, theta 1e6,
                  T=512 (the 512-token row of the transfer-cost table of
                  "Helm Intelligent Routing", section "What the transfer costs").
``qwen3_0p6b_1p7b_off37`` same pair at T=2048 / 8192 with the target shifted
                  by +37 positions.
``qwen3_14b_32b`` 40 -> 64 layers, 8 KV heads, d=128, k=4, bf16, theta 1e6,
                  T=32768 (the 32K latency point of the Qwen3 14B -> 32B
                  article, section "Что на самом деле покрывает главная
                  цифра").
``llama31_8b_70b_paged`` 32 -> 80 layers, 8 KV heads, d=128, k=4, bf16, theta
                  5e5, 16 requests of 1024..16384 tokens, per-request target
                  offset 0..64, paged target cache with 16-token blocks dealt
                  from a randomly permuted shared pool.

Value recipe:
* content vectors: N(0, 1) times a per-(layer, head, channel) log-normal
  (sigma = 1) scale; in the bf16 workloads 4 channels per (layer, head) are
  further scaled x10 (outliers).
* keys are stored as the pilot model would have cached them: the drawn
  content turned by its RoPE at the token's source position p (0 .. len - 1
  within its request), half-split pairs (i, i + d/2) turned by the angle
  p * theta_src^(-2i/d), the angle formed and its cosine and sine taken in
  fp64.  This is part of synthesising a pilot cache, like the value
  distribution; the CUDA library and the oracle each un-rotate the stored
  bytes with their own code and share nothing with this module.
* values are stored as drawn.
* W ~ N(0, 1/(k d)) stored fp32; b ~ N(0, 0.01^2) stored fp32 (tiny) or bf16.
* the layer-index table draws, for each target layer, k distinct source
  layers uniformly without replacement.
* paired calibration caches for layer-selection scoring: see
  ``make_score_inputs``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

CONTIGUOUS = 0
PAGED = 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    src_layers: int
    tgt_layers: int
    kv_heads: int
    head_dim: int
    k: int
    theta_src: float
    theta_tgt: float
    kv_dtype: torch.dtype
    b_dtype: torch.dtype
    seed: int
    seqlens: tuple            # tokens per request
    tgt_offsets: tuple        # target offset per request
    layout: int = CONTIGUOUS
    block_size: int = 16
    outliers: int = 0         # channels per (layer, head) scaled x10

    @property
    def num_requests(self) -> int:
        return len(self.seqlens)

    @property
    def ntok(self) -> int:
        return int(sum(self.seqlens))

    @property
    def max_position(self) -> int:
        """Smallest table length that covers every source and target position."""
        return int(max(n + o for n, o in zip(self.seqlens, self.tgt_offsets)))

    @property
    def dst_capacity(self) -> int:
        return self.max_position

    def blocks_per_request(self):
        bs = self.block_size
        return [(n + o + bs - 1) // bs for n, o in zip(self.seqlens, self.tgt_offsets)]

    @property
    def num_blocks(self) -> int:
        return int(sum(self.blocks_per_request()))

    @property
    def dst_rows(self) -> int:
        if self.layout == PAGED:
            return self.num_blocks * self.block_size
        return self.num_requests * self.dst_capacity

    def with_tokens(self, seqlens, tgt_offsets=None, name=None) -> "Workload":
        """Same pair and value recipe at other sequence lengths (test sizes)."""
        seqlens = tuple(int(n) for n in seqlens)
        if tgt_offsets is None:
            tgt_offsets = tuple([self.tgt_offsets[0]] * len(seqlens))
        return dataclasses.replace(self, seqlens=seqlens,
                                   tgt_offsets=tuple(int(o) for o in tgt_offsets),
                                   name=name or f"{self.name}@{sum(seqlens)}")

    # ---- byte / flop accounting of one transfer -------------------------
    def unique_selected_layers(self, layer_idx: torch.Tensor) -> int:
        return int(torch.unique(layer_idx.flatten()).numel())

    def algorithmic_bytes(self, layer_idx: torch.Tensor) -> int:
        """Unique selected source K+V read once, target K+V written once,
        W and b read once, as stored."""
        eb = torch.empty(0, dtype=self.kv_dtype).element_size()
        row = self.kv_heads * self.head_dim * eb
        src = 2 * self.unique_selected_layers(layer_idx) * self.ntok * row
        dst = 2 * self.tgt_layers * self.ntok * row
        kd = self.k * self.head_dim
        w = self.tgt_layers * self.kv_heads * 2 * kd * self.head_dim * 4
        bb = torch.empty(0, dtype=self.b_dtype).element_size()
        b = self.tgt_layers * self.kv_heads * 2 * self.head_dim * bb
        return int(src + dst + w + b)

    def algorithmic_flops(self) -> int:
        kd = self.k * self.head_dim
        return int(2 * self.ntok * kd * self.head_dim * self.tgt_layers * self.kv_heads * 2)

    # ---- the wide-feature map: one [F x N] map per target layer ----------
    def wide_algorithmic_bytes(self, layer_idx: torch.Tensor) -> int:
        """As ``algorithmic_bytes`` with W [Lt][k*2*H*d][H*2*d] fp32."""
        eb = torch.empty(0, dtype=self.kv_dtype).element_size()
        row = self.kv_heads * self.head_dim * eb
        src = 2 * self.unique_selected_layers(layer_idx) * self.ntok * row
        dst = 2 * self.tgt_layers * self.ntok * row
        F = self.k * 2 * self.kv_heads * self.head_dim
        N = self.kv_heads * 2 * self.head_dim
        bb = torch.empty(0, dtype=self.b_dtype).element_size()
        return int(src + dst + self.tgt_layers * F * N * 4 + self.tgt_layers * N * bb)

    def wide_algorithmic_flops(self) -> int:
        F = self.k * 2 * self.kv_heads * self.head_dim
        N = self.kv_heads * 2 * self.head_dim
        return int(2 * self.ntok * F * N * self.tgt_layers)


def _bf16(name, Ls, Lt, k, theta, seed, seqlens, offsets, **kw):
    return Workload(name=name, src_layers=Ls, tgt_layers=Lt, kv_heads=8, head_dim=128,
                    k=k, theta_src=theta, theta_tgt=theta, kv_dtype=torch.bfloat16,
                    b_dtype=torch.bfloat16, seed=seed, seqlens=tuple(seqlens),
                    tgt_offsets=tuple(offsets), outliers=4, **kw)


def _llama_paged_lengths(seed: int):
    g = torch.Generator().manual_seed(seed * 7919 + 1)
    lens = torch.randint(1024, 16385, (16,), generator=g).tolist()
    offs = torch.randint(0, 65, (16,), generator=g).tolist()
    return tuple(lens), tuple(offs)


_LL, _LO = _llama_paged_lengths(5)

WORKLOADS = {
    "tiny_fp32": Workload(
        name="tiny_fp32", src_layers=4, tgt_layers=6, kv_heads=2, head_dim=64, k=2,
        theta_src=1e4, theta_tgt=1e4, kv_dtype=torch.float32, b_dtype=torch.float32,
        seed=1, seqlens=(128,), tgt_offsets=(0,)),
    "qwen3_0p6b_1p7b": _bf16("qwen3_0p6b_1p7b", 28, 28, 4, 1e6, 2, (512,), (0,)),
    "qwen3_0p6b_1p7b_off37_2k": _bf16("qwen3_0p6b_1p7b_off37_2k", 28, 28, 4, 1e6, 3,
                                      (2048,), (37,)),
    "qwen3_0p6b_1p7b_off37_8k": _bf16("qwen3_0p6b_1p7b_off37_8k", 28, 28, 4, 1e6, 3,
                                      (8192,), (37,)),
    "qwen3_14b_32b": _bf16("qwen3_14b_32b", 40, 64, 4, 1e6, 4, (32768,), (0,)),
    "llama31_8b_70b_paged": _bf16("llama31_8b_70b_paged", 32, 80, 4, 5e5, 5, _LL, _LO,
                                  layout=PAGED, block_size=16),
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def make_inputs(wl: Workload, device="cpu", seed: Optional[int] = None) -> dict:
    """Draw every input tensor of one transfer of workload ``wl``.

    Returns a dict of tensors on ``device``: src_k, src_v [Ls][ntok][H][d]
    (kv dtype), layer_idx int32 [Lt][k], w fp32 [Lt][H][2][k*d][d], b
    [Lt][H][2][d] (b dtype), cu_seqlens int32 [R+1], tgt_offset int32 [R],
    block_table int32 [R][max_blocks] (paged only, -1 padded)."""
    seed = wl.seed if seed is None else seed
    dev = torch.device(device)
    g = _gen(dev, seed)
    gc = _gen("cpu", seed + 1000003)
    Ls, Lt, H, d, k = wl.src_layers, wl.tgt_layers, wl.kv_heads, wl.head_dim, wl.k
    T = wl.ntok
    half = d // 2

    src_k = torch.empty((Ls, T, H, d), dtype=wl.kv_dtype, device=dev)
    src_v = torch.empty((Ls, T, H, d), dtype=wl.kv_dtype, device=dev)
    # the pilot's RoPE at each token's source position, angles in fp64
    pos = torch.cat([torch.arange(n, dtype=torch.float64) for n in wl.seqlens]).to(dev)
    freq = wl.theta_src ** (-2.0 * torch.arange(half, dtype=torch.float64) / d)
    phi = pos[:, None] * freq.to(dev)[None, :]                       # [T][half]
    cos_p = torch.cos(phi).to(torch.float32)[:, None, :]
    sin_p = torch.sin(phi).to(torch.float32)[:, None, :]
    del phi
    for s in range(Ls):
        for dst, is_key in ((src_k, True), (src_v, False)):
            scale = torch.exp(torch.randn((1, H, d), generator=g, device=dev))
            if wl.outliers:
                for h in range(H):
                    ch = torch.randperm(d, generator=gc)[: wl.outliers].to(dev)
                    scale[0, h, ch] *= 10.0
            x = torch.randn((T, H, d), generator=g, device=dev) * scale
            if is_key:
                x0, x1 = x[..., :half], x[..., half:]
                x = torch.cat((x0 * cos_p - x1 * sin_p, x0 * sin_p + x1 * cos_p), dim=-1)
            dst[s].copy_(x.to(wl.kv_dtype))
            del x

    layer_idx = torch.stack([torch.randperm(Ls, generator=gc)[:k] for _ in range(Lt)])
    layer_idx = layer_idx.to(torch.int32).to(dev)

    w = torch.empty((Lt, H, 2, k * d, d), dtype=torch.float32, device=dev)
    std = 1.0 / math.sqrt(k * d)
    for lt in range(Lt):
        w[lt].copy_(torch.randn((H, 2, k * d, d), generator=g, device=dev) * std)
    b = (torch.randn((Lt, H, 2, d), generator=g, device=dev) * 0.01).to(wl.b_dtype)

    lens = torch.tensor(wl.seqlens, dtype=torch.int64)
    cu = torch.zeros(wl.num_requests + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(lens, 0)
    out = dict(src_k=src_k, src_v=src_v, layer_idx=layer_idx, w=w, b=b,
               cu_seqlens=cu.to(torch.int32).to(dev),
               tgt_offset=torch.tensor(wl.tgt_offsets, dtype=torch.int32).to(dev))
    if wl.layout == PAGED:
        out["block_table"] = make_block_table(wl, seed).to(dev)
    return out


def make_wide_weights(wl: Workload, device="cpu", seed: Optional[int] = None) -> torch.Tensor:
    """W of the wide-feature map, fp32 [Lt][F][N] with F = k*2*H*d features
    and N = H*2*d outputs, drawn N(0, 1/F) (the per-head recipe's scale)."""
    seed = (wl.seed if seed is None else seed) + 3000017
    dev = torch.device(device)
    g = _gen(dev, seed)
    F = wl.k * 2 * wl.kv_heads * wl.head_dim
    N = wl.kv_heads * 2 * wl.head_dim
    w = torch.empty((wl.tgt_layers, F, N), dtype=torch.float32, device=dev)
    for lt in range(wl.tgt_layers):
        w[lt].copy_(torch.randn((F, N), generator=g, device=dev) / math.sqrt(F))
    return w


def make_paged_source(wl: Workload, inp: dict, block_size: int, seed: Optional[int] = None,
                      spare_blocks: int = 3):
    """The pilot's own paged cache holding the same tokens as the packed
    source of ``inp``: each request's blocks are dealt from a seeded random
    permutation of a shared pool (plus ``spare_blocks`` unused ones), and the
    token at position p of request r sits in slot p % block_size of its
    request's block p // block_size.  Unused slots hold the all-ones bit
    pattern.  Returns (src_k, src_v, src_block_table [R][max], -1 padded)."""
    seed = (wl.seed if seed is None else seed) + 4000037
    g = _gen("cpu", seed)
    nb = [(n + block_size - 1) // block_size for n in wl.seqlens]
    pool = int(sum(nb)) + spare_blocks
    perm = torch.randperm(pool, generator=g).to(torch.int32)
    table = torch.full((wl.num_requests, max(nb) + 1), -1, dtype=torch.int32)
    at = 0
    rows = []
    for r, n in enumerate(wl.seqlens):
        table[r, :nb[r]] = perm[at: at + nb[r]]
        at += nb[r]
        pos = torch.arange(n)
        rows.append(table[r, pos // block_size].long() * block_size + pos % block_size)
    dev = inp["src_k"].device
    rows = torch.cat(rows).to(dev)
    out = []
    for src in (inp["src_k"], inp["src_v"]):
        paged = sentinel_like((src.shape[0], pool * block_size) + tuple(src.shape[2:]), src.dtype,
                              dev)
        paged[:, rows] = src
        out.append(paged)
    return out[0], out[1], table.to(dev)


def make_ridge_inputs(wl: Workload, batch: int, n: int, device="cpu",
                      seed: Optional[int] = None):
    """Stand-in for the paired observations one calibration batch fits on:
    ``batch`` fits of the per-head map shape (p = k*d features, q = d
    outputs), ``n`` observations each.  Features: N(0, 1) times a
    per-(fit, feature) log-normal (sigma = 0.5) scale plus a per-feature
    offset; targets: the features through a planted N(0, 1/p) map plus an
    offset and N(0, 0.1^2) noise.  fp32 [batch][n][p] and [batch][n][q]."""
    seed = (wl.seed if seed is None else seed) + 5000011
    dev = torch.device(device)
    g = _gen(dev, seed)
    p, q = wl.k * wl.head_dim, wl.head_dim
    x = torch.empty((batch, n, p), dtype=torch.float32, device=dev)
    y = torch.empty((batch, n, q), dtype=torch.float32, device=dev)
    for i in range(batch):
        scale = torch.exp(0.5 * torch.randn((1, p), generator=g, device=dev))
        xi = torch.randn((n, p), generator=g, device=dev) * scale + \
            torch.randn((1, p), generator=g, device=dev)
        wi = torch.randn((p, q), generator=g, device=dev) / math.sqrt(p)
        y[i].copy_(xi @ wi + torch.randn((1, q), generator=g, device=dev) +
                   0.1 * torch.randn((n, q), generator=g, device=dev))
        x[i].copy_(xi)
    return x, y


def make_score_inputs(wl: Workload, device="cpu", seed: Optional[int] = None) -> dict:
    """Stand-in for the paired calibration caches layer selection scores:
    the pilot's and the target model's caches of the same tokens
    (``wl.seqlens`` requests, positions 0 .. len - 1 in each).

    Source content: as ``make_inputs`` (N(0, 1) times a per-(layer, head,
    channel) log-normal scale, outlier channels where the workload has them).
    Target content of layer lt, head h, K|V: the content of its k planted
    source layers ``layer_idx[lt]`` (drawn as in ``make_inputs``) through
    seeded N(0, 1/(k d)) maps, plus N(0, 0.5^2) noise per channel times a
    per-(layer, head, channel) log-normal (sigma = 0.5) scale.  Keys are
    stored turned by each model's own RoPE (theta_src, theta_tgt) at the
    token's position, angles in fp64; values as drawn.  Returns src_k, src_v
    [Ls][ntok][H][d], tgt_k, tgt_v [Lt][ntok][H][d] (kv dtype), layer_idx
    int32 [Lt][k] and cu_seqlens int32 [R+1]."""
    seed = (wl.seed if seed is None else seed) + 7000003
    dev = torch.device(device)
    g = _gen(dev, seed)
    gc = _gen("cpu", seed + 1)
    Ls, Lt, H, d, k = wl.src_layers, wl.tgt_layers, wl.kv_heads, wl.head_dim, wl.k
    T, half = wl.ntok, wl.head_dim // 2
    pos = torch.cat([torch.arange(n, dtype=torch.float64) for n in wl.seqlens]).to(dev)

    def turned(x, theta):
        freq = theta ** (-2.0 * torch.arange(half, dtype=torch.float64) / d)
        phi = pos[:, None] * freq.to(dev)[None, :]
        c = torch.cos(phi).to(torch.float32)[:, None, :]
        s = torch.sin(phi).to(torch.float32)[:, None, :]
        x0, x1 = x[..., :half], x[..., half:]
        return torch.cat((x0 * c - x1 * s, x0 * s + x1 * c), dim=-1)

    content = torch.empty((2, Ls, T, H, d), dtype=torch.float32, device=dev)
    for s in range(Ls):
        for m in range(2):
            scale = torch.exp(torch.randn((1, H, d), generator=g, device=dev))
            if wl.outliers:
                for h in range(H):
                    ch = torch.randperm(d, generator=gc)[: wl.outliers].to(dev)
                    scale[0, h, ch] *= 10.0
            content[m, s] = torch.randn((T, H, d), generator=g, device=dev) * scale
    layer_idx = torch.stack([torch.randperm(Ls, generator=gc)[:k] for _ in range(Lt)])
    out = {}
    for m, name, theta, L in ((0, "src_k", wl.theta_src, Ls), (1, "src_v", 0, Ls)):
        t = torch.empty((L, T, H, d), dtype=wl.kv_dtype, device=dev)
        for s in range(L):
            t[s] = (turned(content[m, s], theta) if m == 0 else content[m, s]).to(wl.kv_dtype)
        out[name] = t
    std = 1.0 / math.sqrt(k * d)
    for m, name in ((0, "tgt_k"), (1, "tgt_v")):
        t = torch.empty((Lt, T, H, d), dtype=wl.kv_dtype, device=dev)
        for lt in range(Lt):
            y = 0.5 * torch.randn((T, H, d), generator=g, device=dev) * \
                torch.exp(0.5 * torch.randn((1, H, d), generator=g, device=dev))
            for s in layer_idx[lt].tolist():
                a = torch.randn((H, d, d), generator=g, device=dev) * std
                y += torch.einsum("thi,hij->thj", content[m, s], a)
            t[lt] = (turned(y, wl.theta_tgt) if m == 0 else y).to(wl.kv_dtype)
            del y
        out[name] = t
    del content
    lens = torch.tensor(wl.seqlens, dtype=torch.int64)
    cu = torch.zeros(wl.num_requests + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(lens, 0)
    out["layer_idx"] = layer_idx.to(torch.int32).to(dev)
    out["cu_seqlens"] = cu.to(torch.int32).to(dev)
    return out


def make_block_table(wl: Workload, seed: int) -> torch.Tensor:
    """Per-request block tables dealt, in request order, from a seeded random
    permutation of the shared pool of ``wl.num_blocks`` blocks; unused
    entries are -1."""
    g = _gen("cpu", seed + 2000003)
    nb = wl.blocks_per_request()
    perm = torch.randperm(wl.num_blocks, generator=g).to(torch.int32)
    table = torch.full((wl.num_requests, max(nb)), -1, dtype=torch.int32)
    at = 0
    for r, n in enumerate(nb):
        table[r, :n] = perm[at: at + n]
        at += n
    return table


def perturbed_like(x: torch.Tensor, seed: int, scale: float = 0.3) -> torch.Tensor:
    """A stand-in for the target model's own cache, to compare a mapped cache
    against: 0.9 x plus seeded Gaussian noise of `scale` times the mean |x|
    (entries that are NaN in x stay NaN), in x's dtype."""
    g = _gen(x.device, seed)
    noise = torch.randn(x.shape, generator=g, device=x.device, dtype=torch.float32)
    xf = x.float()
    return (0.9 * xf + scale * xf.abs().nanmean() * noise).to(x.dtype)


def sentinel_like(shape, dtype, device="cpu") -> torch.Tensor:
    """A destination buffer filled with an all-ones bit pattern (a NaN in
    every float format), so untouched entries can be checked bit for bit."""
    nbytes = torch.empty(0, dtype=dtype).element_size()
    int_dtype = {2: torch.int16, 4: torch.int32, 8: torch.int64}[nbytes]
    return torch.full(shape, -1, dtype=int_dtype, device=device).view(dtype)
