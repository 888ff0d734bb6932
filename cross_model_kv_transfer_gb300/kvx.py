"""ctypes binding of the kvx C ABI (``include/kvx.h``).

Argument marshalling only: the functions below have the C names and pass
device pointers straight through; every step of the transfer runs in the
CUDA kernels of ``libkvx.so``.  There is no fallback: if the library cannot
be loaded (or built with nvcc on first use), importing the symbols raises.

Low level (same names as the C ABI): ``kvx_plan_create``, ``kvx_transfer``,
``kvx_plan_destroy``, ``kvx_status_string``, ``kvx_plan_kernel``,
``kvx_plan_launches``, ``kvx_plan_cta_group``, ``kvx_transfer_static``,
``kvx_kv_diagnostics`` taking the ctypes structures ``PlanDesc`` /
``TransferArgs`` / ``DiagArgs``.

Convenience: ``Plan`` (owns a plan handle), ``Plan.transfer(...)`` which
takes torch CUDA tensors, checks their shapes, dtypes and devices, and calls
``kvx_transfer`` on the current torch stream, and ``Plan.kv_diagnostics(...)``
(fidelity statistics of a mapped cache against the target's own).
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

# --- constants mirrored from include/kvx.h ---------------------------------
KVX_OK = 0
KVX_ERR_INVALID_ARG = 1
KVX_ERR_PAIR_MISMATCH = 2
KVX_ERR_UNSUPPORTED = 3
KVX_ERR_CUDA = 4
KVX_ERR_NO_MEMORY = 5
KVX_ERR_TOO_LARGE = 6

KVX_FLAG_BAD_LAYER_INDEX = 1
KVX_FLAG_BAD_POSITION = 2
KVX_FLAG_BAD_BLOCK = 4
KVX_FLAG_BAD_ROW = 8
KVX_FLAG_TIMEOUT = 16
KVX_FLAG_BAD_SEQLENS = 32
KVX_FLAG_BAD_SRC_BLOCK = 64
KVX_FLAG_NOT_SPD = 128

KVX_F32 = 0
KVX_BF16 = 1
KVX_CONTIGUOUS = 0
KVX_PAGED = 1
KVX_KERNEL_AUTO = 0
KVX_KERNEL_SIMT = 1
KVX_KERNEL_TCGEN05 = 2
KVX_PLAN_TEST_STALL = 1
KVX_PLAN_TC_SINGLE_CTA = 2
KVX_MAPPER_PER_HEAD = 0
KVX_MAPPER_WIDE = 1

EXPORTED = ("kvx_plan_create", "kvx_transfer", "kvx_plan_destroy",
            "kvx_status_string", "kvx_plan_kernel", "kvx_plan_launches",
            "kvx_plan_cta_group", "kvx_transfer_static", "kvx_kv_diagnostics",
            "kvx_ridge_workspace_bytes", "kvx_ridge_fit",
            "kvx_layer_scores_workspace_bytes", "kvx_layer_scores")


class PlanDesc(ctypes.Structure):
    _fields_ = [
        ("src_layers", ctypes.c_int32), ("tgt_layers", ctypes.c_int32),
        ("src_kv_heads", ctypes.c_int32), ("tgt_kv_heads", ctypes.c_int32),
        ("src_head_dim", ctypes.c_int32), ("tgt_head_dim", ctypes.c_int32),
        ("k", ctypes.c_int32),
        ("rope_theta_src", ctypes.c_double), ("rope_theta_tgt", ctypes.c_double),
        ("kv_dtype", ctypes.c_int32), ("w_dtype", ctypes.c_int32), ("b_dtype", ctypes.c_int32),
        ("dst_layout", ctypes.c_int32), ("block_size", ctypes.c_int32),
        ("max_position", ctypes.c_int32), ("kernel", ctypes.c_int32),
        ("tiles_per_item", ctypes.c_int32), ("flags", ctypes.c_int32),
        ("mapper", ctypes.c_int32), ("max_tokens", ctypes.c_int32),
        ("src_layout", ctypes.c_int32), ("src_block_size", ctypes.c_int32),
    ]


class TransferArgs(ctypes.Structure):
    _fields_ = [
        ("src_k", ctypes.c_void_p), ("src_v", ctypes.c_void_p),
        ("ntok", ctypes.c_int64), ("num_requests", ctypes.c_int32),
        ("cu_seqlens", ctypes.c_void_p), ("layer_idx", ctypes.c_void_p),
        ("w", ctypes.c_void_p), ("b", ctypes.c_void_p),
        ("src_pos", ctypes.c_void_p), ("tgt_pos", ctypes.c_void_p),
        ("tgt_offset", ctypes.c_void_p),
        ("dst_k", ctypes.c_void_p), ("dst_v", ctypes.c_void_p),
        ("dst_capacity", ctypes.c_int64), ("num_blocks", ctypes.c_int64),
        ("block_table", ctypes.c_void_p), ("max_blocks_per_req", ctypes.c_int32),
        ("status", ctypes.c_void_p),
        ("src_num_blocks", ctypes.c_int64), ("src_block_table", ctypes.c_void_p),
        ("max_src_blocks_per_req", ctypes.c_int32),
    ]


class DiagArgs(ctypes.Structure):
    _fields_ = [
        ("mapped_k", ctypes.c_void_p), ("mapped_v", ctypes.c_void_p),
        ("ref_k", ctypes.c_void_p), ("ref_v", ctypes.c_void_p),
        ("ntok", ctypes.c_int64), ("num_requests", ctypes.c_int32),
        ("cu_seqlens", ctypes.c_void_p),
        ("src_pos", ctypes.c_void_p), ("tgt_pos", ctypes.c_void_p),
        ("tgt_offset", ctypes.c_void_p),
        ("dst_capacity", ctypes.c_int64), ("num_blocks", ctypes.c_int64),
        ("block_table", ctypes.c_void_p), ("max_blocks_per_req", ctypes.c_int32),
        ("stats", ctypes.c_void_p), ("status", ctypes.c_void_p),
    ]


class RidgeArgs(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("n", ctypes.c_int64),
        ("p", ctypes.c_int32), ("q", ctypes.c_int32),
        ("lambda", ctypes.c_double), ("x_dtype", ctypes.c_int32),
        ("x", ctypes.c_void_p), ("y", ctypes.c_void_p),
        ("w", ctypes.c_void_p), ("b", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("status", ctypes.c_void_p),
    ]


class ScoreArgs(ctypes.Structure):
    _fields_ = [
        ("src_k", ctypes.c_void_p), ("src_v", ctypes.c_void_p),
        ("tgt_k", ctypes.c_void_p), ("tgt_v", ctypes.c_void_p),
        ("ntok", ctypes.c_int64), ("num_requests", ctypes.c_int32),
        ("cu_seqlens", ctypes.c_void_p), ("src_pos", ctypes.c_void_p),
        ("layer_idx", ctypes.c_void_p), ("lambda", ctypes.c_double),
        ("r2", ctypes.c_void_p), ("r2_set", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("status", ctypes.c_void_p),
    ]


class FeatureArgs(ctypes.Structure):
    _fields_ = [
        ("src_k", ctypes.c_void_p), ("src_v", ctypes.c_void_p),
        ("tgt_k", ctypes.c_void_p), ("tgt_v", ctypes.c_void_p),
        ("ntok", ctypes.c_int64), ("num_requests", ctypes.c_int32),
        ("cu_seqlens", ctypes.c_void_p), ("src_pos", ctypes.c_void_p),
        ("layer_idx", ctypes.c_void_p), ("out_dtype", ctypes.c_int32),
        ("x", ctypes.c_void_p), ("y", ctypes.c_void_p),
        ("status", ctypes.c_void_p),
    ]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load():
    """Load ``libkvx.so`` (building it with nvcc if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"kvx CUDA library missing: {path}")
            lib = ctypes.CDLL(path)
            lib.kvx_plan_create.argtypes = [ctypes.POINTER(PlanDesc),
                                            ctypes.POINTER(ctypes.c_void_p)]
            lib.kvx_plan_create.restype = ctypes.c_int
            lib.kvx_transfer.argtypes = [ctypes.c_void_p, ctypes.POINTER(TransferArgs),
                                         ctypes.c_void_p]
            lib.kvx_transfer.restype = ctypes.c_int
            lib.kvx_plan_destroy.argtypes = [ctypes.c_void_p]
            lib.kvx_plan_destroy.restype = ctypes.c_int
            lib.kvx_status_string.argtypes = [ctypes.c_int]
            lib.kvx_status_string.restype = ctypes.c_char_p
            lib.kvx_plan_kernel.argtypes = [ctypes.c_void_p]
            lib.kvx_plan_kernel.restype = ctypes.c_int32
            lib.kvx_plan_launches.argtypes = [ctypes.c_void_p]
            lib.kvx_plan_launches.restype = ctypes.c_int32
            lib.kvx_plan_cta_group.argtypes = [ctypes.c_void_p]
            lib.kvx_plan_cta_group.restype = ctypes.c_int32
            lib.kvx_transfer_static.argtypes = [ctypes.POINTER(PlanDesc),
                                                ctypes.POINTER(TransferArgs), ctypes.c_void_p]
            lib.kvx_transfer_static.restype = ctypes.c_int
            lib.kvx_kv_diagnostics.argtypes = [ctypes.c_void_p, ctypes.POINTER(DiagArgs),
                                               ctypes.c_void_p]
            lib.kvx_kv_diagnostics.restype = ctypes.c_int
            lib.kvx_ridge_workspace_bytes.argtypes = [ctypes.c_int32, ctypes.c_int32,
                                                      ctypes.c_int32]
            lib.kvx_ridge_workspace_bytes.restype = ctypes.c_size_t
            lib.kvx_ridge_fit.argtypes = [ctypes.POINTER(RidgeArgs), ctypes.c_void_p]
            lib.kvx_ridge_fit.restype = ctypes.c_int
            lib.kvx_layer_scores_workspace_bytes.argtypes = [ctypes.c_void_p, ctypes.c_int64]
            lib.kvx_layer_scores_workspace_bytes.restype = ctypes.c_size_t
            lib.kvx_layer_scores.argtypes = [ctypes.c_void_p, ctypes.POINTER(ScoreArgs),
                                             ctypes.c_void_p]
            lib.kvx_layer_scores.restype = ctypes.c_int
            lib.kvx_ridge_features.argtypes = [ctypes.c_void_p, ctypes.POINTER(FeatureArgs),
                                               ctypes.c_void_p]
            lib.kvx_ridge_features.restype = ctypes.c_int
            _lib = lib
    return _lib


def kvx_plan_create(desc: PlanDesc):
    """Returns (status, plan handle or None)."""
    h = ctypes.c_void_p()
    st = load().kvx_plan_create(ctypes.byref(desc), ctypes.byref(h))
    return st, (h.value if st == KVX_OK else None)


def kvx_transfer(plan, args: TransferArgs, stream) -> int:
    return load().kvx_transfer(plan, ctypes.byref(args), stream)


def kvx_plan_destroy(plan) -> int:
    return load().kvx_plan_destroy(plan)


def kvx_status_string(status: int) -> str:
    return load().kvx_status_string(int(status)).decode()


def kvx_plan_kernel(plan) -> int:
    return load().kvx_plan_kernel(plan)


def kvx_plan_launches(plan) -> int:
    return load().kvx_plan_launches(plan)


def kvx_plan_cta_group(plan) -> int:
    return load().kvx_plan_cta_group(plan)


def kvx_transfer_static(desc: PlanDesc, args: TransferArgs, stream) -> int:
    """Allocation-free transfer (SIMT kernel, RoPE tables in the library's
    fixed device array); for callers that may not allocate device memory."""
    return load().kvx_transfer_static(ctypes.byref(desc), ctypes.byref(args), stream)


def kvx_kv_diagnostics(plan, args: DiagArgs, stream) -> int:
    return load().kvx_kv_diagnostics(plan, ctypes.byref(args), stream)


def kvx_ridge_workspace_bytes(batch: int, p: int, q: int) -> int:
    return int(load().kvx_ridge_workspace_bytes(int(batch), int(p), int(q)))


def kvx_ridge_fit(args: RidgeArgs, stream) -> int:
    return load().kvx_ridge_fit(ctypes.byref(args), stream)


def kvx_layer_scores_workspace_bytes(plan, ntok: int) -> int:
    return load().kvx_layer_scores_workspace_bytes(plan, int(ntok))


def kvx_layer_scores(plan, args: ScoreArgs, stream) -> int:
    return load().kvx_layer_scores(plan, ctypes.byref(args), stream)


def kvx_ridge_features(plan, args: FeatureArgs, stream) -> int:
    return load().kvx_ridge_features(plan, ctypes.byref(args), stream)


def ridge_fit(x, y, lam: float = 0.01, w=None, b=None, workspace=None, status=None,
              stream=None):
    """Batched ridge fit of torch CUDA tensors x [batch][n][p], y
    [batch][n][q] (fp32 or bf16, or 2-D for one fit): returns fp32 (w
    [batch][p][q], b [batch][q]), enqueued on ``stream`` (default: torch's
    current stream).  Scratch is allocated here unless ``workspace`` (a
    uint8 CUDA tensor) is given."""
    import torch
    squeeze = x.dim() == 2
    if squeeze:
        x, y = x.unsqueeze(0), y.unsqueeze(0)
    if not (x.is_cuda and y.is_cuda and x.is_contiguous() and y.is_contiguous()):
        raise ValueError("x and y must be contiguous CUDA tensors")
    if x.dtype != y.dtype:
        raise ValueError("x and y must have the same dtype")
    batch, n, p = x.shape
    if tuple(y.shape[:2]) != (batch, n):
        raise ValueError("x and y must have the same batch and observation counts")
    q = y.shape[2]
    dev = x.device
    w = torch.empty((batch, p, q), dtype=torch.float32, device=dev) if w is None else w
    b = torch.empty((batch, q), dtype=torch.float32, device=dev) if b is None else b
    need = kvx_ridge_workspace_bytes(batch, p, q)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    a = RidgeArgs(int(batch), int(n), int(p), int(q), float(lam), _dtype_code(x.dtype),
                  x.data_ptr(), y.data_ptr(), w.data_ptr(), b.data_ptr(), workspace.data_ptr(),
                  workspace.numel(), None if status is None else status.data_ptr())
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    st = kvx_ridge_fit(a, ctypes.c_void_p(stream.cuda_stream))
    if st != KVX_OK:
        raise KvxError(st, "kvx_ridge_fit")
    return (w[0], b[0]) if squeeze else (w, b)


class KvxError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {kvx_status_string(status)} (status {status})")
        self.status = status


def _dtype_code(dt) -> int:
    import torch
    if dt == torch.float32:
        return KVX_F32
    if dt == torch.bfloat16:
        return KVX_BF16
    raise ValueError(f"unsupported dtype {dt}")


class Plan:
    """A kvx plan for one (source, target) model pair on the current device."""

    def __init__(self, *, src_layers, tgt_layers, kv_heads, head_dim, k, rope_theta_src,
                 rope_theta_tgt, max_position, kv_dtype, w_dtype, b_dtype,
                 layout=KVX_CONTIGUOUS, block_size=0, kernel=KVX_KERNEL_AUTO,
                 tgt_kv_heads=None, tgt_head_dim=None, tiles_per_item=0, flags=0,
                 mapper=KVX_MAPPER_PER_HEAD, max_tokens=0, src_layout=KVX_CONTIGUOUS,
                 src_block_size=0):
        self.desc = PlanDesc(
            src_layers, tgt_layers, kv_heads,
            kv_heads if tgt_kv_heads is None else tgt_kv_heads,
            head_dim, head_dim if tgt_head_dim is None else tgt_head_dim, k,
            float(rope_theta_src), float(rope_theta_tgt),
            _dtype_code(kv_dtype), _dtype_code(w_dtype), _dtype_code(b_dtype),
            int(layout), int(block_size), int(max_position), int(kernel),
            int(tiles_per_item), int(flags), int(mapper), int(max_tokens), int(src_layout),
            int(src_block_size))
        self.kv_dtype, self.w_dtype, self.b_dtype = kv_dtype, w_dtype, b_dtype
        st, h = kvx_plan_create(self.desc)
        if st != KVX_OK:
            raise KvxError(st, "kvx_plan_create")
        self.handle = h

    @property
    def kernel(self) -> int:
        return kvx_plan_kernel(self.handle)

    @property
    def cta_group(self) -> int:
        return kvx_plan_cta_group(self.handle)

    @property
    def launches_per_transfer(self) -> int:
        return kvx_plan_launches(self.handle)

    def close(self):
        if getattr(self, "handle", None):
            kvx_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def make_args(self, *, src_k, src_v, layer_idx, w, b, dst_k, dst_v, cu_seqlens=None,
                  src_pos=None, tgt_pos=None, tgt_offset=None,
                  dst_capacity=None, num_blocks=None, block_table=None,
                  status=None, ntok=None, src_block_table=None) -> TransferArgs:
        """Check tensors against the plan and pack a ``TransferArgs``.  A
        paged source ([Ls][src_num_blocks*src_block_size][H][d]) needs
        ``src_block_table`` [R][max] and ``ntok`` (the packed token count)."""
        import torch
        d = self.desc
        Ls, Lt, H, hd, k = d.src_layers, d.tgt_layers, d.src_kv_heads, d.src_head_dim, d.k

        def ptr(t, name, dtype, shape=None, ndim=None):
            if t is None:
                return None
            if not isinstance(t, torch.Tensor) or not t.is_cuda:
                raise ValueError(f"{name} must be a CUDA tensor")
            if t.dtype != dtype:
                raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
            if not t.is_contiguous():
                raise ValueError(f"{name} must be contiguous")
            if shape is not None and tuple(t.shape) != tuple(shape):
                raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
            if ndim is not None and t.dim() != ndim:
                raise ValueError(f"{name} must have {ndim} dims")
            return t.data_ptr()

        R = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
        a = TransferArgs()
        if d.src_layout == KVX_PAGED:
            if ntok is None or src_block_table is None:
                raise ValueError("a paged source needs ntok and src_block_table")
            src_rows = src_k.shape[1]
            if src_rows % d.src_block_size:
                raise ValueError("source rows must be whole blocks")
            a.src_num_blocks = src_rows // d.src_block_size
            a.src_block_table = ptr(src_block_table, "src_block_table", torch.int32, ndim=2)
            a.max_src_blocks_per_req = int(src_block_table.shape[1])
        else:
            ntok = src_k.shape[1] if ntok is None else int(ntok)
            src_rows = ntok
        a.src_k = ptr(src_k, "src_k", self.kv_dtype, (Ls, src_rows, H, hd))
        a.src_v = ptr(src_v, "src_v", self.kv_dtype, (Ls, src_rows, H, hd))
        a.ntok = ntok
        a.num_requests = R
        a.cu_seqlens = ptr(cu_seqlens, "cu_seqlens", torch.int32, (R + 1,))
        a.layer_idx = ptr(layer_idx, "layer_idx", torch.int32, (Lt, k))
        if d.mapper == KVX_MAPPER_WIDE:
            a.w = ptr(w, "w", self.w_dtype, (Lt, k * 2 * H * hd, H * 2 * hd))
        else:
            a.w = ptr(w, "w", self.w_dtype, (Lt, H, 2, k * hd, hd))
        a.b = ptr(b, "b", self.b_dtype, (Lt, H, 2, hd))
        a.src_pos = ptr(src_pos, "src_pos", torch.int32, (ntok,))
        a.tgt_pos = ptr(tgt_pos, "tgt_pos", torch.int32, (ntok,))
        a.tgt_offset = ptr(tgt_offset, "tgt_offset", torch.int32, (R,))
        if d.dst_layout == KVX_CONTIGUOUS:
            cap = int(dst_capacity) if dst_capacity is not None else dst_k.shape[1] // R
            rows = R * cap
            a.dst_capacity = cap
        else:
            nb = int(num_blocks) if num_blocks is not None else dst_k.shape[1] // d.block_size
            rows = nb * d.block_size
            a.num_blocks = nb
            a.block_table = ptr(block_table, "block_table", torch.int32, ndim=2)
            a.max_blocks_per_req = int(block_table.shape[1])
        a.dst_k = ptr(dst_k, "dst_k", self.kv_dtype, (Lt, rows, H, hd))
        a.dst_v = ptr(dst_v, "dst_v", self.kv_dtype, (Lt, rows, H, hd))
        a.status = ptr(status, "status", torch.int32, (1,))
        a._keep = (src_k, src_v, cu_seqlens, layer_idx, w, b, src_pos, tgt_pos, tgt_offset,
                   dst_k, dst_v, block_table, status, src_block_table)
        return a

    def transfer(self, stream=None, **tensors) -> None:
        """Enqueue one transfer on ``stream`` (default: torch's current stream)."""
        import torch
        args = self.make_args(**tensors)
        if stream is None:
            stream = torch.cuda.current_stream()
        st = kvx_transfer(self.handle, args, ctypes.c_void_p(stream.cuda_stream))
        if st != KVX_OK:
            raise KvxError(st, "kvx_transfer")

    def make_diag_args(self, *, mapped_k, mapped_v, ref_k, ref_v, stats, ntok, cu_seqlens=None,
                       src_pos=None, tgt_pos=None, tgt_offset=None, dst_capacity=None,
                       num_blocks=None, block_table=None, status=None) -> DiagArgs:
        """Check tensors against the plan and pack a ``DiagArgs``."""
        import torch
        d = self.desc
        Lt, H, hd = d.tgt_layers, d.tgt_kv_heads, d.tgt_head_dim
        R = 1 if cu_seqlens is None else cu_seqlens.numel() - 1

        def ptr(t, name, dtype, shape=None, ndim=None):
            if t is None:
                return None
            if not isinstance(t, torch.Tensor) or not t.is_cuda:
                raise ValueError(f"{name} must be a CUDA tensor")
            if t.dtype != dtype:
                raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
            if not t.is_contiguous():
                raise ValueError(f"{name} must be contiguous")
            if shape is not None and tuple(t.shape) != tuple(shape):
                raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
            if ndim is not None and t.dim() != ndim:
                raise ValueError(f"{name} must have {ndim} dims")
            return t.data_ptr()

        a = DiagArgs()
        a.ntok = int(ntok)
        a.num_requests = R
        a.cu_seqlens = ptr(cu_seqlens, "cu_seqlens", torch.int32, (R + 1,))
        a.src_pos = ptr(src_pos, "src_pos", torch.int32, (int(ntok),))
        a.tgt_pos = ptr(tgt_pos, "tgt_pos", torch.int32, (int(ntok),))
        a.tgt_offset = ptr(tgt_offset, "tgt_offset", torch.int32, (R,))
        if d.dst_layout == KVX_CONTIGUOUS:
            cap = int(dst_capacity) if dst_capacity is not None else ref_k.shape[1] // R
            rows = R * cap
            a.dst_capacity = cap
        else:
            nb = int(num_blocks) if num_blocks is not None else ref_k.shape[1] // d.block_size
            rows = nb * d.block_size
            a.num_blocks = nb
            a.block_table = ptr(block_table, "block_table", torch.int32, ndim=2)
            a.max_blocks_per_req = int(block_table.shape[1])
        shape = (Lt, rows, H, hd)
        a.mapped_k = ptr(mapped_k, "mapped_k", self.kv_dtype, shape)
        a.mapped_v = ptr(mapped_v, "mapped_v", self.kv_dtype, shape)
        a.ref_k = ptr(ref_k, "ref_k", self.kv_dtype, shape)
        a.ref_v = ptr(ref_v, "ref_v", self.kv_dtype, shape)
        a.stats = ptr(stats, "stats", torch.float64, (Lt, H, 2, hd + 4))
        a.status = ptr(status, "status", torch.int32, (1,))
        a._keep = (mapped_k, mapped_v, ref_k, ref_v, stats, cu_seqlens, src_pos, tgt_pos,
                   tgt_offset, block_table, status)
        return a

    def layer_scores(self, *, src_k, src_v, tgt_k, tgt_v, lam=0.01, cu_seqlens=None,
                     src_pos=None, layer_idx=None, r2=None, r2_set=None, workspace=None,
                     status=None, stream=None):
        """Layer-selection scores (``kvx_layer_scores``) of CUDA tensors:
        src_k / src_v [Ls][ntok][H][d] and tgt_k / tgt_v [Lt][ntok][H][d] of
        the same tokens; returns fp64 r2 [Lt][Ls][H][2] and, with
        ``layer_idx`` [Lt][k], r2_set [Lt][H][2] (else None), enqueued on
        ``stream``.  Scratch is allocated here unless ``workspace`` (a uint8
        CUDA tensor) is given."""
        import torch
        d = self.desc
        Ls, Lt, H, hd = d.src_layers, d.tgt_layers, d.src_kv_heads, d.src_head_dim
        for name, t, L in (("src_k", src_k, Ls), ("src_v", src_v, Ls), ("tgt_k", tgt_k, Lt),
                           ("tgt_v", tgt_v, Lt)):
            if not (isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous()):
                raise ValueError(f"{name} must be a contiguous CUDA tensor")
            if t.dtype != self.kv_dtype or t.dim() != 4 or t.shape[0] != L or \
                    tuple(t.shape[2:]) != (H, hd):
                raise ValueError(f"{name}: expected [{L}][ntok][{H}][{hd}] {self.kv_dtype}")
        ntok = src_k.shape[1]
        if any(t.shape[1] != ntok for t in (src_v, tgt_k, tgt_v)):
            raise ValueError("the four caches must hold the same tokens")
        dev = src_k.device
        R = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
        r2 = torch.empty((Lt, Ls, H, 2), dtype=torch.float64, device=dev) if r2 is None else r2
        if layer_idx is not None and r2_set is None:
            r2_set = torch.empty((Lt, H, 2), dtype=torch.float64, device=dev)
        need = kvx_layer_scores_workspace_bytes(self.handle, ntok)
        if need == 0:
            raise KvxError(KVX_ERR_UNSUPPORTED, "kvx_layer_scores_workspace_bytes")
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        ptr = lambda t: None if t is None else t.data_ptr()
        for name, t, shape in (("cu_seqlens", cu_seqlens, (R + 1,)), ("src_pos", src_pos, (ntok,)),
                               ("layer_idx", layer_idx, (Lt, d.k))):
            if t is not None and (t.dtype != torch.int32 or tuple(t.shape) != shape or
                                  not t.is_cuda or not t.is_contiguous()):
                raise ValueError(f"{name} must be a contiguous int32 CUDA tensor {shape}")
        a = ScoreArgs(src_k.data_ptr(), src_v.data_ptr(), tgt_k.data_ptr(), tgt_v.data_ptr(),
                      int(ntok), int(R), ptr(cu_seqlens), ptr(src_pos), ptr(layer_idx),
                      float(lam), r2.data_ptr(), ptr(r2_set), workspace.data_ptr(),
                      workspace.numel(), ptr(status))
        if stream is None:
            stream = torch.cuda.current_stream(dev)
        st = kvx_layer_scores(self.handle, a, ctypes.c_void_p(stream.cuda_stream))
        if st != KVX_OK:
            raise KvxError(st, "kvx_layer_scores")
        return r2, r2_set

    def ridge_features(self, *, src_k, src_v, layer_idx, tgt_k=None, tgt_v=None,
                       cu_seqlens=None, src_pos=None, out_dtype=None, x=None, y=None,
                       status=None, stream=None):
        """Content-space observations of the maps' ridge fits
        (``kvx_ridge_features``) from CUDA caches src_k / src_v
        [Ls][ntok][H][d] and, for y, tgt_k / tgt_v [Lt][ntok][H][d] of the
        same tokens: returns x [Lt*H*2][ntok][k*d] and y [Lt*H*2][ntok][d]
        (None without the target caches) in ``out_dtype`` (default fp32),
        enqueued on ``stream`` -- the x and y of one ``ridge_fit`` whose W
        and b this plan's transfer reads."""
        import torch
        d = self.desc
        Ls, Lt, H, hd, k = d.src_layers, d.tgt_layers, d.src_kv_heads, d.src_head_dim, d.k
        if layer_idx is None:
            raise ValueError("layer_idx [Lt][k] is required")
        with_y = tgt_k is not None or tgt_v is not None
        caches = [("src_k", src_k, Ls), ("src_v", src_v, Ls)]
        if with_y:
            caches += [("tgt_k", tgt_k, Lt), ("tgt_v", tgt_v, Lt)]
        for name, t, L in caches:
            if not (isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous()):
                raise ValueError(f"{name} must be a contiguous CUDA tensor")
            if t.dtype != self.kv_dtype or t.dim() != 4 or t.shape[0] != L or \
                    tuple(t.shape[2:]) != (H, hd):
                raise ValueError(f"{name}: expected [{L}][ntok][{H}][{hd}] {self.kv_dtype}")
        ntok = src_k.shape[1]
        if any(t.shape[1] != ntok for _, t, _ in caches):
            raise ValueError("the caches must hold the same tokens")
        R = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
        for name, t, shape in (("cu_seqlens", cu_seqlens, (R + 1,)), ("src_pos", src_pos, (ntok,)),
                               ("layer_idx", layer_idx, (Lt, k))):
            if t is not None and (t.dtype != torch.int32 or tuple(t.shape) != shape or
                                  not t.is_cuda or not t.is_contiguous()):
                raise ValueError(f"{name} must be a contiguous int32 CUDA tensor {shape}")
        out_dtype = torch.float32 if out_dtype is None else out_dtype
        dev = src_k.device
        B = Lt * H * 2
        for name, t, shape in (("x", x, (B, ntok, k * hd)), ("y", y, (B, ntok, hd))):
            if t is not None and (t.dtype != out_dtype or tuple(t.shape) != shape or
                                  not t.is_cuda or not t.is_contiguous()):
                raise ValueError(f"{name} must be a contiguous {out_dtype} CUDA tensor {shape}")
        if x is None:
            x = torch.empty((B, ntok, k * hd), dtype=out_dtype, device=dev)
        if with_y and y is None:
            y = torch.empty((B, ntok, hd), dtype=out_dtype, device=dev)
        ptr = lambda t: None if t is None else t.data_ptr()
        a = FeatureArgs(src_k.data_ptr(), src_v.data_ptr(), ptr(tgt_k), ptr(tgt_v), int(ntok),
                        int(R), ptr(cu_seqlens), ptr(src_pos), layer_idx.data_ptr(),
                        _dtype_code(out_dtype), x.data_ptr(), ptr(y if with_y else None),
                        ptr(status))
        if stream is None:
            stream = torch.cuda.current_stream(dev)
        st = kvx_ridge_features(self.handle, a, ctypes.c_void_p(stream.cuda_stream))
        if st != KVX_OK:
            raise KvxError(st, "kvx_ridge_features")
        return x, (y if with_y else None)

    def kv_diagnostics(self, stream=None, **tensors) -> None:
        """Enqueue the fidelity statistics [Lt][H][2][d + 4] (fp64, into
        ``stats``) of a mapped cache against the target's own cache on
        ``stream`` (default: torch's current stream)."""
        import torch
        args = self.make_diag_args(**tensors)
        if stream is None:
            stream = torch.cuda.current_stream()
        st = kvx_kv_diagnostics(self.handle, args, ctypes.c_void_p(stream.cuda_stream))
        if st != KVX_OK:
            raise KvxError(st, "kvx_kv_diagnostics")
