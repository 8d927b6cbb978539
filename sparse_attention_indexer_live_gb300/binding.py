"""Thin ctypes binding of libdsa_select.so (include/dsa_select.h).

Argument marshalling only: torch tensors are turned into device pointers, the
current CUDA stream is passed along, and a non-zero status becomes an
exception.  Every step of the selection path runs in the library's kernels;
there is no fallback of any kind -- if the library is missing, loading fails.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB_PATH

DSA_OK, DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED, DSA_ERR_CUDA, DSA_ERR_TIMEOUT = 0, 1, 2, 3, 4


class dsa_select_cfg(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("width", ctypes.c_int64), ("row_stride", ctypes.c_int64),
                ("col_stride", ctypes.c_int64), ("block_topk", ctypes.c_int32),
                ("row_topk", ctypes.c_int32), ("row_repeat", ctypes.c_int32),
                ("repeat_causal", ctypes.c_int32), ("has_starts", ctypes.c_int32),
                ("split", ctypes.c_int32)]


class dsa_plan_desc(ctypes.Structure):
    _fields_ = [("threads", ctypes.c_int32), ("sm_count", ctypes.c_int32),
                ("nblocks", ctypes.c_int64), ("vector_path", ctypes.c_int32),
                ("stream_capacity", ctypes.c_int32), ("per_round", ctypes.c_int32),
                ("candidate_capacity", ctypes.c_int32), ("smem_select", ctypes.c_int64),
                ("smem_topk_cand", ctypes.c_int64), ("smem_topk_scan", ctypes.c_int64),
                ("ctas_per_sm_select", ctypes.c_int32), ("grid_select", ctypes.c_int32),
                ("split", ctypes.c_int32), ("parts", ctypes.c_int32)]


EXPORTS = ("dsa_select_init", "dsa_select_destroy", "dsa_plan_describe", "dsa_candidate_select",
           "dsa_row_topk", "dsa_select_topk", "dsa_combine_window", "dsa_indexer_logits",
           "dsa_indexer_status", "dsa_indexer_select_workspace", "dsa_indexer_select",
           "dsa_indexer_select_noalloc", "dsa_sparse_attention_workspace", "dsa_group_union",
           "dsa_sparse_attention", "dsa_sparse_attention_ranges_workspace", "dsa_group_union_ranges",
           "dsa_sparse_attention_ranges", "dsa_sparse_attention_status", "dsa_status_string")

# Size of the library's fixed scratch array used by dsa_indexer_select_noalloc
# (DSA_NOALLOC_SCRATCH_BYTES in include/dsa_select.h).
NOALLOC_SCRATCH_BYTES = 8 << 20


class dsa_indexer_cfg(ctypes.Structure):
    _fields_ = [("queries", ctypes.c_int32), ("keys", ctypes.c_int32), ("heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("out_stride", ctypes.c_int64)]

class dsa_attention_cfg(ctypes.Structure):
    _fields_ = [("tokens", ctypes.c_int32), ("heads", ctypes.c_int32), ("keys", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("value_dim", ctypes.c_int32), ("select", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()


class DsaSelectError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def load(path: str | None = None):
    """Load the CUDA library (raises OSError when it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise OSError(f"libdsa_select.so not built at {p}; run "
                              "sparse_attention_indexer_live_gb300.build.build()")
            L = ctypes.CDLL(p)
            vp, i32 = ctypes.c_void_p, ctypes.c_int
            L.dsa_select_init.restype = i32
            L.dsa_select_init.argtypes = [ctypes.POINTER(dsa_select_cfg), i32,
                                          ctypes.POINTER(vp), ctypes.POINTER(ctypes.c_size_t)]
            L.dsa_select_destroy.restype = None
            L.dsa_select_destroy.argtypes = [vp]
            L.dsa_plan_describe.restype = i32
            L.dsa_plan_describe.argtypes = [vp, ctypes.POINTER(dsa_plan_desc)]
            L.dsa_candidate_select.restype = i32
            L.dsa_candidate_select.argtypes = [vp, vp, vp, vp, vp, vp, vp]
            L.dsa_row_topk.restype = i32
            L.dsa_row_topk.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
            L.dsa_select_topk.restype = i32
            L.dsa_select_topk.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
            L.dsa_combine_window.restype = i32
            L.dsa_combine_window.argtypes = [vp, vp, vp, vp, ctypes.c_int32, vp, vp]
            L.dsa_indexer_logits.restype = i32
            L.dsa_indexer_logits.argtypes = [ctypes.POINTER(dsa_indexer_cfg), vp, vp, vp, vp, vp,
                                             vp, vp, vp]
            L.dsa_indexer_status.restype = i32
            L.dsa_indexer_status.argtypes = []
            L.dsa_indexer_select_workspace.restype = i32
            L.dsa_indexer_select_workspace.argtypes = [vp, ctypes.POINTER(ctypes.c_size_t)]
            L.dsa_indexer_select.restype = i32
            L.dsa_indexer_select.argtypes = [vp, ctypes.POINTER(dsa_indexer_cfg), vp, vp, vp, vp,
                                             vp, vp, ctypes.c_size_t, vp, vp, vp]
            L.dsa_sparse_attention_workspace.restype = i32
            L.dsa_sparse_attention_workspace.argtypes = [ctypes.POINTER(dsa_attention_cfg),
                                                         ctypes.POINTER(ctypes.c_size_t)]
            L.dsa_group_union.restype = i32
            L.dsa_group_union.argtypes = [ctypes.POINTER(dsa_attention_cfg), vp, vp, ctypes.c_size_t, vp]
            L.dsa_sparse_attention.restype = i32
            L.dsa_sparse_attention.argtypes = [ctypes.POINTER(dsa_attention_cfg), vp, vp, vp, vp,
                                               ctypes.c_float, vp, ctypes.c_size_t, vp, vp, vp]
            L.dsa_sparse_attention_ranges_workspace.restype = i32
            L.dsa_sparse_attention_ranges_workspace.argtypes = [ctypes.POINTER(dsa_attention_cfg), i32,
                                                                ctypes.POINTER(ctypes.c_size_t)]
            L.dsa_group_union_ranges.restype = i32
            L.dsa_group_union_ranges.argtypes = [ctypes.POINTER(dsa_attention_cfg), vp, i32, vp,
                                                 ctypes.c_size_t, vp]
            L.dsa_sparse_attention_ranges.restype = i32
            L.dsa_sparse_attention_ranges.argtypes = [ctypes.POINTER(dsa_attention_cfg), vp, vp, vp, vp, i32,
                                                      ctypes.c_float, vp, ctypes.c_size_t, vp, vp, vp]
            L.dsa_sparse_attention_status.restype = i32
            L.dsa_sparse_attention_status.argtypes = []
            L.dsa_indexer_select_noalloc.restype = i32
            L.dsa_indexer_select_noalloc.argtypes = [vp, ctypes.POINTER(dsa_indexer_cfg), vp, vp, vp,
                                                     vp, vp, vp, vp, vp]
            L.dsa_status_string.restype = ctypes.c_char_p
            L.dsa_status_string.argtypes = [i32]
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return load().dsa_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != DSA_OK:
        raise DsaSelectError(status, where)


class Plan:
    """A plan for one call-site shape (dsa_select_init)."""

    def __init__(self, cfg: dsa_select_cfg, device: int):
        L = load()
        self._h = ctypes.c_void_p()
        ws = ctypes.c_size_t(0)
        _check(L.dsa_select_init(ctypes.byref(cfg), int(device), ctypes.byref(self._h),
                                 ctypes.byref(ws)), "dsa_select_init")
        self.cfg = cfg
        self.device = int(device)
        self.workspace_bytes = ws.value

    @property
    def handle(self):
        return self._h

    def describe(self) -> dict:
        d = dsa_plan_desc()
        _check(load().dsa_plan_describe(self._h, ctypes.byref(d)), "dsa_plan_describe")
        return {name: getattr(d, name) for name, _ in d._fields_}

    def close(self):
        if self._h:
            load().dsa_select_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def make_cfg(*, rows, width, block_size, block_topk, row_topk, row_stride=None, col_stride=1,
             row_repeat=1, repeat_causal=True, has_starts=False, split=0) -> dsa_select_cfg:
    if row_stride is None:
        row_stride = width * col_stride
    return dsa_select_cfg(rows=rows, block_size=block_size, width=width, row_stride=row_stride,
                          col_stride=col_stride, block_topk=block_topk, row_topk=row_topk,
                          row_repeat=row_repeat, repeat_causal=int(bool(repeat_causal)),
                          has_starts=int(bool(has_starts)), split=int(split))


def dsa_select_init(cfg: dsa_select_cfg | None = None, device: int = 0, **shape) -> Plan:
    """Plan for a shape given as a dsa_select_cfg or as keyword arguments
    (rows, width, block_size, block_topk, row_topk, row_stride, col_stride,
    row_repeat, repeat_causal, has_starts, split)."""
    if cfg is None:
        cfg = make_cfg(**shape)
    return Plan(cfg, device)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


# Argument checks.  The C ABI sees only pointers, so a tensor of the wrong
# type, device or size would reach the kernels as an out-of-bounds access;
# every check below raises (TypeError for a wrong type or dtype, ValueError
# for a wrong device, layout or size) and none of them is an `assert`, so
# they stay in force under `python -O`.

def _tensor(name, t, dtypes, *, numel=0, contiguous=True, device=None):
    """Check one tensor argument: a torch.Tensor of one of `dtypes`, on a CUDA
    device (`device`, when given, is the required device index), contiguous
    unless `contiguous` is False, with at least `numel` elements."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor, got {type(t).__name__}")
    if t.dtype not in dtypes:
        want = " or ".join(str(d) for d in dtypes)
        raise TypeError(f"{name}: dtype {t.dtype}, expected {want}")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor (got device {t.device})")
    if device is not None and t.device.index != device:
        raise ValueError(f"{name}: on cuda:{t.device.index}, the plan is for cuda:{device}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if t.numel() < numel:
        raise ValueError(f"{name}: {t.numel()} elements, at least {numel} needed")
    return t


def _i32(name, t, numel, device=None):
    import torch
    return _tensor(name, t, (torch.int32,), numel=numel, device=device)


def _check_tensors(plan: Plan, logits, starts, ends, outs):
    import torch
    c = plan.cfg
    _tensor("logits", logits, (torch.float32,), contiguous=False, device=plan.device)
    if logits.dim() == 2 and logits.shape[1] == c.width:
        if logits.shape[0] != c.rows:
            raise ValueError(f"logits: {logits.shape[0]} rows, the plan has {c.rows}")
        if (c.rows > 1 and logits.stride(0) != c.row_stride) or logits.stride(1) != c.col_stride:
            raise ValueError(f"logits: strides {tuple(logits.stride())} do not match the plan's "
                             f"({c.row_stride}, {c.col_stride})")
    else:
        need = (c.rows - 1) * c.row_stride + (c.width - 1) * c.col_stride + 1 if c.rows else 0
        if not logits.is_contiguous():
            raise ValueError("logits: a flat logits buffer must be contiguous")
        if logits.numel() < need:
            raise ValueError(f"logits: {logits.numel()} elements, the plan reaches {need}")
    nq = -(-c.rows // c.row_repeat)
    _i32("ends", ends, nq, plan.device)
    if c.has_starts:
        if starts is None:
            raise ValueError("starts: the plan was made with starts")
        _i32("starts", starts, nq, plan.device)
    elif starts is not None:
        raise ValueError("starts: the plan was made without starts")
    for name, t, cols in outs:
        if t is not None:
            _i32(name, t, c.rows * cols, plan.device)


def dsa_candidate_select(plan: Plan, logits, starts, ends, cand, stream=None):
    """Steps 1-4 in place on `logits`; cand [rows, Kb + 1] int32."""
    _check_tensors(plan, logits, starts, ends, [("cand", cand, plan.cfg.block_topk + 1)])
    _check(load().dsa_candidate_select(plan.handle, _ptr(logits), _ptr(starts), _ptr(ends),
                                       _ptr(cand), None, _stream(stream)),
           "dsa_candidate_select")


def dsa_row_topk(plan: Plan, logits, starts, ends, cand, topk, stream=None):
    """Step 5: topk [rows, K] int32; cand=None scans the live span."""
    _check_tensors(plan, logits, starts, ends, [("cand", cand, plan.cfg.block_topk + 1),
                                                ("topk", topk, plan.cfg.row_topk)])
    _check(load().dsa_row_topk(plan.handle, _ptr(logits), _ptr(starts), _ptr(ends), _ptr(cand),
                               _ptr(topk), None, _stream(stream)), "dsa_row_topk")


def dsa_select_topk(plan: Plan, logits, starts, ends, cand, topk, stream=None):
    """Steps 1-5 fused in one launch."""
    _check_tensors(plan, logits, starts, ends, [("cand", cand, plan.cfg.block_topk + 1),
                                                ("topk", topk, plan.cfg.row_topk)])
    _check(load().dsa_select_topk(plan.handle, _ptr(logits), _ptr(starts), _ptr(ends),
                                  _ptr(cand), _ptr(topk), None, _stream(stream)),
           "dsa_select_topk")


def dsa_combine_window(plan: Plan, starts, ends, topk, window: int, out, stream=None):
    """Union of each row's top-k and the last `window` live columns into
    out [rows, K + window] int32 (ascending, -1 padded)."""
    c = plan.cfg
    if int(window) < 0:
        raise ValueError(f"window: {window} is negative")
    nq = -(-c.rows // c.row_repeat)
    _i32("ends", ends, nq, plan.device)
    if c.has_starts:
        if starts is None:
            raise ValueError("starts: the plan was made with starts")
        _i32("starts", starts, nq, plan.device)
    elif starts is not None:
        raise ValueError("starts: the plan was made without starts")
    _i32("topk", topk, c.rows * c.row_topk, plan.device)
    _i32("out", out, c.rows * (c.row_topk + int(window)), plan.device)
    _check(load().dsa_combine_window(plan.handle, _ptr(starts), _ptr(ends), _ptr(topk),
                                     int(window), _ptr(out), _stream(stream)),
           "dsa_combine_window")


def _indexer_args(q, k, k_scale, w, ends, device=None):
    """Check the producer's inputs; returns (T, H, D, S)."""
    import torch
    _tensor("q", q, (torch.uint8,), device=device)
    if q.dim() != 3:
        raise ValueError(f"q: shape {tuple(q.shape)}, expected [queries, heads, head_dim]")
    T, H, D = q.shape
    dev = q.device.index
    _tensor("k", k, (torch.uint8,), device=dev)
    if k.dim() != 2 or k.shape[1] != D:
        raise ValueError(f"k: shape {tuple(k.shape)}, expected [keys, {D}] (q's head_dim)")
    S = k.shape[0]
    _tensor("k_scale", k_scale, (torch.float32,), numel=S, device=dev)
    _tensor("w", w, (torch.float32,), numel=T * H, device=dev)
    _i32("ends", ends, T, dev)
    return T, H, D, S


def dsa_indexer_logits(q, k, k_scale, w, starts, ends, logits, stream=None):
    """Indexer logits on the tensor cores: q [T, 64, 128] and k [S, 128] as
    uint8 e4m3 bytes, k_scale [S] f32, w [T, 64] f32, bounds [T] int32,
    logits [T, ld] f32 written over each query's live span."""
    import torch
    T, H, D, S = _indexer_args(q, k, k_scale, w, ends)
    dev = q.device.index
    if starts is not None:
        _i32("starts", starts, T, dev)
    _tensor("logits", logits, (torch.float32,), contiguous=False, device=dev)
    if logits.dim() != 2 or logits.stride(1) != 1 or logits.shape[0] != T or logits.shape[1] < S:
        raise ValueError(f"logits: shape {tuple(logits.shape)} strides {tuple(logits.stride())}, "
                         f"expected [{T}, >= {S}] with unit column stride")
    cfg = dsa_indexer_cfg(queries=T, keys=S, heads=H, head_dim=D, out_stride=logits.stride(0))
    _check(load().dsa_indexer_logits(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(k_scale), _ptr(w),
                                     _ptr(starts), _ptr(ends), _ptr(logits), _stream(stream)),
           "dsa_indexer_logits")


def dsa_indexer_select_workspace(plan: Plan) -> int:
    """Workspace bytes dsa_indexer_select needs for this plan."""
    n = ctypes.c_size_t(0)
    _check(load().dsa_indexer_select_workspace(plan.handle, ctypes.byref(n)),
           "dsa_indexer_select_workspace")
    return int(n.value)


def _fused_args(plan: Plan, q, k, k_scale, w, ends, cand, topk):
    T, H, D, S = _indexer_args(q, k, k_scale, w, ends, plan.device)
    c = plan.cfg
    if T != c.rows or S != c.width:
        raise ValueError(f"q / k: {T} queries x {S} keys, the plan is {c.rows} rows x {c.width}")
    _i32("cand", cand, c.rows * (c.block_topk + 1), plan.device)
    _i32("topk", topk, c.rows * c.row_topk, plan.device)
    return dsa_indexer_cfg(queries=T, keys=S, heads=H, head_dim=D, out_stride=S)


def dsa_indexer_select(plan: Plan, q, k, k_scale, w, ends, workspace, cand, topk, stream=None):
    """The indexer logits fused with the selection (never materialised):
    q [T, 64, 128] and k [S, 128] uint8 e4m3 bytes, k_scale [S] f32, w [T, 64]
    f32, ends [T] int32; workspace a CUDA uint8 tensor of at least
    dsa_indexer_select_workspace(plan) bytes; cand [T, Kb + 1], topk [T, K]."""
    import torch
    cfg = _fused_args(plan, q, k, k_scale, w, ends, cand, topk)
    _tensor("workspace", workspace, (torch.uint8,), device=plan.device)
    _check(load().dsa_indexer_select(plan.handle, ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(k_scale),
                                     _ptr(w), _ptr(ends), _ptr(workspace), workspace.numel(),
                                     _ptr(cand), _ptr(topk), _stream(stream)),
           "dsa_indexer_select")


def dsa_indexer_select_noalloc(plan: Plan, q, k, k_scale, w, ends, cand, topk, stream=None):
    """dsa_indexer_select for callers that cannot allocate device memory at
    call time (an engine whose pool already owns the free memory, a plugin
    under a host framework's allocator, C code with no allocator): the
    per-query records go to a fixed 8 MiB array inside the library, so no
    workspace is passed and nothing is allocated.  Batches whose workspace
    (dsa_indexer_select_workspace) exceeds that array are refused.  All calls
    on a device share the array: keep them ordered (one stream), and make the
    first call on a device before any stream capture."""
    cfg = _fused_args(plan, q, k, k_scale, w, ends, cand, topk)
    _check(load().dsa_indexer_select_noalloc(plan.handle, ctypes.byref(cfg), _ptr(q), _ptr(k),
                                             _ptr(k_scale), _ptr(w), _ptr(ends), _ptr(cand),
                                             _ptr(topk), _stream(stream)),
           f"dsa_indexer_select_noalloc (fixed scratch of {NOALLOC_SCRATCH_BYTES} bytes)")


def attention_cfg(q, k, idx) -> dsa_attention_cfg:
    T, H, D = q.shape
    return dsa_attention_cfg(tokens=T, heads=H, keys=k.shape[0], head_dim=D, value_dim=D,
                             select=idx.shape[1])


def dsa_sparse_attention_workspace(cfg: dsa_attention_cfg) -> int:
    n = ctypes.c_size_t(0)
    _check(load().dsa_sparse_attention_workspace(ctypes.byref(cfg), ctypes.byref(n)),
           "dsa_sparse_attention_workspace")
    return int(n.value)


def _attention_idx(cfg: dsa_attention_cfg, idx, workspace):
    import torch
    _i32("idx", idx, max(cfg.tokens, 0) * max(cfg.select, 0))
    _tensor("workspace", workspace, (torch.uint8,), device=idx.device.index)


def dsa_group_union(cfg: dsa_attention_cfg, idx, workspace, stream=None):
    """The unions of each group's selections and their token masks, written
    to workspace (layout in include/dsa_select.h)."""
    _attention_idx(cfg, idx, workspace)
    _check(load().dsa_group_union(ctypes.byref(cfg), _ptr(idx), _ptr(workspace), workspace.numel(),
                                  _stream(stream)), "dsa_group_union")


def dsa_sparse_attention(cfg: dsa_attention_cfg, q, k, v, idx, scale: float, workspace, o, lse,
                         stream=None):
    """Grouped masked sparse attention: q [T, H, 128], k / v [S, 128] as bf16
    tensors (or their uint16 bit patterns), idx [T, Kc] int32; writes o
    [T, H, 128] and lse [T, H] (float32)."""
    import torch
    _attention_idx(cfg, idx, workspace)
    dev = idx.device.index
    T, H, S = max(cfg.tokens, 0), max(cfg.heads, 0), max(cfg.keys, 0)
    D, Dv = max(cfg.head_dim, 0), max(cfg.value_dim, 0)
    half = (torch.bfloat16, torch.uint16, torch.int16)
    _tensor("q", q, half, numel=T * H * D, device=dev)
    _tensor("k", k, half, numel=S * D, device=dev)
    _tensor("v", v, half, numel=S * Dv, device=dev)
    _tensor("o", o, (torch.float32,), numel=T * H * Dv, device=dev)
    _tensor("lse", lse, (torch.float32,), numel=T * H, device=dev)
    _check(load().dsa_sparse_attention(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), _ptr(idx),
                                       float(scale), _ptr(workspace), workspace.numel(), _ptr(o),
                                       _ptr(lse), _stream(stream)), "dsa_sparse_attention")


def ranges_attention_cfg(q, k, ranges, select: int) -> dsa_attention_cfg:
    """cfg of the range form: `select` bounds the positions one token's ranges
    cover."""
    T, H, D = q.shape
    return dsa_attention_cfg(tokens=T, heads=H, keys=k.shape[0], head_dim=D, value_dim=D,
                             select=int(select))


def dsa_sparse_attention_ranges_workspace(cfg: dsa_attention_cfg, nranges: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load().dsa_sparse_attention_ranges_workspace(ctypes.byref(cfg), int(nranges), ctypes.byref(n)),
           "dsa_sparse_attention_ranges_workspace")
    return int(n.value)


def _attention_ranges(cfg: dsa_attention_cfg, ranges, workspace) -> int:
    import torch
    if ranges.dim() != 3 or ranges.shape[2] != 2:
        raise ValueError(f"ranges must be [tokens, nranges, 2], got {tuple(ranges.shape)}")
    if ranges.shape[0] != max(cfg.tokens, 0):
        raise ValueError(f"ranges has {ranges.shape[0]} tokens, cfg.tokens = {cfg.tokens}")
    _i32("ranges", ranges, max(cfg.tokens, 0) * ranges.shape[1] * 2)
    _tensor("workspace", workspace, (torch.uint8,), device=ranges.device.index)
    return int(ranges.shape[1])


def dsa_group_union_ranges(cfg: dsa_attention_cfg, ranges, workspace, stream=None):
    """The unions of each group's position ranges and their token masks,
    written to workspace (the record layout of dsa_group_union)."""
    nr = _attention_ranges(cfg, ranges, workspace)
    _check(load().dsa_group_union_ranges(ctypes.byref(cfg), _ptr(ranges), nr, _ptr(workspace),
                                         workspace.numel(), _stream(stream)), "dsa_group_union_ranges")


def dsa_sparse_attention_ranges(cfg: dsa_attention_cfg, q, k, v, ranges, scale: float, workspace, o, lse,
                                stream=None):
    """Grouped masked sparse attention over per-token position ranges:
    ranges [T, nranges, 2] int32 half-open [lo, hi); otherwise as
    dsa_sparse_attention."""
    import torch
    nr = _attention_ranges(cfg, ranges, workspace)
    dev = ranges.device.index
    T, H, S = max(cfg.tokens, 0), max(cfg.heads, 0), max(cfg.keys, 0)
    D, Dv = max(cfg.head_dim, 0), max(cfg.value_dim, 0)
    half = (torch.bfloat16, torch.uint16, torch.int16)
    _tensor("q", q, half, numel=T * H * D, device=dev)
    _tensor("k", k, half, numel=S * D, device=dev)
    _tensor("v", v, half, numel=S * Dv, device=dev)
    _tensor("o", o, (torch.float32,), numel=T * H * Dv, device=dev)
    _tensor("lse", lse, (torch.float32,), numel=T * H, device=dev)
    _check(load().dsa_sparse_attention_ranges(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), _ptr(ranges), nr,
                                              float(scale), _ptr(workspace), workspace.numel(), _ptr(o),
                                              _ptr(lse), _stream(stream)), "dsa_sparse_attention_ranges")


def dsa_sparse_attention_status() -> int:
    return int(load().dsa_sparse_attention_status())


def dsa_indexer_status() -> int:
    """DSA_OK, or DSA_ERR_TIMEOUT once after an indexer kernel gave up a wait
    (synchronises the device)."""
    return int(load().dsa_indexer_status())
