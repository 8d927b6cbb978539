"""CPU oracle for the DSA indexer candidate-selection path -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls it.

The arithmetic lives in ``dsa_oracle.c`` (plain single-threaded C, built here
with gcc); this module only compiles it and marshals numpy arrays into it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "dsa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, EINVAL, ENOMEM = 0, -1, -2


def compile_oracle(src: str, out: str) -> str:
    """gcc -O2 a copy of the oracle source into a shared library at `out`."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, src, "-lm"],
                   check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    if (force or not os.path.exists(_LIB_PATH)
            or os.path.getmtime(_LIB_PATH) < os.path.getmtime(SOURCE)):
        compile_oracle(SOURCE, _LIB_PATH)
    return _LIB_PATH


def _bind(path: str):
    L = ctypes.CDLL(path)
    i32, i64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
    L.oracle_key.restype = ctypes.c_uint32
    L.oracle_key.argtypes = [ctypes.c_float]
    L.oracle_bounds.restype = None
    L.oracle_bounds.argtypes = [i32, vp, vp, i32, i32, i32, vp, vp]
    L.oracle_block_scores.restype = i64
    L.oracle_block_scores.argtypes = [vp, i64, i64, i64, i64, i32, vp]
    L.oracle_block_topk.restype = i32
    L.oracle_block_topk.argtypes = [vp, i64, i32, vp]
    L.oracle_pin.restype = i64
    L.oracle_pin.argtypes = [i64, i64, i32]
    L.oracle_mask.restype = ctypes.c_int
    L.oracle_mask.argtypes = [vp, i64, i64, i64, i64, i32, vp, i32]
    L.oracle_row_topk.restype = i32
    L.oracle_row_topk.argtypes = [vp, i64, i64, i64, i64, i32, vp]
    L.oracle_row.restype = ctypes.c_int
    L.oracle_row.argtypes = [vp, i64, i64, i64, i64, i32, i32, i32, vp, vp]
    L.oracle_combine_window.restype = i32
    L.oracle_combine_window.argtypes = [vp, i32, i64, i64, i64, i32, vp]
    L.oracle_e4m3.restype = ctypes.c_double
    L.oracle_e4m3.argtypes = [ctypes.c_uint8]
    L.oracle_indexer_logits.restype = ctypes.c_int
    L.oracle_indexer_logits.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, i64]
    L.oracle_bf16.restype = ctypes.c_double
    L.oracle_bf16.argtypes = [ctypes.c_uint16]
    L.oracle_group_union.restype = i32
    L.oracle_group_union.argtypes = [vp, i32, i32, i32, i32, vp, vp, i32]
    L.oracle_sparse_attention.restype = ctypes.c_int
    L.oracle_sparse_attention.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                          ctypes.c_double, vp, vp]
    L.oracle_run.restype = ctypes.c_int
    L.oracle_run.argtypes = [vp, i32, i64, i64, i64, vp, vp, i32, i32, i32, i32, i32, i32,
                             vp, vp]
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


class Oracle:
    """numpy-level access to one compiled oracle library (the default one, or a
    deliberately altered copy used by the mutation tests)."""

    def __init__(self, path: str | None = None):
        self.L = lib() if path is None else _bind(path)

    # ---- single steps -------------------------------------------------
    def key(self, x: float) -> int:
        return int(self.L.oracle_key(float(x)))

    def bounds(self, r, starts, ends, rep=1, causal=True):
        s = ctypes.c_int64()
        e = ctypes.c_int64()
        st = None if starts is None else np.ascontiguousarray(starts, dtype=np.int32)
        en = np.ascontiguousarray(ends, dtype=np.int32)
        self.L.oracle_bounds(int(r), None if st is None else st.ctypes.data, en.ctypes.data,
                             int(st is not None), int(rep), int(bool(causal)),
                             ctypes.byref(s), ctypes.byref(e))
        return s.value, e.value

    def block_scores(self, row, width, s, e, B, col_stride=1):
        row = np.ascontiguousarray(row, dtype=np.float32)
        NB = -(-width // B)
        S = np.zeros(max(NB, 1), dtype=np.uint32)
        nb = self.L.oracle_block_scores(row.ctypes.data, width, col_stride, s, e, B,
                                        S.ctypes.data)
        return S[:NB], nb

    def block_topk(self, S, Kb):
        S = np.ascontiguousarray(S, dtype=np.uint32)
        T = np.zeros(Kb, dtype=np.int32)
        n = self.L.oracle_block_topk(S.ctypes.data, len(S), Kb, T.ctypes.data)
        if n < 0:
            raise MemoryError
        return T

    def pin(self, s, e, B):
        return int(self.L.oracle_pin(s, e, B))

    def mask(self, row, width, s, e, B, cand, col_stride=1):
        """Masks `row` (float32, C-contiguous) in place."""
        assert row.dtype == np.float32 and row.flags.c_contiguous
        cand = np.ascontiguousarray(cand, dtype=np.int32)
        rc = self.L.oracle_mask(row.ctypes.data, width, col_stride, s, e, B,
                                cand.ctypes.data, len(cand))
        if rc != OK:
            raise RuntimeError(f"oracle_mask: {rc}")
        return row

    def row_topk(self, row, width, s, e, K, col_stride=1):
        row = np.ascontiguousarray(row, dtype=np.float32)
        out = np.zeros(K, dtype=np.int32)
        n = self.L.oracle_row_topk(row.ctypes.data, width, col_stride, s, e, K,
                                   out.ctypes.data)
        if n < 0:
            raise MemoryError
        return out

    def combine_window(self, topk_row, s, e, width, window):
        """Union of a row's top-k and the last `window` live columns, ascending,
        padded with -1 to K + window."""
        t = np.ascontiguousarray(topk_row, dtype=np.int32)
        out = np.zeros(len(t) + window, dtype=np.int32)
        n = self.L.oracle_combine_window(t.ctypes.data, len(t), s, e, width, window,
                                         out.ctypes.data)
        if n < 0:
            raise MemoryError
        return out

    def e4m3(self, b: int) -> float:
        return float(self.L.oracle_e4m3(int(b)))

    def indexer_logits(self, q, k, k_scale, w, starts, ends, out):
        """q [T, H, D] uint8 (e4m3), k [S, D] uint8, k_scale [S] f32, w [T, H]
        f32, bounds [T]; writes out [T, ld] f32 over each live span."""
        q = np.ascontiguousarray(q, dtype=np.uint8)
        k = np.ascontiguousarray(k, dtype=np.uint8)
        ks = np.ascontiguousarray(k_scale, dtype=np.float32)
        w = np.ascontiguousarray(w, dtype=np.float32)
        T, H, D = q.shape
        S = k.shape[0]
        st = None if starts is None else np.ascontiguousarray(starts, dtype=np.int32)
        en = np.ascontiguousarray(ends, dtype=np.int32)
        assert out.dtype == np.float32 and out.flags.c_contiguous
        rc = self.L.oracle_indexer_logits(q.ctypes.data, k.ctypes.data, ks.ctypes.data,
                                          w.ctypes.data, T, S, H, D,
                                          None if st is None else st.ctypes.data,
                                          en.ctypes.data, out.ctypes.data, out.shape[1])
        if rc != OK:
            raise RuntimeError(f"oracle_indexer_logits: {rc}")
        return out

    def bf16(self, b: int) -> float:
        return float(self.L.oracle_bf16(int(b)))

    def group_union(self, idx, t0, G):
        """Distinct positions selected by tokens [t0, t0 + G) of idx [T, Kc]
        (ascending) and, per position, the mask of the tokens that chose it."""
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        T, Kc = idx.shape
        cap = max(1, G * Kc)
        keys = np.zeros(cap, dtype=np.int32)
        mask = np.zeros(cap, dtype=np.uint32)
        n = self.L.oracle_group_union(idx.ctypes.data, T, Kc, int(t0), int(G), keys.ctypes.data,
                                      mask.ctypes.data, cap)
        if n < 0:
            raise MemoryError
        return keys[:n], mask[:n]

    def sparse_attention(self, q, k, v, idx, scale):
        """q [T, H, D], k [S, D], v [S, Dv] as bf16 bit patterns (uint16),
        idx [T, Kc]; returns (o [T, H, Dv], lse [T, H]) in float64."""
        q = np.ascontiguousarray(q, dtype=np.uint16)
        k = np.ascontiguousarray(k, dtype=np.uint16)
        v = np.ascontiguousarray(v, dtype=np.uint16)
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        T, H, D = q.shape
        S, Dv = v.shape
        Kc = idx.shape[1]
        o = np.zeros((T, H, Dv), dtype=np.float64)
        lse = np.zeros((T, H), dtype=np.float64)
        rc = self.L.oracle_sparse_attention(q.ctypes.data, k.ctypes.data, v.ctypes.data, idx.ctypes.data,
                                            T, H, D, Dv, S, Kc, float(scale), o.ctypes.data,
                                            lse.ctypes.data)
        if rc != OK:
            raise RuntimeError(f"oracle_sparse_attention: {rc}")
        return o, lse

    # ---- whole path -----------------------------------------------------
    def row(self, row, width, s, e, B, Kb, K, col_stride=1):
        """The whole path on one row (masked in place); returns (cand, topk)."""
        assert row.dtype == np.float32 and row.flags.c_contiguous
        cand = np.zeros(Kb + 1, dtype=np.int32)
        topk = np.zeros(K, dtype=np.int32)
        rc = self.L.oracle_row(row.ctypes.data, width, col_stride, s, e, B, Kb, K,
                               cand.ctypes.data, topk.ctypes.data)
        if rc != OK:
            raise RuntimeError(f"oracle_row: {rc}")
        return cand, topk

    def run(self, logits, starts, ends, *, width, block_size, block_topk, row_topk,
            row_repeat=1, causal=True, col_stride=1, row_stride=None):
        """The whole path on every row of `logits` ([rows, row_stride] float32,
        masked in place).  Returns (cand [rows, Kb+1], topk [rows, K])."""
        assert logits.dtype == np.float32 and logits.flags.c_contiguous
        rows = logits.shape[0]
        if row_stride is None:
            row_stride = logits.shape[1]
        st = None if starts is None else np.ascontiguousarray(starts, dtype=np.int32)
        en = np.ascontiguousarray(ends, dtype=np.int32)
        cand = np.zeros((rows, block_topk + 1), dtype=np.int32)
        topk = np.zeros((rows, row_topk), dtype=np.int32)
        rc = self.L.oracle_run(logits.ctypes.data, rows, width, row_stride, col_stride,
                               None if st is None else st.ctypes.data, en.ctypes.data,
                               int(st is not None), row_repeat, int(bool(causal)),
                               block_size, block_topk, row_topk, cand.ctypes.data,
                               topk.ctypes.data)
        if rc != OK:
            raise RuntimeError(f"oracle_run: {rc}")
        return cand, topk


_default = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default
