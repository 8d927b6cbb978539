"""Seeded synthetic workloads for the DSA indexer candidate-selection path.

This module only generates inputs (logits and per-row bounds).  It holds none
of the selection arithmetic, so both the CUDA path and the CPU oracle can be fed
from it without sharing any of the method's code.

The five workloads follow the shapes the vLLM pages discuss for DeepSeek-V4.1
decode and prefill (vLLM PR #57459 "DSA candidate-block kernels walk each row's
live context", Summary; prhub report on vLLM PR #56628, test section):

  tiny          4 rows x 4096, ends U{1..4096}, B=8, Kb=32, K=64
  decode_short  64 rows x 131072, ends log-uniform in [128, 2048]
  decode_1m     96 rows (48 requests x next_n 2, row_repeat 2) x 2^20,
                ends lognormal(median 600) clipped to [1, 16384]
  prefill_1m    2048 causal rows x 2^20, end = 1,046,273 + row,
                64 planted spikes per row
  ragged        128 rows x 262144 at column stride 2, starts U{0..512},
                boundary ends, 1 % exact ties, 0.1 % -inf, B=16

Every value is a pure function of (seed, stream, row, column) through a
Philox4x32-10 counter generator, so single rows can be regenerated on their
own for sampled checks at full size.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libsynth.so")
_lib = None
_lib_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile synth.c with gcc into workloads/_build/libsynth.so."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-fPIC", "-shared",
                    "-pthread", "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lib_lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            L.synth_fill.restype = ctypes.c_int
            L.synth_fill.argtypes = [
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_uint32,
                ctypes.c_uint32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                ctypes.c_double, ctypes.c_int32]
            L.synth_u32.restype = None
            L.synth_u32.argtypes = [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32,
                                    ctypes.c_int64, ctypes.c_void_p]
            L.synth_philox4x32_10.restype = None
            L.synth_philox4x32_10.argtypes = [ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_void_p]
            _lib = L
    return _lib


def philox4x32_10(counter, key) -> np.ndarray:
    """One Philox4x32-10 block (exposed for known-answer tests)."""
    c = np.asarray(counter, dtype=np.uint32)
    k = np.asarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().synth_philox4x32_10(c.ctypes.data, k.ctypes.data, out.ctypes.data)
    return out


def u32(seed: int, stream: int, row: int, n: int) -> np.ndarray:
    out = np.zeros(max(n, 0), dtype=np.uint32)
    if n > 0:
        lib().synth_u32(seed, stream, row, n, out.ctypes.data)
    return out


def _unit(x: np.ndarray) -> np.ndarray:
    return (x.astype(np.float64) + 0.5) * (1.0 / 4294967296.0)


# Streams used for bounds (disjoint from the per-column streams in synth.c).
_S_START = 101
_S_END = 102
_S_END_KIND = 103


@dataclass(frozen=True)
class Workload:
    """One synthetic configuration.  Sizes are in logits elements."""
    name: str
    rows: int
    width: int
    block_size: int
    block_topk: int
    row_topk: int
    seed: int
    row_repeat: int = 1
    col_stride: int = 1
    has_starts: bool = False
    tie_ppm: int = 0
    ninf_ppm: int = 0
    spikes: int = 0
    spike_base: float = 6.0
    note: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def row_stride(self) -> int:
        return self.width * self.col_stride

    @property
    def n_bounds(self) -> int:
        return -(-self.rows // self.row_repeat)

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


WORKLOADS = {
    "tiny": Workload("tiny", rows=4, width=4096, block_size=8, block_topk=32,
                     row_topk=64, seed=0, note="ends U{1..4096}"),
    "decode_short": Workload("decode_short", rows=64, width=131072, block_size=8,
                             block_topk=256, row_topk=2048, seed=1,
                             note="ends log-uniform in [128, 2048]"),
    "decode_1m": Workload("decode_1m", rows=96, width=1 << 20, block_size=8,
                          block_topk=256, row_topk=2048, seed=2, row_repeat=2,
                          note="48 requests x next_n 2; per-request b ~ "
                               "clip(round(lognormal(ln 600, 1)), 1, 16384); "
                               "rows of a request end at b and b+1"),
    "prefill_1m": Workload("prefill_1m", rows=2048, width=1 << 20, block_size=8,
                           block_topk=256, row_topk=2048, seed=3, spikes=64,
                           note="end = 1,046,273 + row; 64 spikes 6+|z| per row"),
    "ragged": Workload("ragged", rows=128, width=262144, block_size=16,
                       block_topk=256, row_topk=2048, seed=4, col_stride=2,
                       has_starts=True, tie_ppm=10000, ninf_ppm=1000,
                       note="starts U{0..512}; boundary and uniform ends; "
                            "1% ties, 0.1% -inf; every 2nd float of [128, 524288]"),
}


def bounds(wl: Workload):
    """Per-bound-entry (starts or None, ends) as int32 arrays of length n_bounds."""
    n = wl.n_bounds
    W, B = wl.width, wl.block_size
    starts = None
    if wl.name.startswith("tiny") or wl.extra.get("ends") == "uniform_full":
        x = u32(wl.seed, _S_END, 0, n)
        ends = 1 + (x.astype(np.int64) % W)
    elif wl.name.startswith("decode_short"):
        u = _unit(u32(wl.seed, _S_END, 0, n))
        ends = np.rint(np.exp(math.log(128) + u * (math.log(2048) - math.log(128))))
    elif wl.name.startswith("decode_1m"):
        a = u32(wl.seed, _S_END, 0, 2 * n)
        u1, u2 = _unit(a[0::2]), _unit(a[1::2])
        z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)
        b = np.clip(np.rint(np.exp(math.log(600.0) + 1.0 * z)), 1, 16384)
        # the request's newest row ends one past its older row (next_n = 2)
        ends = b + (wl.row_repeat - 1)
    elif wl.name.startswith("prefill_1m"):
        base = wl.extra.get("end_base", 1_046_273)
        ends = base + np.arange(n, dtype=np.int64)
    elif wl.name.startswith("ragged"):
        s = u32(wl.seed, _S_START, 0, n).astype(np.int64) % 513
        starts = s
        special = [0, 1, 1023, 1024, 1025, W, W + 1, W + 7, W + B + 3]
        kind = u32(wl.seed, _S_END_KIND, 0, 2 * n)
        ends = np.zeros(n, dtype=np.int64)
        for q in range(n):
            if q < len(special):
                ends[q] = special[q]
                continue
            k = int(kind[2 * q]) % 4
            r = int(kind[2 * q + 1])
            if k == 0:
                ends[q] = special[r % 6]
            elif k == 1:
                ends[q] = special[6 + r % 3]
            else:
                lo = int(s[q])
                ends[q] = lo + r % (W - lo + 1)
    else:
        raise KeyError(wl.name)
    ends = np.asarray(ends, dtype=np.int64)
    if starts is not None:
        starts = np.asarray(starts, dtype=np.int32)
    return starts, ends.astype(np.int32)


def _live_ranges(wl: Workload, rows, starts, ends):
    """[lo, hi) per requested row for tie sources and spike positions: the
    bound entry's [start, min(end, width)) as the bounds generator laid it out
    (workloads with spikes or ties have one bound entry per row)."""
    rows = np.asarray(rows, dtype=np.int64)
    q = rows // wl.row_repeat
    e = ends[q].astype(np.int64)
    s = starts[q].astype(np.int64) if starts is not None else np.zeros_like(e)
    hi = np.minimum(e, wl.width)
    lo = np.minimum(s, hi)
    return lo.astype(np.int64), np.maximum(hi, lo).astype(np.int64)


def fill_rows(wl: Workload, rows, out: np.ndarray, starts=None, ends=None,
              nthreads: int | None = None, bound_rows=None) -> np.ndarray:
    """Write the logits of absolute rows `rows` into `out` ([len(rows), row_stride]
    float32, C-contiguous rows, may be a view of pinned memory).  `bound_rows`
    (default: `rows`) names the row of the bounds each output row is laid out
    for, so replica batches can draw fresh data rows for the same bounds."""
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    if starts is None and ends is None:
        starts, ends = bounds(wl)
    assert out.dtype == np.float32 and out.ndim == 2 and out.shape[0] == len(rows)
    assert out.shape[1] >= wl.row_stride and out.strides[1] == 4
    brows = rows if bound_rows is None else np.asarray(bound_rows, dtype=np.int64)
    assert len(brows) == len(rows)
    lo, hi = _live_ranges(wl, brows, starts, ends)
    lo = np.ascontiguousarray(lo)
    hi = np.ascontiguousarray(hi)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    rc = lib().synth_fill(out.ctypes.data, out.strides[0] // 4, wl.col_stride, wl.width,
                          rows.ctypes.data, len(rows), wl.seed, wl.tie_ppm, wl.ninf_ppm,
                          lo.ctypes.data, hi.ctypes.data, wl.spikes, wl.spike_base,
                          nthreads)
    if rc != 0:
        raise ValueError("synth_fill rejected its arguments")
    return out


def make_rows(wl: Workload, rows, starts=None, ends=None, bound_rows=None) -> np.ndarray:
    rows = list(rows)
    out = np.empty((len(rows), wl.row_stride), dtype=np.float32)
    return fill_rows(wl, rows, out, starts, ends, bound_rows=bound_rows)


def make_all(wl: Workload, out: np.ndarray | None = None):
    """(logits [rows, row_stride] float32, starts, ends) for the whole workload."""
    starts, ends = bounds(wl)
    if out is None:
        out = np.empty((wl.rows, wl.row_stride), dtype=np.float32)
    fill_rows(wl, range(wl.rows), out, starts, ends)
    return out, starts, ends


# ---------------------------------------------------------------------------
# indexer producer inputs: e4m3 bytes for q [T, 64, 128] and k [S, 128]

_S_Q = 111
_S_K = 112
_S_W = 113
_S_KS = 114


def e4m3_bytes(seed: int, stream: int, row: int, n: int) -> np.ndarray:
    """n random OCP E4M3 bytes with exponent field in [3, 9] (|value| in
    [2^-4, 7.5]); no NaN, no subnormal."""
    x = u32(seed, stream, row, n)
    sign = (x >> 31) & 1
    exp = 3 + (x % 7)
    man = (x >> 8) & 7
    return ((sign << 7) | (exp << 3) | man).astype(np.uint8)


def indexer_inputs(T: int, S: int, seed: int = 7, heads: int = 64, dim: int = 128,
                   causal: bool = True):
    """(q, k, k_scale, w, starts, ends) for T queries over S keys; causal ends
    S - T + t + 1 (the last query sees every key), starts 0."""
    q = e4m3_bytes(seed, _S_Q, 0, T * heads * dim).reshape(T, heads, dim)
    k = e4m3_bytes(seed, _S_K, 0, S * dim).reshape(S, dim)
    ks = (0.5 + _unit(u32(seed, _S_KS, 0, S))).astype(np.float32)
    a = u32(seed, _S_W, 0, 2 * T * heads)
    u1, u2 = _unit(a[0::2]), _unit(a[1::2])
    w = (0.1 * np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)).astype(np.float32)
    w = w.reshape(T, heads)
    if causal:
        ends = (S - T + 1 + np.arange(T)).clip(0, S).astype(np.int32)
    else:
        ends = np.full(T, S, dtype=np.int32)
    return q, k, ks, w, None, ends


# OCP E4M3 bytes of small integers (value = 2^(e - 7) * (1 + m / 8)):
# 1 = e 7, 2 = e 8, 3 = e 8 with m 4; bit 7 is the sign.
E4M3_INT = {1: 0x38, 2: 0x40, 3: 0x44, -1: 0xB8, -2: 0xC0, -3: 0xC4}
_S_XQ = 131
_S_XK = 132
_S_XPOOL = 133
_S_XW = 134
_S_XKS = 135


def indexer_exact_inputs(T: int, S: int, seed: int = 3, heads: int = 64, dim: int = 128,
                         pool: int = 48):
    """(q, k, k_scale, w, starts, ends) whose indexer logits are exact in fp32.

    q holds e4m3 integers in {+-1, +-2, +-3}, k in {+-1, +-2}: every product is
    an integer and a head's dot product stays within 128 * 6 = 768.  The head
    weights are powers of two in [1/4, 2] (positive, so no head sum is -0) and
    the key scales powers of two in [1/2, 2] (half of them 1): the weighted
    head sum is a multiple of 1/4 below 2^17, so every partial sum is
    representable in fp32 whatever the order.  Keys are drawn from a pool of
    `pool` distinct rows, so equal logits (ties) are common.  Causal ends."""
    qv = np.array([1, 2, 3, -1, -2, -3])
    kv = np.array([1, 2, -1, -2])
    enc = np.vectorize(E4M3_INT.get, otypes=[np.uint8])
    q = enc(qv[u32(seed, _S_XQ, 0, T * heads * dim) % 6]).reshape(T, heads, dim)
    rows = enc(kv[u32(seed, _S_XK, 0, pool * dim) % 4]).reshape(pool, dim)
    k = np.ascontiguousarray(rows[u32(seed, _S_XPOOL, 0, S) % pool])
    w = (2.0 ** (u32(seed, _S_XW, 0, T * heads) % 4 - 2.0)).astype(np.float32).reshape(T, heads)
    e = u32(seed, _S_XKS, 0, S) % 4
    ks = (2.0 ** np.where(e == 3, 0, e.astype(np.int64) - 1)).astype(np.float32)
    ends = (S - T + 1 + np.arange(T)).clip(0, S).astype(np.int32)
    return q, k, ks, w, None, ends


# ---------------------------------------------------------------------------
# grouped sparse attention inputs

_S_AQ = 121
_S_AK = 122
_S_AV = 123
_S_ASEL = 124
_S_ATOK = 125


def bf16_normal(seed: int, stream: int, n: int, scale: float = 1.0) -> np.ndarray:
    """n N(0, scale^2) values (Box-Muller on Philox words) rounded to bf16,
    returned as their 16-bit patterns (round to nearest, ties to even)."""
    a = u32(seed, stream, 0, 2 * n)
    u1, u2 = _unit(a[0::2]), _unit(a[1::2])
    x = (scale * np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)).astype(np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def attention_inputs(T: int, H: int, S: int, Kc: int, seed: int = 9, dim: int = 128, G: int = 16,
                     own: float = 0.1, fill: float = 1.0):
    """(q [T, H, dim], k [S, dim], v [S, dim] as bf16 bits, idx [T, Kc]).

    Neighbouring tokens select overlapping positions, as the pages observe:
    the tokens of each group of G share a base selection of Kc positions and
    each replaces a fraction `own` of it with positions of its own.  A token
    selects round(fill * Kc) positions (ascending, distinct, -1 padded);
    scores are kept moderate by a 1/4 spread on q."""
    q = bf16_normal(seed, _S_AQ, T * H * dim, 0.25).reshape(T, H, dim)
    k = bf16_normal(seed, _S_AK, S * dim).reshape(S, dim)
    v = bf16_normal(seed, _S_AV, S * dim).reshape(S, dim)
    idx = np.full((T, Kc), -1, dtype=np.int32)
    n = max(0, min(int(round(fill * Kc)), S))
    for g0 in range(0, T, G):
        base = np.unique(u32(seed, _S_ASEL, g0, 4 * Kc + 64) % max(S, 1))
        # n of the distinct draws, spread over their whole range
        base = base[np.linspace(0, len(base) - 1, n).astype(np.int64)] if n else base[:0]
        base = np.unique(base)
        for t in range(g0, min(g0 + G, T)):
            r = u32(seed, _S_ATOK, t, 2 * Kc + 8)
            sel = base.copy()
            m = int(own * len(sel))
            if m:
                swap = np.unique(r[:m] % len(sel))
                sel[swap] = r[Kc:Kc + len(swap)] % S
            sel = np.unique(sel)
            if len(sel) < n:
                # replacements collided: top up with the token's further draws,
                # in draw order, then (tiny key ranges) with the lowest free keys
                extra = r[Kc + m:] % S
                extra = extra[~np.isin(extra, sel)]
                _, first = np.unique(extra, return_index=True)
                sel = np.union1d(sel, extra[np.sort(first)][:n - len(sel)])
                if len(sel) < n:
                    sel = np.union1d(sel, np.setdiff1d(np.arange(S), sel)[:n - len(sel)])
            idx[t, :n] = sel[:n]
    return q, k, v, idx
