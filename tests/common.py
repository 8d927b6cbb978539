"""Helpers shared by the tests: golden-file parsing and exact bit comparison."""
import json
import os
import struct

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

_SPECIAL = {"nan": 0x7FC00000, "-nan": 0xFFC00000}


def value_bits(s: str) -> int:
    """Bit pattern of a golden value string."""
    if s in _SPECIAL:
        return _SPECIAL[s]
    return struct.unpack("<I", struct.pack("<f", float(s)))[0]


def parse_row(values) -> np.ndarray:
    return np.array([value_bits(v) for v in values], dtype=np.uint32).view(np.float32)


def load_golden(name="hand_rows.json"):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def bits(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.float32
    return a.view(np.uint32)


def assert_bits_equal(got, want, what=""):
    g, w = bits(got), bits(want)
    assert g.shape == w.shape, (what, g.shape, w.shape)
    diff = np.nonzero(g != w)
    if len(diff[0]):
        idx = tuple(d[0] for d in diff)
        raise AssertionError(f"{what}: {len(diff[0])} elements differ; first at {idx}: "
                             f"got {g[idx]:#010x} want {w[idx]:#010x}")
