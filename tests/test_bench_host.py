"""bench.py on the host: byte accounting against a direct count from the
oracle's masked output, and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import bench
import oracle
import workloads as wk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("name", ["tiny", "decode_short"])
def test_algorithmic_bytes_match_direct_count(name):
    wl = wk.WORKLOADS[name]
    x, starts, ends = wk.make_all(wl)
    got = x.copy()
    cand, _ = oracle.default().run(got, starts, ends, width=wl.width, block_size=wl.block_size,
                                   block_topk=wl.block_topk, row_topk=wl.row_topk,
                                   row_repeat=wl.row_repeat)
    alg = bench.algorithmic_bytes(wl, starts, ends, cand)
    s, e = bench.row_bounds(wl, starts, ends)
    for r in range(wl.rows):
        ec = min(int(e[r]), wl.width)
        writes = int(np.isneginf(got[r, :max(ec, 0)]).sum())  # finite inputs: -inf == written
        L = max(ec - int(s[r]), 0)
        nb = -(-L // wl.block_size)
        read = 4 * L if nb > wl.block_topk else 0
        assert alg[r] == read + 4 * writes + 4 * (wl.block_topk + 1) + 4 * wl.row_topk + 8


def test_full_width_closed_form():
    # the old design's dead stores at 96 rows x 2^20 columns: 402.65 MB per call
    assert 96 * (1 << 20) * 4 == 402_653_184
    # flags (1 byte per block) against mask bytes (4 per column) at B = 8: 1/32
    assert (1 / 8) / 4 == 1 / 32


def test_reference_arm_prints_one_json_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "2", "--warmup", "1", "--workload", "tiny"],
                         capture_output=True, text=True, env=env, timeout=300, check=True)
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "rows/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0
    for k in ("metric", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config"):
        assert k in d
