"""Pins for the CPU oracle: hand-worked rows, brute force on tiny inputs,
reductions to a library top-K, value independence and mask invariants.

None of these re-runs the oracle's own formula: the expected values are either
worked out by hand (tests/golden/hand_rows.json), computed by an independent
counting formulation (tests/brute.py), or taken from numpy's stable sort.
"""
import random

import numpy as np
import pytest

from oracle import default as oracle_default
from tests import brute
from tests.common import assert_bits_equal, bits, load_golden, parse_row

NEG_INF = np.float32(-np.inf)


@pytest.fixture(scope="module")
def orc():
    return oracle_default()


def _run_case(orc, case):
    x = np.stack([parse_row(r) for r in case["x"]]).astype(np.float32)
    got = x.copy()
    cand, topk = orc.run(got, case["starts"], case["ends"], width=case["width"],
                         block_size=case["block_size"], block_topk=case["block_topk"],
                         row_topk=case["row_topk"], row_repeat=case["row_repeat"],
                         causal=case["causal"])
    return x, got, cand, topk


@pytest.mark.parametrize("case", load_golden()["cases"], ids=lambda c: c["name"])
def test_hand_worked_rows(orc, case):
    _, got, cand, topk = _run_case(orc, case)
    want = np.stack([parse_row(r) for r in case["masked"]])
    assert_bits_equal(got, want, case["name"] + " masked logits")
    assert cand.tolist() == case["cand"], case["name"]
    assert topk.tolist() == case["topk"], case["name"]


def test_hand_worked_block_scores(orc):
    case = next(c for c in load_golden()["cases"] if c["name"] == "ties_and_pin")
    x = parse_row(case["x"][0])
    S, nb = orc.block_scores(x, case["width"], case["starts"][0], case["ends"][0],
                             case["block_size"])
    want = [orc.key(v) for v in parse_row(case["block_scores"][0])]
    assert nb == 3
    assert S.tolist() == want


def test_key_is_total_order(orc):
    # a strictly increasing ladder under IEEE-754 totalOrder
    ladder = [0xFFFFFFFF, 0xFFC00000, 0xFF800001, 0xFF800000, 0xC0000000, 0xBF800000,
              0x80000001, 0x80000000, 0x00000000, 0x00000001, 0x3F800000, 0x7F7FFFFF,
              0x7F800000, 0x7F800001, 0x7FC00000, 0x7FFFFFFF]
    # keys read through a pointer (scores of one-column blocks): a Python float
    # round trip would quiet the signalling NaNs in the ladder
    row = np.array(ladder, dtype=np.uint32).view(np.float32)
    S, _ = orc.block_scores(row, len(ladder), 0, len(ladder), 1)
    keys = S.tolist()
    assert keys == sorted(keys) and len(set(keys)) == len(keys)
    # and the independent brute-force rank agrees on the same ladder
    ranks = [brute.rank(b) for b in ladder]
    assert ranks == sorted(ranks)


def _random_case(rng: random.Random, exotic: bool):
    W = rng.randint(0, 12)
    B = rng.randint(1, 4)
    Kb = rng.randint(1, 5)
    K = rng.randint(1, 6) if rng.random() < 0.8 else rng.randint(7, 16)
    s = rng.choice([0, 0, 0, rng.randint(0, W + 2), -1])
    e = rng.randint(-2, W + 2 * B)
    pool = brute.VALUE_POOL + (brute.EXOTIC_POOL if exotic else [])
    row = []
    for _ in range(W):
        if exotic and rng.random() < 0.08:
            row.append(rng.choice(brute.NAN_BITS))
        else:
            row.append(brute.to_bits(rng.choice(pool)))
    return W, B, Kb, K, s, e, row


@pytest.mark.parametrize("exotic", [False, True])
def test_brute_force_tiny(orc, exotic):
    rng = random.Random(1234 + exotic)
    for _ in range(3000):
        W, B, Kb, K, s, e, row = _random_case(rng, exotic)
        masked, cand, topk = brute.path(row, W, s, e, B, Kb, K)
        x = np.array(row, dtype=np.uint32).view(np.float32).copy() if W else \
            np.zeros(0, dtype=np.float32)
        buf = np.ascontiguousarray(x.reshape(1, W))
        starts = None if s == 0 and rng.random() < 0.5 else [s]
        c, t = orc.run(buf, starts, [e], width=W, block_size=B, block_topk=Kb, row_topk=K)
        ctx = dict(W=W, B=B, Kb=Kb, K=K, s=s, e=e, row=[hex(v) for v in row])
        assert bits(buf[0]).tolist() == masked, ctx
        assert c[0].tolist() == cand, ctx
        assert t[0].tolist() == topk, ctx


def test_brute_force_row_repeat(orc):
    rng = random.Random(99)
    for _ in range(400):
        rep = rng.randint(1, 3)
        causal = rng.random() < 0.5
        rows = rng.randint(1, 5)
        nq = -(-rows // rep)
        W, B, Kb, K = rng.randint(1, 10), rng.randint(1, 3), rng.randint(1, 3), rng.randint(1, 5)
        starts = [rng.randint(0, 3) for _ in range(nq)]
        ends = [rng.randint(-1, W + 3) for _ in range(nq)]
        x = np.array([[brute.to_bits(rng.choice(brute.VALUE_POOL)) for _ in range(W)]
                      for _ in range(rows)], dtype=np.uint32).view(np.float32)
        buf = x.copy()
        c, t = orc.run(buf, starts, ends, width=W, block_size=B, block_topk=Kb, row_topk=K,
                       row_repeat=rep, causal=causal)
        for r in range(rows):
            q = r // rep
            e = ends[q] - (rep - 1) + (r % rep) if causal else ends[q]
            masked, cand, topk = brute.path(bits(x[r]).tolist(), W, starts[q], e, B, Kb, K)
            assert bits(buf[r]).tolist() == masked
            assert c[r].tolist() == cand
            assert t[r].tolist() == topk


def test_b1_reduces_to_stable_topk(orc):
    """With one column per block and Kb >= K, every top-K column of the raw span
    survives the mask, so the row top-k is numpy's stable top-K of the span."""
    rng = np.random.default_rng(7)
    for trial in range(40):
        W = int(rng.integers(50, 3000))
        s = int(rng.integers(0, W // 3))
        e = int(rng.integers(s + 1, W + 5))
        K = int(rng.integers(1, 200))
        Kb = K + int(rng.integers(0, 50))
        x = rng.standard_normal(W).astype(np.float32)
        if trial % 2:
            x = np.round(x * 4) / 4 + np.float32(0.0)  # heavy ties; -0.0 -> +0.0
        buf = x.reshape(1, W).copy()
        _, t = orc.run(buf, [s], [e], width=W, block_size=1, block_topk=Kb, row_topk=K)
        span = x[s:min(e, W)].astype(np.float64)
        order = np.argsort(-span, kind="stable")[:K] + s
        want = np.sort(order)
        want = np.concatenate([want, -np.ones(K - len(want), dtype=np.int64)])
        assert t[0].tolist() == want.tolist()


def test_all_blocks_selected_is_value_independent(orc):
    """When the live span has at most Kb blocks, every live block is chosen
    (finite data), the mask only clears [0, start), and with L <= K the row
    top-k is start..end'-1: the output does not depend on the values."""
    rng = np.random.default_rng(11)
    W, B, Kb, K = 4096, 8, 32, 300
    for _ in range(30):
        s = int(rng.integers(0, 100))
        e = int(rng.integers(s + 1, s + Kb * B))
        outs = []
        for _v in range(2):
            x = rng.standard_normal((1, W)).astype(np.float32)
            buf = x.copy()
            c, t = orc.run(buf, [s], [e], width=W, block_size=B, block_topk=Kb, row_topk=K)
            assert np.all(np.isneginf(buf[0, :s]))
            assert_bits_equal(buf[0, s:], x[0, s:], "live span and tail unchanged")
            outs.append((c.tolist(), t.tolist()))
        assert outs[0] == outs[1]
        nb = -(-(e - s) // B)
        assert outs[0][0][0][:Kb] == list(range(Kb))  # live blocks then padding ids
        assert outs[0][0][0][Kb] == (e - 1 - s) // B
        L = e - s
        if L <= K:
            assert outs[0][1][0] == list(range(s, e)) + [-1] * (K - L)
        assert nb <= Kb


def _invariants(x, got, cand, topk, s, e, W, B, Kb, K):
    ec = min(e, W)
    # columns at or past the clamped end are never written
    assert_bits_equal(got[max(ec, 0):], x[max(ec, 0):], "tail")
    # every column is either unchanged or -inf
    changed = bits(got) != bits(x)
    assert np.all(np.isneginf(got[changed]))
    # a non -inf live column lies in a candidate block or is the edge column
    blocks = set(b for b in cand.tolist() if b >= 0 and s + b * B < W)
    edge = any(b >= 0 and s + b * B >= W for b in cand.tolist())
    for c in np.nonzero(~np.isneginf(got[:max(ec, 0)]))[0]:
        assert c >= s and (((c - s) // B) in blocks or (c == W - 1 and edge))
    assert len(blocks) <= Kb + 1
    # selection certificate: every chosen column beats every other live column
    live = np.arange(s, ec) if ec > s else np.arange(0)
    sel = [c for c in topk.tolist() if c >= 0]
    assert sel == sorted(set(sel)) and all(s <= c < ec for c in sel)
    assert len(sel) == min(K, len(live))
    if sel and len(sel) < len(live):
        keys = [brute.rank(int(b)) for b in bits(got)]
        worst = min(sel, key=lambda c: (keys[c], -c))
        rest = np.setdiff1d(live, sel)
        best_rest = max(rest.tolist(), key=lambda c: (keys[c], -c))
        assert brute.better(keys[worst], worst, keys[best_rest], best_rest)


def test_invariants_and_idempotence_random(orc):
    rng = np.random.default_rng(3)
    for _ in range(25):
        W = int(rng.integers(100, 5000))
        B = int(rng.choice([1, 2, 3, 8, 16]))
        Kb = int(rng.integers(1, 40))
        K = int(rng.integers(1, 300))
        s = int(rng.integers(0, 64))
        e = int(rng.integers(-5, W + 3 * B))
        x = rng.standard_normal(W).astype(np.float32)
        x[rng.random(W) < 0.01] = -np.inf
        got = x.reshape(1, W).copy()
        c, t = orc.run(got, [s], [e], width=W, block_size=B, block_topk=Kb, row_topk=K)
        _invariants(x, got[0], c[0], t[0], s, e, W, B, Kb, K)
        again = got.copy()
        c2, t2 = orc.run(again, [s], [e], width=W, block_size=B, block_topk=Kb, row_topk=K)
        assert_bits_equal(again, got, "idempotent mask")
        assert t2.tolist() == t.tolist()


def test_spikes_always_selected(orc):
    """With 64 spikes far above N(0,1) in distinct blocks, all land in the row top-k."""
    rng = np.random.default_rng(5)
    W, B, Kb, K = 1 << 16, 8, 256, 2048
    x = rng.standard_normal(W).astype(np.float32)
    pos = rng.choice(W // B, size=64, replace=False) * B + 3
    x[pos] = 6 + np.abs(rng.standard_normal(64)).astype(np.float32)
    got = x.reshape(1, W).copy()
    _, t = orc.run(got, None, [W], width=W, block_size=B, block_topk=Kb, row_topk=K)
    assert set(pos.tolist()) <= set(t[0].tolist())
