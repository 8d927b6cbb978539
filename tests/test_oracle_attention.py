"""Pins of the grouped sparse attention oracle against what the
mathematics fixes: softmax over one position, softmax of equal scores,
an independent numpy formulation on small inputs, order independence,
empty selections, and the union against Python sets."""
import math

import numpy as np
import pytest

import workloads as wk
from oracle import default as oracle_default


@pytest.fixture(scope="module")
def orc():
    return oracle_default()


def _f(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_bf16_decoding(orc):
    for b, want in ((0x3F80, 1.0), (0xC000, -2.0), (0x0000, 0.0), (0x3E80, 0.25), (0x7F80, math.inf)):
        assert orc.bf16(b) == want
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 16, 200).astype(np.uint16)
    bits = bits[np.isfinite(_f(bits))]
    assert all(orc.bf16(int(b)) == float(_f(b)) for b in bits)


def test_single_position_is_that_row(orc):
    # softmax over one score is 1: o is the value row, lse the score itself
    q, k, v, _ = wk.attention_inputs(3, 8, 50, 4, seed=1)
    idx = np.array([[7, -1, -1, -1], [-1, 49, -1, -1], [0, -1, -1, -1]], dtype=np.int32)
    scale = 0.125
    o, lse = orc.sparse_attention(q, k, v, idx, scale)
    for t, j in ((0, 7), (1, 49), (2, 0)):
        for h in range(8):
            assert np.array_equal(o[t, h], _f(v[j]))
            assert lse[t, h] == pytest.approx(scale * float(_f(q[t, h]) @ _f(k[j])), rel=1e-14, abs=1e-14)


def test_equal_scores_average_the_values(orc):
    # q = 0: every score is 0, so o is the plain mean and lse = ln(count)
    _, k, v, idx = wk.attention_inputs(4, 8, 300, 32, seed=2, fill=0.75)
    q = np.zeros((4, 8, 128), dtype=np.uint16)
    o, lse = orc.sparse_attention(q, k, v, idx, 0.3)
    for t in range(4):
        sel = idx[t][idx[t] >= 0]
        want = _f(v[sel]).mean(axis=0)
        for h in range(8):
            assert np.allclose(o[t, h], want, rtol=1e-13, atol=1e-13)
            assert lse[t, h] == pytest.approx(math.log(len(sel)), rel=1e-14)


def test_matches_an_independent_numpy_softmax(orc):
    q, k, v, idx = wk.attention_inputs(6, 16, 400, 40, seed=3, fill=0.8)
    scale = 1.0 / math.sqrt(128)
    o, lse = orc.sparse_attention(q, k, v, idx, scale)
    qf, kf, vf = _f(q), _f(k), _f(v)
    for t in range(6):
        sel = idx[t][idx[t] >= 0]
        s = scale * qf[t] @ kf[sel].T          # [H, n]
        mx = s.max(axis=1, keepdims=True)
        w = np.exp(s - mx)
        want_o = (w @ vf[sel]) / w.sum(axis=1, keepdims=True)
        want_lse = mx[:, 0] + np.log(w.sum(axis=1))
        assert np.allclose(o[t], want_o, rtol=1e-12, atol=1e-12)
        assert np.allclose(lse[t], want_lse, rtol=1e-12, atol=1e-12)


def test_order_and_padding_do_not_matter(orc):
    q, k, v, idx = wk.attention_inputs(5, 8, 200, 24, seed=4, fill=0.5)
    o, lse = orc.sparse_attention(q, k, v, idx, 0.2)
    rng = np.random.default_rng(4)
    shuffled = np.full((5, 40), -1, dtype=np.int32)
    for t in range(5):
        sel = idx[t][idx[t] >= 0]
        pos = rng.choice(40, size=len(sel), replace=False)
        shuffled[t, pos] = rng.permutation(sel)
    o2, lse2 = orc.sparse_attention(q, k, v, shuffled, 0.2)
    assert np.allclose(o, o2, rtol=1e-13, atol=1e-13) and np.allclose(lse, lse2, rtol=1e-13)


def test_empty_selection(orc):
    q, k, v, idx = wk.attention_inputs(2, 8, 100, 8, seed=5)
    idx[1] = -1
    o, lse = orc.sparse_attention(q, k, v, idx, 0.1)
    assert np.all(o[1] == 0.0) and np.all(np.isneginf(lse[1]))
    assert np.all(np.isfinite(lse[0]))


def test_union_against_sets(orc):
    _, _, _, idx = wk.attention_inputs(37, 8, 3000, 50, seed=6, fill=0.9)
    idx[5] = -1                      # an empty token inside a group
    for G in (8, 16):
        for t0 in range(0, 37, G):
            keys, mask = orc.group_union(idx, t0, G)
            toks = range(t0, min(t0 + G, 37))
            want = sorted(set().union(*(set(idx[t][idx[t] >= 0].tolist()) for t in toks)))
            assert keys.tolist() == want
            for key, m in zip(keys.tolist(), mask.tolist()):
                bits = {g for g in range(G) if m >> g & 1}
                assert bits == {t - t0 for t in toks if key in set(idx[t].tolist())}


def test_attention_inputs_are_valid_and_seeded():
    a = wk.attention_inputs(20, 8, 1000, 64, seed=7, own=0.2, fill=0.9)
    b = wk.attention_inputs(20, 8, 1000, 64, seed=7, own=0.2, fill=0.9)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    idx = a[3]
    for row in idx:
        sel = row[row >= 0]
        assert len(sel) == round(0.9 * 64) and np.all(np.diff(sel) > 0) and sel.max() < 1000
        assert np.all(row[len(sel):] == -1)
    # bf16 patterns round to nearest: decoding and re-rounding is the identity
    x = _f(a[1][:4])
    assert np.all(np.isfinite(x)) and np.all(np.abs(x) < 8)
