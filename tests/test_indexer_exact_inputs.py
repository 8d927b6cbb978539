"""The exact-arithmetic inputs of the fused producer + selection test, and
the oracle's indexer logits on them.

On these inputs (small e4m3 integers, power-of-two head weights and key
scales) the indexer score of the pages' FP8 MQA indexer (vLLM PR #48726,
Motivation: a score for every query/KV pair) has an exact value that integer
arithmetic gives directly: each head's dot product is an integer, the
weighted head sum a multiple of 1/4 below 2^17.  The oracle's fp64 logits,
rounded to fp32, must equal that value bit for bit -- which is what lets the
GPU path's fused selection be compared with the oracle end to end, with no
GPU value fed to the oracle."""
import numpy as np

import workloads as wk
from oracle import default as oracle_default


def _ints(b):
    dec = {v: k for k, v in wk.E4M3_INT.items()}
    return np.vectorize(dec.get, otypes=[np.int64])(b)


def test_e4m3_table_matches_the_oracle_decoder():
    orc = oracle_default()
    for v, b in wk.E4M3_INT.items():
        assert orc.e4m3(b) == float(v)


def test_oracle_logits_equal_the_integer_formula():
    T, S = 5, 1500
    q, k, ks, w, _, ends = wk.indexer_exact_inputs(T, S, seed=4)
    ends = ends.copy()
    ends[0], ends[1] = 0, S + 9  # an empty span and one past the width
    qi, ki = _ints(q), _ints(k)
    dots = np.einsum("thd,sd->ths", qi, ki)                  # exact integers
    assert np.abs(dots).max() <= 768
    w4 = (w.astype(np.float64) * 4).astype(np.int64)
    assert np.array_equal(w4 / 4.0, w.astype(np.float64))    # powers of two in [1/4, 2]
    total4 = np.einsum("th,ths->ts", w4, np.maximum(dots, 0))  # 4 x the head sum
    assert total4.max() < 4 * 2 ** 17
    exact = (total4 * ks.astype(np.float64)[None, :] / 4.0).astype(np.float32)
    out = np.full((T, S), 1.5, dtype=np.float32)
    oracle_default().indexer_logits(q, k, ks, w, None, ends, out)
    for t in range(T):
        e = min(max(int(ends[t]), 0), S)
        assert np.array_equal(out[t, :e].view(np.uint32), exact[t, :e].view(np.uint32)), t
        assert np.all(out[t, e:] == 1.5), t


def test_inputs_have_ties():
    # equal logits across blocks and inside blocks: the tie-breaks are exercised
    T, S = 3, 4096
    q, k, ks, w, _, ends = wk.indexer_exact_inputs(T, S, seed=5)
    out = np.zeros((T, S), dtype=np.float32)
    oracle_default().indexer_logits(q, k, ks, w, None, ends, out)
    for t in range(T):
        vals, counts = np.unique(out[t, :ends[t]], return_counts=True)
        assert counts.max() >= 20 and (counts > 1).sum() >= 50
