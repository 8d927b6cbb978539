"""The numerics the grouped attention kernel relies on, checked on the CPU.

A model of its per-row arithmetic -- walk the group's union in tiles of 128
positions, fp32 scores, base-2 exponentials against a running maximum that
moves only when the row's maximum rises by more than 8, weights rounded to
bf16 for the P V product while the normaliser sums the fp32 weights, O and
the sum rescaled when the maximum moves -- must stay within the tolerances
the GPU parity tests assert against the fp64 oracle: 2^-8 max|v| for o and
1e-4 + 1e-5 |lse| for lse.  This pins the design (threshold, rounding points),
not the CUDA code, which the GPU tests compare with the oracle directly.
"""
import math

import numpy as np

import workloads as wk
from oracle import default as oracle_default


def _f(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _bf16_round(x):
    # float32 -> nearest-even bf16 value (finite inputs)
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return (((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16).astype(np.uint32).view(np.float32)


def _model(q, k, v, idx, scale, G):
    """Per token/head row: the union tiles in order, fp32 throughout."""
    T, H, _ = q.shape
    qf, kf, vf = _f(q), _f(k), _f(v)
    c2 = np.float32(scale * math.log2(math.e))
    o = np.zeros((T, H, v.shape[1]), np.float64)
    lse = np.full((T, H), -np.inf)
    moves = 0
    for g0 in range(0, T, G):
        toks = range(g0, min(g0 + G, T))
        union = sorted(set().union(*(set(idx[t][idx[t] >= 0].tolist()) for t in toks)))
        for t in toks:
            sel = set(idx[t][idx[t] >= 0].tolist())
            for h in range(H):
                m, l = np.float32(-np.inf), np.float32(0)
                acc = np.zeros(v.shape[1], np.float32)
                for i0 in range(0, len(union), 128):
                    keys = union[i0:i0 + 128]
                    s = (kf[keys] @ qf[t, h]).astype(np.float32)
                    s[[kk not in sel for kk in keys]] = -np.inf
                    smax = np.float32(s.max() * c2)
                    m_new = max(m, smax)
                    alpha = np.float32(1)
                    if m == -np.inf:
                        m = m_new
                    elif m_new > m + 8:
                        alpha = np.float32(2.0 ** float(m - m_new))
                        m = m_new
                        moves += 1
                    if m == -np.inf:
                        continue
                    # the kernel fuses s c - m into one multiply-add; two roundings here
                    p = np.exp2((s * c2 - m).astype(np.float32)).astype(np.float32)
                    l = np.float32(l * alpha + p.sum(dtype=np.float32))
                    acc = (acc * alpha + _bf16_round(p) @ vf[keys]).astype(np.float32)
                if l > 0:
                    o[t, h] = acc / l
                    lse[t, h] = (float(m) + math.log2(float(l))) * math.log(2)
    return o, lse, moves


def _check(q, k, v, idx, scale, G):
    o, lse, moves = _model(q, k, v, idx, scale, G)
    o_ref, lse_ref = oracle_default().sparse_attention(q, k, v, idx, scale)
    vf = _f(v).astype(np.float64)
    for t in range(q.shape[0]):
        sel = idx[t][idx[t] >= 0]
        if len(sel) == 0:
            assert np.all(o[t] == 0) and np.all(np.isneginf(lse[t]))
            continue
        bound = 2.0 ** -8 * np.abs(vf[sel]).max() + 1e-5
        assert np.abs(o[t] - o_ref[t]).max() <= bound
        assert np.all(np.abs(lse[t] - lse_ref[t]) <= 1e-4 + 1e-5 * np.abs(lse_ref[t]))
    return moves


def test_model_within_tolerance_on_ordinary_scores():
    q, k, v, idx = wk.attention_inputs(20, 8, 3000, 200, seed=3, own=0.4, G=16)
    assert _check(q, k, v, idx, 1.0 / math.sqrt(128), 16) == 0  # the maximum never moves


def test_model_within_tolerance_when_the_maximum_moves():
    # scores rising with the position (as in the GPU test of the rescale):
    # the running maximum must move, and the result still meets the bound
    T, H, S, Kc = 16, 8, 6000, 256
    q, k, v, idx = wk.attention_inputs(T, H, S, Kc, seed=13, own=0.5, G=16)
    rng = np.random.default_rng(5)
    kf = (0.55 * np.arange(S) / S)[:, None] + 0.05 * rng.standard_normal(k.shape)
    qf = 0.5 + 0.05 * rng.standard_normal(q.shape)
    qb = (_bf16_round(qf).view(np.uint32) >> 16).astype(np.uint16)
    kb = (_bf16_round(kf).view(np.uint32) >> 16).astype(np.uint16)
    moves = _check(qb, kb, v, idx, 1.0, 16)
    assert moves >= T * H  # at least one move per row on average
