"""Grouped masked sparse attention on the GPU (dsa_group_union,
dsa_sparse_attention) against the oracle: the unions and masks exactly, the
outputs within a bound derived from the arithmetic.

Bound: q, k, v are bf16 (exact in the oracle's doubles).  The scores come
from fp32 tensor-core accumulation (relative error far below 2^-16 of
sum |q||k|); the softmax weights p are computed in fp32 and rounded to bf16
(relative error <= 2^-9) for the P V product, whose fp32 accumulation adds
far less.  o is a weighted mean of value rows, so |o - o_exact| <=
2^-9 * max_j |v_j| + the score error's effect; the test allows 2^-8 *
max_j |v_j| + 1e-5.  lse uses the unrounded fp32 weights: |error| <= 1e-4 +
1e-5 |lse|.
"""
import math

import numpy as np
import pytest

import workloads as wk
from oracle import default as oracle_default

pytestmark = pytest.mark.gpu


def _torch():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return torch


def _f(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _union_from_ws(ws_np, G, Kc, groups):
    cap = G * Kc
    keys_off = 16
    masks_off = keys_off + ((cap * 4 + 15) & ~15)
    rec = masks_off + ((cap * 4 + 15) & ~15)
    out = []
    for g in range(groups):
        r = ws_np[g * rec:(g + 1) * rec]
        n = int(r[:4].view(np.int32)[0])
        keys = r[keys_off:keys_off + 4 * n].view(np.int32)
        masks = r[masks_off:masks_off + 4 * n].view(np.uint32)
        out.append((keys, masks))
    return out


def _run(T, H, S, Kc, seed, own=0.1, fill=1.0, idx_fn=None, check_union=True, qk_fn=None, scale=None):
    torch = _torch()
    import sparse_attention_indexer_live_gb300 as dsa
    q, k, v, idx = wk.attention_inputs(T, H, S, Kc, seed=seed, own=own, fill=fill, G=128 // H)
    if idx_fn is not None:
        idx = idx_fn(idx)
    if qk_fn is not None:
        q, k = qk_fn(q, k)
    dev = "cuda:0"
    qd, kd, vd, idd = (torch.from_numpy(x.view(np.int16) if x.dtype == np.uint16 else x).to(dev)
                       for x in (q, k, v, idx))
    cfg = dsa.attention_cfg(qd, kd, idd)
    ws = torch.zeros(dsa.dsa_sparse_attention_workspace(cfg), dtype=torch.uint8, device=dev)
    o = torch.full((T, H, 128), 7.0, dtype=torch.float32, device=dev)
    lse = torch.full((T, H), 7.0, dtype=torch.float32, device=dev)
    scale = 1.0 / math.sqrt(128) if scale is None else scale
    dsa.dsa_sparse_attention(cfg, qd, kd, vd, idd, scale, ws, o, lse)
    torch.cuda.synchronize()
    assert dsa.dsa_sparse_attention_status() == dsa.DSA_OK
    orc = oracle_default()
    G = 128 // H
    groups = -(-T // G)
    if check_union:
        got = _union_from_ws(ws.cpu().numpy(), G, Kc, groups)
        for g in range(groups):
            keys, masks = orc.group_union(idx, g * G, G)
            assert np.array_equal(got[g][0], keys), f"union keys of group {g}"
            assert np.array_equal(got[g][1], masks), f"union masks of group {g}"
    o_ref, lse_ref = orc.sparse_attention(q, k, v, idx, scale)
    og, lg = o.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)
    _assert_within_bounds(idx, v, og, lg, o_ref, lse_ref)
    return og, lg


def _assert_within_bounds(idx, v, og, lg, o_ref, lse_ref):
    # per token: o within 2^-8 of the largest |v| over the token's own
    # selection (each weight enters P.V rounded to bf16), lse within 1e-4
    vf = _f(v)
    for t in range(idx.shape[0]):
        sel = idx[t][idx[t] >= 0]
        if len(sel) == 0:
            assert np.all(og[t] == 0.0) and np.all(np.isneginf(lg[t])), f"token {t} (empty)"
            continue
        vmax = np.abs(vf[sel]).max()
        err = np.abs(og[t] - o_ref[t]).max()
        assert err <= 2.0 ** -8 * vmax + 1e-5, f"token {t}: o error {err} vs bound {2.0 ** -8 * vmax}"
        lerr = np.abs(lg[t] - lse_ref[t])
        assert np.all(lerr <= 1e-4 + 1e-5 * np.abs(lse_ref[t])), f"token {t}: lse error {lerr.max()}"


def _bf16_bits(x):
    # float32 -> bf16 bit patterns, rounding to nearest even (finite inputs)
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _rising_scores(q, k):
    # scores that rise with the position: k[j] = 0.55 j / S (+ small noise)
    # in every dim and q = 0.5 (+ noise), so q . k climbs from about 0 to
    # about 35 across the key range -- with scale 1 the row maximum rises by
    # some 50 in base 2 over a group's tiles, far past the threshold at which
    # the kernel moves its running maximum and rescales the accumulated output
    S = k.shape[0]
    rng = np.random.default_rng(5)
    kf = (0.55 * np.arange(S) / S)[:, None] + 0.05 * rng.standard_normal(k.shape)
    qf = 0.5 + 0.05 * rng.standard_normal(q.shape)
    return _bf16_bits(qf), _bf16_bits(kf)


def test_running_maximum_rises_across_tiles():
    # exercises the rescale of O (tile maxima rising by more than 2^8)
    _run(32, 8, 20000, 512, seed=13, own=0.5, qk_fn=_rising_scores, scale=1.0)


def test_union_and_attention_small():
    # 37 tokens (a ragged last group), one 128-position tile or two per group
    _run(37, 8, 5000, 64, seed=1)


def test_sixteen_heads():
    _run(29, 16, 3000, 100, seed=2)


def test_many_tiles_and_low_overlap():
    # large unions: 16 tokens x 300 positions with 40 % of each token's own
    _run(40, 8, 60000, 300, seed=3, own=0.4)


def test_edge_selections():
    def f(idx):
        idx = idx.copy()
        idx[3] = -1                       # nothing selected
        idx[4] = -1
        idx[4, 0] = 17                    # one position
        idx[5, 20:] = -1                  # a shorter row
        idx[20] = -1
        idx[20, :3] = [0, 2500, 4999]     # first and last key
        return idx
    _run(33, 8, 5000, 48, seed=4, idx_fn=f)


def test_selection_width_not_a_multiple_of_four():
    # rows of 50 and 37 entries: the union stages them four bytes at a time
    _run(21, 8, 3000, 50, seed=7, own=0.3)
    _run(13, 16, 2000, 37, seed=8, own=0.3, fill=0.9)


def test_full_key_range_and_wide_selection():
    # 2^20 keys and 2048-entry selections (the row top-k's size)
    _run(32, 8, 1 << 20, 2048, seed=5, own=0.05)


def test_widest_group_rows():
    # G * Kc at its limit: 8 tokens x 6144 positions (16 heads)
    _run(16, 16, 1 << 18, 6144, seed=6, own=0.3)


def _union_only(idx, H, S):
    # dsa_group_union alone against the oracle's union, every group
    torch = _torch()
    import sparse_attention_indexer_live_gb300 as dsa
    T, Kc = idx.shape
    G = 128 // H
    cfg = dsa.dsa_attention_cfg(tokens=T, heads=H, keys=S, head_dim=128, value_dim=128, select=Kc)
    ws = torch.full((dsa.dsa_sparse_attention_workspace(cfg),), 0x5A, dtype=torch.uint8, device="cuda:0")
    dsa.dsa_group_union(cfg, torch.from_numpy(np.ascontiguousarray(idx)).to("cuda:0"), ws)
    torch.cuda.synchronize()
    groups = -(-T // G)
    got = _union_from_ws(ws.cpu().numpy(), G, Kc, groups)
    orc = oracle_default()
    for g in range(groups):
        keys, masks = orc.group_union(idx, g * G, G)
        assert np.array_equal(got[g][0], keys), f"union keys of group {g}"
        assert np.array_equal(got[g][1], masks), f"union masks of group {g}"


def test_union_takes_rows_in_any_order():
    # set semantics: shuffled rows, repeated entries and negative values other
    # than -1 anywhere in a row give the oracle's union (16-byte and 4-byte
    # entry loads)
    rng = np.random.default_rng(14)
    for T, H, S, Kc in ((40, 8, 5000, 64), (27, 16, 3001, 37)):
        _, _, _, idx = wk.attention_inputs(T, H, S, Kc, seed=15, own=0.3, G=128 // H)
        idx = idx.copy()
        for t in range(T):
            rng.shuffle(idx[t])
        idx[rng.integers(0, T, 30), rng.integers(0, Kc, 30)] = -5
        idx[rng.integers(0, T, 10), rng.integers(0, Kc, 10)] = np.iinfo(np.int32).min
        rep = rng.integers(0, T, 40)
        idx[rep, rng.integers(0, Kc, 40)] = idx[rep, rng.integers(0, Kc, 40)]
        _union_only(idx, H, S)


def _selections(T, S, Kc, seed, shared=0.5, lo=0):
    # ascending distinct positions in [lo, lo + S) per token, a fraction
    # `shared` of them common to the token's group of 16 (no key or value rows
    # are made: the union alone is checked)
    rng = np.random.default_rng(seed)
    idx = np.full((T, Kc), -1, dtype=np.int32)
    for g0 in range(0, T, 16):
        base = rng.choice(S, size=int(shared * Kc), replace=False)
        for t in range(g0, min(g0 + 16, T)):
            own = rng.choice(S, size=Kc, replace=False)
            sel = np.unique(np.concatenate([base, own]))[:Kc]
            idx[t, :len(sel)] = np.sort(sel) + lo
    return idx


def test_union_over_several_key_chunks_and_mask_windows():
    # 2^22 keys take several chunks of the key-space bitmap (and a first pass
    # for the extreme entries); unions of ~40,000 positions take several
    # windows of 16-bit masks
    S = (1 << 22) + 12345
    _union_only(_selections(32, S, 3072, seed=16, shared=0.2), 8, S)
    # a narrow band of positions far into a huge key range: only the chunks
    # between the smallest and largest entry are scanned
    _union_only(_selections(16, 1 << 20, 512, seed=17, lo=1 << 30), 8, (1 << 31) - 1)


def _expand_ranges(ranges, S):
    # each token's positions: the union of its ranges clipped to [0, S),
    # ascending, then -1 padding (the index-list form the oracle takes)
    sets = []
    for t in range(ranges.shape[0]):
        pos = set()
        for lo, hi in ranges[t]:
            pos.update(range(max(int(lo), 0), min(int(hi), S)))
        sets.append(sorted(pos))
    width = max(1, max(len(x) for x in sets))
    idx = np.full((ranges.shape[0], width), -1, dtype=np.int32)
    for t, x in enumerate(sets):
        idx[t, :len(x)] = x
    return idx


def _run_ranges(T, H, S, ranges, select, seed, scale=None):
    torch = _torch()
    import sparse_attention_indexer_live_gb300 as dsa
    q, k, v, _ = wk.attention_inputs(T, H, S, 8, seed=seed, G=128 // H)
    idx = _expand_ranges(ranges, S)
    assert idx.shape[1] <= select or not (idx >= 0).any()
    dev = "cuda:0"
    qd, kd, vd = (torch.from_numpy(x.view(np.int16)).to(dev) for x in (q, k, v))
    rd = torch.from_numpy(np.ascontiguousarray(ranges, dtype=np.int32)).to(dev)
    cfg = dsa.ranges_attention_cfg(qd, kd, rd, select)
    ws = torch.full((dsa.dsa_sparse_attention_ranges_workspace(cfg, ranges.shape[1]),), 0x5A,
                    dtype=torch.uint8, device=dev)
    o = torch.full((T, H, 128), 7.0, dtype=torch.float32, device=dev)
    lse = torch.full((T, H), 7.0, dtype=torch.float32, device=dev)
    scale = 1.0 / math.sqrt(128) if scale is None else scale
    dsa.dsa_sparse_attention_ranges(cfg, qd, kd, vd, rd, scale, ws, o, lse)
    torch.cuda.synchronize()
    assert dsa.dsa_sparse_attention_status() == dsa.DSA_OK
    orc = oracle_default()
    G = 128 // H
    groups = -(-T // G)
    got = _union_from_ws(ws.cpu().numpy(), G, select, groups)
    for g in range(groups):
        keys, masks = orc.group_union(idx, g * G, G)
        assert np.array_equal(got[g][0], keys), f"union keys of group {g}"
        assert np.array_equal(got[g][1], masks), f"union masks of group {g}"
    o_ref, lse_ref = orc.sparse_attention(q, k, v, idx, scale)
    _assert_within_bounds(idx, v, o.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
                          o_ref, lse_ref)


def test_ranges_compressed_prefix_and_window():
    # the C128A shape the pages describe: keys [0, Sc) are the compressed
    # prefix (one entry per 128 positions), keys [Sc, Sc + Sr) the raw
    # positions; token t at position p attends to the compressed entries of
    # the blocks before it and to a sliding window of the last w raw positions
    Sr, w, blk = 4096, 256, 128
    Sc = Sr // blk
    T, H = 40, 8
    pos = 3000 + np.arange(T)
    ranges = np.zeros((T, 2, 2), dtype=np.int32)
    ranges[:, 0, 1] = (pos + 1) // blk
    ranges[:, 1, 0] = Sc + np.maximum(0, pos - w + 1)
    ranges[:, 1, 1] = Sc + pos + 1
    _run_ranges(T, H, Sc + Sr, ranges, select=Sc + w, seed=18)


def test_ranges_overlapping_empty_and_clipped():
    # three ranges a token, some overlapping each other or a neighbour's,
    # some empty or reversed, some reaching below 0 or past S; 16 heads
    rng = np.random.default_rng(19)
    T, H, S = 27, 16, 3000
    lo = rng.integers(-200, S, size=(T, 3))
    ln = rng.integers(-50, 400, size=(T, 3))
    ranges = np.stack([lo, lo + ln], axis=2).astype(np.int32)
    ranges[5] = [[10, 10], [200, 100], [-30, -1]]  # nothing selected
    ranges[6] = [[S - 5, S + 50], [0, 3], [1, 2]]  # the first and last keys
    _run_ranges(T, H, S, ranges, select=3 * 450, seed=20)


def test_ranges_at_the_limits():
    # 8 ranges a token and 16 tokens a group: 256 end points, the most the
    # sweep takes; end points shared between tokens (ties in the sort),
    # ranges touching inside a token (merged), and a ragged last group
    rng = np.random.default_rng(25)
    T, H, S = 37, 8, 2000
    grid = np.arange(0, S + 1, 50)  # shared end points
    lo = rng.choice(grid[:-1], size=(T, 8))
    ln = 50 * rng.integers(0, 4, size=(T, 8))
    ranges = np.stack([lo, lo + ln], axis=2).astype(np.int32)
    ranges[3, :, 0] = np.arange(8) * 100  # touching pairs inside one token
    ranges[3, :, 1] = np.arange(8) * 100 + 100
    _run_ranges(T, H, S, ranges, select=8 * 150 + 800, seed=26)


def test_ranges_graph_replay_follows_new_ranges():
    # the range form captured once replays on new ranges written into the
    # captured buffer, and gives what a direct call gives
    torch = _torch()
    import sparse_attention_indexer_live_gb300 as dsa
    T, H, S = 33, 8, 5000
    q, k, v, _ = wk.attention_inputs(T, H, S, 8, seed=23)
    rng = np.random.default_rng(24)

    def ranges():
        lo = rng.integers(0, S, size=(T, 2))
        return np.stack([lo, lo + rng.integers(0, 300, size=(T, 2))], axis=2).astype(np.int32)

    dev = "cuda:0"
    qd, kd, vd = (torch.from_numpy(x.view(np.int16)).to(dev) for x in (q, k, v))
    r0 = ranges()
    rd = torch.from_numpy(r0).to(dev)
    cfg = dsa.ranges_attention_cfg(qd, kd, rd, 600)
    ws = torch.zeros(dsa.dsa_sparse_attention_ranges_workspace(cfg, 2), dtype=torch.uint8, device=dev)
    o = torch.empty((T, H, 128), dtype=torch.float32, device=dev)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    scale = 1.0 / math.sqrt(128)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        dsa.dsa_sparse_attention_ranges(cfg, qd, kd, vd, rd, scale, ws, o, lse, stream=stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        dsa.dsa_sparse_attention_ranges(cfg, qd, kd, vd, rd, scale, ws, o, lse, stream=stream)
    for sel in (ranges(), r0):
        rd.copy_(torch.from_numpy(sel))
        graph.replay()
        torch.cuda.synchronize()
        og, lg = o.clone(), lse.clone()
        dsa.dsa_sparse_attention_ranges(cfg, qd, kd, vd, rd, scale, ws, o, lse)
        torch.cuda.synchronize()
        assert torch.equal(og, o) and torch.equal(lg, lse)
    assert dsa.dsa_sparse_attention_status() == dsa.DSA_OK
    idx = _expand_ranges(r0, S)
    o_ref, lse_ref = oracle_default().sparse_attention(q, k, v, idx, scale)
    _assert_within_bounds(idx, v, og.cpu().numpy().astype(np.float64), lg.cpu().numpy().astype(np.float64),
                          o_ref, lse_ref)


def test_graph_replay_follows_new_selections():
    # both launches take their grids from the shapes only: a captured call
    # replays on new selections (written into the captured buffers) and gives
    # what a direct call gives
    torch = _torch()
    import sparse_attention_indexer_live_gb300 as dsa
    T, H, S, Kc = 40, 8, 20000, 256
    q, k, v, idx0 = wk.attention_inputs(T, H, S, Kc, seed=10, own=0.2)
    _, _, _, idx1 = wk.attention_inputs(T, H, S, Kc, seed=11, own=0.6, fill=0.7)
    dev = "cuda:0"
    qd, kd, vd = (torch.from_numpy(x.view(np.int16)).to(dev) for x in (q, k, v))
    idd = torch.from_numpy(idx0).to(dev)
    cfg = dsa.attention_cfg(qd, kd, idd)
    ws = torch.zeros(dsa.dsa_sparse_attention_workspace(cfg), dtype=torch.uint8, device=dev)
    o = torch.empty((T, H, 128), dtype=torch.float32, device=dev)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    scale = 1.0 / math.sqrt(128)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        dsa.dsa_sparse_attention(cfg, qd, kd, vd, idd, scale, ws, o, lse, stream=stream)  # warm-up
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        dsa.dsa_sparse_attention(cfg, qd, kd, vd, idd, scale, ws, o, lse, stream=stream)
    for sel in (idx1, idx0):
        idd.copy_(torch.from_numpy(sel))
        graph.replay()
        torch.cuda.synchronize()
        og, lg = o.clone(), lse.clone()
        dsa.dsa_sparse_attention(cfg, qd, kd, vd, idd, scale, ws, o, lse)
        torch.cuda.synchronize()
        assert torch.equal(og, o) and torch.equal(lg, lse)
    assert dsa.dsa_sparse_attention_status() == dsa.DSA_OK
    # and the replayed result is the oracle's (selection idx0)
    o_ref, lse_ref = oracle_default().sparse_attention(q, k, v, idx0, scale)
    _assert_within_bounds(idx0, v, og.cpu().numpy().astype(np.float64),
                          lg.cpu().numpy().astype(np.float64), o_ref, lse_ref)


def test_no_keys_and_no_tokens():
    # zero key rows: every selection is empty (o = 0, lse = -inf) and the
    # key / value pointers are never read; zero tokens: nothing runs
    torch = _torch()
    import sparse_attention_indexer_live_gb300 as dsa
    dev = "cuda:0"
    T, H, Kc = 20, 16, 32
    q, _, _, _ = wk.attention_inputs(T, H, 100, Kc, seed=12)
    qd = torch.from_numpy(q.view(np.int16)).to(dev)
    kd = torch.empty((0, 128), dtype=torch.int16, device=dev)
    vd = torch.empty((0, 128), dtype=torch.int16, device=dev)
    idd = torch.full((T, Kc), -1, dtype=torch.int32, device=dev)
    cfg = dsa.attention_cfg(qd, kd, idd)
    ws = torch.full((dsa.dsa_sparse_attention_workspace(cfg),), 0x5A, dtype=torch.uint8, device=dev)
    o = torch.full((T, H, 128), 7.0, dtype=torch.float32, device=dev)
    lse = torch.full((T, H), 7.0, dtype=torch.float32, device=dev)
    dsa.dsa_sparse_attention(cfg, qd, kd, vd, idd, 0.1, ws, o, lse)
    torch.cuda.synchronize()
    assert dsa.dsa_sparse_attention_status() == dsa.DSA_OK
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
    q0 = torch.empty((0, H, 128), dtype=torch.int16, device=dev)
    i0 = torch.empty((0, Kc), dtype=torch.int32, device=dev)
    cfg0 = dsa.attention_cfg(q0, kd, i0)
    assert dsa.dsa_sparse_attention_workspace(cfg0) == 0
    ws0 = torch.empty(0, dtype=torch.uint8, device=dev)
    o0 = torch.empty((0, H, 128), dtype=torch.float32, device=dev)
    l0 = torch.empty((0, H), dtype=torch.float32, device=dev)
    dsa.dsa_sparse_attention(cfg0, q0, kd, vd, i0, 0.1, ws0, o0, l0)
    torch.cuda.synchronize()
    assert dsa.dsa_sparse_attention_status() == dsa.DSA_OK


def test_unsupported_shapes():
    torch = _torch()
    import sparse_attention_indexer_live_gb300 as dsa
    n = torch.empty(1)
    for kw in (dict(heads=4), dict(head_dim=64), dict(select=3073)):
        c = dict(tokens=8, heads=8, keys=1000, head_dim=128, value_dim=128, select=16)
        c.update(kw)
        with pytest.raises(dsa.DsaSelectError) as e:
            dsa.dsa_sparse_attention_workspace(dsa.dsa_attention_cfg(**c))
        assert e.value.status == dsa.DSA_ERR_UNSUPPORTED
    del n
