"""The indexer producer fused with the selection (dsa_indexer_select).

Its cand and topk must equal, bit for bit, (a) the two-step path on the same
inputs -- the producer's materialised logits, then dsa_select_topk -- and (b)
the oracle's selection run on those same logits (the oracle computes logits in
fp64, so the selection is compared on the GPU's fp32 logits, which both paths
share exactly).
"""
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


def _inputs(T, S, seed, ends=None, ks_fn=None):
    q, k, ks, w, _, en = wk.indexer_inputs(T, S, seed)
    if ends is not None:
        en = np.asarray(ends, dtype=np.int32)
    if ks_fn is not None:
        ks = np.ascontiguousarray(ks_fn(ks.copy()), dtype=np.float32)
    return q, k, ks, w, en


def _run(T, S, B, Kb, K, seed, ends=None, ks_fn=None, oracle_rows=None):
    torch = _torch()
    import sparse_attention_indexer_live_gb300 as dsa
    q, k, ks, w, en = _inputs(T, S, seed, ends, ks_fn)
    dev = "cuda:0"
    qd, kd, ksd, wd, end = (torch.from_numpy(x).to(dev) for x in (q, k, ks, w, en))
    plan = dsa.dsa_select_init(rows=T, width=S, block_size=B, block_topk=Kb, row_topk=K)
    # two-step reference path
    logits = torch.full((T, S), 3.0, dtype=torch.float32, device=dev)
    dsa.dsa_indexer_logits(qd, kd, ksd, wd, None, end, logits)
    raw = logits.clone()
    cand_ref = torch.empty((T, Kb + 1), dtype=torch.int32, device=dev)
    topk_ref = torch.empty((T, K), dtype=torch.int32, device=dev)
    dsa.dsa_select_topk(plan, logits, None, end, cand_ref, topk_ref)
    # fused path, on a workspace full of junk (it must not need zeroing)
    nbytes = dsa.dsa_indexer_select_workspace(plan)
    g = torch.Generator(device="cpu").manual_seed(seed)
    ws = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, generator=g).to(dev)
    cand = torch.full((T, Kb + 1), -7, dtype=torch.int32, device=dev)
    topk = torch.full((T, K), -7, dtype=torch.int32, device=dev)
    dsa.dsa_indexer_select(plan, qd, kd, ksd, wd, end, ws, cand, topk)
    torch.cuda.synchronize()
    assert dsa.dsa_indexer_status() == dsa.DSA_OK
    assert torch.equal(cand, cand_ref), "cand differs from the two-step path"
    assert torch.equal(topk, topk_ref), "topk differs from the two-step path"
    # the oracle's selection on the producer's logits
    rows = range(T) if oracle_rows is None else oracle_rows
    raw_np = raw.cpu().numpy()
    orc = oracle_default()
    c_got, t_got = cand.cpu().numpy(), topk.cpu().numpy()
    for r in rows:
        row = np.ascontiguousarray(raw_np[r:r + 1])
        c_o, t_o = orc.run(row, None, en[r:r + 1], width=S, block_size=B, block_topk=Kb,
                           row_topk=K)
        assert np.array_equal(c_got[r], c_o[0]), f"cand row {r}"
        assert np.array_equal(t_got[r], t_o[0]), f"topk row {r}"
    return plan, c_got, t_got


def test_decode_shape_causal():
    # 128K keys, block 8, Kb 256, k 2048; a ragged last CTA (37 = 9 * 4 + 1)
    _run(37, 131072, 8, 256, 2048, seed=11)


def test_edge_ends():
    # empty rows, spans inside one block, one tile, exactly the width, past the
    # width (the pin lies past W: edge flag), a negative end; S not a multiple
    # of the 128-key tile
    ends = [0, 1, 7, 8, 9, 127, 128, 129, 4999, 5000, 5003, -3]
    _run(len(ends), 5000, 8, 32, 64, seed=12, ends=ends)


@pytest.mark.parametrize("B,Kb,K", [(1, 40, 128), (2, 100, 300), (4, 256, 700), (8, 1, 16),
                                    (1, 1000, 1500)])
def test_block_sizes(B, Kb, K):
    ends = [3001, 2500, 1, 0, 3001, 64, 1000, 2999, 3005]
    _run(len(ends), 3001, B, Kb, K, seed=13 + B, ends=ends)


def test_fewer_blocks_than_kb():
    # NB = 13 < Kb: -inf padding blocks fill the block top-k
    _run(5, 100, 8, 32, 40, seed=14, ends=[100, 50, 3, 0, 101])


def test_ascending_scores_many_compactions():
    # key scales rising with the key: most blocks beat the running threshold,
    # so the streaming buffer compacts every few tiles
    _run(16, 65536, 8, 256, 2048, seed=15,
         ks_fn=lambda ks: np.linspace(0.5, 50.0, ks.size))


def test_zero_scale_ties_and_signed_zeros():
    # long runs of zero scale: +0 / -0 logits, block maxima tied across blocks
    def f(ks):
        ks[1000:40000] = 0.0
        ks[50000:50100] = 0.0
        return ks
    _run(12, 65536, 8, 256, 2048, seed=16, ks_fn=f)


def test_infinite_scales():
    # +-inf logits where the scale is inf (and NaN where the head sum is zero)
    def f(ks):
        ks[[5, 777, 20000, 65535]] = np.inf
        return ks
    _run(8, 65536, 8, 256, 2048, seed=17, ks_fn=f)


def test_full_width_1m():
    # the 1M-key width of the long-context workloads; the oracle checks 3 rows
    _run(8, 1 << 20, 8, 256, 2048, seed=18, oracle_rows=[0, 5, 7])


def test_bench_shape_sampled():
    # the benchmark's shape (608 queries x 131072 keys); every row against the
    # two-step path, sampled rows against the oracle
    _run(608, 131072, 8, 256, 2048, seed=19, oracle_rows=[0, 151, 303, 607])


def test_graph_replay_follows_new_ends():
    torch = _torch()
    import sparse_attention_indexer_live_gb300 as dsa
    T, S, B, Kb, K = 20, 40000, 8, 256, 2048
    q, k, ks, w, en = _inputs(T, S, seed=20)
    dev = "cuda:0"
    qd, kd, ksd, wd, end = (torch.from_numpy(x).to(dev) for x in (q, k, ks, w, en))
    plan = dsa.dsa_select_init(rows=T, width=S, block_size=B, block_topk=Kb, row_topk=K)
    ws = torch.empty(dsa.dsa_indexer_select_workspace(plan), dtype=torch.uint8, device=dev)
    cand = torch.empty((T, Kb + 1), dtype=torch.int32, device=dev)
    topk = torch.empty((T, K), dtype=torch.int32, device=dev)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dsa.dsa_indexer_select(plan, qd, kd, ksd, wd, end, ws, cand, topk, stream=s)  # warm
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            dsa.dsa_indexer_select(plan, qd, kd, ksd, wd, end, ws, cand, topk, stream=s)
    rng = np.random.default_rng(20)
    for _ in range(3):
        new = rng.integers(-2, S + 5, size=T).astype(np.int32)
        end.copy_(torch.from_numpy(new))
        g.replay()
        torch.cuda.synchronize()
        c_eager = torch.empty_like(cand)
        t_eager = torch.empty_like(topk)
        dsa.dsa_indexer_select(plan, qd, kd, ksd, wd, end, ws, c_eager, t_eager)
        torch.cuda.synchronize()
        assert torch.equal(cand, c_eager) and torch.equal(topk, t_eager)
    assert dsa.dsa_indexer_status() == dsa.DSA_OK


def test_unsupported_and_invalid():
    torch = _torch()
    import sparse_attention_indexer_live_gb300 as dsa
    dev = "cuda:0"
    T, S = 4, 1000
    q, k, ks, w, en = _inputs(T, S, seed=21)
    qd, kd, ksd, wd, end = (torch.from_numpy(x).to(dev) for x in (q, k, ks, w, en))
    cand = torch.empty((T, 33), dtype=torch.int32, device=dev)
    topk = torch.empty((T, 64), dtype=torch.int32, device=dev)
    for shape in (dict(block_size=16, block_topk=32), dict(block_size=8, block_topk=32, row_repeat=2),
                  dict(block_size=6, block_topk=32), dict(block_size=8, block_topk=32,
                                                          has_starts=True)):
        plan = dsa.dsa_select_init(rows=T, width=S, row_topk=64, **shape)
        with pytest.raises(dsa.DsaSelectError) as e:
            dsa.dsa_indexer_select_workspace(plan)
        assert e.value.status == dsa.DSA_ERR_UNSUPPORTED
    plan = dsa.dsa_select_init(rows=T, width=S, block_size=8, block_topk=32, row_topk=64)
    need = dsa.dsa_indexer_select_workspace(plan)
    small = torch.empty(need - 16, dtype=torch.uint8, device=dev)
    with pytest.raises(dsa.DsaSelectError) as e:
        dsa.dsa_indexer_select(plan, qd, kd, ksd, wd, end, small, cand, topk)
    assert e.value.status == dsa.DSA_ERR_INVALID_ARG
    # the plan's width must be the key count: the binding refuses it on the
    # host, and so does the C ABI when called directly
    other = dsa.dsa_select_init(rows=T, width=S + 1, block_size=8, block_topk=32, row_topk=64)
    ws = torch.empty(dsa.dsa_indexer_select_workspace(other), dtype=torch.uint8, device=dev)
    with pytest.raises(ValueError):
        dsa.dsa_indexer_select(other, qd, kd, ksd, wd, end, ws, cand, topk)
    import ctypes
    from sparse_attention_indexer_live_gb300 import binding
    icfg = binding.dsa_indexer_cfg(queries=T, keys=S, heads=64, head_dim=128, out_stride=S)
    ptr = binding._ptr
    st = dsa.load().dsa_indexer_select(other.handle, ctypes.byref(icfg), ptr(qd), ptr(kd), ptr(ksd),
                                       ptr(wd), ptr(end), ptr(ws), ws.numel(), ptr(cand), ptr(topk),
                                       binding._stream(None))
    assert st == dsa.DSA_ERR_INVALID_ARG
    # undersized outputs never reach the library
    with pytest.raises(ValueError):
        dsa.dsa_indexer_select(plan, qd, kd, ksd, wd, end, ws, cand[:3], topk)
    torch.cuda.synchronize()
    assert dsa.dsa_indexer_status() == dsa.DSA_OK
