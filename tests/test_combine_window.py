"""The top-k / sliding-window combine: oracle pins (closed forms, hand-worked
rows, a set-union formulation) and GPU parity through the C ABI."""
import random

import numpy as np
import pytest

from oracle import default as oracle_default


@pytest.fixture(scope="module")
def orc():
    return oracle_default()


def test_hand_worked(orc):
    # topk {2, 5, 9} and the last 3 of [0, 12) = {9, 10, 11}: 9 appears once
    assert orc.combine_window([2, 5, 9, -1, -1], 0, 12, 16, 3).tolist() == \
        [2, 5, 9, 10, 11, -1, -1, -1]
    # end 20 past W = 16: the window is the last 3 columns of [0, 16)
    assert orc.combine_window([2, 5, 14], 0, 20, 16, 3).tolist() == [2, 5, 13, 14, 15, -1]
    # start 4, end 6: the window cannot reach below the start
    assert orc.combine_window([4, -1], 4, 6, 16, 5).tolist() == [4, 5, -1, -1, -1, -1, -1]
    # empty row: only padding
    assert orc.combine_window([-1, -1], 3, 3, 16, 2).tolist() == [-1, -1, -1, -1]


def test_window_zero_is_the_topk(orc):
    rng = np.random.default_rng(1)
    for _ in range(50):
        t = np.sort(rng.choice(1000, size=int(rng.integers(0, 20)), replace=False))
        K = len(t) + int(rng.integers(0, 5))
        row = np.concatenate([t, -np.ones(K - len(t), dtype=np.int64)])
        assert orc.combine_window(row, 0, 1000, 1000, 0).tolist() == row.tolist()


def test_full_window_is_the_span(orc):
    rng = np.random.default_rng(2)
    for _ in range(50):
        s = int(rng.integers(0, 50))
        e = s + int(rng.integers(1, 200))
        t = np.sort(rng.choice(np.arange(s, e), size=min(8, e - s), replace=False))
        out = orc.combine_window(t, s, e, 10_000, e - s + int(rng.integers(0, 10)))
        n = e - s
        assert out[:n].tolist() == list(range(s, e)) and np.all(out[n:] == -1)


def test_set_union_on_random_rows(orc):
    rng = random.Random(3)
    for _ in range(2000):
        W = rng.randint(1, 40)
        s = rng.randint(0, W + 2)
        e = rng.randint(-2, W + 5)
        ec = min(e, W)
        K = rng.randint(1, 12)
        live = list(range(s, ec)) if ec > s else []
        t = sorted(rng.sample(live, min(len(live), rng.randint(0, K))))
        row = t + [-1] * (K - len(t))
        window = rng.randint(0, 10)
        w1 = max(ec, s)
        want = sorted(set(t) | set(range(max(s, w1 - window), w1)))
        want += [-1] * (K + window - len(want))
        assert orc.combine_window(row, s, e, W, window).tolist() == want


@pytest.mark.gpu
def test_gpu_matches_oracle(orc):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import sparse_attention_indexer_live_gb300 as dsa
    import workloads as wk
    dsa.build()
    rng = np.random.default_rng(4)
    for name in ("tiny", "ragged", "decode_1m"):
        wl = wk.WORKLOADS[name]
        x, starts, ends = wk.make_all(wl)
        plan = dsa.dsa_select_init(rows=wl.rows, width=wl.width, block_size=wl.block_size,
                                   block_topk=wl.block_topk, row_topk=wl.row_topk,
                                   row_stride=wl.row_stride, col_stride=wl.col_stride,
                                   row_repeat=wl.row_repeat, has_starts=starts is not None)
        dev = "cuda:0"
        buf = torch.from_numpy(x).to(dev)
        logits = buf.as_strided((wl.rows, wl.width), (wl.row_stride, wl.col_stride))
        st = None if starts is None else torch.from_numpy(starts).to(dev)
        en = torch.from_numpy(ends).to(dev)
        cand = torch.empty((wl.rows, wl.block_topk + 1), dtype=torch.int32, device=dev)
        topk = torch.empty((wl.rows, wl.row_topk), dtype=torch.int32, device=dev)
        dsa.dsa_select_topk(plan, logits, st, en, cand, topk)
        for window in (0, 1, 64, 4096, int(rng.integers(2, 3000))):
            out = torch.full((wl.rows, wl.row_topk + window), -7, dtype=torch.int32, device=dev)
            dsa.dsa_combine_window(plan, st, en, topk, window, out)
            torch.cuda.synchronize()
            got = out.cpu().numpy()
            tk = topk.cpu().numpy()
            for r in range(wl.rows):
                s, e = orc.bounds(r, starts, ends, wl.row_repeat, True)
                want = orc.combine_window(tk[r], s, e, wl.width, window)
                assert np.array_equal(got[r], want), (name, window, r)
