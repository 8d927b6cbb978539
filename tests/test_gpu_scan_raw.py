"""Scan-mode row top-k (dsa_row_topk with cand = NULL) on raw, unmasked logits
against the oracle's row top-k of the same rows; and a CUDA-graph replay of
the cluster-split path with changing ends."""
import random

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import workloads as wk
from tests import brute

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import sparse_attention_indexer_live_gb300 as dsa
    dsa.build()


def _scan(x, starts, ends, W, K, cs=1, rep=1, causal=True):
    import sparse_attention_indexer_live_gb300 as dsa
    rows = x.shape[0]
    plan = dsa.dsa_select_init(rows=rows, width=W, block_size=8, block_topk=16, row_topk=K,
                               row_stride=x.shape[1], col_stride=cs, row_repeat=rep,
                               repeat_causal=causal, has_starts=starts is not None)
    buf = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    logits = buf.as_strided((rows, W), (x.shape[1], cs))
    st = None if starts is None else torch.tensor(starts, dtype=torch.int32).cuda()
    en = torch.tensor(ends, dtype=torch.int32).cuda()
    topk = torch.full((rows, K), -7, dtype=torch.int32).cuda()
    dsa.dsa_row_topk(plan, logits, st, en, None, topk)
    torch.cuda.synchronize()
    # bit patterns (the data holds NaNs, which never compare equal as floats)
    assert np.array_equal(buf.cpu().numpy().view(np.uint32),
                          np.ascontiguousarray(x).view(np.uint32)), "scan mode wrote logits"
    return topk.cpu().numpy()


def _want(x, starts, ends, W, K, cs=1, rep=1, causal=True):
    orc = oracle.default()
    out = []
    for r in range(x.shape[0]):
        s, e = orc.bounds(r, starts, ends, rep, causal)
        out.append(orc.row_topk(x[r], W, s, e, K, col_stride=cs))
    return np.stack(out)


def test_scan_on_raw_workload_rows():
    for name in ("tiny", "ragged", "decode_short"):
        wl = wk.WORKLOADS[name]
        x, starts, ends = wk.make_all(wl)
        got = _scan(x, starts, ends, wl.width, wl.row_topk, wl.col_stride, wl.row_repeat)
        assert np.array_equal(got, _want(x, starts, ends, wl.width, wl.row_topk, wl.col_stride,
                                         wl.row_repeat)), name


def test_scan_on_raw_heavy_ties_and_specials():
    rng = random.Random(5)
    for trial in range(40):
        W = rng.choice([37, 1000, 5003, 70_000])
        rows = rng.randint(1, 6)
        K = rng.choice([1, 7, 64, 2048, 4096])
        pool = brute.VALUE_POOL + brute.EXOTIC_POOL
        x = np.array([[brute.to_bits(rng.choice(pool)) for _ in range(W)] for _ in range(rows)],
                     dtype=np.uint32)
        x[np.array([[rng.random() < 0.01 for _ in range(W)] for _ in range(rows)])] = \
            rng.choice(brute.NAN_BITS)
        x = x.view(np.float32)
        starts = [rng.randint(0, W // 2) for _ in range(rows)]
        ends = [rng.randint(-1, W + 9) for _ in range(rows)]
        got = _scan(x, starts, ends, W, K)
        assert np.array_equal(got, _want(x, starts, ends, W, K)), trial


def test_cluster_path_graph_replay():
    import sparse_attention_indexer_live_gb300 as dsa
    from tests.gpu_util import Case, DeviceRun, assert_run_matches
    rng = np.random.default_rng(9)
    W, rows = 1 << 19, 3
    x = rng.standard_normal((rows, W)).astype(np.float32)
    case = Case(x, None, [W, 100_000, 3000], width=W, block_size=8, block_topk=256,
                row_topk=2048, split=8)
    run = DeviceRun(case)
    assert run.plan.describe()["split"] == 8
    base = run.buf.clone()
    dsa.dsa_select_topk(run.plan, run.logits, None, run.ends, run.cand, run.topk)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        dsa.dsa_select_topk(run.plan, run.logits, None, run.ends, run.cand, run.topk, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for replay in ([1, W, 0], [W + 3, 7, 400_001], [250_000, 250_001, W]):
        run.ends.copy_(torch.tensor(replay, dtype=torch.int32))
        run.buf.copy_(base)
        g.replay()
        torch.cuda.synchronize()
        c2 = Case(x, None, replay, width=W, block_size=8, block_topk=256, row_topk=2048)
        want = c2.oracle()
        assert_run_matches(run, *want, what=f"cluster replay {replay}")
