"""GPU parity: the CUDA path through the C ABI against the CPU oracle, element
by element, on the same seeded inputs.  Logits are compared as uint32 bit
patterns over the whole allocation (guard bands included), cand and topk
exactly.  Every mode is checked: fused select+top-k, select then candidate-
mode top-k, and scan-mode top-k on the masked logits."""
import random

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads as wk
from tests import brute
from tests.common import load_golden, parse_row
from tests.gpu_util import Case, DeviceRun, assert_run_matches

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import sparse_attention_indexer_live_gb300 as dsa
    dsa.build()
    dsa.load()


def check_all_modes(case: Case, misalign=0, what=""):
    want_logits, want_cand, want_topk = case.oracle()
    # fused
    run = DeviceRun(case, misalign=misalign).fused()
    assert_run_matches(run, want_logits, want_cand, want_topk, what + " [fused]")
    # separate: select, then candidate-mode row top-k
    run = DeviceRun(case, misalign=misalign).select().topk_cand()
    assert_run_matches(run, want_logits, want_cand, want_topk, what + " [select+cand]")
    # scan mode on the masked logits gives the same top-k
    scan = torch.full_like(run.topk, -7)
    run.topk_scan(scan)
    torch.cuda.synchronize()
    assert np.array_equal(scan.cpu().numpy(), want_topk), what + " [scan]"


@pytest.mark.parametrize("case", load_golden()["cases"], ids=lambda c: c["name"])
def test_hand_worked_rows_on_gpu(case):
    x = np.stack([parse_row(r) for r in case["x"]])
    c = Case(x, case["starts"], case["ends"], width=case["width"],
             block_size=case["block_size"], block_topk=case["block_topk"],
             row_topk=case["row_topk"], row_repeat=case["row_repeat"], causal=case["causal"])
    want_logits, want_cand, want_topk = c.oracle()
    assert want_cand.tolist() == case["cand"] and want_topk.tolist() == case["topk"]
    check_all_modes(c, what=case["name"])


def _random_small(rng: random.Random, exotic: bool):
    W = rng.randint(1, 80)
    B = rng.choice([1, 2, 3, 4, 5, 8, 16])
    Kb = rng.randint(1, 12)
    K = rng.randint(1, 40)
    rep = rng.choice([1, 1, 2, 3])
    causal = rng.random() < 0.7
    rows = rng.randint(1, 12)
    nq = -(-rows // rep)
    has_starts = rng.random() < 0.5
    starts = [rng.choice([0, 0, rng.randint(0, W + 3), -1]) for _ in range(nq)] if has_starts \
        else None
    ends = [rng.randint(-2, W + 3 * B) for _ in range(nq)]
    pool = brute.VALUE_POOL + (brute.EXOTIC_POOL if exotic else [])
    x = np.empty((rows, W), dtype=np.uint32)
    for r in range(rows):
        for c in range(W):
            if exotic and rng.random() < 0.05:
                x[r, c] = rng.choice(brute.NAN_BITS)
            else:
                x[r, c] = brute.to_bits(rng.choice(pool))
    return Case(x.view(np.float32), starts, ends, width=W, block_size=B, block_topk=Kb,
                row_topk=K, row_repeat=rep, causal=causal)


@pytest.mark.parametrize("exotic", [False, True])
def test_random_small_shapes(exotic):
    rng = random.Random(2024 + exotic)
    for i in range(60):
        case = _random_small(rng, exotic)
        check_all_modes(case, misalign=rng.choice([0, 0, 1, 2]), what=f"small#{i}")


@pytest.mark.parametrize("B", [1, 3, 4, 8, 12, 16, 32, 64, 128])
@pytest.mark.parametrize("aligned", [True, False])
def test_block_sizes_multi_tile(B, aligned):
    """Rows spanning many streaming rounds (several buffer compactions), odd
    widths, starts that break 16-byte alignment, pins past W."""
    rng = np.random.default_rng(B * 7 + aligned)
    rows, W = 6, 50_003 if not aligned else 65_536
    x = rng.standard_normal((rows, W)).astype(np.float32)
    starts = [0, 4, 5, 0, 64, 1] if not aligned else [0, 4, 8, 0, 64, 16]
    ends = [W, W - 3, 40_000, W + 5, 10, W + B + 1]
    case = Case(x, starts, ends, width=W, block_size=B, block_topk=37, row_topk=300)
    check_all_modes(case, what=f"B={B}")


def test_ascending_values_force_many_compactions():
    """Increasing values make every block beat the running threshold: the
    streaming buffer compacts every few rounds."""
    W = 200_000
    x = np.tile(np.arange(W, dtype=np.float32) / W, (3, 1))
    x[1] = x[1][::-1]
    x[2] = 1.0  # all ties: lowest ids win everywhere
    case = Case(x, None, [W, W, W], width=W, block_size=8, block_topk=256, row_topk=2048)
    check_all_modes(case, what="monotone")


@pytest.mark.parametrize("split", [2, 4, 16, 32, 64, 128])
@pytest.mark.parametrize("layout", ["aligned", "misaligned", "stride2", "b1"])
def test_cluster_split_rows(split, layout):
    """k CTAs per row in a thread-block cluster: each streams a share of the
    blocks, the leader merges the shares over distributed shared memory.
    split 32 / 64 / 128: the wide split -- the row streamed in that many parts by a
    first launch, their top-Kb lists merged by a 16-CTA cluster."""
    rng = np.random.default_rng(split * 13 + len(layout))
    W, B, cs, starts = 200_000, 8, 1, [0, 4, 0, 100]
    if layout == "misaligned":
        starts = [1, 5, 3, 6]
    elif layout == "stride2":
        B, cs = 16, 2
    elif layout == "b1":
        W, B = 60_000, 1
    x = rng.standard_normal((4, W * cs)).astype(np.float32)
    x[1, ::97] = -np.inf
    ends = [W, W + 3 * B + 1, 150_001, 3000]
    case = Case(x, starts, ends, width=W, block_size=B, block_topk=256, row_topk=2048,
                col_stride=cs, row_stride=W * cs, split=split)
    run = DeviceRun(case)
    desc = run.plan.describe()
    if split <= 16:
        assert desc["split"] == split and desc["parts"] == 0
    else:
        assert desc["split"] == 16 and desc["parts"] == split
    check_all_modes(case, what=f"split={split} {layout}")


def test_cluster_split_edge_rows():
    """Cluster path on the hand-worked edge shapes scaled up: start past W,
    empty rows, pins past W, -NaN blocks, few candidates (-inf tier)."""
    rng = np.random.default_rng(77)
    W = 70_001
    x = rng.standard_normal((8, W)).astype(np.float32)
    x[3, 10_000:10_800] = np.array([0xFFC00000], dtype=np.uint32).view(np.float32)[0]
    starts = [W + 5, 0, 0, 0, 17, 0, 3, 0]
    ends = [W + 20, 0, -4, W, W + 9, 1, 65_000, W + 16]
    for Kb, K in ((256, 2048), (3, 40), (1, 4096)):
        for split in (8, 32):
            case = Case(x, starts, ends, width=W, block_size=8, block_topk=Kb, row_topk=K, split=split)
            check_all_modes(case, what=f"cluster edges Kb={Kb} K={K} split={split}")


def test_auto_split_for_few_long_rows():
    import sparse_attention_indexer_live_gb300 as dsa
    few = dsa.dsa_select_init(rows=1, width=1 << 20, block_size=8, block_topk=256, row_topk=2048)
    many = dsa.dsa_select_init(rows=2048, width=1 << 20, block_size=8, block_topk=256,
                               row_topk=2048)
    assert few.describe()["split"] >= 8
    assert many.describe()["split"] == 1 and many.describe()["parts"] == 0
    # one 1M-column row leaves most SMs idle even with a 16-CTA cluster: the
    # wide split streams it in 128 parts first (64 a row for two rows)
    two = dsa.dsa_select_init(rows=2, width=1 << 20, block_size=8, block_topk=256, row_topk=2048)
    sms = few.describe()["sm_count"]
    if sms >= 128 and few.describe()["split"] == 16:
        assert few.describe()["parts"] == 128
    if sms >= 128 and two.describe()["split"] == 16:
        assert two.describe()["parts"] == 64


@pytest.mark.parametrize("split", [64, 128])
def test_wide_split_large_kb(split):
    """The wide split with Kb = 1000, K = 4096 on two 1M-column rows: a
    cluster CTA's lists (8000 slots at 128 parts) are more than its threads
    load in one round, and each part keeps up to 1000 of its 1024 or 2048
    blocks."""
    W = 1 << 20
    rng = np.random.default_rng(300 + split)
    x = rng.standard_normal((2, W)).astype(np.float32)
    x[1, 500_000:520_000] = 7.0  # a run of equal maxima across parts
    case = Case(x, [0, 40], [W, W - 12_345], width=W, block_size=8, block_topk=1000, row_topk=4096,
                split=split)
    desc = DeviceRun(case).plan.describe()
    if desc["split"] == 16:  # a 16-CTA cluster of this shared memory fits on GB300
        assert desc["parts"] == split
    check_all_modes(case, what=f"wide split {split}, Kb 1000")


def test_wide_split_graph_replay():
    """The wide split captured in a CUDA graph (the cluster launch is a
    programmatic dependent of the parts' launch, an edge of the graph) and
    replayed with new ends: a full row, a short one that leaves most parts
    empty, one with the pin past W, one of five columns."""
    import sparse_attention_indexer_live_gb300 as dsa
    W = 1 << 20
    rng = np.random.default_rng(41)
    x = rng.standard_normal((1, W)).astype(np.float32)
    x[0, rng.integers(0, W, 64)] = 6.0 + np.abs(rng.standard_normal(64)).astype(np.float32)
    case = Case(x, None, [W], width=W, block_size=8, block_topk=256, row_topk=2048, split=128)
    run = DeviceRun(case)
    if run.plan.describe()["parts"] != 128:
        pytest.skip("this device does not run the wide split")
    base = run.buf.clone()
    dsa.dsa_select_topk(run.plan, run.logits, None, run.ends, run.cand, run.topk)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        dsa.dsa_select_topk(run.plan, run.logits, None, run.ends, run.cand, run.topk, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for replay in ([W], [300_001], [W + 5], [5], [W - 777]):
        run.ends.copy_(torch.tensor(replay, dtype=torch.int32))
        run.buf.copy_(base)
        g.replay()
        torch.cuda.synchronize()
        c2 = Case(x, None, replay, width=W, block_size=8, block_topk=256, row_topk=2048)
        assert_run_matches(run, *c2.oracle(), what=f"wide split replay {replay}")


@pytest.mark.parametrize("rows", [1, 2])
def test_one_or_two_1m_rows_auto_plan(rows):
    """P1's test plan: a single row over a 1M-column buffer -- in the plan the
    device picks for it (on GB300 the wide split: 128 parts for one row, 64
    for two, then a 16-CTA cluster per row), every column and index compared with the oracle in all
    three modes.  The second row has a start, an end short of W and a spike
    mix; a third shape puts the pin past W."""
    W = 1 << 20
    rng = np.random.default_rng(90 + rows)
    x = rng.standard_normal((rows, W)).astype(np.float32)
    x[:, rng.integers(0, W, 64)] = 6.0 + np.abs(rng.standard_normal(64)).astype(np.float32)
    if rows == 1:
        cases = [(None, [W]), (None, [W + 5])]  # full width; pin past W (edge column)
    else:
        x[1, 300_000:300_800] = -np.inf
        cases = [([0, 17], [W, 900_001]), ([3, 0], [W + 9, W])]
    for starts, ends in cases:
        case = Case(x, starts, ends, width=W, block_size=8, block_topk=256, row_topk=2048)
        check_all_modes(case, what=f"{rows} x 1M rows, starts {starts}, ends {ends}")


def test_tiny_workload_full():
    wl = wk.WORKLOADS["tiny"]
    x, s, e = wk.make_all(wl)
    check_all_modes(Case.from_workload(wl, x, s, e), what="tiny")


def test_decode_short_workload_full():
    wl = wk.WORKLOADS["decode_short"]
    x, s, e = wk.make_all(wl)
    check_all_modes(Case.from_workload(wl, x, s, e), what="decode_short")


def test_ragged_workload_full():
    wl = wk.WORKLOADS["ragged"]
    x, s, e = wk.make_all(wl)
    check_all_modes(Case.from_workload(wl, x, s, e), what="ragged")


def test_decode_1m_workload_full():
    wl = wk.WORKLOADS["decode_1m"]
    x, s, e = wk.make_all(wl)
    check_all_modes(Case.from_workload(wl, x, s, e), what="decode_1m")


def test_row_repeat_shared_end_reading():
    rng = np.random.default_rng(8)
    W = 30_000
    x = rng.standard_normal((7, W)).astype(np.float32)
    for causal in (True, False):
        case = Case(x, None, [5000, 2049, 29_999], width=W, block_size=8, block_topk=64,
                    row_topk=500, row_repeat=3, causal=causal)
        check_all_modes(case, what=f"rep3 causal={causal}")


def test_sentinel_tail_untouched():
    """Columns at or past each row's end keep a sentinel (the pages' 1.5 fill)."""
    W = 262_144
    ends = [0, 1, 1025, W // 2, W - 1, W]
    x = np.full((len(ends), W), 1.5, dtype=np.float32)
    case = Case(x, None, ends, width=W, block_size=8, block_topk=256, row_topk=2048)
    run = DeviceRun(case).fused()
    allbits, _, _ = run.result()
    got = allbits[run.offset:run.offset + len(ends) * W].view(np.float32).reshape(len(ends), W)
    for r, e in enumerate(ends):
        assert np.all(got[r, e:] == 1.5), f"row {r} written past end {e}"
    want_logits, want_cand, want_topk = case.oracle()
    assert_run_matches(run, want_logits, want_cand, want_topk, "sentinel")


def test_cuda_graph_replay_tracks_changing_ends():
    """A graph captured with one set of ends replays correctly with others:
    the grid is fixed by the shapes, the work follows the bounds."""
    import sparse_attention_indexer_live_gb300 as dsa
    rng = np.random.default_rng(21)
    W, rows = 262_144, 4
    x = rng.standard_normal((rows, W)).astype(np.float32)
    captured = [1024, 4096, 8192, 2048]
    case = Case(x, None, captured, width=W, block_size=8, block_topk=256, row_topk=2048)
    run = DeviceRun(case)
    base = run.buf.clone()
    # warm up outside the capture
    dsa.dsa_select_topk(run.plan, run.logits, None, run.ends, run.cand, run.topk)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            dsa.dsa_select_topk(run.plan, run.logits, None, run.ends, run.cand, run.topk,
                                stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for replay in ([1, 131_072, W, 0], [W, 1025, 3, 65_536], [W + 9, 0, 2049, 2048]):
        run.ends.copy_(torch.tensor(replay, dtype=torch.int32))
        run.buf.copy_(base)
        g.replay()
        torch.cuda.synchronize()
        c2 = Case(x, None, replay, width=W, block_size=8, block_topk=256, row_topk=2048)
        want_logits, want_cand, want_topk = c2.oracle()
        assert_run_matches(run, want_logits, want_cand, want_topk, f"replay {replay}")


def test_zero_rows_is_a_no_op():
    import sparse_attention_indexer_live_gb300 as dsa
    plan = dsa.dsa_select_init(rows=0, width=1024, block_size=8, block_topk=4, row_topk=8)
    logits = torch.zeros((0, 1024), device="cuda")
    ends = torch.zeros(0, dtype=torch.int32, device="cuda")
    cand = torch.zeros((0, 5), dtype=torch.int32, device="cuda")
    topk = torch.zeros((0, 8), dtype=torch.int32, device="cuda")
    dsa.dsa_select_topk(plan, logits, None, ends, cand, topk)
    torch.cuda.synchronize()


def test_large_kb_and_k():
    rng = np.random.default_rng(4)
    W = 400_000
    x = rng.standard_normal((3, W)).astype(np.float32)
    case = Case(x, [0, 3, 100], [W, 300_001, W + 77], width=W, block_size=8, block_topk=1000,
                row_topk=4096)
    check_all_modes(case, what="Kb=1000 K=4096")
