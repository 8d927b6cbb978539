"""The 1M-context prefill workload at full size (2048 x 1,048,576 fp32, 8 GiB),
in the launch configuration the benchmark times: sampled rows element by
element against the oracle, and properties that hold at any size on every row
(tail untouched, kept columns bounded, top-k valid, planted spikes found)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import workloads as wk

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def prefill_run():
    import sparse_attention_indexer_live_gb300 as dsa
    dsa.build()
    wl = wk.WORKLOADS["prefill_1m"]
    starts, ends = wk.bounds(wl)
    host = torch.empty((wl.rows, wl.row_stride), dtype=torch.float32, pin_memory=True)
    wk.fill_rows(wl, np.arange(wl.rows), host.numpy(), starts, ends)
    dev = torch.device("cuda:0")
    logits = host.to(dev)
    ends_d = torch.from_numpy(ends).to(dev)
    cand = torch.full((wl.rows, wl.block_topk + 1), -7, dtype=torch.int32, device=dev)
    topk = torch.full((wl.rows, wl.row_topk), -7, dtype=torch.int32, device=dev)
    plan = dsa.dsa_select_init(device=0, rows=wl.rows, width=wl.width, block_size=wl.block_size,
                               block_topk=wl.block_topk, row_topk=wl.row_topk)
    dsa.dsa_select_topk(plan, logits, None, ends_d, cand, topk)
    torch.cuda.synchronize()
    yield wl, host.numpy(), ends, logits, cand.cpu().numpy(), topk.cpu().numpy()
    del logits


def test_sampled_rows_match_oracle(prefill_run):
    wl, host, ends, logits, cand, topk = prefill_run
    rows = [0, 1, 2, 777, 1023, 1024, 1500, 2046, 2047] + \
        np.random.default_rng(0).choice(2048, 7, replace=False).tolist()
    orc = oracle.default()
    for r in rows:
        want = host[r].copy()
        c, t = orc.row(want, wl.width, 0, int(ends[r]), wl.block_size, wl.block_topk,
                       wl.row_topk)
        got = logits[r].cpu().numpy()
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), f"row {r} logits"
        assert np.array_equal(cand[r], c), f"row {r} cand"
        assert np.array_equal(topk[r], t), f"row {r} topk"


def test_every_row_properties(prefill_run):
    wl, host, ends, logits, cand, topk = prefill_run
    W, B, Kb, K = wl.width, wl.block_size, wl.block_topk, wl.row_topk
    # tails past each end are untouched (ends are >= W - 2303)
    tail0 = W - 2560
    got_tail = logits[:, tail0:].cpu().numpy()
    for r in range(wl.rows):
        e = int(ends[r])
        assert np.array_equal(got_tail[r, e - tail0:].view(np.uint32),
                              host[r, e:].view(np.uint32)), f"row {r} tail written"
    # kept (non -inf) live columns: at most Kb + 1 blocks
    for r0 in range(0, wl.rows, 256):
        blk = logits[r0:r0 + 256]
        kept = (~torch.isneginf(blk)).sum(dim=1).cpu().numpy()
        for i, k in enumerate(kept):
            r = r0 + i
            tail = W - int(ends[r])
            assert k - tail <= (Kb + 1) * B + 1, f"row {r} keeps {k - tail} live columns"
    # top-k: K distinct ascending columns inside the span; the pin is the last block
    assert np.all(np.diff(topk, axis=1) > 0)
    assert np.all(topk[:, 0] >= 0) and np.all(topk.max(axis=1) < ends)
    assert np.array_equal(cand[:, Kb], (ends - 1) // B)
    # every planted spike (+6 sigma) is among the row's top-k
    for r in range(0, wl.rows, 64):
        spikes = np.nonzero(host[r, :ends[r]] >= 6.0)[0]
        assert len(spikes) >= 60
        assert np.isin(spikes, topk[r]).all(), f"row {r} lost a spike"
