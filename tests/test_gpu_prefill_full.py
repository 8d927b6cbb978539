"""The 1M-context prefill workload at full size (2048 x 1,048,576 fp32, 8 GiB),
in the launch configuration the benchmark times, against the oracle on EVERY
row: the masked logits as uint32 bit patterns over the whole row (the tail
past each end included), cand and topk exactly -- for the fused launch, for
select + candidate-mode top-k, and for scan mode on the masked logits.  The
oracle's rows run on all host cores (its C code releases the GIL), a chunk of
rows at a time."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import workloads as wk

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

CHUNK = 128  # rows per comparison chunk (512 MB of logits)


@pytest.fixture(scope="module")
def prefill_run():
    import sparse_attention_indexer_live_gb300 as dsa
    dsa.build()
    wl = wk.WORKLOADS["prefill_1m"]
    starts, ends = wk.bounds(wl)
    host = torch.empty((wl.rows, wl.row_stride), dtype=torch.float32, pin_memory=True)
    wk.fill_rows(wl, np.arange(wl.rows), host.numpy(), starts, ends)
    dev = torch.device("cuda:0")
    ends_d = torch.from_numpy(ends).to(dev)
    plan = dsa.dsa_select_init(device=0, rows=wl.rows, width=wl.width, block_size=wl.block_size,
                               block_topk=wl.block_topk, row_topk=wl.row_topk)

    def outs():
        return (torch.full((wl.rows, wl.block_topk + 1), -7, dtype=torch.int32, device=dev),
                torch.full((wl.rows, wl.row_topk), -7, dtype=torch.int32, device=dev))

    # the benchmark's call: one fused launch
    fused = host.to(dev)
    cand_f, topk_f = outs()
    dsa.dsa_select_topk(plan, fused, None, ends_d, cand_f, topk_f)
    # the two-call form, then scan mode on its masked logits
    split = host.to(dev)
    cand_s, topk_s = outs()
    dsa.dsa_candidate_select(plan, split, None, ends_d, cand_s)
    dsa.dsa_row_topk(plan, split, None, ends_d, cand_s, topk_s)
    topk_scan = torch.full_like(topk_s, -7)
    dsa.dsa_row_topk(plan, split, None, ends_d, None, topk_scan)
    torch.cuda.synchronize()
    yield dict(wl=wl, host=host.numpy(), ends=ends, fused=fused, split=split,
               cand_f=cand_f.cpu().numpy(), topk_f=topk_f.cpu().numpy(),
               cand_s=cand_s.cpu().numpy(), topk_s=topk_s.cpu().numpy(),
               topk_scan=topk_scan.cpu().numpy())
    del fused, split


def test_every_row_matches_oracle(prefill_run):
    d = prefill_run
    wl, host, ends = d["wl"], d["host"], d["ends"]
    orc = oracle.default()
    want_cand = np.zeros((wl.rows, wl.block_topk + 1), dtype=np.int32)
    want_topk = np.zeros((wl.rows, wl.row_topk), dtype=np.int32)
    threads = max(1, min(32, os.cpu_count() or 1))
    with ThreadPoolExecutor(threads) as ex:
        for r0 in range(0, wl.rows, CHUNK):
            r1 = min(r0 + CHUNK, wl.rows)
            want = host[r0:r1].copy()

            def one(i):
                c, t = orc.row(want[i], wl.width, 0, int(ends[r0 + i]), wl.block_size,
                               wl.block_topk, wl.row_topk)
                want_cand[r0 + i] = c
                want_topk[r0 + i] = t

            list(ex.map(one, range(r1 - r0)))
            wbits = want.view(np.uint32)
            for name in ("fused", "split"):
                got = d[name][r0:r1].cpu().numpy().view(np.uint32)
                bad = np.nonzero((got != wbits).any(axis=1))[0]
                assert len(bad) == 0, (f"[{name}] logits of row {r0 + bad[0]} differ at "
                                       f"{np.nonzero(got[bad[0]] != wbits[bad[0]])[0][:8]}")
    for name, got, want in (("fused cand", d["cand_f"], want_cand),
                            ("fused topk", d["topk_f"], want_topk),
                            ("select cand", d["cand_s"], want_cand),
                            ("candidate-mode topk", d["topk_s"], want_topk),
                            ("scan-mode topk", d["topk_scan"], want_topk)):
        bad = np.nonzero((got != want).any(axis=1))[0]
        assert len(bad) == 0, f"{name}: {len(bad)} rows differ, first {bad[0]}"


def test_every_row_properties(prefill_run):
    d = prefill_run
    wl, host, ends, topk, cand = d["wl"], d["host"], d["ends"], d["topk_f"], d["cand_f"]
    B, Kb = wl.block_size, wl.block_topk
    # top-k: K distinct ascending columns inside the span; the pin is the last block
    assert np.all(np.diff(topk, axis=1) > 0)
    assert np.all(topk[:, 0] >= 0) and np.all(topk.max(axis=1) < ends)
    assert np.array_equal(cand[:, Kb], (ends - 1) // B)
    # every planted spike (+6 sigma) is among the row's top-k
    for r in range(0, wl.rows, 64):
        spikes = np.nonzero(host[r, :ends[r]] >= 6.0)[0]
        assert len(spikes) >= 60
        assert np.isin(spikes, topk[r]).all(), f"row {r} lost a spike"
