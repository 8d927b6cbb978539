"""Row sharding on one GPU: the selector without a process group, and the
shards of a 2- and 4-way split run one after another and concatenated, each
against the oracle (the multi-rank gather itself is covered by the gloo
tests; a box has one GPU)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import workloads as wk

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def decode_case():
    import sparse_attention_indexer_live_gb300 as dsa
    dsa.build()
    wl = wk.WORKLOADS["decode_1m"].with_(width=1 << 17)
    x, starts, ends = wk.make_all(wl)
    want = x.copy()
    cand, topk = oracle.default().run(want, starts, ends, width=wl.width,
                                      block_size=wl.block_size, block_topk=wl.block_topk,
                                      row_topk=wl.row_topk, row_repeat=wl.row_repeat)
    return wl, x, ends, want, cand, topk


def test_selector_without_group(decode_case):
    from sparse_attention_indexer_live_gb300 import ShardedSelector
    wl, x, ends, want, cand_w, topk_w = decode_case
    sel = ShardedSelector(total_rows=wl.rows, width=wl.width, block_size=wl.block_size,
                          block_topk=wl.block_topk, row_topk=wl.row_topk,
                          row_repeat=wl.row_repeat)
    dev = "cuda:0"
    logits = torch.from_numpy(x).to(dev)
    cand = torch.empty((wl.rows, wl.block_topk + 1), dtype=torch.int32, device=dev)
    topk = torch.empty((wl.rows, wl.row_topk), dtype=torch.int32, device=dev)
    topk_all = torch.empty_like(topk)
    got = sel(logits, None, torch.from_numpy(ends).to(dev), cand, topk, topk_all)
    assert np.array_equal(got.cpu().numpy(), topk_w)
    assert np.array_equal(logits.cpu().numpy().view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("world", [2, 4])
def test_shards_concatenate_to_the_whole(decode_case, world):
    import sparse_attention_indexer_live_gb300 as dsa
    wl, x, ends, want, cand_w, topk_w = decode_case
    dev = "cuda:0"
    rep = wl.row_repeat
    parts_t, parts_c, parts_x = [], [], []
    for r in range(world):
        sh = dsa.shard_rows(wl.rows, world, r, rep)
        per = sh.rows_per_rank
        xs = np.zeros((per, wl.width), dtype=np.float32)
        xs[:sh.rows] = x[sh.row0:sh.row0 + sh.rows]
        es = np.zeros(sh.bounds, dtype=np.int32)  # padding rows end at 0
        real = sh.rows // rep
        es[:real] = ends[sh.bound0:sh.bound0 + real]
        plan = dsa.dsa_select_init(rows=per, width=wl.width, block_size=wl.block_size,
                                   block_topk=wl.block_topk, row_topk=wl.row_topk, row_repeat=rep)
        lg = torch.from_numpy(xs).to(dev)
        cand = torch.empty((per, wl.block_topk + 1), dtype=torch.int32, device=dev)
        topk = torch.empty((per, wl.row_topk), dtype=torch.int32, device=dev)
        dsa.dsa_select_topk(plan, lg, None, torch.from_numpy(es).to(dev), cand, topk)
        torch.cuda.synchronize()
        t = topk.cpu().numpy()
        assert np.all(t[sh.rows:] == -1)  # padding rows are empty
        parts_t.append(t[:sh.rows])
        parts_c.append(cand.cpu().numpy()[:sh.rows])
        parts_x.append(lg.cpu().numpy()[:sh.rows])
    assert np.array_equal(np.concatenate(parts_t), topk_w)
    assert np.array_equal(np.concatenate(parts_c), cand_w)
    assert np.array_equal(np.concatenate(parts_x).view(np.uint32), want.view(np.uint32))
