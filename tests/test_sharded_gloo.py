"""Row-sharded selection across ranks (world size 2, gloo, CPU): shard
arithmetic, the all-gather of every rank's row top-k, and the fail-closed
status check when one rank's local call fails.  The local step is a stand-in
on CPU (a copy of the oracle's rows, or a raised DsaSelectError); the GPU
step itself is covered by the GPU tests."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from sparse_attention_indexer_live_gb300 import shard_rows


@pytest.mark.parametrize("total,world,rep", [(2048, 2, 1), (96, 8, 2), (7, 3, 1), (5, 4, 2),
                                             (0, 2, 1), (1, 8, 1)])
def test_shards_cover_rows_once(total, world, rep):
    shards = [shard_rows(total, world, r, rep) for r in range(world)]
    per = shards[0].rows_per_rank
    assert all(s.rows_per_rank == per for s in shards) and per % rep == 0
    covered = [row for s in shards for row in range(s.row0, s.row0 + s.rows)]
    assert covered == list(range(total))
    for s in shards:
        assert s.row0 % rep == 0 and 0 <= s.rows <= per


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, fail_rank, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    import oracle
    import workloads as wk
    from sparse_attention_indexer_live_gb300 import DsaSelectError, ShardedSelector
    dist.init_process_group("gloo", rank=rank, world_size=world)
    wl = wk.WORKLOADS["tiny"].with_(rows=7)
    starts, ends = wk.bounds(wl)
    x = wk.make_rows(wl, range(wl.rows), starts, ends)
    _, want = oracle.default().run(x.copy(), starts, ends, width=wl.width,
                                   block_size=wl.block_size, block_topk=wl.block_topk,
                                   row_topk=wl.row_topk)

    def fake_local(plan, logits, st, en, cand, topk):
        # stand-in for the GPU call: this rank's rows from the oracle, or a failure
        if rank == fail_rank:
            raise DsaSelectError(3, "dsa_select_topk")
        sh = sel.shard
        topk.fill_(-1)
        topk[:sh.rows] = torch.from_numpy(want[sh.row0:sh.row0 + sh.rows])

    sel = ShardedSelector(total_rows=wl.rows, width=wl.width, block_size=wl.block_size,
                          block_topk=wl.block_topk, row_topk=wl.row_topk, plan=False,
                          local_fn=fake_local)
    per = sel.shard.rows_per_rank
    topk = torch.empty((per, wl.row_topk), dtype=torch.int32)
    cand = torch.empty((per, wl.block_topk + 1), dtype=torch.int32)
    topk_all = torch.empty((world * per, wl.row_topk), dtype=torch.int32)
    try:
        got = sel(None, None, None, cand, topk, topk_all)
        q.put((rank, "ok", bool(np.array_equal(got.numpy(), want))))
    except RuntimeError as e:
        q.put((rank, "raised", str(e)))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
@pytest.mark.parametrize("fail_rank", [None, 1])
def test_gather_and_fail_closed(fail_rank):
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, fail_rank, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=100) for _ in range(world))
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    if fail_rank is None:
        assert out == [(0, "ok", True), (1, "ok", True)]
    else:
        # every rank refuses the gathered result and names the failed rank
        for rank, kind, msg in out:
            assert kind == "raised" and f"rank(s) [{fail_rank}]" in msg
