"""The N > 1 host logic of bench.py on CPU: world-size-2 gloo ranks, each with
its own replica rows (weak scaling), a barrier and the max over ranks.  The
data path has no collective, so this is all there is to test without GPUs."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    import oracle
    import workloads as wk
    w, r = bench.dist_init("gloo")
    assert (w, r) == (world, rank)
    bench.barrier()
    wl = wk.WORKLOADS["tiny"]
    rows = bench.replica_rows(rank, wl.rows)
    starts, ends = wk.bounds(wl)
    x = wk.make_rows(wl, rows, starts, ends, bound_rows=np.arange(wl.rows))
    cand, topk = oracle.default().run(x, starts, ends, width=wl.width, block_size=wl.block_size,
                                      block_topk=wl.block_topk, row_topk=wl.row_topk)
    slowest = bench.max_over_ranks(float(rank + 1))
    gathered = [None] * world
    dist.all_gather_object(gathered, rows.tolist())
    q.put((rank, slowest, gathered, topk.sum()))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_weak_scaling():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=100) for _ in range(world)]
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    out.sort()
    # the max over ranks is seen by every rank
    assert [o[1] for o in out] == [2.0, 2.0]
    # replica rows are disjoint across ranks and cover rank * rows + [0, rows)
    rows = out[0][2]
    assert set(rows[0]).isdisjoint(rows[1])
    assert sorted(rows[0] + rows[1]) == list(range(2 * len(rows[0])))
    # different data per rank (different row ids) -> different selections
    assert out[0][3] != out[1][3]
