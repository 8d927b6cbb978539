"""Row-sharded selection across ranks with a fail-closed status check.

Rows are independent, so a batch of query rows can be split over the ranks of
a process group: every rank runs the fused selection on its own shard and the
row top-k lists are all-gathered so that each rank holds the whole batch.
This follows the tensor-parallel query sharding discussed for LiteTopK (vLLM
PR #48726, review of `sparse_attn_indexer.py`): the shard's indices are
gathered with `all_gather_into_tensor`, a one-word status per rank is gathered
beside them, and -- as the review asks instead of a device-side assert -- the
host reads the gathered status and raises a `RuntimeError` naming every rank
that failed, so no rank consumes a shard of -1 rows silently.

Shards are equal (padded) so that `all_gather_into_tensor` applies; padding
rows carry end 0 and come back as all -1.  The shard size is a multiple of
`row_repeat`, so rows sharing a bound entry never straddle two ranks.
"""
from __future__ import annotations

from dataclasses import dataclass

from .binding import DsaSelectError, dsa_select_init, dsa_select_topk


@dataclass(frozen=True)
class Shard:
    rank: int
    world: int
    row0: int           # first global row of this rank's shard
    rows: int           # real rows in this shard (the rest is padding)
    rows_per_rank: int  # padded shard size, equal on every rank
    row_repeat: int = 1

    @property
    def bound0(self) -> int:
        """First bound entry of the shard."""
        return self.row0 // self.row_repeat

    @property
    def bounds(self) -> int:
        """Bound entries of the padded shard."""
        return self.rows_per_rank // self.row_repeat


def shard_rows(total_rows: int, world: int, rank: int, row_repeat: int = 1) -> Shard:
    """Contiguous equal shards of ceil(total / world) rows, rounded up to a
    multiple of row_repeat."""
    if world < 1 or not 0 <= rank < world or total_rows < 0 or row_repeat < 1:
        raise ValueError("bad shard arguments")
    per = -(-total_rows // world) if total_rows else 0
    per = -(-per // row_repeat) * row_repeat
    row0 = rank * per
    rows = max(0, min(total_rows - row0, per))
    return Shard(rank=rank, world=world, row0=row0, rows=rows, rows_per_rank=per,
                 row_repeat=row_repeat)


class ShardedSelector:
    """Fused selection on this rank's shard, then an all-gather of the row
    top-k lists and of a status word, checked on the host (fail-closed).

    `local_fn(plan, logits, starts, ends, cand, topk)` runs the local step; it
    defaults to the C ABI's `dsa_select_topk`.  Any `DsaSelectError` it raises
    marks this rank as failed: its shard is sent as -1 rows and every rank
    raises after the gather.
    """

    def __init__(self, *, total_rows, width, block_size, block_topk, row_topk, row_repeat=1,
                 repeat_causal=True, has_starts=False, group=None, device=0, local_fn=None,
                 plan=True):
        import torch.distributed as dist
        self.group = group
        self.dist = dist if (group is not None or (dist.is_available() and
                                                   dist.is_initialized())) else None
        world = self.dist.get_world_size(group) if self.dist else 1
        rank = self.dist.get_rank(group) if self.dist else 0
        self.shard = shard_rows(total_rows, world, rank, row_repeat)
        self.total_rows = total_rows
        self.row_topk = row_topk
        self.block_topk = block_topk
        self.local_fn = local_fn or dsa_select_topk
        self.plan = None
        if plan and self.shard.rows_per_rank > 0:
            self.plan = dsa_select_init(device=device, rows=self.shard.rows_per_rank, width=width,
                                        block_size=block_size, block_topk=block_topk,
                                        row_topk=row_topk, row_repeat=row_repeat,
                                        repeat_causal=repeat_causal, has_starts=has_starts)

    def __call__(self, logits, starts, ends, cand, topk, topk_all):
        """logits/cand/topk: this rank's padded shard ([rows_per_rank, ...]);
        starts/ends: the shard's bound entries; topk_all: [world * rows_per_rank, K]
        on every rank.  Returns topk_all[:total_rows]."""
        import torch
        ok = 1
        err = ""
        try:
            self.local_fn(self.plan, logits, starts, ends, cand, topk)
        except DsaSelectError as e:
            ok, err = 0, str(e)
            topk.fill_(-1)
        if self.dist is None:
            if not ok:
                raise RuntimeError(f"row-sharded selection failed on rank 0: {err}")
            topk_all[:topk.shape[0]].copy_(topk)
            return topk_all[:self.total_rows]
        self.dist.all_gather_into_tensor(topk_all, topk, group=self.group)
        status = torch.tensor([ok], dtype=torch.int32, device=topk.device)
        status_all = torch.empty(self.shard.world, dtype=torch.int32, device=topk.device)
        self.dist.all_gather_into_tensor(status_all, status, group=self.group)
        bad = [r for r, v in enumerate(status_all.tolist()) if v != 1]  # host read: fail closed
        if bad:
            raise RuntimeError(f"row-sharded selection failed on rank(s) {bad}"
                               + (f": {err}" if err else "") + "; the gathered top-k is not usable")
        return topk_all[:self.total_rows]
