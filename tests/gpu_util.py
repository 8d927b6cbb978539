"""Helpers for the GPU parity tests: run the CUDA path through the C ABI on a
guard-banded device buffer and run the oracle on the same host bytes."""
from __future__ import annotations

import numpy as np

GUARD = 1024             # floats of sentinel before and after the logits
SENTINEL = 0x7FC0DEAD    # a quiet NaN no input ever holds


class Case:
    """One call: logits [rows, row_stride] float32 (host) + bounds + shape."""

    def __init__(self, logits, starts, ends, *, width, block_size, block_topk, row_topk,
                 row_repeat=1, causal=True, col_stride=1, row_stride=None, split=0):
        self.logits = np.ascontiguousarray(logits, dtype=np.float32)
        self.rows = self.logits.shape[0]
        self.starts = None if starts is None else np.asarray(starts, dtype=np.int32)
        self.ends = np.asarray(ends, dtype=np.int32)
        self.width = width
        self.B = block_size
        self.Kb = block_topk
        self.K = row_topk
        self.rep = row_repeat
        self.causal = causal
        self.cs = col_stride
        self.row_stride = self.logits.shape[1] if row_stride is None else row_stride
        self.split = split

    @classmethod
    def from_workload(cls, wl, logits, starts, ends):
        return cls(logits, starts, ends, width=wl.width, block_size=wl.block_size,
                   block_topk=wl.block_topk, row_topk=wl.row_topk, row_repeat=wl.row_repeat,
                   causal=True, col_stride=wl.col_stride, row_stride=wl.row_stride)

    def cfg_kwargs(self):
        return dict(rows=self.rows, width=self.width, block_size=self.B, block_topk=self.Kb,
                    row_topk=self.K, row_stride=self.row_stride, col_stride=self.cs,
                    row_repeat=self.rep, repeat_causal=self.causal,
                    has_starts=self.starts is not None, split=self.split)

    def oracle(self):
        from oracle import default
        got = self.logits.copy()
        cand, topk = default().run(got, self.starts, self.ends, width=self.width,
                                   block_size=self.B, block_topk=self.Kb, row_topk=self.K,
                                   row_repeat=self.rep, causal=self.causal,
                                   col_stride=self.cs, row_stride=self.row_stride)
        return got, cand, topk


class DeviceRun:
    """Device copies of a Case, with guard bands around the logits."""

    def __init__(self, case: Case, device="cuda:0", misalign=0):
        import torch
        import sparse_attention_indexer_live_gb300 as dsa
        self.case = case
        self.torch = torch
        self.dsa = dsa
        n = case.rows * case.row_stride
        host = np.empty(2 * GUARD + n + misalign, dtype=np.uint32)
        host[:] = SENTINEL
        host[GUARD + misalign:GUARD + misalign + n] = case.logits.reshape(-1).view(np.uint32)
        self.host = host
        self.offset = GUARD + misalign
        self.buf = torch.from_numpy(host.view(np.float32).copy()).to(device)
        self.logits = self.buf.as_strided((case.rows, case.width), (case.row_stride, case.cs),
                                          self.offset)
        self.starts = None if case.starts is None else torch.from_numpy(case.starts).to(device)
        self.ends = torch.from_numpy(case.ends).to(device)
        self.cand = torch.full((case.rows, case.Kb + 1), -7, dtype=torch.int32, device=device)
        self.topk = torch.full((case.rows, case.K), -7, dtype=torch.int32, device=device)
        self.plan = dsa.dsa_select_init(device=torch.device(device).index or 0,
                                        **case.cfg_kwargs())

    def fused(self):
        self.dsa.dsa_select_topk(self.plan, self.logits, self.starts, self.ends, self.cand,
                                 self.topk)
        return self

    def select(self):
        self.dsa.dsa_candidate_select(self.plan, self.logits, self.starts, self.ends, self.cand)
        return self

    def topk_cand(self):
        self.dsa.dsa_row_topk(self.plan, self.logits, self.starts, self.ends, self.cand, self.topk)
        return self

    def topk_scan(self, out=None):
        out = self.topk if out is None else out
        self.dsa.dsa_row_topk(self.plan, self.logits, self.starts, self.ends, None, out)
        return self

    def result(self):
        self.torch.cuda.synchronize()
        allbits = self.buf.cpu().numpy().view(np.uint32)
        return allbits, self.cand.cpu().numpy(), self.topk.cpu().numpy()

    def expected_buffer(self, masked_logits):
        want = self.host.copy()
        n = self.case.rows * self.case.row_stride
        want[self.offset:self.offset + n] = masked_logits.reshape(-1).view(np.uint32)
        return want


def assert_run_matches(run: DeviceRun, want_logits, want_cand, want_topk, what=""):
    allbits, cand, topk = run.result()
    want = run.expected_buffer(want_logits)
    bad = np.nonzero(allbits != want)[0]
    if len(bad):
        i = int(bad[0])
        off = i - run.offset
        rs = run.case.row_stride
        where = f"guard[{i}]" if off < 0 or off >= run.case.rows * rs else \
            f"row {off // rs} elem {off % rs}"
        raise AssertionError(f"{what}: {len(bad)} logits words differ; first at {where}: "
                             f"got {allbits[i]:#010x} want {want[i]:#010x}")
    if not np.array_equal(cand, want_cand):
        r = int(np.nonzero((cand != want_cand).any(axis=1))[0][0])
        raise AssertionError(f"{what}: cand row {r}: got {cand[r][:12]}... pin {cand[r][-1]}; "
                             f"want {want_cand[r][:12]}... pin {want_cand[r][-1]}")
    if not np.array_equal(topk, want_topk):
        r = int(np.nonzero((topk != want_topk).any(axis=1))[0][0])
        d = np.nonzero(topk[r] != want_topk[r])[0]
        raise AssertionError(f"{what}: topk row {r}: {len(d)} slots differ, first {d[0]}: "
                             f"got {topk[r][d[0]]} want {want_topk[r][d[0]]}")
