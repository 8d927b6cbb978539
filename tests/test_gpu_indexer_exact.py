"""The fused producer + selection against the oracle end to end.

On inputs whose indexer logits are exact in fp32 (small e4m3 integers,
power-of-two head weights and key scales; see workloads.indexer_exact_inputs)
the oracle's fp64 logits round to the very bits the tensor cores produce, so
nothing from the GPU is fed to the oracle: the oracle computes the logits
from q, k, k_scale and w, then runs the selection on them, and

  * dsa_indexer_logits must equal the oracle's logits bit for bit over every
    live span and leave the rest of each row untouched;
  * dsa_indexer_select's cand and topk must equal the oracle's exactly.

The inputs repeat key rows, so equal logits -- ties between blocks and inside
blocks -- are common, and the lower-index tie-break is exercised throughout.
(The pages' FP8 MQA indexer score: vLLM PR #48726, Motivation.)"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import workloads as wk
from oracle import default as oracle_default

pytestmark = pytest.mark.gpu


def _torch():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return torch


def _pool():
    return ThreadPoolExecutor(max(1, min(32, os.cpu_count() or 1)))


def _oracle(q, k, ks, w, ends, B, Kb, K, fill):
    T, S = q.shape[0], k.shape[0]
    orc = oracle_default()
    logits = np.full((T, S), fill, dtype=np.float32)

    def produce(t):
        orc.indexer_logits(q[t:t + 1], k, ks, w[t:t + 1], None, ends[t:t + 1], logits[t:t + 1])

    masked = None
    cand = np.zeros((T, Kb + 1), dtype=np.int32)
    topk = np.zeros((T, K), dtype=np.int32)
    with _pool() as ex:
        list(ex.map(produce, range(T)))
        masked = logits.copy()

        def select(t):
            cand[t], topk[t] = orc.row(masked[t], S, 0, int(ends[t]), B, Kb, K)

        list(ex.map(select, range(T)))
    return logits, cand, topk


CASES = {
    # the decode shape: 2500 blocks per row at B 8, causal ends
    "causal_20000": (48, 20000, 8, 256, 2048, None),
    # empty rows, spans inside one block or tile, exactly / past the width, a negative end
    "edge_ends": (12, 5000, 8, 32, 64, [0, 1, 7, 8, 9, 127, 128, 129, 4999, 5000, 5003, -3]),
    "block_4": (9, 3001, 4, 100, 300, [3001, 2500, 1, 0, 3001, 64, 1000, 2999, 3005]),
    "block_2": (9, 3001, 2, 100, 300, [3001, 2500, 1, 0, 3001, 64, 1000, 2999, 3005]),
    "block_1": (9, 3001, 1, 500, 700, [3001, 2500, 1, 0, 3001, 64, 1000, 2999, 3005]),
    # fewer blocks than Kb: -inf padding blocks fill the block top-k
    "few_blocks": (5, 100, 8, 32, 40, [100, 50, 3, 0, 101]),
    # the full 1M-key width of the long-context workloads
    "width_1m": (4, 1 << 20, 8, 256, 2048, None),
}


@pytest.mark.parametrize("name", list(CASES))
def test_fused_selection_matches_oracle_end_to_end(name):
    torch = _torch()
    import sparse_attention_indexer_live_gb300 as dsa
    T, S, B, Kb, K, ends = CASES[name]
    q, k, ks, w, _, en = wk.indexer_exact_inputs(T, S, seed=30 + len(name))
    if ends is not None:
        en = np.asarray(ends, dtype=np.int32)
    fill = 1.5
    want_logits, want_cand, want_topk = _oracle(q, k, ks, w, en, B, Kb, K, fill)
    dev = "cuda:0"
    qd, kd, ksd, wd, end = (torch.from_numpy(x).to(dev) for x in (q, k, ks, w, en))
    # the producer alone: bit-exact logits, nothing written outside the spans
    logits = torch.full((T, S), fill, dtype=torch.float32, device=dev)
    dsa.dsa_indexer_logits(qd, kd, ksd, wd, None, end, logits)
    # the fused call
    plan = dsa.dsa_select_init(rows=T, width=S, block_size=B, block_topk=Kb, row_topk=K)
    ws = torch.full((dsa.dsa_indexer_select_workspace(plan),), 0xA5, dtype=torch.uint8, device=dev)
    cand = torch.full((T, Kb + 1), -7, dtype=torch.int32, device=dev)
    topk = torch.full((T, K), -7, dtype=torch.int32, device=dev)
    dsa.dsa_indexer_select(plan, qd, kd, ksd, wd, end, ws, cand, topk)
    torch.cuda.synchronize()
    assert dsa.dsa_indexer_status() == dsa.DSA_OK
    got = logits.cpu().numpy()
    for t in range(T):
        bad = np.nonzero(got[t].view(np.uint32) != want_logits[t].view(np.uint32))[0]
        assert len(bad) == 0, (f"logits of query {t} (end {en[t]}) differ at {bad[:6]}: "
                               f"{got[t, bad[:3]]} vs {want_logits[t, bad[:3]]}")
    c, tk = cand.cpu().numpy(), topk.cpu().numpy()
    for t in range(T):
        assert np.array_equal(c[t], want_cand[t]), f"cand of query {t} (end {en[t]})"
        assert np.array_equal(tk[t], want_topk[t]), f"topk of query {t} (end {en[t]})"
