"""The allocation-free fused selection, dsa_indexer_select_noalloc.

Some callers of this library cannot allocate device memory when they call it:
an engine that gave all free device memory to its own pool before serving, a
plugin running under a host framework that owns the device allocator, or C
code with no allocator at hand.  For them the fused producer + selection keeps
its per-query records in a fixed array inside the library instead of a
workspace the caller allocates.

These tests call it through the C ABI and check that it returns exactly what
dsa_indexer_select returns with a caller workspace (indices, compared bit for
bit like every selection test here), on two calls in a row with different
inputs -- the second call runs on whatever the first left in the shared array.
The file is named to be collected last.
"""
import numpy as np
import pytest

import workloads as wk

pytestmark = pytest.mark.gpu


def _torch():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return torch


def test_noalloc_matches_the_workspace_call_twice_in_a_row():
    torch = _torch()
    import sparse_attention_indexer_live_gb300 as dsa
    dev = "cuda:0"
    # 96 queries of 65,536 keys at block size 8 fit the fixed array (about 4 MB of records)
    T, S, B, Kb, K = 96, 65536, 8, 256, 2048
    plan = dsa.dsa_select_init(rows=T, width=S, block_size=B, block_topk=Kb, row_topk=K)
    need = dsa.dsa_indexer_select_workspace(plan)
    assert need <= dsa.NOALLOC_SCRATCH_BYTES
    rng = np.random.default_rng(33)
    for call, seed in enumerate((31, 32)):
        q, k, ks, w, _, en = wk.indexer_inputs(T, S, seed)
        if call == 1:
            # other spans (some empty, some past the width) on the second call
            en = rng.integers(-3, S + 9, size=T).astype(np.int32)
        qd, kd, ksd, wd, end = (torch.from_numpy(x).to(dev) for x in (q, k, ks, w, en))
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
        cand_ref = torch.empty((T, Kb + 1), dtype=torch.int32, device=dev)
        topk_ref = torch.empty((T, K), dtype=torch.int32, device=dev)
        dsa.dsa_indexer_select(plan, qd, kd, ksd, wd, end, ws, cand_ref, topk_ref)
        cand = torch.full((T, Kb + 1), -9, dtype=torch.int32, device=dev)
        topk = torch.full((T, K), -9, dtype=torch.int32, device=dev)
        dsa.dsa_indexer_select_noalloc(plan, qd, kd, ksd, wd, end, cand, topk)
        torch.cuda.synchronize()
        assert dsa.dsa_indexer_status() == dsa.DSA_OK
        assert torch.equal(cand, cand_ref), f"cand differs on call {call + 1}"
        assert torch.equal(topk, topk_ref), f"topk differs on call {call + 1}"


def test_noalloc_refuses_a_batch_larger_than_its_array():
    torch = _torch()
    import sparse_attention_indexer_live_gb300 as dsa
    dev = "cuda:0"
    T, S = 40, 1 << 19  # 40 records of about 260 KB: more than the 8 MiB array
    plan = dsa.dsa_select_init(rows=T, width=S, block_size=8, block_topk=32, row_topk=64)
    assert dsa.dsa_indexer_select_workspace(plan) > dsa.NOALLOC_SCRATCH_BYTES
    q, k, ks, w, _, en = wk.indexer_inputs(T, S, seed=34)
    qd, kd, ksd, wd, end = (torch.from_numpy(x).to(dev) for x in (q, k, ks, w, en))
    cand = torch.empty((T, 33), dtype=torch.int32, device=dev)
    topk = torch.empty((T, 64), dtype=torch.int32, device=dev)
    with pytest.raises(dsa.DsaSelectError) as e:
        dsa.dsa_indexer_select_noalloc(plan, qd, kd, ksd, wd, end, cand, topk)
    assert e.value.status == dsa.DSA_ERR_UNSUPPORTED
    assert "fixed scratch" in str(e.value)
    torch.cuda.synchronize()
    assert dsa.dsa_indexer_status() == dsa.DSA_OK
