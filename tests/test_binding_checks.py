"""The binding's argument checks run on the host, before any pointer reaches
the C ABI (which cannot see tensor sizes): wrong types raise TypeError, wrong
devices, layouts or sizes raise ValueError -- and none of them is an
`assert`, so `python -O` keeps them.  No GPU is needed: a tensor subclass that
reports a CUDA device stands in for device tensors, and every check fires
before the library is called."""
import os
import subprocess
import sys
import types

import pytest

torch = pytest.importorskip("torch")

from sparse_attention_indexer_live_gb300 import binding as B  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


class _OnCuda(torch.Tensor):
    """A host tensor that reports cuda:0 (for the checks only; never launched)."""

    @property
    def is_cuda(self):
        return True

    @property
    def device(self):
        return torch.device("cuda", 0)


def dev(t):
    return torch.Tensor._make_subclass(_OnCuda, t)


def plan(**kw):
    shape = dict(rows=4, width=1000, block_size=8, block_topk=16, row_topk=32)
    shape.update(kw)
    return types.SimpleNamespace(cfg=B.make_cfg(**shape), device=0)


def sel_args(p, rows=4, width=1000, cand_cols=17, topk_cols=32, ends_n=4):
    return (dev(torch.zeros(rows, width)), None, dev(torch.zeros(ends_n, dtype=torch.int32)),
            [("cand", dev(torch.zeros(rows, cand_cols, dtype=torch.int32)), 17),
             ("topk", dev(torch.zeros(rows, topk_cols, dtype=torch.int32)), 32)])


def test_well_formed_selection_arguments_pass():
    p = plan()
    B._check_tensors(p, *sel_args(p))


@pytest.mark.parametrize("bad,exc", [
    (dict(topk_cols=31), ValueError),      # topk one column short
    (dict(cand_cols=16), ValueError),      # cand one column short
    (dict(ends_n=3), ValueError),          # fewer ends than rows
    (dict(rows=3), ValueError),            # logits rows differ from the plan
])
def test_undersized_selection_arguments_raise(bad, exc):
    p = plan()
    with pytest.raises(exc):
        B._check_tensors(p, *sel_args(p, **bad))


def test_wrong_dtype_device_and_starts():
    p = plan()
    logits, starts, ends, outs = sel_args(p)
    with pytest.raises(TypeError):
        B._check_tensors(p, dev(torch.zeros(4, 1000, dtype=torch.float64)), None, ends, outs)
    with pytest.raises(ValueError):  # a host tensor
        B._check_tensors(p, torch.zeros(4, 1000), None, ends, outs)
    with pytest.raises(TypeError):
        B._check_tensors(p, logits, None, dev(torch.zeros(4, dtype=torch.int64)), outs)
    with pytest.raises(ValueError):  # starts given to a plan made without them
        B._check_tensors(p, logits, dev(torch.zeros(4, dtype=torch.int32)), ends, outs)
    ps = plan(has_starts=True)
    with pytest.raises(ValueError):  # and missing for a plan made with them
        B._check_tensors(ps, logits, None, ends, outs)
    with pytest.raises(ValueError):  # a plan for another device
        B._check_tensors(types.SimpleNamespace(cfg=p.cfg, device=1), logits, None, ends, outs)


def _indexer(T=3, S=500, H=64, D=128, **short):
    n = dict(ks=S, w=T * H, ends=T)
    n.update(short)
    q = dev(torch.zeros(T, H, D, dtype=torch.uint8))
    k = dev(torch.zeros(S, D, dtype=torch.uint8))
    return (q, k, dev(torch.zeros(n["ks"])), dev(torch.zeros(n["w"])),
            dev(torch.zeros(n["ends"], dtype=torch.int32)))


def test_producer_arguments():
    assert B._indexer_args(*_indexer()) == (3, 64, 128, 500)
    for short in (dict(ks=499), dict(w=3 * 64 - 1), dict(ends=2)):
        with pytest.raises(ValueError):
            B._indexer_args(*_indexer(**short))
    q, k, ks, w, ends = _indexer()
    with pytest.raises(ValueError):  # k's row length differs from q's head_dim
        B._indexer_args(q, dev(torch.zeros(500, 64, dtype=torch.uint8)), ks, w, ends)
    with pytest.raises(TypeError):
        B._indexer_args(q, k, dev(torch.zeros(500, dtype=torch.float16)), w, ends)


def test_fused_selection_checks_the_plan_shape():
    p = plan(rows=3, width=500)
    q, k, ks, w, ends = _indexer()
    cand = dev(torch.zeros(3, 17, dtype=torch.int32))
    topk = dev(torch.zeros(3, 32, dtype=torch.int32))
    cfg = B._fused_args(p, q, k, ks, w, ends, cand, topk)
    assert (cfg.queries, cfg.keys) == (3, 500)
    with pytest.raises(ValueError):  # plan width differs from the key count
        B._fused_args(plan(rows=3, width=501), q, k, ks, w, ends, cand, topk)
    with pytest.raises(ValueError):
        B._fused_args(p, q, k, ks, w, ends, cand, dev(torch.zeros(3, 31, dtype=torch.int32)))


def test_attention_arguments():
    cfg = B.dsa_attention_cfg(tokens=4, heads=8, keys=100, head_dim=128, value_dim=128, select=16)
    ws = dev(torch.zeros(64, dtype=torch.uint8))
    B._attention_idx(cfg, dev(torch.zeros(4, 16, dtype=torch.int32)), ws)
    with pytest.raises(ValueError):
        B._attention_idx(cfg, dev(torch.zeros(4, 15, dtype=torch.int32)), ws)
    with pytest.raises(TypeError):
        B._attention_idx(cfg, dev(torch.zeros(4, 16, dtype=torch.int32)),
                         dev(torch.zeros(64, dtype=torch.int8)))


def test_attention_range_arguments():
    cfg = B.dsa_attention_cfg(tokens=4, heads=8, keys=100, head_dim=128, value_dim=128, select=16)
    ws = dev(torch.zeros(64, dtype=torch.uint8))
    assert B._attention_ranges(cfg, dev(torch.zeros(4, 2, 2, dtype=torch.int32)), ws) == 2
    for shape in ((4, 2), (4, 2, 3), (3, 2, 2)):
        with pytest.raises(ValueError):
            B._attention_ranges(cfg, dev(torch.zeros(*shape, dtype=torch.int32)), ws)
    with pytest.raises(TypeError):
        B._attention_ranges(cfg, dev(torch.zeros(4, 2, 2, dtype=torch.int64)), ws)


def test_attention_range_workspace_limits():
    # the C ABI's own checks (no device call): 1..8 ranges a token, and a
    # record bound far above the index-list form's
    cfg = B.dsa_attention_cfg(tokens=2048, heads=8, keys=1 << 20, head_dim=128, value_dim=128,
                              select=8704)
    n = B.dsa_sparse_attention_ranges_workspace(cfg, 2)
    G, cap = 16, 16 * 8704
    assert n == 128 * (16 + 2 * ((cap * 4 + 15) & ~15))
    for nr, status in ((0, B.DSA_ERR_INVALID_ARG), (9, B.DSA_ERR_UNSUPPORTED)):
        with pytest.raises(B.DsaSelectError) as e:
            B.dsa_sparse_attention_ranges_workspace(cfg, nr)
        assert e.value.status == status
    # the index-list form refuses this select (its union is built in shared memory)
    with pytest.raises(B.DsaSelectError) as e:
        B.dsa_sparse_attention_workspace(cfg)
    assert e.value.status == B.DSA_ERR_UNSUPPORTED
    del G


def test_checks_survive_python_O():
    # under -O every assert statement is stripped; the checks must still raise
    code = ("import sys, torch; sys.path.insert(0, %r)\n"
            "from sparse_attention_indexer_live_gb300 import binding as B\n"
            "try:\n"
            "    B._tensor('x', torch.zeros(3), (torch.int32,))\n"
            "except TypeError:\n"
            "    print('raised')\n" % ROOT)
    out = subprocess.run([sys.executable, "-O", "-c", code], capture_output=True, text=True,
                         timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    assert out.stdout.strip() == "raised"
