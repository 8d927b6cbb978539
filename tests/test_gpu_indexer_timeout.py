"""Failure detection of the tensor-core kernels without a GPU fault.

A test build of the library (compile-time hooks, never in the product build)
shortens the bounded waits to 20 M cycles and starves one barrier of each
tcgen05 kernel: the producer's first K stage expects one chunk more than its
copy delivers, and the grouped attention's Q barrier expects one arrival more
than the Q copy makes.  The waits then run out, every role of the kernel
winds down and frees its tensor memory, the kernel's status call reports
DSA_ERR_TIMEOUT once, and the CUDA context stays usable.  The same holds for
the fused producer + selection form."""
import os
import subprocess
import sys
import textwrap

import pytest

torch = pytest.importorskip("torch")

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def starved_lib(tmp_path_factory):
    import importlib
    B = importlib.import_module("sparse_attention_indexer_live_gb300.build")
    tmp = tmp_path_factory.mktemp("starved")
    so = tmp / "libdsa_timeout.so"
    objs = []
    for src in B.SOURCES:
        obj = tmp / (os.path.basename(src) + ".o")
        subprocess.run([B.nvcc_path(), *B.ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-c",
                        "-DDSA_INDEXER_TEST_WAIT_CYCLES=20000000ll", "-DDSA_INDEXER_TEST_STARVE",
                        "-DDSA_ATTENTION_TEST_STARVE", "-I", B.INCLUDE, "-o", str(obj), src],
                       check=True)
        objs.append(str(obj))
    subprocess.run([B.nvcc_path(), *B.ARCH, "-shared", "-o", str(so), *objs], check=True)
    return str(so)


def _run(script):
    res = subprocess.run([sys.executable, "-c", textwrap.dedent(script)], capture_output=True,
                         text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    return res.stdout.split()


def test_bounded_wait_reports_timeout(starved_lib):
    so = starved_lib
    script = f"""
        import sys, torch
        sys.path.insert(0, {ROOT!r})
        from sparse_attention_indexer_live_gb300 import binding
        binding.load({str(so)!r})
        import sparse_attention_indexer_live_gb300 as dsa
        import workloads as wk
        q, k, ks, w, st, en = wk.indexer_inputs(8, 4096, seed=5)
        d = "cuda:0"
        out = torch.full((8, 4096), 1.5, device=d)
        dsa.dsa_indexer_logits(torch.from_numpy(q).to(d), torch.from_numpy(k).to(d),
                               torch.from_numpy(ks).to(d), torch.from_numpy(w).to(d), None,
                               torch.from_numpy(en).to(d), out)
        torch.cuda.synchronize()
        first = dsa.dsa_indexer_status()
        second = dsa.dsa_indexer_status()
        # the fused form: its epilogue warps meet at named barriers every tile,
        # so after the first wait gives up they must still walk every tile
        plan = dsa.dsa_select_init(rows=8, width=4096, block_size=8, block_topk=32, row_topk=64)
        ws = torch.zeros(dsa.dsa_indexer_select_workspace(plan), dtype=torch.uint8, device=d)
        cand = torch.empty((8, 33), dtype=torch.int32, device=d)
        topk = torch.empty((8, 64), dtype=torch.int32, device=d)
        dsa.dsa_indexer_select(plan, torch.from_numpy(q).to(d), torch.from_numpy(k).to(d),
                               torch.from_numpy(ks).to(d), torch.from_numpy(w).to(d),
                               torch.from_numpy(en).to(d), ws, cand, topk)
        torch.cuda.synchronize()
        third = dsa.dsa_indexer_status()
        fourth = dsa.dsa_indexer_status()
        alive = float(torch.ones(1024, device=d).sum().item())
        print(first, second, third, fourth, alive)
    """
    first, second, third, fourth, alive = _run(script)[-5:]
    import sparse_attention_indexer_live_gb300 as dsa
    assert int(first) == dsa.DSA_ERR_TIMEOUT
    assert int(second) == dsa.DSA_OK       # reported once, then cleared
    assert int(third) == dsa.DSA_ERR_TIMEOUT  # the fused form winds down the same way
    assert int(fourth) == dsa.DSA_OK
    assert float(alive) == 1024.0          # the context is still usable


def test_attention_bounded_wait_reports_timeout(starved_lib):
    so = starved_lib
    script = f"""
        import sys, math, torch
        import numpy as np
        sys.path.insert(0, {ROOT!r})
        from sparse_attention_indexer_live_gb300 import binding
        binding.load({so!r})
        import sparse_attention_indexer_live_gb300 as dsa
        import workloads as wk
        d = "cuda:0"
        # 3 groups of 16 tokens x 8 heads, unions of several 128-position tiles
        q, k, v, idx = wk.attention_inputs(40, 8, 4096, 256, seed=7, own=0.5, G=16)
        qd, kd, vd = (torch.from_numpy(x.view(np.int16)).to(d) for x in (q, k, v))
        idd = torch.from_numpy(idx).to(d)
        cfg = dsa.attention_cfg(qd, kd, idd)
        ws = torch.zeros(dsa.dsa_sparse_attention_workspace(cfg), dtype=torch.uint8, device=d)
        o = torch.zeros((40, 8, 128), dtype=torch.float32, device=d)
        lse = torch.zeros((40, 8), dtype=torch.float32, device=d)
        dsa.dsa_sparse_attention(cfg, qd, kd, vd, idd, 1.0 / math.sqrt(128), ws, o, lse)
        torch.cuda.synchronize()
        first = dsa.dsa_sparse_attention_status()
        second = dsa.dsa_sparse_attention_status()
        # a second launch on the same context winds down the same way
        dsa.dsa_sparse_attention(cfg, qd, kd, vd, idd, 1.0 / math.sqrt(128), ws, o, lse)
        torch.cuda.synchronize()
        third = dsa.dsa_sparse_attention_status()
        alive = float(torch.ones(1024, device=d).sum().item())
        print(first, second, third, alive)
    """
    first, second, third, alive = _run(script)[-4:]
    import sparse_attention_indexer_live_gb300 as dsa
    assert int(first) == dsa.DSA_ERR_TIMEOUT
    assert int(second) == dsa.DSA_OK       # reported once, then cleared
    assert int(third) == dsa.DSA_ERR_TIMEOUT
    assert float(alive) == 1024.0          # the context is still usable
