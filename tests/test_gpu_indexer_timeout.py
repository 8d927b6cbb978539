"""Failure detection of the tensor-core producer without a GPU fault: a test
build of the library (compile-time hooks, never in the product build) makes
the first K stage's mbarrier expect one chunk more than its copy delivers, so
the bounded waits run out; the kernel then winds down, dsa_indexer_status()
reports DSA_ERR_TIMEOUT once, and the CUDA context stays usable.  The same
holds for the fused producer + selection form."""
import os
import subprocess
import sys
import textwrap

import pytest

torch = pytest.importorskip("torch")

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bounded_wait_reports_timeout(tmp_path):
    import importlib
    B = importlib.import_module("sparse_attention_indexer_live_gb300.build")
    so = tmp_path / "libdsa_timeout.so"
    objs = []
    for src in B.SOURCES:
        obj = tmp_path / (os.path.basename(src) + ".o")
        subprocess.run([B.nvcc_path(), *B.ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-c",
                        "-DDSA_INDEXER_TEST_WAIT_CYCLES=20000000ll", "-DDSA_INDEXER_TEST_STARVE",
                        "-I", B.INCLUDE, "-o", str(obj), src], check=True)
        objs.append(str(obj))
    subprocess.run([B.nvcc_path(), *B.ARCH, "-shared", "-o", str(so), *objs], check=True)
    script = textwrap.dedent(f"""
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
    """)
    res = subprocess.run([sys.executable, "-c", script], capture_output=True, text=True,
                         timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    first, second, third, fourth, alive = res.stdout.split()[-5:]
    import sparse_attention_indexer_live_gb300 as dsa
    assert int(first) == dsa.DSA_ERR_TIMEOUT
    assert int(second) == dsa.DSA_OK       # reported once, then cleared
    assert int(third) == dsa.DSA_ERR_TIMEOUT  # the fused form winds down the same way
    assert int(fourth) == dsa.DSA_OK
    assert float(alive) == 1024.0          # the context is still usable
