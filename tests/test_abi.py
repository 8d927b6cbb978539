"""The C ABI without a GPU: the library loads, exports every function the
header declares, validates shapes before touching CUDA, rejects NULL
arguments, and the binding's structs match the C layout."""
import ctypes
import os
import re
import subprocess

import pytest

import sparse_attention_indexer_live_gb300 as dsa
from sparse_attention_indexer_live_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    dsa.build()
    return dsa.load()


def declared_functions():
    names = set()
    for h in HEADERS:
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(dsa_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 7
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(binding.EXPORTS) <= set(names)


def test_exports_are_c_linkage():
    out = subprocess.run(["nm", "-D", "--defined-only", dsa.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for n in declared_functions():
        assert n in syms


def _init(lib, **kw):
    base = dict(rows=4, width=4096, block_size=8, block_topk=32, row_topk=64)
    raw = {k: kw.pop(k) for k in ("has_starts", "repeat_causal", "split") if k in kw}
    base.update(kw)
    cfg = dsa.make_cfg(**base)
    for k, v in raw.items():  # set the raw C fields, bypassing make_cfg's normalisation
        setattr(cfg, k, v)
    h = ctypes.c_void_p()
    ws = ctypes.c_size_t(123)
    rc = lib.dsa_select_init(ctypes.byref(cfg), 0, ctypes.byref(h), ctypes.byref(ws))
    if rc == dsa.DSA_OK:
        lib.dsa_select_destroy(h)
    return rc


@pytest.mark.parametrize("kw", [dict(width=0), dict(width=-1), dict(width=1 << 31),
                                dict(block_size=0), dict(block_topk=0), dict(row_topk=0),
                                dict(rows=-1), dict(row_repeat=0), dict(col_stride=0),
                                dict(row_stride=100), dict(has_starts=2), dict(repeat_causal=3),
                                dict(split=3), dict(split=-2)])
def test_invalid_shapes_rejected_before_cuda(lib, kw):
    assert _init(lib, **kw) == dsa.DSA_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(row_topk=4097), dict(block_topk=5000),
                                dict(block_size=5000), dict(split=512)])
def test_out_of_range_shapes_unsupported(lib, kw):
    assert _init(lib, **kw) == dsa.DSA_ERR_UNSUPPORTED


def test_valid_shape_reaches_cuda(lib):
    import torch
    rc = _init(lib)
    if torch.cuda.is_available():
        assert rc == dsa.DSA_OK
    else:
        assert rc == dsa.DSA_ERR_CUDA


def test_null_arguments(lib):
    vp = ctypes.c_void_p
    assert lib.dsa_select_init(None, 0, ctypes.byref(vp()), None) == dsa.DSA_ERR_INVALID_ARG
    cfg = dsa.make_cfg(rows=1, width=8, block_size=4, block_topk=1, row_topk=1)
    assert lib.dsa_select_init(ctypes.byref(cfg), 0, None, None) == dsa.DSA_ERR_INVALID_ARG
    for fn, nargs in (("dsa_candidate_select", 7), ("dsa_row_topk", 8), ("dsa_select_topk", 8)):
        assert getattr(lib, fn)(*([None] * nargs)) == dsa.DSA_ERR_INVALID_ARG
    d = dsa.dsa_plan_desc()
    assert lib.dsa_plan_describe(None, ctypes.byref(d)) == dsa.DSA_ERR_INVALID_ARG
    lib.dsa_select_destroy(None)


def test_status_strings(lib):
    for s in range(5):
        assert dsa.status_string(s) != "unknown status"
    assert dsa.status_string(99) == "unknown status"


def test_struct_layout_matches_header(tmp_path):
    prog = tmp_path / "layout.c"
    fields_cfg = [f for f, _ in binding.dsa_select_cfg._fields_]
    fields_desc = [f for f, _ in binding.dsa_plan_desc._fields_]
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "dsa_select.h"',
             'int main(void) {',
             'printf("cfg %zu\\n", sizeof(dsa_select_cfg));',
             'printf("desc %zu\\n", sizeof(dsa_plan_desc));']
    lines += [f'printf("cfg.{f} %zu\\n", offsetof(dsa_select_cfg, {f}));' for f in fields_cfg]
    lines += [f'printf("desc.{f} %zu\\n", offsetof(dsa_plan_desc, {f}));' for f in fields_desc]
    lines += ["return 0; }"]
    prog.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(prog)],
                   check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True,
                                                       text=True).stdout.splitlines())
    assert int(got["cfg"]) == ctypes.sizeof(binding.dsa_select_cfg)
    assert int(got["desc"]) == ctypes.sizeof(binding.dsa_plan_desc)
    for f in fields_cfg:
        assert int(got[f"cfg.{f}"]) == getattr(binding.dsa_select_cfg, f).offset
    for f in fields_desc:
        assert int(got[f"desc.{f}"]) == getattr(binding.dsa_plan_desc, f).offset


def test_product_path_does_not_import_oracle():
    pkg = os.path.join(ROOT, "sparse_attention_indexer_live_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in src.replace("the oracle", ""), f


def test_attention_shapes_checked_without_cuda(lib):
    # the workspace query validates the shape on the host only
    def ws(**kw):
        c = dict(tokens=37, heads=8, keys=5000, head_dim=128, value_dim=128, select=64)
        c.update(kw)
        n = ctypes.c_size_t(123)
        rc = lib.dsa_sparse_attention_workspace(ctypes.byref(binding.dsa_attention_cfg(**c)), ctypes.byref(n))
        return rc, n.value
    rc, n = ws()
    # 3 groups of 16 tokens: header 16 + keys 16 * 64 * 4 + masks 16 * 64 * 4 bytes each
    assert rc == dsa.DSA_OK and n == 3 * (16 + 2 * 16 * 64 * 4)
    rc, n = ws(heads=16)
    assert rc == dsa.DSA_OK and n == 5 * (16 + 2 * 8 * 64 * 4)
    for kw in (dict(heads=4), dict(heads=32), dict(head_dim=64), dict(value_dim=256),
               dict(select=3073), dict(heads=16, select=6145)):
        assert ws(**kw)[0] == dsa.DSA_ERR_UNSUPPORTED, kw
    for kw in (dict(tokens=-1), dict(select=-2), dict(keys=-5)):
        assert ws(**kw)[0] == dsa.DSA_ERR_INVALID_ARG, kw
    assert lib.dsa_sparse_attention_workspace(None, ctypes.byref(ctypes.c_size_t())) == dsa.DSA_ERR_INVALID_ARG
