"""Compile the sm_103a CUDA library in-tree (nvcc, no torch extension machinery).

Output: sparse_attention_indexer_live_gb300/_build/libdsa_select.so, plus the
ptxas resource report (registers, spills, shared memory) next to it.
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
INCLUDE = os.path.join(ROOT, "include")
SOURCES = [os.path.join(PKG, "csrc", "dsa_select.cu"), os.path.join(PKG, "csrc", "dsa_indexer.cu"),
           os.path.join(PKG, "csrc", "dsa_attention.cu")]
HEADERS = [os.path.join(INCLUDE, "dsa_select.h"), os.path.join(PKG, "csrc", "dsa_internal.h")]
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libdsa_select.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return os.path.join(cand, "bin", "nvcc")
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found: the CUDA library cannot be built")
    return found


def stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in SOURCES + HEADERS)


def build(force: bool = False) -> str:
    """Compile every translation unit in parallel, then link the library."""
    from concurrent.futures import ThreadPoolExecutor
    if not force and not stale():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = nvcc_path()
    pid = os.getpid()

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.basename(src) + f".{pid}.o")
        cmd = [nvcc, *ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xptxas", "-v",
               "-Xcompiler", "-fPIC", "-c", "-I", INCLUDE, "-o", obj, src]
        res = subprocess.run(cmd, capture_output=True, text=True)
        return obj, " ".join(cmd) + "\n" + res.stdout + res.stderr, res.returncode

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    with open(os.path.join(BUILD_DIR, "ptxas.txt"), "w") as f:
        f.write("\n".join(log for _, log, _ in results))
    bad = [log for _, log, rc in results if rc != 0]
    if bad:
        raise RuntimeError("nvcc failed:\n" + bad[0][-4000:])
    tmp = LIB_PATH + f".tmp{pid}"
    res = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *[o for o, _, _ in results]],
                         capture_output=True, text=True)
    for o, _, _ in results:
        os.remove(o)
    if res.returncode != 0:
        raise RuntimeError("nvcc link failed:\n" + res.stderr[-4000:])
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True))
