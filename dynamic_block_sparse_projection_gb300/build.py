"""Build libdsv.so (the C-ABI library) for sm_103a with nvcc, in-tree.

One nvcc process per translation unit, run in parallel, then one link step.
Output: dynamic_block_sparse_projection_gb300/_build/libdsv.so.  Rebuilds only
when a source or header is newer than the library.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
OUT = PKG / "_build"
LIB = OUT / "libdsv.so"
SOURCES = ["dsv_api.cu", "predict.cu", "topk.cu", "attn_fwd.cu", "attn_bwd.cu", "topk_noalloc.cu", "cube.cu",
           "predict_max.cu", "predict_topk.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdsv")


def _inputs():
    return [CSRC / s for s in SOURCES] + list(CSRC.glob("*.cuh")) + list(CSRC.glob("*.h")) + list(INCLUDE.glob("*.h"))


def up_to_date() -> bool:
    if not LIB.exists():
        return False
    t = LIB.stat().st_mtime
    return all(p.stat().st_mtime <= t for p in _inputs())


def build(force: bool = False, ptxas_verbose: bool = False, quiet: bool = False) -> Path:
    if not force and not ptxas_verbose and up_to_date():
        return LIB
    OUT.mkdir(exist_ok=True)
    nvcc = _nvcc()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", str(INCLUDE), "-I", str(CSRC)]
    if ptxas_verbose:
        flags += ["-Xptxas", "-v"]

    def compile_one(src: str):
        obj = OUT / (Path(src).stem + ".o")
        cmd = [nvcc, "-c", str(CSRC / src), "-o", str(obj)] + flags
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    failed = [(s, r) for s, _, r in results if r.returncode != 0]
    for s, _, r in results:
        if (ptxas_verbose or r.returncode != 0) and not quiet:
            sys.stderr.write(f"--- {s}\n{r.stdout}{r.stderr}")
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(s for s, _ in failed))
    tmp = OUT / "libdsv.so.tmp"
    cmd = [nvcc, "-shared", "-o", str(tmp)] + [str(o) for _, o, _ in results] + ARCH
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, ptxas_verbose="-v" in sys.argv)
    print(LIB)
