"""Build libdgcanvas.so in-tree with nvcc for sm_103a (cross-compiles without a GPU).

    python -m uniform_state_denoising_vocab_b300.build [--force]
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
CSRC = PKG / "csrc"
INCLUDE = PKG.parent / "include"
OUT = PKG / "libdgcanvas.so"
OBJ = PKG / "_build"
SOURCES = ["dg_abi.cu", "dg_head_tc.cu", "dg_head_tc2.cu", "dg_head_fp4.cu", "dg_nvfp4.cu", "dg_head_simt.cu",
           "dg_sampler.cu", "dg_noalloc.cu", "dg_host.cu"]
HEADERS = ["dg_common.cuh", "dg_head_epi.cuh", "dg_ptx.cuh", "dg_internal.h", "dg_nvtx.h"]
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
         "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden", "-I", str(INCLUDE),
         "--expt-relaxed-constexpr"]


def _stale(target: Path, deps) -> bool:
    if not target.exists():
        return True
    t = target.stat().st_mtime
    return any(Path(d).stat().st_mtime > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> Path:
    OBJ.mkdir(exist_ok=True)
    hdrs = [CSRC / h for h in HEADERS] + [INCLUDE / "dgcanvas.h"]
    objs = []
    jobs = []
    for src in SOURCES:
        s = CSRC / src
        o = OBJ / (src + ".o")
        objs.append(o)
        if force or _stale(o, [s, *hdrs]):
            jobs.append([NVCC, *FLAGS, "-c", str(s), "-o", str(o)])

    def run(cmd):
        if verbose:
            print(" ".join(cmd), flush=True)
        subprocess.run(cmd, check=True)

    with ThreadPoolExecutor(max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        list(ex.map(run, jobs))
    if force or jobs or _stale(OUT, objs):
        tmp = OUT.with_suffix(f".{os.getpid()}.tmp")
        run([NVCC, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-cudart", "static",
             "-o", str(tmp), *map(str, objs)])
        os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
    print(OUT)
