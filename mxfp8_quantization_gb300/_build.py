"""Builds the CUDA library librn.so in-tree with nvcc (sm_103a only).

Each translation unit is compiled in parallel, then linked into one shared
object next to this file, with the CUDA runtime linked statically so the
library carries no runtime dependency beyond the driver.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "librn.so")
SOURCES = ["rn_api.cu", "rn_fwd.cu", "rn_fwd_res.cu", "rn_mx.cu", "rn_bwd.cu", "rn_scaling.cu", "rn_act.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build librn.so")
    return cand


def _stale(objs) -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(os.path.dirname(HERE), "include", "rn.h"))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile librn.so if a source is newer than it; return its path."""
    build_dir = os.path.join(HERE, "_build")
    os.makedirs(build_dir, exist_ok=True)
    objs = [os.path.join(build_dir, s.replace(".cu", ".o")) for s in SOURCES]
    if not force and not _stale(objs):
        return LIB
    nvcc = _nvcc()

    def compile_one(src_obj):
        src, obj = src_obj
        cmd = [nvcc, *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        logs = list(ex.map(compile_one, zip(SOURCES, objs)))
    tmp = LIB + ".tmp"
    # export only the rn_* entry points: the statically linked CUDA runtime
    # stays private, so another runtime loaded in the process cannot
    # interpose on it
    vscript = os.path.join(build_dir, "exports.map")
    with open(vscript, "w") as f:
        f.write("{ global: rn_*; local: *; };\n")
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs,
           "-Xlinker", f"--version-script={vscript}", "-lpthread", "-ldl", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    if verbose:
        for log in logs:
            print(log)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
