"""Build libsdpa_gb300.so in-tree with nvcc for sm_103a.

Usage: ``python -m attention_sm_flash_attn_gb300.build`` (or ``build()``).
The library is rebuilt when any source under csrc/ or the public header is
newer than it.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_NAME = "libsdpa_gb300.so"
LIB_PATH = os.path.join(HERE, LIB_NAME)
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def _nvcc() -> str:
    cuda_home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(cuda_home, "bin", "nvcc")
    if os.path.exists(cand):
        return cand
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found (set CUDA_HOME)")
    return found


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + glob.glob(os.path.join(INCLUDE, "*.h")))


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(s) <= t for s in _sources())


def _flags():
    return [ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xptxas", "-v", "-Xcompiler", "-fPIC",
            "-I", INCLUDE]


def compile_commands(out: str):
    """One `nvcc -c` per translation unit (run in parallel), then the link."""
    nvcc = _nvcc()
    cuda_lib = os.path.join(os.path.dirname(os.path.dirname(nvcc)), "lib64")
    obj_dir = os.path.join(HERE, "_build")
    units = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    objs = [os.path.join(obj_dir, os.path.basename(u)[:-3] + f".{os.getpid()}.o") for u in units]
    compiles = [[nvcc, *_flags(), "-c", u, "-o", o] for u, o in zip(units, objs)]
    link = [nvcc, ARCH, "-shared", "-cudart", "shared", "-Xlinker", f"-rpath,{cuda_lib}",
            "-o", out, *objs]
    return compiles, link, objs


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    compiles, link, objs = compile_commands(tmp)
    os.makedirs(os.path.join(HERE, "_build"), exist_ok=True)
    log = []
    try:
        procs = [(c, subprocess.Popen(c, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                      text=True)) for c in compiles]
        failed = None
        for c, pr in procs:
            out, _ = pr.communicate()
            log.append(out)
            if pr.returncode != 0 and failed is None:
                failed = (c, out)
        if failed:
            raise RuntimeError("nvcc failed:\n" + " ".join(failed[0]) + "\n" + failed[1])
        res = subprocess.run(link, capture_output=True, text=True)
        log.append(res.stdout + res.stderr)
        if res.returncode != 0:
            raise RuntimeError("link failed:\n" + " ".join(link) + "\n" + res.stdout + res.stderr)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
    if verbose:
        print("".join(log))
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
