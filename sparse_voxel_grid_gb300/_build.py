"""Builds libvbm.so in-tree for sm_103a (nvcc + g++, translation units compiled
in parallel).  `python -m sparse_voxel_grid_gb300._build [--force]`."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libvbm.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CU_SOURCES = ["vbm_api.cu", "vbm_decode.cu", "vbm_box.cu", "vbm_cross.cu", "vbm_brick.cu", "vbm_weno.cu", "vbm_weno_brick.cu", "vbm_build_dev.cu", "vbm_probe.cu", "vbm_host.cu", "vbm_shard.cu"]
CPP_SOURCES = ["vbm_build.cpp"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _cuda_include() -> str:
    nvcc = os.path.realpath(_nvcc())
    return os.path.join(os.path.dirname(os.path.dirname(nvcc)), "include")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "vbm.h"))
    files.append(os.path.abspath(__file__))
    return files


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _deps())


def _run(cmd, log):
    r = subprocess.run(cmd, capture_output=True, text=True)
    with open(log, "w") as fh:
        fh.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError(f"build failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every translation unit and link libvbm.so; returns its path."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    jobs = []
    # Optional extra nvcc flags (e.g. -D tuning constants) from VBM_NVCC_FLAGS.
    extra = os.environ.get("VBM_NVCC_FLAGS", "").split()
    for src in CU_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        cmd = [nvcc, "-std=c++20", "-O3", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC", "-Xptxas", "-v", *extra,
               "-I", INCLUDE, "-c", os.path.join(CSRC, src), "-o", obj]
        jobs.append((cmd, obj, os.path.join(BUILD, src + ".log")))
    for src in CPP_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        cmd = ["g++", "-std=c++20", "-O3", "-fPIC", "-Wall", "-I", INCLUDE, "-I", _cuda_include(),
               "-c", os.path.join(CSRC, src), "-o", obj]
        jobs.append((cmd, obj, os.path.join(BUILD, src + ".log")))
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        futs = [ex.submit(_run, cmd, log) for cmd, _, log in jobs]
        for f in futs:
            out = f.result()
            if verbose:
                print(out)
    objs = [obj for _, obj, _ in jobs]
    tmp = LIB + f".tmp{os.getpid()}"
    _run([nvcc, "-shared", *ARCH, "-o", tmp, *objs], os.path.join(BUILD, "link.log"))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
