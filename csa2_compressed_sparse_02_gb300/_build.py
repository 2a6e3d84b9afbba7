"""Builds the in-tree native libraries (no cmake, no setuptools):

* ``libcsa2.so``      — the CSA2 kernels and their C ABI (``include/csa2.h``), sm_103a;
* ``libcsa2synth.so`` — the GPU twin of the seeded input generator (``synth.py``).

Each translation unit compiles in its own nvcc process, in parallel, then one
link. A unit is recompiled only when it or a header is newer than its object.
"""
from __future__ import annotations

import glob
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libcsa2.so")
SYNTH_LIB = os.path.join(PKG, "libcsa2synth.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                "-I" + os.path.join(ROOT, "include")]


def _newer(src_paths, out):
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(p) > t for p in src_paths)


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("build failed: %s\n%s%s" % (" ".join(cmd), r.stdout, r.stderr))
    return r.stdout + r.stderr


def build(verbose: bool = False, ptxas_info: bool = False) -> list[str]:
    os.makedirs(OBJ, exist_ok=True)
    headers = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(ROOT, "include", "*.h"))
    units = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    jobs = []
    for u in units:
        o = os.path.join(OBJ, os.path.basename(u)[:-3] + ".o")
        if ptxas_info or _newer([u] + headers, o):
            jobs.append(FLAGS + extra + ["-c", u, "-o", o])
    synth_src = os.path.join(CSRC, "synth", "synth.cu")
    synth_job = None
    if _newer([synth_src], SYNTH_LIB):
        synth_job = FLAGS + ["-shared", synth_src, "-o", SYNTH_LIB + ".tmp"]
    logs = []
    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        futs = [ex.submit(_run, [NVCC] + j) for j in jobs]
        if synth_job:
            futs.append(ex.submit(_run, [NVCC] + synth_job))
        for f in futs:
            logs.append(f.result())
    if synth_job:
        os.replace(SYNTH_LIB + ".tmp", SYNTH_LIB)
    objs = [os.path.join(OBJ, os.path.basename(u)[:-3] + ".o") for u in units]
    if jobs or _newer(objs, LIB):
        _run([NVCC] + ARCH + ["-shared", "-o", LIB + ".tmp"] + objs)
        os.replace(LIB + ".tmp", LIB)
    if verbose:
        for line in logs:
            if line.strip():
                print(line)
    return logs
