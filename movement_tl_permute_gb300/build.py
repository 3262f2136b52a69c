"""Builds libtl_permute.so in-tree: nvcc for sm_103a, one object per source, in parallel.

Usage: ``python -m movement_tl_permute_gb300.build [--force] [--verbose]``.
The library links the CUDA runtime statically and resolves the driver's tensor-map
encoder at run time, so it needs no libcuda at link time and loads on CPU-only
hosts (its host-only entry points work there).
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libtl_permute.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return path


def _sources():
    cu = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    cpp = sorted(glob.glob(os.path.join(CSRC, "*.cpp")))
    deps = (sorted(glob.glob(os.path.join(CSRC, "*.h"))) + sorted(glob.glob(os.path.join(CSRC, "*.cuh")))
            + sorted(glob.glob(os.path.join(INCLUDE, "*.h")))
            + sorted(glob.glob(os.path.join(INCLUDE, "*.cuh"))))
    return cu, cpp, deps


def _stale(cu, cpp, deps):
    if not os.path.exists(LIB):
        return True
    newest = max(os.path.getmtime(p) for p in cu + cpp + deps + [os.path.abspath(__file__)])
    return os.path.getmtime(LIB) < newest


def _compile(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    return cmd, r.returncode, r.stdout


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    cu, cpp, deps = _sources()
    if not force and not _stale(cu, cpp, deps):
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    common = ["-O3", "-std=c++17", "-I", INCLUDE, "-I", CSRC, "-Xcompiler", "-fvisibility=hidden"]
    jobs = []
    objs = []
    for src in cu:
        obj = os.path.join(BUILD_DIR, os.path.basename(src) + ".o")
        cmd = [nvcc] + ARCH + common + ["-lineinfo", "-Xcompiler", "-fPIC", "-c", src, "-o", obj]
        if ptxas_info:
            cmd += ["-Xptxas", "-v"]
        jobs.append(cmd)
        objs.append(obj)
    for src in cpp:
        obj = os.path.join(BUILD_DIR, os.path.basename(src) + ".o")
        jobs.append([nvcc] + common + ["-Xcompiler", "-fPIC", "-x", "c++", "-c", src, "-o", obj])
        objs.append(obj)
    workers = max(1, min(len(jobs), os.cpu_count() or 4))
    with cf.ThreadPoolExecutor(workers) as ex:
        results = list(ex.map(_compile, jobs))
    failed = [(c, out) for c, rc, out in results if rc != 0]
    for c, rc, out in results:
        if verbose or ptxas_info or rc != 0:
            sys.stderr.write(" ".join(os.path.basename(x) for x in c[-3:]) + "\n" + out)
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(c[-3] for c, _ in failed))
    tmp = LIB + ".tmp%d" % os.getpid()
    link = [nvcc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout)
    os.replace(tmp, LIB)
    return LIB


def kernel_resources() -> list:
    """Spill bytes of every kernel and device function, as ptxas reports them (-v) for each
    CUDA source compiled on its own into a scratch directory (the library is not touched):
    a list of {"name", "spill_stores", "spill_loads"}."""
    import re
    import tempfile
    cu, _, _ = _sources()
    nvcc = _nvcc()
    common = ["-O3", "-std=c++17", "-I", INCLUDE, "-I", CSRC, "-Xptxas", "-v"]
    with tempfile.TemporaryDirectory() as tmp:
        jobs = [[nvcc] + ARCH + common + ["-c", src, "-o", os.path.join(tmp, os.path.basename(src) + ".o")]
                for src in cu]
        with cf.ThreadPoolExecutor(max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
            results = list(ex.map(_compile, jobs))
    out, name = [], None
    for c, rc, text in results:
        if rc != 0:
            raise RuntimeError("nvcc failed for " + c[-3] + ":\n" + text)
        for line in text.splitlines():
            m = re.search(r"Function properties for (\S+)", line)
            if m:
                name = m.group(1)
                continue
            m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
            if m and name:
                out.append({"name": name, "spill_stores": int(m.group(1)),
                            "spill_loads": int(m.group(2))})
                name = None
    return out


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true")
    args = ap.parse_args(argv)
    print(build(force=args.force, verbose=args.verbose, ptxas_info=args.ptxas_info))


if __name__ == "__main__":
    main()
