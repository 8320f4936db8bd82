"""Build the L³ CUDA library in-tree: ``static_token_routed_csr_b300/libl3.so`` (sm_103a).

Usage: ``python -m static_token_routed_csr_b300.build [--force] [--debug]``. Every ``.cu``
under ``csrc/`` is compiled by nvcc for ``sm_103a`` only, every ``.cpp`` by g++ (with
``-ffp-contract=off`` so host arithmetic is not fused), and the objects are linked into
one shared library against the CUDA runtime and cuBLASLt (the backward's plain GEMMs). Objects are rebuilt when a source or header
is newer than them.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libl3.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _cuda_home() -> str:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if home and os.path.isdir(home):
        return home
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def _headers():
    return glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale(obj: str, src: str, newest_header: float) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return os.path.getmtime(src) > t or newest_header > t


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("build failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def build(force: bool = False, debug: bool = False, verbose: bool = False) -> str:
    cuda = _cuda_home()
    nvcc = os.path.join(cuda, "bin", "nvcc")
    os.makedirs(BUILD, exist_ok=True)
    headers = _headers()
    newest = max([os.path.getmtime(h) for h in headers] + [0.0])
    opt = ["-O0", "-G"] if debug else ["-O3", "-lineinfo"]
    jobs = []
    objs = []
    for src in sorted(glob.glob(os.path.join(CSRC, "*.cu"))):
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        objs.append(obj)
        if force or _stale(obj, src, newest):
            jobs.append([nvcc, *ARCH, *opt, "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
                         "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj])
    for src in sorted(glob.glob(os.path.join(CSRC, "*.cpp"))):
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        objs.append(obj)
        if force or _stale(obj, src, newest):
            jobs.append(["g++", "-O2", "-fPIC", "-std=c++17", "-ffp-contract=off", "-Wall",
                         "-I", INCLUDE, "-I", os.path.join(cuda, "include"), "-c", src, "-o", obj])
    logs = []
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
            logs = list(ex.map(_run, jobs))
    if jobs or not os.path.exists(LIB) or force:
        libdir = os.path.join(cuda, "lib64")
        _run([nvcc, *ARCH, "-shared", "-o", LIB, *objs, "-L", libdir, "-lcudart", "-lcublasLt",
              "-Xlinker", "-rpath", "-Xlinker", libdir])
    if verbose:
        for lg in logs:
            sys.stdout.write(lg)
    return LIB


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--debug", action="store_true")
    ap.add_argument("-v", "--verbose", action="store_true")
    a = ap.parse_args(argv)
    print(build(force=a.force, debug=a.debug, verbose=a.verbose))


if __name__ == "__main__":
    main()
