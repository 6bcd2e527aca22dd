"""Compile the CUDA library (``libfa_gb300.so``) in-tree for sm_103a.

Each ``csrc/*.cu`` translation unit is compiled by its own nvcc process (in
parallel), then linked into one shared library next to this file. The CUDA
runtime is linked statically, so the library needs only the NVIDIA driver at
run time. The same sources are also built with ``-DFA_DEBUG`` into
``libfa_gb300_debug.so``: device-side index checks that report
FA_ERR_DEVICE_CHECK through the workspace status word (both libraries are
compiled at once, in parallel).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_NAME = "libfa_gb300.so"
LIB_PATH = os.path.join(PKG_DIR, LIB_NAME)
DEBUG_BUILD_DIR = os.path.join(PKG_DIR, "_build_debug")
DEBUG_LIB_PATH = os.path.join(PKG_DIR, "libfa_gb300_debug.so")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH_FLAGS + [
    "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O3",
    "-I", INCLUDE, "-I", CSRC,
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfa_gb300.so")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return files + [os.path.abspath(__file__)]


def up_to_date() -> bool:
    for lib in (LIB_PATH, DEBUG_LIB_PATH):
        if not os.path.exists(lib):
            return False
        t = os.path.getmtime(lib)
        if any(os.path.getmtime(f) > t for f in _deps()):
            return False
    return True


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    """Build both libraries if any source is newer than them; return the
    release library's path."""
    if not force and up_to_date():
        return LIB_PATH
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    variants = ((BUILD_DIR, LIB_PATH, []), (DEBUG_BUILD_DIR, DEBUG_LIB_PATH, ["-DFA_DEBUG"]))
    for d, _, _ in variants:
        os.makedirs(d, exist_ok=True)

    def compile_one(job):
        src, (d, _, flags) = job
        obj = os.path.join(d, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *NVCC_FLAGS, *flags, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src} {' '.join(flags)}:\n{r.stderr}")
        return obj, r.stderr

    srcs = _sources()
    jobs = [(src, v) for v in variants for src in srcs]
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        results = list(ex.map(compile_one, jobs))
    if verbose or ptxas_verbose:
        for _, err in results[:len(srcs)]:
            if err:
                print(err)
    for i, (_, lib, _) in enumerate(variants):
        objs = [o for o, _ in results[i * len(srcs):(i + 1) * len(srcs)]]
        tmp = lib + ".tmp"
        cmd = [cc, *ARCH_FLAGS, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB_PATH


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv))
