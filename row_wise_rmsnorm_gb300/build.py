"""Compile the CUDA library (libmt_norm.so) in-tree for sm_103a.

    python -m row_wise_rmsnorm_gb300.build [--force] [--verbose]

Each translation unit under csrc/ is compiled in parallel with nvcc
(``-gencode arch=compute_103a,code=sm_103a -lineinfo -O3``, never fast-math), then
linked into ``_build/libmt_norm.so`` with the CUDA runtime linked statically.
ptxas register/spill reports go to ``_build/ptxas.log``.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libmt_norm.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "-Xptxas", "-v", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmt_norm.so")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers() -> list[str]:
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return hs


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Build libmt_norm.so if any source is newer; return its path."""
    nvcc = _nvcc()
    objdir = os.path.join(BUILD, "obj")
    os.makedirs(objdir, exist_ok=True)
    srcs = sources()
    hdrs = _headers()
    objs = [os.path.join(objdir, os.path.basename(s)[:-3] + ".o") for s in srcs]

    def compile_one(src_obj):
        src, obj = src_obj
        if not force and not _stale(obj, [src] + hdrs + [__file__]):
            return obj, ""
        cmd = [nvcc, *NVCC_FLAGS, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stderr}")
        return obj, r.stderr

    logs = []
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        for obj, log in ex.map(compile_one, zip(srcs, objs)):
            if log:
                logs.append(f"== {os.path.basename(obj)}\n{log}")
    if logs:
        with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
            f.write("\n".join(logs))
        if verbose:
            print("\n".join(logs))
    if force or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


HOOKS_LIB = os.path.join(BUILD, "libmt_norm_hooks.so")
HOOKS_SOURCE = os.path.join(CSRC, "api.cu")


def build_test_hooks() -> str:
    """Build the test-only variant libmt_norm_hooks.so: the library with api.cu compiled
    with -DMT_TEST_HOOKS (host-side launch-failure injection, mt_test_*), every other
    object shared with libmt_norm.so. The product library never contains the hooks."""
    build()
    nvcc = _nvcc()
    objdir = os.path.join(BUILD, "obj")
    hookdir = os.path.join(BUILD, "hooks")
    os.makedirs(hookdir, exist_ok=True)
    hobj = os.path.join(hookdir, "api.o")
    if _stale(hobj, [HOOKS_SOURCE] + _headers() + [__file__]):
        cmd = [nvcc, *NVCC_FLAGS, "-DMT_TEST_HOOKS", "-c", HOOKS_SOURCE, "-o", hobj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for the test-hook api.cu:\n{r.stderr}")
    objs = [hobj] + [os.path.join(objdir, os.path.basename(s)[:-3] + ".o") for s in sources()
                     if os.path.basename(s) != "api.cu"]
    if _stale(HOOKS_LIB, objs):
        tmp = HOOKS_LIB + f".tmp{os.getpid()}"
        r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True,
                           text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(tmp, HOOKS_LIB)
    return HOOKS_LIB


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    args = ap.parse_args(argv)
    print(build(force=args.force, verbose=args.verbose))


if __name__ == "__main__":
    sys.exit(main())
