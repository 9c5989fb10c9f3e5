"""Compile the CUDA library ``librelattn.so`` (sm_103a) in-tree.

Each ``csrc/*.cu`` translation unit is compiled in parallel with nvcc, then
linked into a shared library next to this file.  No CMake, no torch extension
machinery: the library exposes only the C ABI in ``include/relattn.h``.

A second library, ``librelattn_test.so``, links the same kernel objects with
``api.cu`` compiled once more under ``RELATTN_TEST_HOOKS``: it adds the
``relattn_test_*`` entry points the failure-path tests use.  The product
library has no test hooks.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "librelattn.so")
TEST_LIB = os.path.join(HERE, "librelattn_test.so")
TEST_DEFINE = "-DRELATTN_TEST_HOOKS"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the relative-attention library cannot be built")


def _flags(extra=()):
    return [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
            f"-I{os.path.join(ROOT, 'include')}", "--expt-relaxed-constexpr", *extra]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(CSRC, "*.h")) + [os.path.join(ROOT, "include", "relattn.h")]


def up_to_date() -> bool:
    if not (os.path.exists(LIB) and os.path.exists(TEST_LIB)):
        return False
    t = min(os.path.getmtime(LIB), os.path.getmtime(TEST_LIB))
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    srcs = _sources()

    def compile_one(job):
        src, test = job
        obj = os.path.join(BUILD, os.path.basename(src) + (".test.o" if test else ".o"))
        cmd = [cc, *_flags(extra_flags), *([TEST_DEFINE] if test else []), "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    api = os.path.join(CSRC, "api.cu")
    jobs = [(s_, False) for s_ in srcs] + [(api, True)]
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(compile_one, jobs))
    prod = objs[:len(srcs)]
    test = [o for o, s_ in zip(prod, srcs) if s_ != api] + [objs[-1]]
    for out, group in ((LIB, prod), (TEST_LIB, test)):
        tmp = out + f".tmp{os.getpid()}"
        cmd = [cc, *ARCH, "-shared", "-o", tmp, *group, "-lcudart"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, out)
    return LIB


if __name__ == "__main__":
    v = "-v" in sys.argv
    print(build(force=True, verbose=v, extra_flags=["-Xptxas", "-v"] if v else ()))
