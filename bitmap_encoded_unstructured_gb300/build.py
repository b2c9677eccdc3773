"""Build libbsp.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

Each .cu file is compiled to an object in parallel, then linked into
``bitmap_encoded_unstructured_gb300/libbsp.so``.  The test library
``libbsp_test.so`` links the same objects except the tuning unit, which is
compiled a second time with BSP_TESTING defined: only that build exports the
switches of ``include/bsp_testing.h`` (stalled copies, a short spin cap) that
the timeout tests use.  Run as a module or call ``build_library()``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
ROOT = os.path.dirname(PKG)
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libbsp.so")
TEST_LIB = os.path.join(PKG, "libbsp_test.so")
TESTING_UNIT = "bsp_tuning.cu"  # the only source compiled differently for the test library

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    files = sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return files


def _up_to_date() -> bool:
    if not (os.path.exists(LIB) and os.path.exists(TEST_LIB)):
        return False
    t = min(os.path.getmtime(LIB), os.path.getmtime(TEST_LIB))
    return all(os.path.getmtime(f) <= t for f in _deps())


def build_library(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    if not force and not extra_flags and _up_to_date():
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    objs = []
    cmds = []
    test_objs = []
    for src in sources():
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmds.append([nvcc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj])
        if os.path.basename(src) == TESTING_UNIT:
            tobj = os.path.join(BUILD, os.path.basename(src)[:-3] + "_testing.o")
            cmds.append([nvcc, *ARCH, *NVCC_FLAGS, *extra_flags, "-DBSP_TESTING=1", "-c", src, "-o", tobj])
            test_objs.append(tobj)
        else:
            test_objs.append(obj)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode:
            raise RuntimeError(f"nvcc failed on {cmd[-3]}")
        return r

    with cf.ThreadPoolExecutor(max_workers=min(8, len(cmds))) as ex:
        list(ex.map(run, cmds))
    for target, parts in ((LIB, objs), (TEST_LIB, test_objs)):
        tmp = target + f".tmp{os.getpid()}"
        run([nvcc, *ARCH, "-shared", "-o", tmp, *parts])
        os.replace(tmp, target)
    return LIB


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose="-v" in sys.argv))
