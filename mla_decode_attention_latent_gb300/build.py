"""Build the in-tree CUDA library ``libmla_decode_gb300.so`` for sm_103a.

Each ``csrc/*.cu`` is compiled in parallel with nvcc into ``_build/`` and the
objects are linked into one shared library next to this file.  The library
exports only the ``extern "C"`` calls of ``include/mla_decode.h``.

    python -m mla_decode_attention_latent_gb300.build [--force]
"""
from __future__ import annotations

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
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_NAME = "libmla_decode_gb300.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-Xptxas", "-v"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the MLA decode library")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                  glob.glob(os.path.join(INCLUDE, "*.h")))


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src, obj, log):
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    with open(log, "w") as f:
        f.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr[-4000:]}")
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every CUDA source for sm_103a and link the shared library. Returns its path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    srcs = _sources()
    headers = _headers()
    objs = []
    jobs = []
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        for src in srcs:
            stem = os.path.splitext(os.path.basename(src))[0]
            obj = os.path.join(BUILD_DIR, stem + ".o")
            objs.append(obj)
            if force or _stale(obj, [src, *headers]):
                jobs.append(ex.submit(_compile, src, obj, os.path.join(BUILD_DIR, stem + ".log")))
        for j in jobs:
            j.result()
    if force or _stale(LIB_PATH, objs):
        tmp = LIB_PATH + ".tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", *objs, "-o", tmp]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
        os.replace(tmp, LIB_PATH)
    if verbose:
        for src in srcs:
            stem = os.path.splitext(os.path.basename(src))[0]
            log = os.path.join(BUILD_DIR, stem + ".log")
            if os.path.exists(log):
                sys.stdout.write(open(log).read())
    return LIB_PATH


# test-only library: the same objects, but the bf16 d = 576 split kernel built
# with a 1 ms wait limit and part 0 skipping one chunk load, so that a bounded
# wait runs out on purpose (never the product library)
TIMEOUT_TEST_LIB = os.path.join(BUILD_DIR, "libmla_decode_gb300_timeout_test.so")
TIMEOUT_TEST_DEFINES = ["-DMLA_WAIT_LIMIT_NS=1000000ull", "-DMLA_TEST_SKIP_ONE_LOAD"]


def build_timeout_test_lib(force: bool = False) -> str:
    """Build the test-only library for the bounded-wait timeout test; returns its path."""
    build()
    src = os.path.join(CSRC, "mla_split_tc.cu")
    obj = os.path.join(BUILD_DIR, "mla_split_tc_timeout_test.o")
    if force or _stale(obj, [src, *_headers()]):
        cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *TIMEOUT_TEST_DEFINES, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on the timeout test object:\n{r.stderr[-4000:]}")
    objs = [os.path.join(BUILD_DIR, os.path.splitext(os.path.basename(x))[0] + ".o") for x in _sources()
            if os.path.basename(x) != "mla_split_tc.cu"] + [obj]
    if force or _stale(TIMEOUT_TEST_LIB, objs):
        cmd = [nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", *objs, "-o", TIMEOUT_TEST_LIB]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
    return TIMEOUT_TEST_LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
