"""Build libaq.so in-tree with nvcc for sm_103a.

Each .cu file is compiled in parallel, then linked into
quantized_matmul_affine_gb300/_build/libaq.so (the CUDA runtime is linked
statically, so the library loads on machines without a GPU driver; kernels
need one to run).  Usage: ``python -m quantized_matmul_affine_gb300.build``.

The same sources are also built, in the same pool, into
_build/test/libaq_test.so with AQ_TEST_HOOKS defined and the pipeline wait
limit cut to 1 ms: a test-only library in which a producer can be told to
withhold the copies of its first stage (aq_test_withhold), so that a test
can watch a bounded wait give up.  The package never loads it.
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libaq.so")
TEST_BUILD = os.path.join(BUILD, "test")
TEST_LIB = os.path.join(TEST_BUILD, "libaq_test.so")
TEST_FLAGS = ["-DAQ_TEST_HOOKS=1", "-DAQ_WAIT_LIMIT_NS=1000000ull"]
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "--expt-relaxed-constexpr", "-I", INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=None) -> str:
    """Build libaq.so (and the test-only libaq_test.so) unless up to date."""
    targets = [(LIB, BUILD, [])]
    if extra_flags is None:
        targets.append((TEST_LIB, TEST_BUILD, TEST_FLAGS))
    targets = [t for t in targets if force or not up_to_date(t[0])]
    if not targets:
        return LIB
    cc = nvcc()
    jobs, links = [], []
    for lib, out_dir, defs in targets:
        os.makedirs(out_dir, exist_ok=True)
        flags = NVCC_FLAGS + defs + list(extra_flags or [])
        objs = []
        for src in _sources():
            obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
            objs.append(obj)
            jobs.append([cc] + flags + ["-c", src, "-o", obj])
        links.append((lib, objs))

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with concurrent.futures.ThreadPoolExecutor(max_workers=max(4, os.cpu_count() or 4)) as ex:
        for cmd, r in ex.map(run, jobs):
            if verbose or r.returncode != 0:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError("nvcc failed: " + " ".join(cmd))
    for lib, objs in links:
        tmp = lib + f".tmp{os.getpid()}"
        link = [cc] + ARCH + ["-shared", "-Xcompiler", "-fPIC", "-o", tmp] + objs
        r = subprocess.run(link, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("link failed")
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra_flags=["-Xptxas", "-v"] if "--ptxas" in sys.argv else None))
