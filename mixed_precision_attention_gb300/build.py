"""Builds libapa.so in-tree (mixed_precision_attention_gb300/_lib/) with nvcc for sm_103a.

Each translation unit is compiled in parallel, then linked into one shared
library with the CUDA runtime linked statically.  Rebuilds only when a source
is newer than the library.
"""
from __future__ import annotations

import glob
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIBDIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIBDIR, "libapa.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr", "-I", INCLUDE]


def _nvcc():
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.isabs(c) and os.path.exists(c) or not os.path.isabs(c)):
            return c
    return "nvcc"


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in _deps())


# The test-hook variant (tests only, never loaded by the package): the same sources
# with APA_TEST_HOOKS, which exports a switch that makes pass 1's wait for the
# in-launch quantizer run out, and a short wait limit (~0.5 s at 2 GHz).
TEST_HOOKS_LIB = os.path.join(LIBDIR, "libapa_testhooks.so")
TEST_HOOKS_FLAGS = ["-DAPA_TEST_HOOKS", "-DAPA_WAIT_LIMIT_CYCLES=1000000000ull"]


def build_test_hooks(force: bool = False) -> str:
    """Builds the test-hook variant of the library (for the timeout test)."""
    if not force and os.path.exists(TEST_HOOKS_LIB) and \
            all(os.path.getmtime(p) <= os.path.getmtime(TEST_HOOKS_LIB) for p in _deps()):
        return TEST_HOOKS_LIB
    return _build(TEST_HOOKS_LIB, os.path.join(LIBDIR, "testhooks"), TEST_HOOKS_FLAGS)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not needs_build():
        return LIB
    return _build(LIB, LIBDIR, [], verbose)


def _build(lib: str, objdir: str, extra: list, verbose: bool = False) -> str:
    os.makedirs(objdir, exist_ok=True)
    nvcc = _nvcc()
    objs = []

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
        if verbose:
            cmd += ["-Xptxas", "-v"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=len(sources())) as ex:
        for obj, log in ex.map(compile_one, sources()):
            objs.append(obj)
            if verbose and log:
                print(log)
    tmp = lib + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
