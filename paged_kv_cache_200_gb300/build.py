"""Build ``libpkv.so`` in-tree with nvcc for sm_103a (no cmake, no torch extension).

``build()`` compiles each translation unit under ``csrc/`` in parallel into
``_build/`` and links the shared library next to this file.  It is a no-op
when the library is newer than every source and header.
"""

from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libpkv.so")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH_FLAGS + [
    "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC,
]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpkv")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _newest_input() -> float:
    files = sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]
    return max(os.path.getmtime(f) for f in files)


TEST_BUILD_DIR = os.path.join(BUILD_DIR, "test")
TEST_LIB_PATH = os.path.join(TEST_BUILD_DIR, "libpkv_test.so")
# Test-only variant: every bounded wait inside a kernel gives up after 1 ms
# instead of 2 s, and host-set hooks can withhold one TMA copy so that a wait
# runs out (the failure-detection tests).  Never the product library.
TEST_FLAGS = ["-DPKV_TEST_HOOKS", "-DPKV_TEST_WAIT_NS=1000000ull"]


def build_test_library(verbose: bool = False) -> str:
    """Compile the test-only variant of the library (see TEST_FLAGS); return its path."""
    return build(verbose=verbose, extra_flags=TEST_FLAGS, out_path=TEST_LIB_PATH, build_dir=TEST_BUILD_DIR)


def build(verbose: bool = False, force: bool = False, extra_flags=None, out_path: str = LIB_PATH,
          build_dir: str = BUILD_DIR) -> str:
    """Compile and link libpkv.so (or a variant at out_path); return its path."""
    if not force and os.path.exists(out_path) and os.path.getmtime(out_path) >= _newest_input():
        if not extra_flags or out_path != LIB_PATH:
            return out_path
    nvcc = _nvcc()
    os.makedirs(build_dir, exist_ok=True)
    flags = NVCC_FLAGS + list(extra_flags or [])

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src) + ".o")
        cmd = [nvcc] + flags + ["-c", src, "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
        if verbose and (res.stdout or res.stderr):
            print(res.stdout + res.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = out_path + ".tmp"
    cmd = [nvcc] + ARCH_FLAGS + ["-shared", "-o", tmp] + objs
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, out_path)
    return out_path


if __name__ == "__main__":
    print(build(verbose=True, force=True))
