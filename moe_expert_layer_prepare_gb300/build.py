"""Build the CUDA library ``libmoe_prep.so`` in-tree (sm_103a only).

Each ``csrc/*.cu`` is compiled in parallel with nvcc, then linked into one
shared library next to this file.  No cmake, no PyTorch extension machinery.
"""
from __future__ import annotations

import os
import platform
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build", platform.machine())
LIB_NAME = "libmoe_prep.so"
LIB_PATH = os.path.join(HERE, LIB_NAME)

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         f"-I{INCLUDE}", f"-I{CSRC}", "--expt-relaxed-constexpr"]


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers_mtime():
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    paths.append(os.path.join(INCLUDE, "moe_prep.h"))
    return max(os.path.getmtime(p) for p in paths)


def _compile(src, verbose_ptxas=False, build_dir=BUILD_DIR, defines=()):
    obj = os.path.join(build_dir, os.path.basename(src) + ".o")
    dep = max(os.path.getmtime(src), _headers_mtime())
    if os.path.exists(obj) and os.path.getmtime(obj) >= dep and not verbose_ptxas:
        return obj, ""
    cmd = [NVCC, *ARCH, *FLAGS, *[f"-D{d}" for d in defines], "-c", src, "-o", obj]
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    os.makedirs(BUILD_DIR, exist_ok=True)
    if force:
        for f in os.listdir(BUILD_DIR):
            if os.path.isfile(os.path.join(BUILD_DIR, f)):
                os.remove(os.path.join(BUILD_DIR, f))
    srcs = sources()
    with ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose_ptxas), srcs))
    objs = [o for o, _ in results]
    if verbose_ptxas:
        for (_, log), s in zip(results, srcs):
            sys.stderr.write(f"== {os.path.basename(s)}\n{log}")
    newest = max(os.path.getmtime(o) for o in objs)
    if force or not os.path.exists(LIB_PATH) or os.path.getmtime(LIB_PATH) < newest:
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        cmd = [NVCC, *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


# Test-only builds of the library with compile-time knobs (for example the
# failure-detection test's shortened wait limit and withheld pipeline stage).
# They go to their own folder and file name; build() above never uses them.
TEST_VARIANTS = {
    "timeout": ("MOE_WAIT_LIMIT_NS=5000000ull", "MOE_TEST_WITHHOLD_STAGE"),
}


def build_test_variant(name: str) -> str:
    defines = TEST_VARIANTS[name]
    bdir = os.path.join(BUILD_DIR, "test_" + name)
    os.makedirs(bdir, exist_ok=True)
    srcs = sources()
    with ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = [o for o, _ in ex.map(lambda s: _compile(s, False, bdir, defines), srcs)]
    lib = os.path.join(bdir, f"libmoe_prep_test_{name}.so")
    newest = max(os.path.getmtime(o) for o in objs)
    if not os.path.exists(lib) or os.path.getmtime(lib) < newest:
        tmp = lib + f".tmp{os.getpid()}"
        r = subprocess.run([NVCC, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True,
                           text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
