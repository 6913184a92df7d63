"""Build ``libpagedkv.so`` in-tree: nvcc for sm_103a, translation units in parallel.

Usage: ``python -m paged_kv_cache_145_gb300.build [--force] [--verbose]``.
Objects go to ``paged_kv_cache_145_gb300/_build/``; the library is written
next to this file.  No CMake; one ``-gencode`` (sm_103a only).
"""

import argparse
import concurrent.futures
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libpagedkv.so")

CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "--expt-relaxed-constexpr", "-I" + INCLUDE]
CXX_FLAGS = ["-O2", "-fPIC", "-std=c++17", "-Wall", "-I" + INCLUDE,
             "-I" + os.path.join(CUDA_HOME, "include")]


def _tool(name):
    cand = os.path.join(CUDA_HOME, "bin", name)
    return cand if os.path.exists(cand) else (shutil.which(name) or name)


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src, verbose):
    obj = os.path.join(BUILD_DIR, os.path.basename(src) + ".o")
    if src.endswith(".cu"):
        cmd = [_tool("nvcc")] + NVCC_FLAGS + (["-Xptxas", "-v"] if verbose else []) + ["-c", src, "-o", obj]
    else:
        cmd = [os.environ.get("CXX", "g++")] + CXX_FLAGS + ["-c", src, "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("compile failed: %s\n%s%s" % (" ".join(cmd), res.stdout, res.stderr))
    return obj, res.stderr


def build(force=False, verbose=False):
    """Compile every CUDA/C++ source and link the shared library; returns its path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    headers = _headers()
    srcs = _sources()
    todo = [s for s in srcs
            if force or _stale(os.path.join(BUILD_DIR, os.path.basename(s) + ".o"), [s] + headers)]
    logs = []
    if todo:
        with concurrent.futures.ThreadPoolExecutor(max_workers=len(todo)) as pool:
            for obj, log in pool.map(lambda s: _compile(s, verbose), todo):
                logs.append(log)
    objs = [os.path.join(BUILD_DIR, os.path.basename(s) + ".o") for s in srcs]
    if force or todo or _stale(LIB_PATH, objs):
        cmd = [_tool("nvcc")] + ARCH + ["-shared", "-o", LIB_PATH] + objs
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("link failed: %s\n%s%s" % (" ".join(cmd), res.stdout, res.stderr))
    if verbose:
        sys.stderr.write("".join(logs))
    return LIB_PATH


if __name__ == "__main__":
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true", help="print ptxas resource usage")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose))
