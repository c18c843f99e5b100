"""In-tree build of libnvfp4kv.so (sm_103a only).

Each CUDA / C++ translation unit compiles in its own process (in parallel),
then nvcc links the shared library.  Outputs go to ``_build/`` beside this
file.  ``python -m nvfp4_paged_kv_nvfp4kv_gb300.build`` builds from the
command line.
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
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libnvfp4kv.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _cuda_home() -> str:
    home = os.environ.get("CUDA_HOME") or "/usr/local/cuda"
    if not os.path.exists(os.path.join(home, "bin", "nvcc")):
        nvcc = shutil.which("nvcc")
        if nvcc:
            home = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return home


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) +
                  glob.glob(os.path.join(CSRC, "*.cpp")))


def _deps():
    return sources() + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(INCLUDE, "nvfp4kv.h"),
                                                  os.path.abspath(__file__)]


def _compile(src: str, cuda: str, verbose: bool, build_dir: str = BUILD,
             defines=()) -> str:
    obj = os.path.join(build_dir, os.path.basename(src) + ".o")
    inc = ["-I", INCLUDE, "-I", CSRC, "-I", os.path.join(cuda, "include")]
    if src.endswith(".cu"):
        cmd = [os.path.join(cuda, "bin", "nvcc"), *ARCH, "-lineinfo", "-O3",
               "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
               *["-D" + d for d in defines], *inc, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
    else:
        cmd = [os.environ.get("CXX", "g++"), "-O2", "-std=c++17", "-fPIC", "-Wall",
               *inc, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("compile failed: %s\n%s%s" % (" ".join(cmd), r.stdout, r.stderr))
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False, defines=(), out: str = None) -> str:
    """Compile and link the library if any source is newer than it.

    ``defines`` adds -D flags to the CUDA sources (the kernels' launch-shape
    defaults can be overridden that way) and ``out`` builds into another
    path instead of the package's own library."""
    lib = out or LIB
    build_dir = os.path.dirname(lib)
    if not force and os.path.exists(lib):
        t = os.path.getmtime(lib)
        if all(os.path.getmtime(d) <= t for d in _deps()):
            return lib
    cuda = _cuda_home()
    os.makedirs(build_dir, exist_ok=True)
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(s, cuda, verbose, build_dir, defines), srcs))
    tmp = lib + ".tmp%d" % os.getpid()
    cmd = [os.path.join(cuda, "bin", "nvcc"), *ARCH, "-shared", "-o", tmp, *objs,
           "-cudart=static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed: %s\n%s%s" % (" ".join(cmd), r.stdout, r.stderr))
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
