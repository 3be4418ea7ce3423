"""In-tree build of ``libtpk.so`` (planner + C ABI + sm_103a kernels).

Compiles every ``csrc/*.cpp`` and ``csrc/*.cu`` with nvcc for
``-gencode arch=compute_103a,code=sm_103a`` in parallel and links one shared
library with the CUDA runtime linked statically, so the library has no
link-time dependency on libcuda (the driver entry point for tensor-map
encoding is looked up at run time).  A stamp file records the sources' hash,
the flags and the machine architecture; an up-to-date library is not rebuilt.
"""
import concurrent.futures
import hashlib
import os
import platform
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libtpk.so")
STAMP = LIB + ".stamp"

GENCODE = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def _nvcc():
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the tpk library needs the CUDA 13 toolkit to build")
    return cand


def _sources():
    files = sorted(f for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))
    return [os.path.join(CSRC, f) for f in files]


def _headers():
    files = sorted(f for f in os.listdir(CSRC) if f.endswith((".h", ".cuh")))
    return [os.path.join(CSRC, f) for f in files] + [os.path.join(INCLUDE, "tpk.h")]


def _stamp(extra):
    h = hashlib.sha256()
    for p in _sources() + _headers():
        h.update(p.encode())
        with open(p, "rb") as f:
            h.update(f.read())
    h.update(" ".join(GENCODE + COMMON + extra).encode())
    h.update(platform.machine().encode())
    return h.hexdigest()


def build_library(quiet=False, force=False, verbose_ptxas=False, jobs=None):
    """Build (if needed) and return the path of libtpk.so."""
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    stamp = _stamp(extra)
    if not force and os.path.exists(LIB) and os.path.exists(STAMP):
        with open(STAMP) as f:
            if f.read().strip() == stamp:
                return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        cmd = [nvcc] + GENCODE + COMMON + extra + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("compile failed: %s\n%s%s" % (" ".join(cmd), r.stdout, r.stderr))
        return obj, r.stdout + r.stderr

    srcs = _sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=jobs or min(8, len(srcs))) as ex:
        results = list(ex.map(compile_one, srcs))
    if not quiet or verbose_ptxas:
        for _, log in results:
            if log.strip():
                sys.stderr.write(log)
    tmp = LIB + ".tmp"
    cmd = [nvcc] + GENCODE + ["-shared", "-cudart", "static", "-o", tmp] + [o for o, _ in results] + ["-lrt", "-ldl", "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed: %s\n%s%s" % (" ".join(cmd), r.stdout, r.stderr))
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(stamp)
    return LIB


if __name__ == "__main__":
    print(build_library(quiet=False, force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
