"""Compile the CUDA sources of this package into libra.so, in-tree, for sm_103a.

Each translation unit is compiled in parallel with nvcc, then linked into one
shared library next to this file.  Objects go to ``_build/`` (not versioned).
The debug build, libra_debug.so, is the same library compiled with RA_DEBUG_BOUNDS:
the kernels check their tensor-memory, shared-memory and global indices and report
a failed check through the status word (RA_ERR_BOUNDS) instead of faulting.
"""

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OBJDIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libra.so")
LIB_DEBUG = os.path.join(HERE, "libra_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def _nvcc():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _build(variants, verbose=False, ptxas_info=False):
    """Compile and link each variant (debug flag -> library path); one pool for all objects."""
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(job):
        debug, src = job
        objdir = os.path.join(OBJDIR, "debug" if debug else "release")
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        defs = ["-DRA_DEBUG_BOUNDS"] if debug else []
        cmd = [nvcc, *ARCH, *FLAGS, *defs, *extra, "-c", src, "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}{' (debug)' if debug else ''}:\n{res.stderr}")
        return debug, obj, res.stderr

    jobs = [(debug, src) for debug in variants for src in sources()]
    for debug in variants:
        os.makedirs(os.path.join(OBJDIR, "debug" if debug else "release"), exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 2)) as ex:
        results = list(ex.map(compile_one, jobs))
    if verbose or ptxas_info:
        for _, _, log in results:
            if log.strip():
                print(log)
    out = []
    for debug in variants:
        lib = LIB_DEBUG if debug else LIB
        tmp = lib + ".tmp"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *[o for d, o, _ in results if d == debug]]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stderr}")
        os.replace(tmp, lib)
        out.append(lib)
    return out


def build(verbose=False, ptxas_info=False, debug=False):
    """Build libra.so (libra_debug.so with debug=True); returns its path.  Raises
    RuntimeError on a compiler error."""
    return _build([debug], verbose, ptxas_info)[0]


def build_all(verbose=False):
    """Build libra.so and libra_debug.so together; returns both paths."""
    return tuple(_build([False, True], verbose))


if __name__ == "__main__":
    print(build_all(verbose=True))
