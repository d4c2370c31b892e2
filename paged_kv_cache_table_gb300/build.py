"""Build the C-ABI shared library ``libpa_gb300.so`` in-tree, for sm_103a only.

Each CUDA / C++ translation unit is compiled in parallel; the link uses nvcc with the static
CUDA runtime, so the library depends on nothing but the driver.  ``build()`` is idempotent:
it recompiles only when a source or header is newer than the library.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_PATH = os.path.join(PKG_DIR, "libpa_gb300.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-Wall"]


def _cuda_home() -> str:
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return cand
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(nvcc))
    raise RuntimeError("nvcc not found: set CUDA_HOME")


def sources():
    cu = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))
    cpp = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cpp"))
    return cu, cpp


def _headers():
    hs = [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    hs += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return hs


def _stale(target, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr, flush=True)
    return r


def build(verbose: bool = False, force: bool = False, ptxas_verbose: bool = False,
          defines=(), lib_path: str | None = None, build_dir: str | None = None) -> str:
    """Compile and link the library; returns its path.

    ``defines`` (e.g. ``("PA_PREFETCH_STAGES=2",)``) override compile-time tuning constants;
    use them together with a separate ``lib_path`` and ``build_dir``.
    """
    lib_out = lib_path or LIB_PATH
    bdir = build_dir or BUILD_DIR
    dflags = [f"-D{d}" for d in defines]
    cuda = _cuda_home()
    nvcc = os.path.join(cuda, "bin", "nvcc")
    cxx = os.environ.get("CXX", "g++")
    cu, cpp = sources()
    headers = _headers()
    os.makedirs(bdir, exist_ok=True)
    jobs = []
    objs = []
    for src in cu:
        obj = os.path.join(bdir, os.path.basename(src) + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + headers):
            cmd = [nvcc, *ARCH, *NVCC_FLAGS, *dflags, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
            if ptxas_verbose:
                cmd += ["-Xptxas", "-v"]
            jobs.append(cmd)
    for src in cpp:
        obj = os.path.join(bdir, os.path.basename(src) + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + headers):
            jobs.append([cxx, *CXX_FLAGS, "-I", INCLUDE, "-I", CSRC, "-I", os.path.join(cuda, "include"),
                         "-c", src, "-o", obj])
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            results = list(ex.map(lambda c: _run(c, verbose or ptxas_verbose), jobs))
        del results
    if force or jobs or _stale(lib_out, objs):
        tmp = lib_out + ".tmp"
        _run([nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs], verbose)
        os.replace(tmp, lib_out)
    return lib_out


if __name__ == "__main__":
    force = "--force" in sys.argv
    print(build(verbose=True, force=force, ptxas_verbose="--ptxas" in sys.argv))
