"""Build libtwell.so in-tree with nvcc for sm_103a (GB300).

Each translation unit compiles in parallel to an object under ``_build/``, then
nvcc links the shared library next to this file.  Rebuilds only when a source
or header is newer than the library.

Besides the product library, two variants of the same sources serve the tests
and the benchmark only (they are never loaded by the Python binding's
entry points):

* ``libtwell_hooks.so`` -- adds two measurement hooks (``TWELL_TEST_HOOKS``):
  the tensor-core GEMM engine with a plain fp32 epilogue, and the random-row
  gather probe that the benchmark reads the gather kernels against.
* ``libtwell_timeout.so`` -- the pipeline waits of the tensor-core kernels
  limited to 1 ns, so that every wait that is not satisfied at once runs out
  on a sane input and the timeout path (status, drain, exit) can be tested
  without a fault.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(PKG, "_build")

SOURCES = ["twell_abi.cu", "pack.cu", "simt_gemm.cu", "updown.cu", "tc_gemm.cu", "backward.cu",
           "rowell.cu", "static_split.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]

# variant -> (library file, extra sources, extra nvcc flags)
VARIANTS = {
    "": ("libtwell.so", [], []),
    "hooks": ("libtwell_hooks.so", ["probe.cu"], ["-DTWELL_TEST_HOOKS"]),
    "timeout": ("libtwell_timeout.so", [], ["-DTWELL_WAIT_LIMIT_NS=1ull"]),
}
LIB = os.path.join(PKG, VARIANTS[""][0])


def lib_path(variant: str = "") -> str:
    return os.path.join(PKG, VARIANTS[variant][0])


def nvcc_path() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtwell.so")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "twell.h"))
    files.append(os.path.abspath(__file__))
    return files


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _deps())


def _jobs(variant: str):
    name, extra_src, flags = VARIANTS[variant]
    objdir = os.path.join(OBJDIR, variant or "lib")
    return [(src, os.path.join(objdir, os.path.splitext(src)[0] + ".o"), flags)
            for src in SOURCES + extra_src], objdir, os.path.join(PKG, name)


def build(force: bool = False, verbose: bool = False, extra_flags=(), variants=("",)) -> str:
    """Build the requested library variants ("" = libtwell.so); returns the
    path of the first one."""
    todo = [v for v in variants if force or _stale(lib_path(v))]
    if not todo:
        return lib_path(variants[0])
    nvcc = nvcc_path()
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                     "-I", CSRC, "--expt-relaxed-constexpr"] + list(extra_flags)

    def compile_one(job):
        src, obj, flags = job
        cmd = [nvcc, "-c", os.path.join(CSRC, src), "-o", obj] + common + flags
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    plans = []
    jobs = []
    for v in todo:
        js, objdir, lib = _jobs(v)
        os.makedirs(objdir, exist_ok=True)
        plans.append((js, lib))
        jobs += js
    workers = max(1, min(len(jobs), os.cpu_count() or 8))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(compile_one, jobs))
    for js, lib in plans:
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc, "-shared", "-o", tmp] + [o for _, o, _ in js] + ARCH + ["-ldl"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib_path(variants[0])


def build_all(force: bool = False, verbose: bool = False) -> None:
    """The product library and both test variants, compiled together."""
    build(force=force, verbose=verbose, variants=tuple(VARIANTS))


if __name__ == "__main__":
    build_all(force="--force" in sys.argv, verbose=True)
    print("\n".join(lib_path(v) for v in VARIANTS))
