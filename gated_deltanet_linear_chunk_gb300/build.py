"""Builds the CUDA library (libgdn) in-tree for sm_103a with nvcc.

Each .cu under csrc/ compiles to an object in parallel; the objects link into
one shared library with the CUDA runtime linked statically, so the library
loads on a machine without a GPU (only the C ABI symbols are exported).  A
second variant, libgdn_debug, is built with GDN_DEBUG: the same kernels plus
device-side checks of the inputs' preconditions and of the kernels' indices.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import platform
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-fvisibility=hidden",
              "-Xptxas", "-warn-spills", "--expt-relaxed-constexpr"]


def library_path(debug: bool = False) -> str:
    """The release library, or with `debug` the GDN_DEBUG one (device-side
    checks of the inputs' preconditions and of the kernels' indices)."""
    name = "libgdn_debug" if debug else "libgdn"
    return os.path.join(BUILD, f"{name}_{platform.machine()}.so")


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def _stale(out: str) -> bool:
    if not os.path.exists(out):
        return True
    newest = max(os.path.getmtime(p) for p in _deps())
    return os.path.getmtime(out) < newest


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug=None) -> str:
    """Compile every CUDA source and link the library: debug=None builds the
    release and the GDN_DEBUG variants (their sources compiled in one
    parallel pool), True or False one of them.  Returns the path of the
    release library (or of the one variant asked for)."""
    variants = [False, True] if debug is None else [bool(debug)]
    todo = [v for v in variants if force or _stale(library_path(v))]
    if todo:
        nvcc = _nvcc()
        srcs = _sources()

        def obj_dir(dbg):
            return os.path.join(BUILD, "debug") if dbg else BUILD

        def compile_one(job):
            dbg, src = job
            obj = os.path.join(obj_dir(dbg), os.path.basename(src) + f".{platform.machine()}.o")
            flags = [*NVCC_FLAGS, *extra_flags] + (["-DGDN_DEBUG"] if dbg else [])
            cmd = [nvcc, *ARCH, *flags, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
            if verbose and r.stderr:
                print(r.stderr)
            return obj

        for dbg in todo:
            os.makedirs(obj_dir(dbg), exist_ok=True)
        jobs = [(dbg, src) for dbg in todo for src in srcs]
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            objs = list(ex.map(compile_one, jobs))
        for dbg in todo:
            out = library_path(dbg)
            mine = [o for (d, _), o in zip(jobs, objs) if d == dbg]
            tmp = out + ".tmp"
            cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-Xcompiler", "-fPIC", *mine,
                   "-o", tmp]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"link failed:\n{r.stderr}")
            os.replace(tmp, out)
    return library_path(False if debug is None else bool(debug))


if __name__ == "__main__":
    print(build(force=True, verbose=True))
