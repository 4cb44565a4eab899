"""Build libdsa.so in-tree with nvcc for sm_103a.

Every translation unit under ``csrc/`` is compiled in parallel to an object
file under ``_lib/obj`` and linked into ``_lib/libdsa.so``.  Objects are
rebuilt when their source or any header under ``csrc/`` or ``include/`` is
newer.  No CMake, one ``-gencode``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIBDIR = os.path.join(PKG, "_lib")
OBJDIR = os.path.join(LIBDIR, "obj")
LIB = os.path.join(LIBDIR, "libdsa.so")
# the checked build: device-side input checks compiled in (-DDSA_CHECKS=1)
OBJDIR_CHECKED = os.path.join(LIBDIR, "obj_checked")
LIB_CHECKED = os.path.join(LIBDIR, "libdsa_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
          "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libdsa")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    inc = os.path.join(ROOT, "include")
    hs += [os.path.join(inc, f) for f in os.listdir(inc) if f.endswith(".h")]
    return hs


def _stale(obj: str, src: str, newest_header: float) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return os.path.getmtime(src) > t or newest_header > t


def build(verbose: bool = False, jobs: int | None = None, extra_flags=None,
          checked: bool = False) -> str:
    """Compile (if needed) and return the path of libdsa.so (checked: libdsa_checked.so,
    with the device-side input checks compiled in)."""
    nvcc = _nvcc()
    objdir = OBJDIR_CHECKED if checked else OBJDIR
    lib = LIB_CHECKED if checked else LIB
    os.makedirs(objdir, exist_ok=True)
    srcs = _sources()
    newest_header = max((os.path.getmtime(h) for h in _headers()), default=0.0)
    flags = COMMON + list(extra_flags or []) + (["-DDSA_CHECKS=1"] if checked else [])
    todo = []
    objs = []
    for src in srcs:
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        objs.append(obj)
        if _stale(obj, src, newest_header):
            todo.append((src, obj))

    def compile_one(job):
        src, obj = job
        cmd = [nvcc, *ARCH, *flags, "-c", src, "-o", obj]
        if src.endswith(".cu"):
            cmd[1:1] = ["-Xptxas", "-v"] if verbose else []
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        return r.stderr if verbose else ""

    if todo:
        with ThreadPoolExecutor(max_workers=jobs or min(len(todo), os.cpu_count() or 4)) as ex:
            for msg in ex.map(compile_one, todo):
                if msg:
                    print(msg)
    if todo or not os.path.exists(lib):
        tmp = lib + ".tmp"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of {os.path.basename(lib)} failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(verbose="-v" in sys.argv))
