"""Build libmedusa.so in-tree with nvcc for sm_103a (GB300).

Each CUDA source is compiled to an object in parallel, then linked into one
shared library next to this file. Rebuilds only when a source or header is
newer than the library. The same sources compiled with -DMEDUSA_CHECKED give
libmedusa_checked.so, whose kernels also record every out-of-range index they
meet (a debug build; see medusa_poll_checks in include/medusa.h).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libmedusa.so")
LIB_CHECKED = os.path.join(PKG, "libmedusa_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmedusa")
    return exe


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(ROOT, "include", "*.h"))


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=(), checked: bool = True) -> str:
    """Build libmedusa.so (and, unless checked=False, libmedusa_checked.so); returns the first's path."""
    variants = [(LIB, os.path.join(BUILD, "lib"), [])]
    if checked:
        variants.append((LIB_CHECKED, os.path.join(BUILD, "checked"), ["-DMEDUSA_CHECKED"]))
    variants = [v for v in variants if force or not up_to_date(v[0])]
    if not variants:
        return LIB
    exe = nvcc()
    for _, d, _ in variants:
        os.makedirs(d, exist_ok=True)

    def compile_one(job):
        src, out_dir, flags = job
        obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [exe, *ARCH, *NVCC_FLAGS, *flags, *extra_flags, "-I", os.path.join(ROOT, "include"), "-c", src,
               "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    jobs = [(src, d, flags) for _, d, flags in variants for src in sources()]
    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, jobs))
    n = len(sources())
    for i, (lib, _, _) in enumerate(variants):
        tmp = lib + ".tmp"
        r = subprocess.run([exe, *ARCH, "-shared", "-o", tmp, *objs[i * n:(i + 1) * n]], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
