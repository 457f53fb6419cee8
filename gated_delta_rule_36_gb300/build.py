"""In-tree build of the KDA C-ABI library (``libkda.so``) for sm_103a.

Each ``csrc/*.cu`` translation unit is compiled by nvcc in parallel, then linked
into one shared library next to this file.  The CUDA runtime is linked
statically, so the library only needs the driver at run time.

Two more builds of the same sources serve the tests only:
``build(variant="checked")`` makes ``libkda_checked.so`` (``-DKDA_CHECKED``: a bad index
sets KDA_DEVERR_INTERNAL instead of faulting), and ``build(variant="waittest")`` makes
``libkda_waittest.so`` (``-DKDA_WAIT_TEST``: short wait limits and one arrival skipped on
request, to exercise the timeout path).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libkda.so")
# test-only builds: name -> extra nvcc flag
VARIANTS = {"checked": "-DKDA_CHECKED", "waittest": "-DKDA_WAIT_TEST"}
LIB_PATH_CHECKED = os.path.join(HERE, "libkda_checked.so")


def lib_path(variant=None) -> str:
    return LIB_PATH if variant is None else os.path.join(HERE, f"libkda_{variant}.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = [os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the KDA library needs the CUDA toolkit to build")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
                               + glob.glob(os.path.join(INCLUDE, "*.h"))) + [os.path.abspath(__file__)]


def needs_build(variant=None) -> bool:
    lib = lib_path(variant)
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(d) > t for d in _deps())


def compile_flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
                   "--expt-relaxed-constexpr", *extra]


def build(force: bool = False, verbose: bool = False, extra_flags=(), variant=None) -> str:
    """Compile every CUDA source for sm_103a and link ``libkda.so`` in-tree (with a
    ``variant`` of VARIANTS, the test-only ``libkda_<variant>.so``)."""
    out_path = lib_path(variant)
    build_dir = BUILD_DIR if variant is None else os.path.join(HERE, f"_build_{variant}")
    if not force and not needs_build(variant):
        return out_path
    nvcc = _nvcc()
    os.makedirs(build_dir, exist_ok=True)
    flags = compile_flags(tuple(extra_flags) + ((VARIANTS[variant],) if variant else ()))

    def cc(src):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *flags, "-Xptxas", "-v", "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stderr)
        return obj

    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(cc, srcs))
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static", "-ldl", "-lrt", "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out_path)
    return out_path


if __name__ == "__main__":
    import sys
    v = [a[2:] for a in sys.argv[1:] if a[2:] in VARIANTS]
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, variant=v[0] if v else None))
