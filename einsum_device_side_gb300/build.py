"""Build libtropical_gb300.so in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel, then linked into
``einsum_device_side_gb300/_build/libtropical_gb300.so``.  No cmake, no torch
extension machinery: the library has a plain C ABI (include/tropical.h).

Numerics flags: no fast-math, ``-fmad=false`` (no multiply-add contraction),
``-ftz=false`` (subnormals kept), so every tropical product rounds once.

``build(variant="debug")`` makes the bounds-checked library instead, in
``_build_debug/`` (``-DTROP_DEBUG_BOUNDS=1``): every global access of every kernel is
tested against the byte range of its tensor and a violation is recorded, not made
(``tropical_debug_bounds_report``).  It has no CPython binding; the package loads it,
through ctypes, when ``TROP_LIBRARY=debug`` is set.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libtropical_gb300.so")
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(BUILD_DEBUG, "libtropical_gb300.so")
VARIANTS = {"release": (BUILD, LIB, []), "debug": (BUILD_DEBUG, LIB_DEBUG, ["-DTROP_DEBUG_BOUNDS=1"])}
SOURCES = ["runtime.cpp", "api.cpp", "unary.cu", "gemm.cu", "gemm64.cu", "gemm_int.cu", "backtrack.cu", "backward.cu",
           "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fno-strict-aliasing",
          "-ftz=false", "-prec-div=true", "-prec-sqrt=true", "-fmad=false",
          "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    deps = [src, os.path.join(CSRC, "internal.h"), os.path.join(CSRC, "bounds.h"),
            os.path.join(ROOT, "include", "tropical.h")]
    return any(os.path.getmtime(d) > os.path.getmtime(obj) for d in deps)


def _compile(src: str, verbose: bool, variant: str = "release") -> str:
    out_dir, _, defs = VARIANTS[variant]
    path = os.path.join(CSRC, src)
    obj = os.path.join(out_dir, src + ".o")
    if not _stale(obj, path):
        return obj
    cmd = [nvcc(), *ARCH, *COMMON, *defs, "-c", path, "-o", obj + ".tmp"]
    if verbose and src.endswith(".cu"):
        cmd.insert(1, "-Xptxas=-v")
    if src.endswith(".cpp"):
        cmd[1:1] = ["-x", "cu"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    os.replace(obj + ".tmp", obj)
    return obj


def _ext_path() -> str:
    import sysconfig
    return os.path.join(BUILD, "_fastcall" + (sysconfig.get_config_var("EXT_SUFFIX") or ".so"))


def build_fastcall(force: bool = False) -> str | None:
    """The CPython binding of the hot entry points (csrc/fastcall.c), linked against the
    library in the same folder.  Returns its path, or None when this Python has no
    development headers (the ctypes binding then serves every call)."""
    import sysconfig
    src = os.path.join(CSRC, "fastcall.c")
    out = _ext_path()
    inc = sysconfig.get_paths().get("include", "")
    if not os.path.exists(os.path.join(inc, "Python.h")):
        return None
    deps = [src, LIB, os.path.join(ROOT, "include", "tropical.h")]
    if not force and os.path.exists(out) and all(os.path.getmtime(d) <= os.path.getmtime(out) for d in deps):
        return out
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        return None
    tmp = out + f".tmp{os.getpid()}"
    cmd = [cc, "-O2", "-shared", "-fPIC", "-std=c11", "-I", inc, "-I", os.path.join(ROOT, "include"), src,
           "-o", tmp, "-L", BUILD, "-l:" + os.path.basename(LIB), "-Wl,-rpath,$ORIGIN"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"fastcall build failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


def build(verbose: bool = False, force: bool = False, variant: str = "release") -> str:
    out_dir, lib, _ = VARIANTS[variant]
    os.makedirs(out_dir, exist_ok=True)
    if force:
        for f in os.listdir(out_dir):
            os.remove(os.path.join(out_dir, f))
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, variant), SOURCES))
    if os.path.exists(lib) and all(os.path.getmtime(o) <= os.path.getmtime(lib) for o in objs):
        if variant == "release":
            build_fastcall(force=force)
        return lib
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static", "-lrt", "-ldl", "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    if variant == "release":
        build_fastcall(force=True)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv,
                variant="debug" if "--debug" in sys.argv else "release"))
