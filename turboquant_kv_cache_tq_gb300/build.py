"""Build ``libtq.so`` (the C ABI of include/tq.h) in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` translation unit is compiled in parallel and the objects
are linked with the static CUDA runtime, so the library only needs the
driver at run time. Usage: ``python -m turboquant_kv_cache_tq_gb300.build``.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libtq.so")
# The debug variant: the same library compiled with device-side index checks
# (TQ_DEBUG_CHECKS: an index outside its buffer sets the device error word
# read by tq_device_status and skips the access).
DEBUG_BUILD_DIR = os.path.join(PKG, "_build_debug")
DEBUG_LIB_PATH = os.path.join(PKG, "libtq_debug.so")
DEBUG_FLAGS = ("-DTQ_DEBUG_CHECKS",)
ARCH = ("-gencode", "arch=compute_103a,code=sm_103a")
NVCC_FLAGS = (
    "-O3", "-std=c++17", "-lineinfo", *ARCH,
    # one IEEE rounding per operation: no FMA contraction, IEEE div and sqrt
    "-fmad=false", "-prec-div=true", "-prec-sqrt=true", "-ftz=false",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-ffp-contract=off",
    # only the C ABI (TQ_API in include/tq.h) is exported: template statics
    # and the static CUDA runtime stay private to each build, so the library
    # and its debug variant can be loaded in one process
    "-Xcompiler", "-fvisibility=hidden",
    "--expt-relaxed-constexpr",
)


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the TurboQuant CUDA library cannot be built")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(PKG, "..", "include", "tq.h")]


def _stale(lib_path: str = LIB_PATH) -> bool:
    if not os.path.exists(lib_path):
        return True
    t = os.path.getmtime(lib_path)
    return any(os.path.getmtime(p) > t for p in _deps() + [os.path.abspath(__file__)])


def _compile(src: str, extra: tuple[str, ...], build_dir: str = BUILD_DIR) -> str:
    obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed on %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
    return obj


def build(force: bool = False, verbose: bool = False, extra: tuple[str, ...] = (), debug: bool = False) -> str:
    """Compile and link the library (or its debug variant); returns the path
    of libtq.so (libtq_debug.so)."""
    lib_path = DEBUG_LIB_PATH if debug else LIB_PATH
    build_dir = DEBUG_BUILD_DIR if debug else BUILD_DIR
    extra = tuple(extra) + (DEBUG_FLAGS if debug else ())
    if not (force or _stale(lib_path) or (extra and not debug)):
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    srcs = _sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, build_dir), srcs))
    tmp = lib_path + ".tmp%d" % os.getpid()
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-Xlinker", "--exclude-libs,ALL", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
    os.replace(tmp, lib_path)
    if verbose:
        print("built", lib_path)
    return lib_path


if __name__ == "__main__":
    flags = tuple(a for a in sys.argv[1:] if a.startswith("-X") or a.startswith("--"))
    build(force=True, verbose=True, extra=tuple(a for a in flags if a not in ("--force", "--debug")),
          debug="--debug" in flags)
