"""Builds libcb.so in-tree from csrc/*.cu with nvcc for sm_103a.

Each translation unit compiles in parallel (nvcc -c), then one link step
produces ``conv_bn_activation_gb300/libcb.so`` with the CUDA runtime linked
statically.  The build is incremental: an object is rebuilt when its source
or any header in csrc/ or include/ is newer.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libcb.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
_lock = threading.Lock()


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libcb.so")
    return exe


def _flags():
    extra = os.environ.get("CB_NVCC_EXTRA", "").split()  # e.g. -DCB_IGEMM_TRACE (profiling builds)
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-I", INCLUDE, "-I", CSRC,
                   "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"] + extra


def _flag_tag():
    import hashlib
    return hashlib.sha1(" ".join(_flags()).encode()).hexdigest()[:8]


def _headers():
    return glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, verbose: bool) -> str:
    obj = os.path.join(BUILD, os.path.basename(src) + "." + _flag_tag() + ".o")
    if _stale(obj, [src] + _headers()):
        cmd = [nvcc()] + _flags() + ["-c", src, "-o", obj + ".tmp"]
        if verbose:
            cmd += ["-Xptxas", "-v"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        os.replace(obj + ".tmp", obj)
    return obj


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libcb.so; returns its path."""
    with _lock:
        os.makedirs(BUILD, exist_ok=True)
        srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
        stamp = os.path.join(BUILD, "last_flags")
        tag = _flag_tag()
        if os.path.exists(stamp) and open(stamp).read() != tag:
            force = True
        if force:
            for o in glob.glob(os.path.join(BUILD, "*.o")):
                os.remove(o)
        with ThreadPoolExecutor(max_workers=max(1, min(os.cpu_count() or 8, len(srcs)))) as ex:
            objs = list(ex.map(lambda s: _compile(s, verbose), srcs))
        if force or _stale(LIB, objs):
            tmp = LIB + f".tmp{os.getpid()}"
            cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs + ["-lpthread", "-ldl", "-lrt"]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
            os.replace(tmp, LIB)
        open(stamp, "w").write(tag)
        return LIB


if __name__ == "__main__":
    import sys
    print(build_library(force="--force" in sys.argv, verbose="-v" in sys.argv))
