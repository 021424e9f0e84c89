"""Build libcsa.so (the C-ABI library) from csrc/*.cu for sm_103a.

Each translation unit is compiled by nvcc in parallel, then linked into a
shared library next to this file.  Rebuilds only what changed.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import hashlib
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libcsa.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xptxas", "-O3", "-I", INCLUDE]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps_mtime() -> float:
    files = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
    files += glob.glob(os.path.join(INCLUDE, "*.h"))
    return max((os.path.getmtime(f) for f in files), default=0.0)


def _obj_dir(extra: list) -> str:
    """Objects built with different extra flags live apart, so a flag change rebuilds."""
    if not extra:
        return BUILD
    return os.path.join(BUILD, hashlib.sha1(" ".join(extra).encode()).hexdigest()[:12])


def _compile(nvcc: str, src: str, extra: list) -> str:
    obj = os.path.join(_obj_dir(extra), os.path.basename(src).replace(".cu", ".o"))
    if os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(src), _deps_mtime()):
        return obj
    cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj + ".tmp"]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{p.stdout}\n{p.stderr}")
    os.replace(obj + ".tmp", obj)
    return obj


def build(verbose: bool = False, extra: list | None = None) -> str:
    """Compile every csrc/*.cu and link libcsa.so; returns its path."""
    extra = list(extra or [])
    os.makedirs(_obj_dir(extra), exist_ok=True)
    nvcc = _nvcc()
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(nvcc, s, extra), srcs))
    newest = max(os.path.getmtime(o) for o in objs)
    stamp = os.path.join(BUILD, "last_link")  # which object set the library was linked from
    linked_from = open(stamp).read() if os.path.exists(stamp) else ""
    if not os.path.exists(LIB) or os.path.getmtime(LIB) < newest or linked_from != _obj_dir(extra):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]  # static cudart (nvcc default)
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"link failed:\n{p.stdout}\n{p.stderr}")
        os.replace(tmp, LIB)
        with open(stamp, "w") as fh:
            fh.write(_obj_dir(extra))
    if verbose:
        print(LIB)
    return LIB


if __name__ == "__main__":
    build(verbose=True, extra=sys.argv[1:])
