"""In-tree build of the CUDA library ``_lib/libqps.so`` for sm_103a.

Each translation unit is compiled by nvcc in parallel, then linked into one shared
library against the shared CUDA runtime.  IEEE division and square root are kept
(no fast-math): the encoders are bit-exact contracts.  ``variant="checked"`` builds the
same sources with ``-DQPS_CHECK_BOUNDS=1`` into ``_lib/libqps_checked.so``: every
kernel then tests its staged and addressed accesses against their extents (a debug
build; loaded with ``QPS_LIB_VARIANT=checked``).

Usage: ``python -m quantized_position_split_gb300.build [--force] [-j N] [--checked]``.
"""

from __future__ import annotations

import argparse
import concurrent.futures
import hashlib
import os
import platform
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "_lib")
VARIANTS = {  # build directory, library, extra compiler flags
    "default": (os.path.join(PKG, "_build"), os.path.join(LIBDIR, "libqps.so"), []),
    "checked": (os.path.join(PKG, "_build_checked"), os.path.join(LIBDIR, "libqps_checked.so"),
                ["-DQPS_CHECK_BOUNDS=1"]),
}
BUILD, LIB, _ = VARIANTS["default"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = [
    "-O3",
    "-lineinfo",
    "-std=c++17",
    "-Xcompiler", "-fPIC",
    "-Xcompiler", "-fvisibility=hidden",
    "--expt-relaxed-constexpr",
    "-Xptxas", "-warn-spills",
]


def nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(cuda, "bin", "nvcc")
    if os.path.exists(cand):
        return cand
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found (set CUDA_HOME)")
    return found


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _digest(paths, extra):
    h = hashlib.sha256()
    for p in paths:
        with open(p, "rb") as f:
            h.update(f.read())
    h.update(" ".join(extra).encode())
    h.update(platform.machine().encode())  # objects never cross host architectures
    return h.hexdigest()


def _headers():
    hs = [os.path.join(INCLUDE, "qps.h")]
    hs += sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh")))
    return hs


def compile_one(src: str, verbose: bool, build_dir: str = BUILD, extra=()) -> str:
    obj = os.path.join(build_dir, os.path.basename(src) + ".o")
    stamp = obj + ".sha"
    flags = ARCH + NVCC_FLAGS + list(extra) + ["-I", INCLUDE, "-I", CSRC]
    key = _digest([src] + _headers(), flags)
    if os.path.exists(obj) and os.path.exists(stamp) and open(stamp).read() == key:
        return obj
    cmd = [nvcc()] + flags + ["-c", src, "-o", obj]
    if verbose:
        print(" ".join(cmd), flush=True)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{res.stdout}\n{res.stderr}")
    if verbose and (res.stdout or res.stderr):
        print(res.stdout + res.stderr, flush=True)
    with open(stamp, "w") as f:
        f.write(key)
    return obj


def build(force: bool = False, jobs: int = 0, verbose: bool = False, variant: str = "default") -> str:
    build_dir, lib_path, extra = VARIANTS[variant]
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    if force:
        for f in os.listdir(build_dir):
            os.remove(os.path.join(build_dir, f))
    srcs = sources()
    jobs = jobs or min(len(srcs), os.cpu_count() or 4)
    with concurrent.futures.ThreadPoolExecutor(max_workers=jobs) as ex:
        objs = list(ex.map(lambda s: compile_one(s, verbose, build_dir, extra), srcs))
    key = _digest(objs, ["link"])
    LIB = lib_path
    stamp = LIB + ".sha"
    if not force and os.path.exists(LIB) and os.path.exists(stamp) and open(stamp).read() == key:
        return LIB
    tmp = LIB + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(key)
    return LIB


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("-j", "--jobs", type=int, default=0)
    ap.add_argument("-v", "--verbose", action="store_true")
    ap.add_argument("--checked", action="store_true", help="build the bounds-checked variant")
    args = ap.parse_args(argv)
    print(build(args.force, args.jobs, args.verbose, "checked" if args.checked else "default"))


if __name__ == "__main__":
    sys.exit(main())
