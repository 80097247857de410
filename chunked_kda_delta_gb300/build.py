"""Build the KDA CUDA library (``_build/libkda.so``) with nvcc for sm_103a.

Each ``csrc/*.cu`` file is compiled in parallel with
``-gencode arch=compute_103a,code=sm_103a`` and linked into one shared
library against the shared CUDA runtime (so a process that already loaded
torch's ``libcudart.so.13`` shares a single runtime with it).  Run as
``python -m chunked_kda_delta_gb300.build``.
"""
from __future__ import annotations

import concurrent.futures
import glob
import hashlib
import os
import platform
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libkda.so")
STAMP_PATH = LIB_PATH + ".stamp"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found; the KDA library needs the CUDA 13 toolkit")


def cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + [
        os.path.join(INCLUDE, "kda.h"), os.path.abspath(__file__)]


def _stamp(flags) -> str:
    """Digest of everything the library is built from: the source and header bytes,
    the compiler flags, the host architecture and the nvcc version line.  A library
    whose stamp differs (other sources, flags, or a library built on another machine
    and copied here) is rebuilt."""
    h = hashlib.sha256()
    for d in _deps():
        h.update(os.path.basename(d).encode())
        with open(d, "rb") as f:
            h.update(f.read())
    h.update(" ".join(flags).encode())
    h.update(platform.machine().encode())
    try:
        ver = subprocess.run([nvcc_path(), "--version"], capture_output=True, text=True).stdout
    except (OSError, RuntimeError):
        ver = ""
    h.update(ver.encode())
    return h.hexdigest()


def _up_to_date(stamp: str) -> bool:
    if not (os.path.exists(LIB_PATH) and os.path.exists(STAMP_PATH)):
        return False
    with open(STAMP_PATH) as f:
        return f.read().strip() == stamp


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile every CUDA source and link ``libkda.so``; returns the library path."""
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                    "--expt-relaxed-constexpr",
                    "-I", INCLUDE, "-I", CSRC, "-DKDA_BUILDING_LIBRARY"] + list(extra_flags)
    stamp = _stamp(flags)
    if not force and _up_to_date(stamp):
        return LIB_PATH
    nvcc = nvcc_path()
    os.makedirs(BUILD_DIR, exist_ok=True)
    if verbose:
        flags += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.basename(src) + ".o")
        cmd = [nvcc] + flags + ["-c", src, "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
        return obj, res.stderr

    srcs = _sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, len(srcs))) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    objs = [o for o, _ in results]
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    libdir = cuda_lib_dir(nvcc)
    cmd = [nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs + [
        "-Xlinker", f"-rpath={libdir}"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB_PATH)
    with open(STAMP_PATH, "w") as f:
        f.write(stamp + "\n")
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
