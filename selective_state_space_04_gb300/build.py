"""Compile libssd.so in-tree with nvcc (sm_103a only).

Translation units are compiled in parallel and linked into
``selective_state_space_04_gb300/_build/libssd.so``.  The CUDA runtime is
linked statically; the driver API is reached through the runtime's
entry-point query, so the library needs no libcuda at link time.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libssd.so")
SOURCES = ["ssd_api.cu", "ssd_seq.cu", "ssd_chunk.cu", "ssd_decode.cu", "ssd_trap.cu", "ssd_neighbors.cu", "ssd_bwd.cu", "ssd_bwd_chunk.cu", "ssd_bwd_tc.cu", "ssd_complex.cu", "ssd_complex_tc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; libssd needs the CUDA 13 toolkit to build")
    return cand


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "ssd.h"))
    files.append(os.path.abspath(__file__))
    return files


FLAGS_STAMP = os.path.join(BUILD_DIR, "flags")


def option_flags() -> list:
    """Compile-time options chosen by the environment: SSD_NVTX=1 compiles in the
    NVTX ranges around every entry point and launch function."""
    return ["-DSSD_NVTX"] if os.environ.get("SSD_NVTX") == "1" else []


def _stamp(flags) -> str:
    return " ".join(flags)


def is_stale(flags=()) -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    try:
        with open(FLAGS_STAMP) as f:
            if f.read() != _stamp(flags):
                return True
    except OSError:
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    flags = [*option_flags(), *extra_flags]
    if not force and not is_stale(flags):
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    common = [*ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-I", INCLUDE, "-I", CSRC, *flags]
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [nvcc(), *common, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, pr in procs:
        out, _ = pr.communicate()
        if pr.returncode != 0:
            failed.append((src, out.decode(errors="replace")))
        elif verbose and out:
            print(out.decode(errors="replace"), file=sys.stderr)
    if failed:
        msg = "\n".join(f"--- {s}\n{o}" for s, o in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, LIB_PATH)
    with open(FLAGS_STAMP, "w") as f:
        f.write(_stamp(flags))
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
