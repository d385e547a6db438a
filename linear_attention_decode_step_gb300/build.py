"""Builds the KDA CUDA library (libkda_gb300.so) in-tree for sm_103a.

Each .cu under csrc/ is compiled in parallel with nvcc, then linked into one
shared library next to this file. The C ABI it exports is include/kda.h.
Rebuilds only when a source or header is newer than the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libkda_gb300.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the KDA library needs the CUDA toolkit to build")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps() -> list[str]:
    return (sources() + glob.glob(os.path.join(CSRC, "*.cuh")) +
            glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None) -> str:
    """Compile and link libkda_gb300.so; returns its path."""
    if not force and up_to_date():
        return LIB
    os.makedirs(OBJ_DIR, exist_ok=True)
    cc = nvcc()
    flags = NVCC_FLAGS + list(extra_flags or [])

    def compile_one(src: str) -> str:
        obj = os.path.join(OBJ_DIR, os.path.basename(src)[:-3] + ".o")
        cmd = [cc] + flags + ["-c", src, "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, res.stdout, res.stderr))
        if verbose and (res.stdout or res.stderr):
            sys.stderr.write(res.stdout + res.stderr)
        return obj

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = LIB + ".tmp%d" % os.getpid()
    res = subprocess.run([cc] + ARCH + ["-shared", "-o", tmp] + objs,
                         capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (res.stdout, res.stderr))
    os.replace(tmp, LIB)
    return LIB


def build_variant(tag: str, defines: list[str], only: list[str]) -> str:
    """A second build of the library for tests: the sources named in `only`
    (file names under csrc/) compiled with extra preprocessor definitions
    (`defines`, e.g. ["KDA_WAIT_BUDGET=0"]), linked with the regular objects
    of the other sources into libkda_gb300_<tag>.so next to the regular
    library. Returns its path. The regular library is built first."""
    build()
    cc = nvcc()
    obj_dir = os.path.join(PKG, "_build_" + tag)
    os.makedirs(obj_dir, exist_ok=True)
    flags = NVCC_FLAGS + ["-D" + d for d in defines]
    lib = os.path.join(PKG, "libkda_gb300_%s.so" % tag)

    def obj_for(src: str) -> str:
        name = os.path.basename(src)
        if name in only:
            obj = os.path.join(obj_dir, name[:-3] + ".o")
            res = subprocess.run([cc] + flags + ["-c", src, "-o", obj], capture_output=True, text=True)
            if res.returncode != 0:
                raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, res.stdout, res.stderr))
            return obj
        return os.path.join(OBJ_DIR, name[:-3] + ".o")

    srcs = sources()
    missing = [n for n in only if os.path.join(CSRC, n) not in srcs]
    if missing:
        raise ValueError("no such source: %s" % ", ".join(missing))
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(obj_for, srcs))
    tmp = lib + ".tmp%d" % os.getpid()
    res = subprocess.run([cc] + ARCH + ["-shared", "-o", tmp] + objs, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (res.stdout, res.stderr))
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    v = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas" in sys.argv else None
    print(build(force=True, verbose=v or bool(extra), extra_flags=extra))
