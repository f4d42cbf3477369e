"""Build libtb.so (the C-ABI CUDA library) in-tree for sm_103a with nvcc.

    python -m predicted_token_importance_tb_b300.build [--force]

The library is rebuilt only when a source or header changed (content hash).
"""
from __future__ import annotations

import glob
import hashlib
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libtb.so")
STAMP = LIB + ".buildhash"

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-shared", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "--expt-relaxed-constexpr",
]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + [os.path.join(INCLUDE, "tb.h"), __file__]


def _hash() -> str:
    h = hashlib.sha256()
    for p in _inputs():
        h.update(os.path.basename(p).encode())
        with open(p, "rb") as f:
            h.update(f.read())
    h.update(" ".join(NVCC_FLAGS).encode())
    return h.hexdigest()


def strip_comments(src: str) -> str:
    """C/C++/CUDA source without its comments, whitespace runs folded to one
    space: two sources that compile to the same code (up to line numbers)
    give the same text."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":                          # string or character literal, escapes kept
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def code_hash(units=None) -> str:
    """Hash of the library's code: the sources (all, or only the translation
    units named in `units`, e.g. ("fused_fast.cu", "tb_api.cu")) and every
    header, with comments and layout removed, plus the compiler flags. A
    profile of a kernel stays valid across builds whose code hash over that
    kernel's units is the same."""
    srcs = _sources() if units is None else [os.path.join(CSRC, u) for u in sorted(units)]
    h = hashlib.sha256()
    for p in srcs + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + [os.path.join(INCLUDE, "tb.h")]:
        h.update(os.path.basename(p).encode())
        with open(p, encoding="utf-8") as f:
            h.update(strip_comments(f.read()).encode())
    h.update(" ".join(NVCC_FLAGS).encode())
    return h.hexdigest()


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.sep not in c or os.path.exists(c)):
            return c
    return "nvcc"


OBJ_DIR = os.path.join(PKG, "_build")


def _unit_hash(src: str) -> str:
    """A translation unit's object is current when this matches: its source, every header, the flags."""
    h = hashlib.sha256()
    for p in [src] + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + [os.path.join(INCLUDE, "tb.h")]:
        h.update(os.path.basename(p).encode())
        with open(p, "rb") as f:
            h.update(f.read())
    h.update(" ".join(NVCC_FLAGS).encode())
    return h.hexdigest()


def _compile(src: str, verbose: bool) -> str:
    """nvcc -c of one translation unit into _build/ (skipped when its object is current)."""
    os.makedirs(OBJ_DIR, exist_ok=True)
    obj = os.path.join(OBJ_DIR, os.path.basename(src) + ".o")
    stamp = obj + ".buildhash"
    h = _unit_hash(src)
    if os.path.exists(obj) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == h:
                return obj
    flags = [f for f in NVCC_FLAGS if f != "-shared"]
    tmp = obj + f".tmp{os.getpid()}"
    cmd = [nvcc(), *flags, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", tmp]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    os.replace(tmp, obj)
    with open(stamp, "w") as f:
        f.write(h)
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every translation unit (in parallel, each only when it changed) and link libtb.so."""
    h = _hash()
    if not force and os.path.exists(LIB) and os.path.exists(STAMP):
        with open(STAMP) as f:
            if f.read().strip() == h:
                return LIB
    from concurrent.futures import ThreadPoolExecutor
    srcs = _sources()
    if force:
        for src in srcs:
            stamp = os.path.join(OBJ_DIR, os.path.basename(src) + ".o.buildhash")
            if os.path.exists(stamp):
                os.remove(stamp)
    with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose), srcs))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-Xcompiler", "-fPIC",
           "-o", tmp, *objs]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(h)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
