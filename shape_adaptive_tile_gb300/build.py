"""Builds the CUDA library ``_lib/libsatgemm.so`` in-tree with nvcc for sm_103a.

Translation units compile in parallel; the previous library is deleted
before linking, so a failed build never leaves a stale one behind, and a
stamp records the nvcc version and flags, so a toolchain or flag change
forces a rebuild.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import re
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIB_DIR, "libsatgemm.so")
STAMP = os.path.join(LIB_DIR, "libsatgemm.stamp")

# The kernel variants come as three translation units per dtype (they take
# most of the build); the longest units are listed first.
SOURCES = [f"kernels_{dt}{grp}.cu" for grp in ("", "_alt", "_trans") for dt in ("tf32", "bf16", "fp16")] + [
    "device_call.cu", "api.cu", "aux_kernels.cu", "dispatch.cpp", "tensor_map.cpp", "noalloc.cu", "rowops.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]
# The GEMM kernel units: an explicit register ceiling (the launch bounds of
# a 320-thread, one-CTA-per-SM kernel allow 200) keeps ptxas from spilling
# the epilogue at its own default of 168 registers.
EXTRA = {f: ["-maxrregcount=200"] for f in SOURCES if f.startswith("kernels_") or f == "device_call.cu"}


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _inputs():
    files = [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC))]
    files += [os.path.join(INCLUDE, "gemm.h"), os.path.join(INCLUDE, "rowops.h"), os.path.join(INCLUDE, "gemm_device.cuh")]
    return [f for f in files if os.path.isfile(f)]


# A C/C++ comment or a string or character literal (kept whole, so that a
# comment marker inside a literal is not taken for a comment).
_TOKEN = re.compile(rb'//[^\n]*|/\*.*?\*/|"(?:\\.|[^"\\\n])*"|\'(?:\\.|[^\'\\\n])*\'', re.S)


def _code_text(data: bytes) -> bytes:
    """The source with comments removed and runs of whitespace collapsed: a
    profile stays valid across edits that change neither."""
    data = _TOKEN.sub(lambda m: b" " if m.group(0)[:1] == b"/" else m.group(0), data)
    return b" ".join(data.split())


def source_hash() -> str:
    """SHA-256 of the kernel and ABI sources (what a profile was taken of),
    comments and layout aside."""
    h = hashlib.sha256()
    for f in _inputs():
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode() + b"\0" + _code_text(fh.read()))
    return h.hexdigest()[:16]


# Sources of the row operators only: no GEMM kernel includes or calls them.
_ROWOP_ONLY = ("rowops.cu", "rowops.h")


def gemm_source_hash() -> str:
    """SHA-256 of the sources the GEMM kernels are built from: every input but
    the row operators' own files, comments and layout aside. A profile of a
    GEMM kernel stays valid as long as this is unchanged."""
    h = hashlib.sha256()
    for f in _inputs():
        if os.path.basename(f) in _ROWOP_ONLY:
            continue
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode() + b"\0" + _code_text(fh.read()))
    return h.hexdigest()[:16]


def _key(nvcc: str) -> str:
    ver = subprocess.run([nvcc, "--version"], capture_output=True, text=True, check=True).stdout
    h = hashlib.sha256()
    h.update(ver.encode())
    h.update(" ".join(FLAGS).encode())
    h.update(repr(sorted(EXTRA.items())).encode())
    for f in _inputs():
        with open(f, "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()


def build(force: bool = False, jobs: int | None = None, verbose: bool = False) -> str:
    """Compile (if needed) and return the path of the shared library."""
    nvcc = _nvcc()
    key = _key(nvcc)
    if not force and os.path.exists(LIB) and os.path.exists(STAMP):
        with open(STAMP) as f:
            if f.read().strip() == key:
                return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    for stale in (LIB, STAMP):
        if os.path.exists(stale):
            os.remove(stale)

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
        if os.path.exists(obj):
            os.remove(obj)
        cmd = [nvcc, *FLAGS, *EXTRA.get(src, []), "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    jobs = jobs or min(len(SOURCES), os.cpu_count() or 1)
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(key + "\n")
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
