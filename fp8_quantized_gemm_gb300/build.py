"""Build libfp8gemm.so in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` is compiled to an object in ``_build/`` (in parallel),
then linked with the static CUDA runtime into
``fp8_quantized_gemm_gb300/libfp8gemm.so``.  Objects are rebuilt when the
source, a header or the flags change.  No cmake, no torch extension machinery.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import platform
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfp8gemm.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-fvisibility=hidden", "-I" + INCLUDE,
                     "--expt-relaxed-constexpr", "-diag-suppress", "177"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps_digest() -> str:
    h = hashlib.sha256()
    for d in (CSRC, INCLUDE):
        for f in sorted(os.listdir(d)):
            if f.endswith((".cuh", ".h")):
                with open(os.path.join(d, f), "rb") as fh:
                    h.update(f.encode() + fh.read())
    h.update(" ".join(NVCC_FLAGS).encode())
    h.update(platform.machine().encode())  # host objects differ per architecture
    return h.hexdigest()[:16]


def _compile(nvcc: str, src: str, digest: str) -> str:
    with open(src, "rb") as fh:
        tag = hashlib.sha256(fh.read() + digest.encode()).hexdigest()[:16]
    obj = os.path.join(BUILD, os.path.basename(src)[:-3] + "." + tag + ".o")
    if not os.path.exists(obj):
        tmp = obj + ".tmp"
        cmd = [nvcc] + NVCC_FLAGS + ["-c", src, "-o", tmp]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
        os.replace(tmp, obj)
    return obj


def build(verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    digest = _deps_digest()
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(nvcc, s, digest), srcs))
    stamp = hashlib.sha256(("".join(objs) + platform.machine()).encode()).hexdigest()[:16]
    stamp_file = os.path.join(BUILD, "lib.stamp")
    if os.path.exists(LIB) and os.path.exists(stamp_file):
        with open(stamp_file) as fh:
            if fh.read().strip() == stamp:
                return LIB
    tmp = LIB + ".tmp"
    cmd = [nvcc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    with open(stamp_file, "w") as fh:
        fh.write(stamp)
    if verbose:
        print("built", LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
