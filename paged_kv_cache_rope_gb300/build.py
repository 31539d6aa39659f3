"""Build libpaged_kv.so in-tree for sm_103a (GB300).

    python -m paged_kv_cache_rope_gb300.build [--force] [--verbose-ptxas]

Each translation unit under csrc/ is compiled in parallel by nvcc into _build/, then linked
into paged_kv_cache_rope_gb300/libpaged_kv.so against the shared CUDA runtime (the same one
PyTorch loads).  Only one -gencode is used: compute_103a -> sm_103a.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libpaged_kv.so")
SOURCES = ["api.cpp", "append_rope.cu", "decode_attn.cu", "context_attn.cu", "noalloc.cu"]
HEADERS = ["common.cuh", "internal.h", "tcgen05.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpaged_kv.so")
    return cand


def _flags(verbose_ptxas: bool) -> list[str]:
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O3", "-I", INCLUDE, "-I", CSRC,
                "--expt-relaxed-constexpr"]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _fingerprint(verbose_ptxas: bool) -> str:
    h = hashlib.sha256()
    for name in SOURCES + HEADERS:
        with open(os.path.join(CSRC, name), "rb") as fh:
            h.update(name.encode() + fh.read())
    with open(os.path.join(INCLUDE, "paged_kv.h"), "rb") as fh:
        h.update(fh.read())
    h.update(" ".join(_flags(False)).encode())
    return h.hexdigest()


# The self-test build: the same sources with the producer of the context kernel issuing no K / V
# copies and every bounded wait given about a millisecond, so that a test can watch a wait run
# out and the kernel wind down (error bit set, TMEM freed, the context still usable).  Only the
# tests build and load it; it is never part of libpaged_kv.so.
SELFTEST_LIB = os.path.join(PKG, "libpaged_kv_selftest.so")
SELFTEST_DEFS = ["-DPKV_SELFTEST", "-DPKV_WAIT_BUDGET=2000000LL"]


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    return _build_lib(LIB, BUILD, [], force, verbose_ptxas)


def build_selftest(force: bool = False) -> str:
    return _build_lib(SELFTEST_LIB, os.path.join(BUILD, "selftest"), SELFTEST_DEFS, force, False)


def _build_lib(lib: str, build_dir: str, defs: list[str], force: bool, verbose_ptxas: bool) -> str:
    os.makedirs(build_dir, exist_ok=True)
    stamp = os.path.join(build_dir, os.path.basename(lib) + ".stamp")
    fp = _fingerprint(verbose_ptxas) + " ".join(defs)
    if not force and os.path.exists(lib) and os.path.exists(stamp) and open(stamp).read() == fp:
        return lib
    nvcc = _nvcc()
    flags = _flags(verbose_ptxas) + defs

    def compile_one(name: str) -> str:
        src = os.path.join(CSRC, name)
        obj = os.path.join(build_dir, name + ".o")
        cmd = [nvcc] + flags + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {name}:\n{r.stdout}\n{r.stderr}")
        if verbose_ptxas and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(stamp, "w") as fh:
        fh.write(fp)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="--verbose-ptxas" in sys.argv))
