"""Build libbsa.so in-tree with nvcc for sm_103a.

The translation units compile in parallel, then link into
``block_sparse_long_kv_gb300/libbsa.so``.  Objects go to ``_build/`` next to the
sources (git-ignored), with the key the library was built under: a hash of the
sources and headers, the flags and the nvcc version, so a change to any of them
rebuilds.  Run ``python -m block_sparse_long_kv_gb300.build``.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libbsa.so")
SOURCES = ["bsa_api.cu", "bsa_mask.cu", "bsa_score.cu", "bsa_token_score.cu", "bsa_attn.cu", "bsa_decode.cu",
           "bsa_select_noalloc.cu", "bsa_selftest.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr", "-I" + INCLUDE]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libbsa")


KEY = os.path.join(OBJ, "libbsa.key")


def _build_key(nvcc: str) -> str:
    """Hash of everything the library is built from: every source and header,
    the file list, the architecture and compiler flags, and the nvcc version."""
    h = hashlib.sha256()
    ver = subprocess.run([nvcc, "--version"], capture_output=True, text=True).stdout
    h.update(ver.encode())
    h.update(repr((SOURCES, ARCH, FLAGS)).encode())
    deps = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)) + [os.path.join(INCLUDE, "bsa.h")]
    for d in deps:
        h.update(os.path.basename(d).encode())
        with open(d, "rb") as f:
            h.update(hashlib.sha256(f.read()).digest())
    return h.hexdigest()


def _stale(key: str) -> bool:
    if not os.path.exists(LIB) or not os.path.exists(KEY):
        return True
    with open(KEY) as f:
        return f.read().strip() != key


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libbsa.so unless it was built from exactly these sources, flags and nvcc."""
    nvcc = _nvcc()
    key = _build_key(nvcc)
    if not force and not _stale(key):
        return LIB
    os.makedirs(OBJ, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(OBJ, src.replace(".cu", ".o"))
        cmd = [nvcc, "-c", *ARCH, *FLAGS, os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stdout.write(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + ".tmp"
    cmd = [nvcc, "-shared", *ARCH, "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(KEY, "w") as f:
        f.write(key + "\n")
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
