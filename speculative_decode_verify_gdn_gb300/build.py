"""In-tree build of the sm_103a GDN verify library (``libgdn_sm103a.so``).

Compiles every ``csrc/*.cu`` translation unit in parallel with nvcc for
``sm_103a`` only and links one shared library next to this file.  A stamp of
the sources' and flags' hash skips rebuilds when nothing changed.

    python -m speculative_decode_verify_gdn_gb300.build [--force] [--verbose]
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
REPO_DIR = os.path.dirname(PKG_DIR)
CSRC_DIR = os.path.join(PKG_DIR, "csrc")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_PATH = os.path.join(PKG_DIR, "libgdn_sm103a.so")
HEADER = os.path.join(REPO_DIR, "include", "gdn.h")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v"] + ARCH_FLAGS


def nvcc_path() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    p = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(p):
        return p
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is needed to build the sm_103a library")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC_DIR, f) for f in os.listdir(CSRC_DIR) if f.endswith(".cu"))


def _digest() -> str:
    h = hashlib.sha256()
    files = sources() + sorted(os.path.join(CSRC_DIR, f) for f in os.listdir(CSRC_DIR)
                               if f.endswith((".cuh", ".h"))) + [HEADER]
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(NVCC_FLAGS).encode())
    return h.hexdigest()


def _code_only(text: str) -> str:
    """C/C++/CUDA source without its comments and with blank runs collapsed (string and
    character literals kept as they are)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def _code_digest(files) -> str:
    h = hashlib.sha256()
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    h.update(" ".join(NVCC_FLAGS).encode())
    return h.hexdigest()[:16]


def kernel_source_digest() -> str:
    """Hash of all CUDA sources without their comments, and of the flags: identifies the
    kernels a profile was taken on, and stays put when only commentary changes."""
    return _code_digest(sources() + sorted(os.path.join(CSRC_DIR, f) for f in os.listdir(CSRC_DIR)
                                           if f.endswith((".cuh", ".h"))) + [HEADER])


# the translation unit of the verify kernels and everything it includes
VERIFY_SOURCES = ("gdn_verify.cu", "gdn_common.cuh", "gdn_kernels.h")


def verify_kernel_digest() -> str:
    """The same hash over the verify kernels' sources only (gdn_verify.cu, the headers it
    includes, and gdn.h): a profile of those kernels stays valid across edits elsewhere."""
    return _code_digest([os.path.join(CSRC_DIR, f) for f in VERIFY_SOURCES] + [HEADER])


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Build libgdn_sm103a.so if missing or stale; returns its path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    stamp = os.path.join(BUILD_DIR, "stamp")
    digest = _digest()
    if not force and os.path.exists(LIB_PATH) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return LIB_PATH
    nvcc = nvcc_path()
    objs = []

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD_DIR, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, "-c", src, "-o", obj, "-I", os.path.join(REPO_DIR, "include")] + NVCC_FLAGS
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        with open(obj + ".log", "w") as f:
            f.write(r.stdout + r.stderr)
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc, "-shared", "-o", tmp] + objs + ARCH_FLAGS + ["-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    with open(stamp, "w") as f:
        f.write(digest)
    return LIB_PATH


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    args = ap.parse_args()
    print(build_library(force=args.force, verbose=args.verbose))


if __name__ == "__main__":
    main()
