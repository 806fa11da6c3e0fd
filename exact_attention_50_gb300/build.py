"""Builds libattn_gb300.so in-tree from csrc/*.cu with nvcc for sm_103a (no torch extension
machinery: the library has a plain C ABI).  Translation units compile in parallel; a stamp
of the sources and flags skips the build when nothing changed."""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libattn_gb300.so")

SOURCES = ["attn_api.cu", "fwd_tc_bf16.cu", "fwd_tc_f16.cu", "bwd_tc_bf16.cu", "bwd_tc_f16.cu", "kv_combine.cu",
           "simt_f32.cu", "bwd_aux.cu", "attn_noalloc.cu", "fwd_short.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build the library")
    return cand


def _stamp() -> str:
    h = hashlib.sha256()
    h.update(" ".join(FLAGS).encode())
    for d in (CSRC, INCLUDE):
        for name in sorted(os.listdir(d)):
            if name.endswith((".cu", ".cuh", ".h")):
                with open(os.path.join(d, name), "rb") as f:
                    h.update(name.encode())
                    h.update(f.read())
    return h.hexdigest()


# Host-only sources: the C ABI entry points (argument checks, tensor maps, launches).  Their
# device code is the status word alone; include/attn.h reaches the kernels only through the
# ATTN_ status and flag constants.
HOST_SOURCES = ("attn_api.cu",)


def _portable_flags() -> list:
    """The compile flags without the include directories, which name absolute paths of the
    checkout: the same sources compiled in another directory give the same stamp."""
    return [f for f in FLAGS if not f.startswith("-I")]


def code_stamp(read=None) -> str:
    """Hash of the device code: every CUDA source and header that holds kernels or device
    functions, with comments and blank lines removed, the device declarations of the host-only
    sources, the ATTN_ constants of the C header, and the flags.  Kernel profiles stay valid
    while it is unchanged: edits to comments, to host-side entry points or to declarations do
    not change it.  `read(path)` returns a file's text (default: the working tree)."""
    import re
    read = read or (lambda path: open(path).read())

    def strip(text):
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        return [ln.rstrip() for ln in text.splitlines() if ln.strip()]

    h = hashlib.sha256()
    h.update(" ".join(_portable_flags()).encode())
    for name in sorted(os.listdir(CSRC)):
        if not name.endswith((".cu", ".cuh", ".h")):
            continue
        lines = strip(read(os.path.join(CSRC, name)))
        if name in HOST_SOURCES:
            lines = [ln for ln in lines if "__device__" in ln or "__global__" in ln]
        h.update(name.encode())
        h.update("\n".join(lines).encode())
    for name in sorted(os.listdir(INCLUDE)):
        if name.endswith(".h"):
            lines = [ln for ln in strip(read(os.path.join(INCLUDE, name))) if re.search(r"\bATTN_\w+\s*(=|\d)", ln)]
            h.update(name.encode())
            h.update("\n".join(lines).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every translation unit and link the shared library; returns its path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    stamp_path = os.path.join(BUILD_DIR, "stamp")
    stamp = _stamp()
    if not force and os.path.exists(LIB_PATH) and os.path.exists(stamp_path):
        with open(stamp_path) as f:
            if f.read() == stamp:
                return LIB_PATH
    cc = nvcc()

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        cmd = [cc, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    with open(stamp_path, "w") as f:
        f.write(stamp)
    return LIB_PATH


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
