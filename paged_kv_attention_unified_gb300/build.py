"""Build libua.so (the C-ABI library) in-tree with nvcc for sm_103a.

Every translation unit is compiled in parallel, then linked into one shared
library next to this file. A hash of the sources and flags is stored beside
the library; an unchanged tree is not rebuilt.
"""
from __future__ import annotations

import concurrent.futures
import hashlib
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libua.so")
STAMP = LIB + ".hash"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "--expt-relaxed-constexpr", "-I" + INCLUDE, "-I" + CSRC]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found (CUDA 13 toolkit required)")
    return cand


def sources():
    out = []
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cpp")):
            out.append(os.path.join(CSRC, name))
    return out


_SOURCE_SUFFIXES = (".cu", ".cuh", ".cpp", ".h")


# What a kernel's DRAM traffic depends on: its own source, the shared device
# headers, the scheduler (the tiles it launches) and the TMA map encoding.
_KERNEL_SOURCES = {
    "decode": ("decode.cu",),
    "prefill": ("prefill.cu",),
    "prefill_wide": ("prefill_wide.cu",),
    "append": ("append.cu",),
    "stage": ("stage.cu",),
}
_SHARED_SOURCES = ("sm100.cuh", "ua_device.cuh", "ua_kernels.h", "tma_host.cu", "planner.cpp",
                   "planner.h", "ua.h")


def kernel_digest(kernel: str) -> str:
    """Digest of the code one kernel's DRAM traffic depends on (committed ncu
    traffic records are keyed by it); comments do not count."""
    return _digest(only=_KERNEL_SOURCES[kernel] + _SHARED_SOURCES, code_only=True)


def _strip_comments(text: str) -> str:
    """C / C++ source without its comments (string and character literals
    kept as they are)."""
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
    return "".join(out)


def _digest(extra=(), only=None, code_only=False):
    """Hash of the library's sources (by file name, not path) and its compile
    flags with the include paths taken out: the same tree gives the same
    digest wherever it is checked out. only: restrict to these file names;
    code_only: hash the sources without their comments."""
    h = hashlib.sha256()
    files = [(f, CSRC) for f in os.listdir(CSRC)] + [(f, INCLUDE) for f in os.listdir(INCLUDE)]
    for name, base in sorted(files):
        if not name.endswith(_SOURCE_SUFFIXES) or (only is not None and name not in only):
            continue
        with open(os.path.join(base, name), "rb") as fh:
            data = fh.read()
        if code_only:
            data = _strip_comments(data.decode("utf-8")).encode("utf-8")
        h.update(name.encode())
        h.update(data)
    h.update(" ".join(f for f in NVCC_FLAGS if not f.startswith("-I")).encode())
    for e in extra:
        h.update(str(e).encode())
    return h.hexdigest()


def build(verbose: bool = False, force: bool = False) -> str:
    """Compile and link libua.so; return its path."""
    digest = _digest()
    if not force and os.path.exists(LIB) and os.path.exists(STAMP):
        with open(STAMP) as f:
            if f.read().strip() == digest:
                return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.basename(src) + ".o")
        cmd = [nvcc] + NVCC_FLAGS + ["-c", src, "-o", obj]
        if src.endswith(".cpp"):
            cmd = [nvcc, "-x", "c++"] + NVCC_FLAGS[len(ARCH):] + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    srcs = sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = LIB + ".tmp"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(digest)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True, force="--force" in sys.argv))
