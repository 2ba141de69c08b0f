"""Build libkvq.so (the CUDA kernels + C ABI) in-tree for sm_103a.

Each translation unit is compiled by nvcc in parallel, then linked into
``bit_quantized_kv_store_gb300/_build/libkvq.so``.  A unit is rebuilt only when
its source or a header is newer than its object file.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
# KVQ_SANITIZE=1: a separate build of the host code with AddressSanitizer and
# UndefinedBehaviorSanitizer, for checking the C ABI's argument validation on
# the CPU (device code as PTX only: that build never launches a kernel).
SANITIZE = os.environ.get("KVQ_SANITIZE") == "1"
BUILD = os.path.join(PKG, "_build_san" if SANITIZE else "_build")
LIB = os.path.join(BUILD, "libkvq.so")

ARCH = ["-gencode", "arch=compute_103a,code=compute_103a" if SANITIZE else "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", f"-I{os.path.join(ROOT, 'include')}"]
SAN_FLAGS = ["-Xcompiler", "-fsanitize=address", "-Xcompiler", "-fsanitize=undefined",  # (-Xcompiler splits at commas)
             "-Xcompiler", "-fno-sanitize-recover=undefined", "-Xcompiler", "-fno-omit-frame-pointer"]
if SANITIZE:
    FLAGS = FLAGS + SAN_FLAGS
# The store computes codes that must be bit-exact: no fused multiply-adds there.
PER_FILE = {"store.cu": ["-fmad=false"], "tq4.cu": ["-fmad=false"]}


def _tool_env():
    """The environment for the compilers: without a preloaded sanitizer runtime
    (a sanitized test process preloads one, and nvcc's own tools crash under it)."""
    return {k: v for k, v in os.environ.items() if k != "LD_PRELOAD"}


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers_mtime():
    hs = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(ROOT, "include", "*.h"))
    return max(os.path.getmtime(h) for h in hs)


def _compile(src, verbose_ptxas=False):
    obj = os.path.join(BUILD, os.path.basename(src).replace(".cu", ".o"))
    if os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(src), _headers_mtime()):
        return obj, ""
    cmd = [_nvcc(), *ARCH, *FLAGS, *PER_FILE.get(os.path.basename(src), []), "-c", src, "-o", obj + ".tmp"]
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True, env=_tool_env())
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    os.replace(obj + ".tmp", obj)
    return obj, r.stderr


def build(verbose_ptxas=False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose_ptxas), srcs))
    objs = [o for o, _ in results]
    if verbose_ptxas:
        for _, log in results:
            if log:
                print(log)
    if not os.path.exists(LIB) or os.path.getmtime(LIB) < max(os.path.getmtime(o) for o in objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp, *objs, *(SAN_FLAGS if SANITIZE else [])]
        r = subprocess.run(cmd, capture_output=True, text=True, env=_tool_env())
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(verbose_ptxas="-v" in sys.argv))
