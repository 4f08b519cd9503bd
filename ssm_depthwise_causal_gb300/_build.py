"""Builds libccc.so (the CUDA library behind include/ccc.h) in-tree.

Each .cu translation unit is compiled by nvcc for sm_103a in parallel, then
linked into ``ssm_depthwise_causal_gb300/libccc.so`` with the CUDA runtime
linked statically (the library needs no libcudart on the loader path).
Objects go to ``ssm_depthwise_causal_gb300/_build/``; a unit is recompiled when
it, a header, or the flags changed.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libccc.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
                     f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libccc.so")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return sorted(hs)


def _stamp(src: str, extra: list[str]) -> str:
    h = hashlib.sha256()
    for p in [src] + _headers():
        with open(p, "rb") as f:
            h.update(f.read())
    h.update(" ".join(NVCC_FLAGS + extra).encode())
    return h.hexdigest()


def _compile(src: str, extra: list[str], verbose: bool, build_dir: str = BUILD) -> str:
    obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
    stamp_path = obj + ".stamp"
    stamp = _stamp(src, extra)
    if os.path.exists(obj) and os.path.exists(stamp_path) and open(stamp_path).read() == stamp:
        return obj
    cmd = [nvcc()] + NVCC_FLAGS + extra + ["-c", src, "-o", obj]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    if verbose and r.stderr.strip():
        print(r.stderr, flush=True)
    with open(stamp_path, "w") as f:
        f.write(stamp)
    return obj


def build(verbose: bool = False, extra_flags: list[str] | None = None, lib_path: str = LIB,
          build_dir: str = BUILD) -> str:
    """Compile every CUDA unit and link the library (by default
    ssm_depthwise_causal_gb300/libccc.so); returns its path.  `extra_flags`
    (e.g. -DCCC_BWD_UNROLL=8) with another `lib_path` / `build_dir` builds a
    variant beside the default one."""
    extra = list(extra_flags or [])
    # Optional extra defines for experiments, e.g.
    # CCC_EXTRA_NVCC_FLAGS="-DCCC_BWD_UNROLL=2"; unset in normal builds.
    extra += os.environ.get("CCC_EXTRA_NVCC_FLAGS", "").split()
    os.makedirs(build_dir, exist_ok=True)
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, verbose, build_dir), srcs))
    newest = max(os.path.getmtime(o) for o in objs)
    LIB_OUT = lib_path
    if not os.path.exists(LIB_OUT) or os.path.getmtime(LIB_OUT) < newest:
        tmp = LIB_OUT + f".tmp{os.getpid()}"
        cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of libccc.so failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB_OUT)
    return LIB_OUT


if __name__ == "__main__":
    print(build(verbose=True))
