"""Compile libattnmask.so in-tree with nvcc for sm_103a.

Each .cu translation unit is compiled in parallel, then linked into one
shared library next to this file.  Objects go to ``_build/`` (not tracked).
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB_NAME = "libattnmask.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)

SOURCES = ["api.cu", "blockmask.cu", "blockmask_noalloc.cu", "attn_fwd_bf16.cu", "attn_fwd_f32.cu",
           "attn_bwd_bf16.cu"]
HEADERS = ["common.cuh", "ptx.cuh", "tile_pipeline.cuh"]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-lineinfo", "-O3", "-std=c++17",
    "--expt-relaxed-constexpr",
    "-Xcompiler", "-fPIC,-fvisibility=hidden",
    "-I" + INCLUDE, "-I" + CSRC,
]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libattnmask")


def _inputs():
    return ([os.path.join(CSRC, s) for s in SOURCES + HEADERS] +
            [os.path.join(INCLUDE, "attn_block_mask.h"), os.path.abspath(__file__)])


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(p) > t for p in _inputs())


def _compile_and_link(out_path: str, obj_dir: str, extra_flags=(), verbose: bool = False) -> str:
    nvcc = _nvcc()
    os.makedirs(obj_dir, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *NVCC_FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
        if verbose and (res.stdout or res.stderr):
            sys.stderr.write(res.stdout + res.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = out_path + ".tmp"
    cmd = [nvcc, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-o", tmp, *objs,
           "-lcudart"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Build the library if missing or out of date; return its path."""
    if not force and not _stale():
        return LIB_PATH
    return _compile_and_link(LIB_PATH, BUILD, extra_flags, verbose)


def build_variant(tag: str, defines: dict) -> str:
    """Build a copy of the library with extra preprocessor definitions (for
    tests of compile-time settings, e.g. a short pipeline-wait bound) as
    ``lib<name>_<tag>.so`` next to the regular one; return its path."""
    out = os.path.join(PKG, f"{os.path.splitext(LIB_NAME)[0]}_{tag}.so")
    if os.path.exists(out) and all(os.path.getmtime(p) <= os.path.getmtime(out) for p in _inputs()):
        return out
    flags = [f"-D{k}={v}" for k, v in sorted(defines.items())]
    return _compile_and_link(out, os.path.join(BUILD, tag), flags)


def ensure_built() -> str:
    return build(force=False)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else []))
