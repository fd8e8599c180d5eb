"""Builds libfatattn.so (the CUDA library behind include/fat_attn.h) in-tree with nvcc for
sm_103a. Translation units compile in parallel; the link uses nvcc with the static CUDA runtime."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OBJ_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(PKG, "libfatattn.so")
SOURCES = ["fat_attn_api.cu", "fat_attn_fwd.cu", "fat_attn_bwd.cu", "fat_attn_decode.cu",
           "fat_attn_noalloc.cu", "fat_rope.cu", "fat_norm_ce.cu"]
HEADERS = ["sm103_ptx.cuh", "fat_attn_internal.cuh"]
PUBLIC_HEADERS = [os.path.join(ROOT, "include", h) for h in ("fat_attn.h", "fat_attn_debug.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfatattn.so")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, log_dir: str) -> str:
    obj = os.path.join(OBJ_DIR, src.replace(".cu", ".o"))
    deps = [os.path.join(CSRC, src)] + [os.path.join(CSRC, h) for h in HEADERS] + PUBLIC_HEADERS
    if not _stale(obj, deps):
        return obj
    cmd = [nvcc()] + ARCH + FLAGS + ["-c", os.path.join(CSRC, src), "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    with open(os.path.join(log_dir, src + ".log"), "w") as f:
        f.write(" ".join(cmd) + "\n" + res.stdout + res.stderr)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{res.stderr[-4000:]}")
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(OBJ_DIR, exist_ok=True)
    if force:
        for s in SOURCES:
            o = os.path.join(OBJ_DIR, s.replace(".cu", ".o"))
            if os.path.exists(o):
                os.remove(o)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, OBJ_DIR), SOURCES))
    if force or _stale(LIB_PATH, objs):
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stderr[-4000:]}")
        os.replace(tmp, LIB_PATH)
    if verbose:
        for s in SOURCES:
            p = os.path.join(OBJ_DIR, s + ".log")
            if os.path.exists(p):
                print(open(p).read())
    return LIB_PATH


if __name__ == "__main__":
    print(build(verbose=True))
