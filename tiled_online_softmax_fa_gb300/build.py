"""Build the sm_103a C-ABI library in-tree with nvcc (one translation unit, one -gencode)."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
OUT_DIR = os.path.join(PKG_DIR, "_build")
LIB_NAME = "libfa_sm103.so"
LIB_PATH = os.path.join(OUT_DIR, LIB_NAME)
SOURCES = [os.path.join(CSRC, "fa_api.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, "fa_fwd_kernel.cuh"), os.path.join(CSRC, "ptx_sm103.cuh"),
                     os.path.join(CSRC, "fa_merge_kernel.cuh"), os.path.join(CSRC, "fa_fwd_1tile_kernel.cuh"),
                     os.path.join(CSRC, "fa_fwd_row_kernel.cuh"),
                     os.path.join(CSRC, "fa_materialised_kernel.cuh"),
                     os.path.join(ROOT, "include", "fa.h"), os.path.abspath(__file__)]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (os.environ.get("CUDA_HOME"), os.environ.get("CUDA_PATH"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return os.path.join(cand, "bin", "nvcc")
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found: the sm_103a library cannot be built")
    return found


def is_stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(p) > t for p in DEPENDS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile csrc/ into _build/libfa_sm103.so (skipped when up to date). Returns the path."""
    if not force and not is_stale():
        return LIB_PATH
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB_PATH + f".{os.getpid()}.tmp"
    cmd = [nvcc_path(), *ARCH_FLAGS, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
           "-shared", "-o", tmp, *SOURCES, "-lcublas"]
    if verbose:
        cmd[1:1] = ["-Xptxas", "-v"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + res.stdout + res.stderr)
    if verbose:
        print(res.stdout + res.stderr)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
