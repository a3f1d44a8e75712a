"""Build the sm_103a C-ABI libraries in-tree with nvcc (one -gencode, compiled in parallel).

libfa_sm103.so    the tiled forward pass (include/fa.h): csrc/fa_api.cu and the kernels.
libfa_baseline.so the materialised baseline (include/fa_baseline.h): csrc/fa_baseline.cu,
                  linked with cuBLAS, which the forward library does not link.

ptxas reports every kernel's register allocation (-Xptxas -v).  The two-tile kernel
(fa_fwd_row_kernel) moves registers between its warpgroups with setmaxnreg and needs the
allocation its split is written for; the build fails if ptxas reports another count,
before any GPU could meet the unbounded setmaxnreg wait.  (The library checks the same
thing again at run time with cudaFuncGetAttributes.)
"""
from __future__ import annotations

import os
import re
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
OUT_DIR = os.path.join(PKG_DIR, "_build")
LIB_NAME = "libfa_sm103.so"
LIB_PATH = os.path.join(OUT_DIR, LIB_NAME)
BASELINE_LIB_PATH = os.path.join(OUT_DIR, "libfa_baseline.so")
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
# registers per thread the two-tile kernel's setmaxnreg split is written for
ROW_KERNEL_REGS = 128


def _csrc(*names):
    return [os.path.join(CSRC, n) for n in names]


# library -> (sources, files whose change triggers a rebuild, extra link flags)
TARGETS = {
    LIB_PATH: (_csrc("fa_api.cu"),
               _csrc("fa_api.cu", "fa_fwd_kernel.cuh", "ptx_sm103.cuh", "fa_merge_kernel.cuh",
                     "fa_fwd_1tile_kernel.cuh", "fa_fwd_row_kernel.cuh")
               + [os.path.join(ROOT, "include", "fa.h")], []),
    BASELINE_LIB_PATH: (_csrc("fa_baseline.cu"),
                        _csrc("fa_baseline.cu", "fa_materialised_kernel.cuh")
                        + [os.path.join(ROOT, "include", "fa.h"),
                           os.path.join(ROOT, "include", "fa_baseline.h")], ["-lcublas"]),
}


def nvcc_path() -> str:
    for cand in (os.environ.get("CUDA_HOME"), os.environ.get("CUDA_PATH"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return os.path.join(cand, "bin", "nvcc")
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found: the sm_103a library cannot be built")
    return found


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = TARGETS[lib][1] + [os.path.abspath(__file__)]
    return any(os.path.getmtime(p) > t for p in deps)


def is_stale() -> bool:
    return any(_stale(lib) for lib in TARGETS)


def kernel_registers(ptxas_log: str) -> dict:
    """Registers per thread of every kernel in a `-Xptxas -v` log: {mangled name: count}."""
    regs, current = {}, None
    for line in ptxas_log.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            current = m.group(1)
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and current is not None:
            regs[current] = int(m.group(1))
            current = None
    return regs


def check_row_kernel_registers(ptxas_log: str) -> None:
    """Fail unless every fa_fwd_row_kernel instantiation got ROW_KERNEL_REGS registers."""
    regs = {k: v for k, v in kernel_registers(ptxas_log).items() if "fa_fwd_row_kernel" in k}
    if not regs:
        raise RuntimeError("ptxas reported no fa_fwd_row_kernel instantiation")
    bad = {k: v for k, v in regs.items() if v != ROW_KERNEL_REGS}
    if bad:
        raise RuntimeError(
            "fa_fwd_row_kernel must be compiled to exactly %d registers per thread (its "
            "setmaxnreg split hands out 512 x %d); ptxas gave %s" % (ROW_KERNEL_REGS, ROW_KERNEL_REGS, bad))


def _compile(lib: str, verbose: bool) -> str:
    sources, _, link = TARGETS[lib]
    tmp = lib + f".{os.getpid()}.tmp"
    cmd = [nvcc_path(), *ARCH_FLAGS, "-O3", "-std=c++17", "-lineinfo", "-Xptxas", "-v",
           "-Xcompiler", "-fPIC", "-shared", "-o", tmp, *sources, *link]
    res = subprocess.run(cmd, capture_output=True, text=True)
    log = res.stdout + res.stderr
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + log)
    if lib == LIB_PATH:
        try:
            check_row_kernel_registers(log)
        except RuntimeError:
            os.remove(tmp)
            raise
    if verbose:
        print(log)
    os.replace(tmp, lib)
    return log


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile csrc/ into _build/ (each library skipped when up to date).  Returns the
    forward library's path."""
    os.makedirs(OUT_DIR, exist_ok=True)
    todo = [lib for lib in TARGETS if force or _stale(lib)]
    if todo:
        with ThreadPoolExecutor(len(todo)) as ex:
            list(ex.map(lambda lib: _compile(lib, verbose), todo))
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
