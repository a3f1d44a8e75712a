"""CPU fp64 oracle for the FlashAttention forward pass -- TEST INFRASTRUCTURE ONLY.

Only the tests, the package's ``smoke()`` check and the benchmark's CPU-baseline /
reference legs import this package.  The product path (the C-ABI library and its
Python binding) never imports, links or runs anything here, and this package
imports nothing from the product.

* ``attn_rows``      materialised fp64 attention for chosen query rows (C, threaded)
* ``ref``            page-style fp64 restatements (dense, tiled, traffic models)

Every function here is pinned by ``tests/test_oracle.py`` to values the pages
print, closed forms, invariants and brute force (no function is parity-unpinned).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libattn_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (portable flags, no FP contraction). Returns the .so path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_attn_rows.restype = ctypes.c_int
            lib.oracle_attn_rows.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.oracle_default_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def default_threads() -> int:
    return int(_load().oracle_default_threads())


def _as_heads(x):
    """Accept a torch bf16 tensor, a uint16 bit array or a float64 array; return (array, kind)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            if x.dtype == torch.bfloat16:
                bits = x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
                return bits, 1
            return x.detach().cpu().to(torch.float64).contiguous().numpy(), 0
    except ImportError:  # pragma: no cover
        pass
    a = np.asarray(x)
    if a.dtype == np.uint16:
        return np.ascontiguousarray(a), 1
    return np.ascontiguousarray(a, dtype=np.float64), 0


def attn_rows(q, k, v, rows, causal: bool, scale: float, nthreads: int = 0):
    """fp64 attention output and logsumexp for selected query rows.

    q, k, v : [..., N, d] (leading dims flattened to heads); torch bf16 tensors or
              uint16 bf16 bits are widened exactly, anything else is taken as float64.
    rows    : int array of (bh, i) pairs, bh indexing the flattened heads.
    Returns (o [len(rows), d] float64, lse [len(rows)] float64).
    """
    qa, kind = _as_heads(q)
    ka, kk = _as_heads(k)
    va, vk = _as_heads(v)
    if not (kind == kk == vk):
        raise TypeError("q, k and v must share one element type")
    N, d = qa.shape[-2], qa.shape[-1]
    BH = int(np.prod(qa.shape[:-2])) if qa.ndim > 2 else 1
    for a in (ka, va):
        if a.shape != qa.shape:
            raise ValueError("q, k and v must have one shape")
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 2))
    n = rows.shape[0]
    o = np.empty((n, d), dtype=np.float64)
    lse = np.empty(n, dtype=np.float64)
    rc = _load().oracle_attn_rows(
        qa.ctypes.data, ka.ctypes.data, va.ctypes.data, kind, BH, N, d,
        rows.ctypes.data, n, int(bool(causal)), float(scale),
        o.ctypes.data, lse.ctypes.data, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_rows failed with code {rc}")
    return o, lse


def attn_full(q, k, v, causal: bool, scale: float, nthreads: int = 0):
    """Every row of every head: (o [BH, N, d], lse [BH, N])."""
    qa, _ = _as_heads(q)
    N, d = qa.shape[-2], qa.shape[-1]
    BH = int(np.prod(qa.shape[:-2])) if qa.ndim > 2 else 1
    bh, i = np.meshgrid(np.arange(BH), np.arange(N), indexing="ij")
    rows = np.stack([bh.ravel(), i.ravel()], axis=1)
    o, lse = attn_rows(q, k, v, rows, causal, scale, nthreads)
    return o.reshape(BH, N, d), lse.reshape(BH, N)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 (ties to even), returned as float64.

    Used to state the representability floor of a bf16 output: the error that
    rounding the exact answer alone would make.  Goes through float32 first only
    when that is exact for the bf16 decision (values already in fp32 range).
    """
    a = np.asarray(x, dtype=np.float64)
    f = a.astype(np.float32)
    # correct the double rounding f64->f32->bf16: decide on the f64 value directly
    u = f.view(np.uint32).astype(np.uint64)
    lo = (u & 0xFFFF0000).astype(np.uint32).view(np.float32).astype(np.float64)
    hi_bits = ((u & 0xFFFF0000) + 0x10000).astype(np.uint32)
    hi = hi_bits.view(np.float32).astype(np.float64)
    # candidates are the two bf16 neighbours bracketing |a| (same sign as a)
    lo_err = np.abs(a - lo)
    hi_err = np.abs(a - hi)
    even_lo = ((u >> 16) & 1) == 0
    pick_hi = (hi_err < lo_err) | ((hi_err == lo_err) & ~even_lo)
    out = np.where(pick_hi, hi, lo)
    return np.where(np.isfinite(a), out, a)
