"""Python binding of the GB300 (sm_103a) attention forward library.

Argument marshalling only: every step of the computation runs in the CUDA kernels
behind the C ABI of ``include/fa.h`` (libfa_sm103.so).  The materialised baseline,
``fa_fwd_materialised``, lives in a separate library (``include/fa_baseline.h``,
libfa_baseline.so, linked with cuBLAS) loaded only when it is called.  PyTorch supplies
device memory and the stream.  There is no fallback: if a compiled library cannot be
loaded, every call into it raises.
"""
from __future__ import annotations

import ctypes
import math
import threading

from . import build as _build

__all__ = ["fa_fwd", "fa_fwd_raw", "fa_fwd_splitkv", "fa_fwd_splitkv_raw",
           "splitkv_workspace_bytes", "splitkv_auto_splits", "fa_fwd_splitkv_noalloc_raw",
           "noalloc_scratch_bytes", "fa_fwd_materialised", "fa_fwd_materialised_raw",
           "materialised_workspace_bytes", "get_device_status", "strerror", "last_error", "version",
           "load_library", "load_baseline_library", "row_kernel_register_check",
           "override_kernel_registers_for_test", "FAError", "FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED",
           "FA_ERR_MISALIGNED", "FA_ERR_ARCH", "FA_ERR_CUDA", "FA_ERR_DEVICE_TIMEOUT",
           "FwdOptions", "SUPPORTED_HEAD_DIMS"]

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_MISALIGNED = 3
FA_ERR_ARCH = 4
FA_ERR_CUDA = 5
FA_ERR_DEVICE_TIMEOUT = 6
SUPPORTED_HEAD_DIMS = (16, 32, 64, 128, 256)
FA_KERNEL_AUTO = 0
FA_KERNEL_TWO_TILE = 1  # 256 query rows per work unit; head dims 16-128; split-KV
FA_KERNEL_ONE_TILE = 2  # 128 query rows per work unit; head dims 32 to 256
FA_ORDER_AUTO = 0
FA_ORDER_ONE_SNAKE = 1     # one snake over all work units
FA_ORDER_GROUP_SNAKES = 2  # a snake per head group, odd groups mirrored
FA_ORDER_SHIFTED_SNAKES = 3  # a snake per head group, each starting where the last left off


class FwdOptions(ctypes.Structure):
    """Mirror of ``fa_fwd_options``."""
    _fields_ = [("wait_budget_cycles", ctypes.c_int64),
                ("inject_skip_kv_load", ctypes.c_int32),
                ("max_ctas", ctypes.c_int32),
                ("kernel", ctypes.c_int32),
                ("order", ctypes.c_int32),
                ("block_kv", ctypes.c_int32)]


class FAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = last_error()
        super().__init__(f"{where}: {strerror(status)} (status {status})"
                         + (f": {detail}" if detail else ""))


class BaselineError(FAError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = load_baseline_library().fa_baseline_last_error().decode()
        RuntimeError.__init__(self, f"{where}: {strerror(status)} (status {status})"
                              + (f": {detail}" if detail else ""))


_lib = None
_baseline_lib = None
_lock = threading.Lock()


def load_library(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load (building first if needed) the in-tree libfa_sm103.so."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.build() if build_if_missing else _build.LIB_PATH
        lib = ctypes.CDLL(path)
        vp, i64 = ctypes.c_void_p, ctypes.c_int64
        sig = [vp, vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_int, ctypes.c_float, vp]
        lib.fa_fwd.argtypes = sig
        lib.fa_fwd.restype = ctypes.c_int
        lib.fa_fwd_opts.argtypes = sig + [ctypes.POINTER(FwdOptions)]
        lib.fa_fwd_opts.restype = ctypes.c_int
        lib.fa_strerror.argtypes = [ctypes.c_int]
        lib.fa_strerror.restype = ctypes.c_char_p
        lib.fa_last_error.argtypes = []
        lib.fa_last_error.restype = ctypes.c_char_p
        lib.fa_get_device_status.argtypes = [vp]
        lib.fa_get_device_status.restype = ctypes.c_int
        lib.fa_version.argtypes = []
        lib.fa_version.restype = ctypes.c_int
        lib.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_int,
                                       ctypes.c_float, ctypes.c_int, vp, ctypes.c_size_t, vp]
        lib.fa_fwd_splitkv.restype = ctypes.c_int
        lib.fa_fwd_splitkv_opts.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_int,
                                            ctypes.c_float, ctypes.c_int, vp, ctypes.c_size_t, vp,
                                            ctypes.POINTER(FwdOptions)]
        lib.fa_fwd_splitkv_opts.restype = ctypes.c_int
        lib.fa_splitkv_workspace_bytes.argtypes = [i64, i64, i64, i64, ctypes.c_int]
        lib.fa_splitkv_workspace_bytes.restype = ctypes.c_int64
        lib.fa_splitkv_auto_splits.argtypes = [i64, i64, i64, ctypes.c_int]
        lib.fa_splitkv_auto_splits.restype = ctypes.c_int
        lib.fa_fwd_plan.argtypes = [i64, i64, i64, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int),
                                    ctypes.POINTER(ctypes.c_int)]
        lib.fa_fwd_plan.restype = ctypes.c_int
        lib.fa_fwd_splitkv_noalloc.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64,
                                               ctypes.c_int, ctypes.c_float, ctypes.c_int, vp]
        lib.fa_fwd_splitkv_noalloc.restype = ctypes.c_int
        lib.fa_noalloc_scratch_bytes.argtypes = []
        lib.fa_noalloc_scratch_bytes.restype = ctypes.c_int64
        lib.fa_row_kernel_register_check.argtypes = [ctypes.c_int, ctypes.c_int]
        lib.fa_row_kernel_register_check.restype = ctypes.c_int
        lib.fa_test_override_kernel_registers.argtypes = [ctypes.c_int]
        lib.fa_test_override_kernel_registers.restype = None
        _lib = lib
        return lib


def load_baseline_library(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load (building first if needed) the in-tree libfa_baseline.so (materialised path)."""
    global _baseline_lib
    with _lock:
        if _baseline_lib is not None:
            return _baseline_lib
        if build_if_missing:
            _build.build()
        lib = ctypes.CDLL(_build.BASELINE_LIB_PATH)
        vp, i64 = ctypes.c_void_p, ctypes.c_int64
        lib.fa_fwd_materialised.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_int,
                                            ctypes.c_float, vp, ctypes.c_size_t, vp]
        lib.fa_fwd_materialised.restype = ctypes.c_int
        lib.fa_materialised_workspace_bytes.argtypes = [i64, i64, i64, i64]
        lib.fa_materialised_workspace_bytes.restype = ctypes.c_int64
        lib.fa_baseline_last_error.argtypes = []
        lib.fa_baseline_last_error.restype = ctypes.c_char_p
        _baseline_lib = lib
        return lib


def row_kernel_register_check(num_regs: int, max_threads_per_block: int) -> int:
    """The two-tile kernel's launch check on its compiled register allocation (pure)."""
    return int(load_library().fa_row_kernel_register_check(int(num_regs), int(max_threads_per_block)))


def override_kernel_registers_for_test(num_regs: int) -> None:
    """Test hook: launches of the two-tile kernel check `num_regs` instead of the compiled
    register count while it is > 0; 0 restores normal operation."""
    load_library().fa_test_override_kernel_registers(int(num_regs))


def strerror(status: int) -> str:
    return load_library().fa_strerror(int(status)).decode()


def last_error() -> str:
    return load_library().fa_last_error().decode()


def version() -> int:
    return int(load_library().fa_version())


def fa_fwd_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int, B: int, H: int,
               N: int, d: int, causal: bool, scale: float, stream: int = 0,
               options: FwdOptions | None = None) -> int:
    """Call the C entry point with raw device addresses; returns the status code."""
    lib = load_library()
    args = (q_ptr or None, k_ptr or None, v_ptr or None, o_ptr or None, lse_ptr or None,
            int(B), int(H), int(N), int(d), int(bool(causal)), float(scale), stream or None)
    if options is None:
        return int(lib.fa_fwd(*args))
    return int(lib.fa_fwd_opts(*args, ctypes.byref(options)))


def _stream_handle(stream, device) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream)


def fa_fwd(q, k, v, o=None, lse=None, causal: bool = True, scale: float | None = None,
           want_lse: bool = True, stream=None, options: FwdOptions | None = None):
    """O = softmax(scale * q k^T + mask) v and its row logsumexp, on the GPU.

    q, k, v : CUDA bf16 tensors [B, H, N, d], contiguous, d in {16, 32, 64, 128, 256}.
    o, lse  : optional outputs ([B, H, N, d] bf16, [B, H, N] fp32); allocated if None.
    scale   : defaults to 1/sqrt(d), rounded to fp32.
    Returns (o, lse) (lse is None when ``want_lse`` is False and none was given).
    """
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.bfloat16:
            raise TypeError(f"{name} must be a CUDA bf16 tensor")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [B, H, N, d] tensor")
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k and v must have the same shape")
    B, H, N, d = q.shape
    if scale is None:
        scale = float(torch.tensor(1.0 / math.sqrt(d), dtype=torch.float32))
    if o is None:
        o = torch.empty_like(q)
    elif o.shape != q.shape or o.dtype != torch.bfloat16 or not o.is_contiguous() or not o.is_cuda:
        raise ValueError("o must be a contiguous CUDA bf16 tensor shaped like q")
    if lse is None and want_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    elif lse is not None and (tuple(lse.shape) != (B, H, N) or lse.dtype != torch.float32
                              or not lse.is_contiguous() or not lse.is_cuda):
        raise ValueError("lse must be a contiguous CUDA fp32 tensor [B, H, N]")
    rc = fa_fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                    lse.data_ptr() if lse is not None else 0, B, H, N, d, causal, scale,
                    _stream_handle(stream, q.device), options)
    if rc != FA_OK:
        raise FAError(rc, "fa_fwd")
    return o, lse


def splitkv_workspace_bytes(B: int, H: int, N: int, d: int, splits: int) -> int:
    return int(load_library().fa_splitkv_workspace_bytes(B, H, N, d, splits))


def splitkv_auto_splits(B: int, H: int, N: int, causal: bool = True) -> int:
    return int(load_library().fa_splitkv_auto_splits(B, H, N, int(bool(causal))))


def fwd_plan(B: int, H: int, N: int, d: int, causal: bool = True, allow_split: bool = False,
             num_sms: int = 0, with_order: bool = False):
    """(kernel, splits) the library picks for these sizes (fa_fwd_plan), or
    (kernel, splits, order) with ``with_order``.

    allow_split=False gives fa_fwd's choice, True that of fa_fwd_splitkv with splits=0.
    num_sms=0 asks the current device; a positive count plans without touching CUDA.
    """
    kernel, splits, order = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    rc = load_library().fa_fwd_plan(int(B), int(H), int(N), int(d), int(bool(causal)),
                                    int(bool(allow_split)), int(num_sms), ctypes.byref(kernel),
                                    ctypes.byref(splits), ctypes.byref(order))
    if rc != FA_OK:
        raise FAError(rc, "fa_fwd_plan")
    if with_order:
        return kernel.value, splits.value, order.value
    return kernel.value, splits.value


def fa_fwd_splitkv_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, N, d, causal, scale, splits,
                       ws_ptr, ws_bytes, stream: int = 0, options: FwdOptions | None = None) -> int:
    """Call fa_fwd_splitkv (fa_fwd_splitkv_opts with ``options``) with raw device
    addresses; returns the status code."""
    lib = load_library()
    args = (q_ptr or None, k_ptr or None, v_ptr or None, o_ptr or None, lse_ptr or None, int(B),
            int(H), int(N), int(d), int(bool(causal)), float(scale), int(splits), ws_ptr or None,
            int(ws_bytes), stream or None)
    if options is None:
        return int(lib.fa_fwd_splitkv(*args))
    return int(lib.fa_fwd_splitkv_opts(*args, ctypes.byref(options)))


def fa_fwd_splitkv(q, k, v, o=None, lse=None, causal: bool = True, scale: float | None = None,
                   splits: int = 0, workspace=None, stream=None, options: FwdOptions | None = None):
    """fa_fwd with each query block's key range split across CTAs and merged by lse.

    splits = 0 lets the library choose.  ``workspace`` (a CUDA uint8 tensor) is
    allocated here when not given.  ``options`` may pin the kernel (with splits >= 1)
    and the unit order.  Returns (o, lse).
    """
    import torch
    B, H, N, d = q.shape
    if scale is None:
        scale = float(torch.tensor(1.0 / math.sqrt(d), dtype=torch.float32))
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    # splits = 0: the library plans the launch (kernel and pieces) itself; the workspace
    # is sized for the pieces that plan takes
    use = splits if splits > 0 else fwd_plan(B, H, N, d, causal, allow_split=True)[1]
    need = splitkv_workspace_bytes(B, H, N, d, use) if use > 1 else 0
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else 0
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.bfloat16 \
                or not t.is_contiguous() or t.shape != q.shape:
            raise TypeError(f"{name} must be a contiguous CUDA bf16 tensor shaped like q")
    rc = fa_fwd_splitkv_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                            lse.data_ptr(), B, H, N, d, causal, scale, splits, ws_ptr, ws_bytes,
                            _stream_handle(stream, q.device), options)
    if rc != FA_OK:
        raise FAError(rc, "fa_fwd_splitkv")
    return o, lse


def fa_fwd_splitkv_noalloc_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, N, d, causal, scale,
                               splits, stream: int = 0) -> int:
    """Split-KV forward using the library's built-in scratch (no workspace, no
    allocation); raw device addresses in, status code out."""
    lib = load_library()
    return int(lib.fa_fwd_splitkv_noalloc(q_ptr or None, k_ptr or None, v_ptr or None,
                                          o_ptr or None, lse_ptr or None, int(B), int(H), int(N),
                                          int(d), int(bool(causal)), float(scale), int(splits),
                                          stream or None))


def noalloc_scratch_bytes() -> int:
    return int(load_library().fa_noalloc_scratch_bytes())


def materialised_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(load_baseline_library().fa_materialised_workspace_bytes(B, H, N, d))


def fa_fwd_materialised_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, N, d, causal, scale,
                            ws_ptr, ws_bytes, stream: int = 0) -> int:
    """Call fa_fwd_materialised with raw device addresses; returns the status code."""
    lib = load_baseline_library()
    return int(lib.fa_fwd_materialised(q_ptr or None, k_ptr or None, v_ptr or None, o_ptr or None,
                                       lse_ptr or None, int(B), int(H), int(N), int(d),
                                       int(bool(causal)), float(scale), ws_ptr or None,
                                       int(ws_bytes), stream or None))


def fa_fwd_materialised(q, k, v, o=None, lse=None, causal: bool = True,
                        scale: float | None = None, workspace=None, stream=None):
    """The materialised baseline (N x N scores and probabilities in device memory).

    ``workspace`` (a CUDA uint8 tensor of at least materialised_workspace_bytes) is
    allocated here when not given.  Returns (o, lse).
    """
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.bfloat16 \
                or t.dim() != 4 or not t.is_contiguous() or t.shape != q.shape:
            raise TypeError(f"{name} must be a contiguous CUDA bf16 tensor shaped like q")
    B, H, N, d = q.shape
    if scale is None:
        scale = float(torch.tensor(1.0 / math.sqrt(d), dtype=torch.float32))
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    need = materialised_workspace_bytes(B, H, N, d)
    if need < 0:
        raise BaselineError(FA_ERR_UNSUPPORTED, "fa_fwd_materialised")
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    rc = fa_fwd_materialised_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), B, H, N, d, causal, scale, workspace.data_ptr(),
                                 workspace.numel() * workspace.element_size(),
                                 _stream_handle(stream, q.device))
    if rc != FA_OK:
        raise BaselineError(rc, "fa_fwd_materialised")
    return o, lse


def get_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status (FA_OK or a timeout)."""
    import torch
    handle = _stream_handle(stream, torch.cuda.current_device())
    return int(load_library().fa_get_device_status(handle or None))
