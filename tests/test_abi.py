"""Host-side checks of the C ABI that need no GPU: the library loads, exports every
function ``include/fa.h`` declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

import tiled_online_softmax_fa_gb300 as fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for fn in os.listdir(inc):
        if fn.endswith(".h"):
            with open(os.path.join(inc, fn)) as f:
                text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
            names |= set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", text))
    return sorted(names)


def test_library_builds_and_loads():
    lib = fa.load_library()
    assert isinstance(lib, ctypes.CDLL)
    assert fa.version() == 200


def test_every_declared_symbol_is_exported():
    names = _declared_functions()
    assert {"fa_fwd", "fa_fwd_opts", "fa_strerror", "fa_last_error", "fa_get_device_status",
            "fa_version", "fa_fwd_splitkv", "fa_splitkv_workspace_bytes",
            "fa_splitkv_auto_splits"} <= set(names)
    lib = fa.load_library()
    for name in names:
        assert hasattr(lib, name), name


def test_strerror_covers_every_status():
    for code in range(7):
        assert fa.strerror(code) and fa.strerror(code) != "unknown status"
    assert fa.strerror(99) == "unknown status"


def _call(**kw):
    args = dict(q_ptr=0x10000, k_ptr=0x20000, v_ptr=0x30000, o_ptr=0x40000, lse_ptr=0,
                B=1, H=1, N=128, d=64, causal=True, scale=0.125)
    args.update(kw)
    return fa.fa_fwd_raw(**args)


@pytest.mark.parametrize("kw,want", [
    (dict(B=-1), fa.FA_ERR_INVALID_ARG),
    (dict(N=-5), fa.FA_ERR_INVALID_ARG),
    (dict(d=48), fa.FA_ERR_UNSUPPORTED),
    (dict(d=512), fa.FA_ERR_UNSUPPORTED),
    (dict(d=192), fa.FA_ERR_UNSUPPORTED),
    (dict(q_ptr=0), fa.FA_ERR_INVALID_ARG),
    (dict(o_ptr=0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=-0.5), fa.FA_ERR_INVALID_ARG),
    (dict(q_ptr=0x10008), fa.FA_ERR_MISALIGNED),
    (dict(o_ptr=0x40002), fa.FA_ERR_MISALIGNED),
    (dict(lse_ptr=0x50002), fa.FA_ERR_MISALIGNED),
    (dict(o_ptr=0x10000 + 4096), fa.FA_ERR_INVALID_ARG),          # o overlaps q
    (dict(lse_ptr=0x40000 + 64), fa.FA_ERR_INVALID_ARG),          # lse overlaps o
    (dict(N=(1 << 30) + 1), fa.FA_ERR_UNSUPPORTED),
    (dict(B=1 << 20, H=1 << 12), fa.FA_ERR_UNSUPPORTED),
])
def test_argument_errors(kw, want):
    assert _call(**kw) == want
    assert fa.last_error() != ""


@pytest.mark.parametrize("kw", [dict(B=0), dict(H=0), dict(N=0),
                                dict(B=0, q_ptr=0, k_ptr=0, v_ptr=0, o_ptr=0)])
def test_empty_is_a_noop_without_cuda(kw):
    assert _call(**kw) == fa.FA_OK


def test_options_are_checked():
    opts = fa.FwdOptions(wait_budget_cycles=-1)
    assert _call(options=opts) == fa.FA_ERR_INVALID_ARG


def test_python_wrapper_rejects_cpu_tensors():
    torch = pytest.importorskip("torch")
    t = torch.zeros((1, 1, 8, 16), dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        fa.fa_fwd(t, t, t)


def test_splitkv_workspace_bytes():
    # 256-row units, per item 256 rows of (d fp32 partial O + 1 fp32 lse)
    units = 1 * 32 * (1024 // 256)
    assert fa.splitkv_workspace_bytes(1, 32, 1024, 128, 4) == units * 4 * 256 * (128 + 1) * 4
    assert fa.splitkv_workspace_bytes(1, 32, 1024, 128, 1) == 0
    assert fa.splitkv_workspace_bytes(1, 32, 1024, 48, 4) == -1
    assert fa.splitkv_workspace_bytes(1, 32, 1024, 128, 0) == -1
    assert fa.splitkv_workspace_bytes(0, 32, 1024, 128, 4) == 0
    assert fa.splitkv_workspace_bytes(1, 32, 1024, 256, 1) == 0
    # head dim 256 splits on the one-tile kernel: 128-row items, the same total rows
    assert fa.splitkv_workspace_bytes(1, 32, 1024, 256, 4) == units * 4 * 256 * (256 + 1) * 4


def _split(**kw):
    args = dict(q_ptr=0x10000, k_ptr=0x20000, v_ptr=0x30000, o_ptr=0x40000, lse_ptr=0, B=1, H=1,
                N=128, d=64, causal=True, scale=0.1, splits=3, ws_ptr=0x100000, ws_bytes=10 ** 9)
    args.update(kw)
    return fa.fa_fwd_splitkv_raw(**args)


@pytest.mark.parametrize("kw,want", [
    (dict(ws_ptr=0), fa.FA_ERR_INVALID_ARG),
    (dict(ws_bytes=100), fa.FA_ERR_INVALID_ARG),
    (dict(ws_ptr=0x100008), fa.FA_ERR_MISALIGNED),
    (dict(splits=65), fa.FA_ERR_INVALID_ARG),
    (dict(splits=-1), fa.FA_ERR_INVALID_ARG),
    (dict(ws_ptr=0x20000), fa.FA_ERR_INVALID_ARG),      # workspace overlaps k
    (dict(d=40), fa.FA_ERR_UNSUPPORTED),
])
def test_splitkv_argument_errors(kw, want):
    assert _split(**kw) == want
    assert fa.last_error() != ""


def test_materialised_workspace_bytes():
    def r256(x):
        return (x + 255) // 256 * 256
    # fp32 S | bf16 P ([B*H, N, N]) | fp32 acc [B*H, N, d] | fp32 row sums [B*H, N]
    for B, H, N, d in ((1, 32, 1024, 128), (8, 32, 8192, 128), (2, 3, 129, 16)):
        BH = B * H
        want = r256(BH * N * N * 4) + r256(BH * N * N * 2) + r256(BH * N * d * 4) + r256(BH * N * 4)
        assert fa.materialised_workspace_bytes(B, H, N, d) == want
    assert fa.materialised_workspace_bytes(0, 32, 1024, 128) == 0
    assert fa.materialised_workspace_bytes(-1, 32, 1024, 128) == -1
    assert fa.materialised_workspace_bytes(1, 32, 1024, 40) == -1
    assert fa.materialised_workspace_bytes(1, 1, (1 << 20) + 1, 128) == -1


def _mat(**kw):
    args = dict(q_ptr=0x10000, k_ptr=0x20000, v_ptr=0x30000, o_ptr=0x40000, lse_ptr=0, B=1, H=1,
                N=128, d=64, causal=True, scale=0.1, ws_ptr=0x1000000, ws_bytes=10 ** 9)
    args.update(kw)
    return fa.fa_fwd_materialised_raw(**args)


@pytest.mark.parametrize("kw,want", [
    (dict(ws_ptr=0), fa.FA_ERR_INVALID_ARG),
    (dict(ws_bytes=128 * 128 * 6), fa.FA_ERR_INVALID_ARG),    # no room for acc and row sums
    (dict(ws_ptr=0x1000080), fa.FA_ERR_MISALIGNED),     # workspace must be 256-byte aligned
    (dict(ws_ptr=0x20000 - 256), fa.FA_ERR_INVALID_ARG),  # workspace overlaps k
    (dict(q_ptr=0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(d=40), fa.FA_ERR_UNSUPPORTED),
    (dict(o_ptr=0x40008), fa.FA_ERR_MISALIGNED),
])
def test_materialised_argument_errors(kw, want):
    assert _mat(**kw) == want
    assert fa.last_error() != ""


def test_materialised_empty_is_a_noop():
    assert _mat(B=0) == fa.FA_OK
    assert _mat(N=0, ws_ptr=0) == fa.FA_OK
