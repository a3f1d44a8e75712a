"""Host-side checks of the C ABI that need no GPU: both libraries load, each exports every
function its header declares (``include/fa.h``: libfa_sm103.so, ``include/fa_baseline.h``:
libfa_baseline.so), and they reject bad arguments before touching CUDA."""
import ctypes
import os
import re
import subprocess

import pytest

import tiled_online_softmax_fa_gb300 as fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions(header):
    with open(os.path.join(ROOT, "include", header)) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", text)))


def test_every_header_belongs_to_a_library():
    assert sorted(fn for fn in os.listdir(os.path.join(ROOT, "include")) if fn.endswith(".h")) == \
        ["fa.h", "fa_baseline.h"]


def test_library_builds_and_loads():
    lib = fa.load_library()
    assert isinstance(lib, ctypes.CDLL)
    assert fa.version() == 300


def test_every_declared_symbol_is_exported():
    names = _declared_functions("fa.h")
    assert {"fa_fwd", "fa_fwd_opts", "fa_strerror", "fa_last_error", "fa_get_device_status",
            "fa_version", "fa_fwd_splitkv", "fa_splitkv_workspace_bytes",
            "fa_splitkv_auto_splits", "fa_row_kernel_register_check"} <= set(names)
    lib = fa.load_library()
    for name in names:
        assert hasattr(lib, name), name
    base = _declared_functions("fa_baseline.h")
    assert set(base) == {"fa_fwd_materialised", "fa_materialised_workspace_bytes",
                         "fa_baseline_last_error"}
    blib = fa.load_baseline_library()
    for name in base:
        assert hasattr(blib, name), name


def _needed(path):
    out = subprocess.run(["readelf", "-d", path], capture_output=True, text=True, check=True).stdout
    return re.findall(r"\(NEEDED\)\s+Shared library: \[([^\]]+)\]", out)


def test_forward_library_links_no_blas():
    from tiled_online_softmax_fa_gb300 import build
    fa.load_library()
    fa.load_baseline_library()
    assert not any("cublas" in n for n in _needed(build.LIB_PATH)), _needed(build.LIB_PATH)
    assert any("cublas" in n for n in _needed(build.BASELINE_LIB_PATH))
    # and it exports none of the baseline's entry points
    assert not hasattr(fa.load_library(), "fa_fwd_materialised")


def test_register_split_check():
    # the allocation the two-tile kernel's setmaxnreg split is written for
    assert fa.row_kernel_register_check(128, 512) == fa.FA_OK
    assert fa.last_error() == ""
    # anything else would leave setmaxnreg.inc waiting forever: refused
    for regs, threads in ((120, 512), (96, 512), (127, 1024), (168, 384), (128, 384), (0, 512)):
        assert fa.row_kernel_register_check(regs, threads) == fa.FA_ERR_UNSUPPORTED
        assert "setmaxnreg" in fa.last_error()


def test_build_rejects_other_register_counts():
    from tiled_online_softmax_fa_gb300 import build
    name = "_ZN8fa_sm1034rowk17fa_fwd_row_kernelILi128ELb0EEEv14CUtensorMap_stS2_S2_NS_6ParamsE"
    log = (f"ptxas info    : Compiling entry function '{name}' for 'sm_103a'\n"
           f"ptxas info    : Function properties for {name}\n"
           "    0 bytes stack frame, 0 bytes spill stores, 0 bytes spill loads\n"
           "ptxas info    : Used {regs} registers, used 1 barriers, 6400 bytes smem\n")
    build.check_row_kernel_registers(log.format(regs=128))
    assert build.kernel_registers(log.format(regs=120)) == {name: 120}
    with pytest.raises(RuntimeError, match="setmaxnreg"):
        build.check_row_kernel_registers(log.format(regs=120))
    with pytest.raises(RuntimeError, match="no fa_fwd_row_kernel"):
        build.check_row_kernel_registers("")


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
    # sizes beyond the kernels' 32-bit indices: -1, never a wrapped (small) byte count
    assert fa.splitkv_workspace_bytes(1 << 20, 1 << 12, 1, 128, 2) == -1   # B*H > 2^31
    assert fa.splitkv_workspace_bytes(1, 1, (1 << 30) + 1, 128, 2) == -1    # N > 2^30
    assert fa.splitkv_workspace_bytes(1 << 15, 1 << 15, 1 << 14, 128, 64) == -1  # units
    assert fa.splitkv_workspace_bytes(1 << 14, 1 << 10, 1 << 10, 128, 64) == -1  # items


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
    assert fa.load_baseline_library().fa_baseline_last_error().decode() != ""


def test_materialised_empty_is_a_noop():
    assert _mat(B=0) == fa.FA_OK
    assert _mat(N=0, ws_ptr=0) == fa.FA_OK


@pytest.mark.parametrize("B,H,N,splits", [
    (1 << 15, 1 << 15, 1 << 14, 2),    # work units beyond int32
    (1 << 14, 1 << 10, 1 << 10, 64),   # units x splits beyond int32
    (1 << 20, 1 << 12, 128, 2),        # B*H beyond int32
])
def test_noalloc_range_checks_come_before_any_size_arithmetic(B, H, N, splits):
    # rejected on the host, before planning or sizing the scratch (no CUDA call needed)
    rc = fa.fa_fwd_splitkv_noalloc_raw(0x10000, 0x20000, 0x30000, 0x40000, 0, B, H, N, 128,
                                       True, 0.088, splits)
    assert rc == fa.FA_ERR_UNSUPPORTED
    assert fa.last_error() != ""


@pytest.mark.parametrize("block_kv,d,kernel,want", [
    (32, 128, 0, fa.FA_ERR_INVALID_ARG),       # neither 64 nor 128
    (256, 64, 0, fa.FA_ERR_INVALID_ARG),
    (-64, 64, 0, fa.FA_ERR_INVALID_ARG),
    (64, 256, 0, fa.FA_ERR_UNSUPPORTED),       # 64-key tiles: the two-tile kernel only
    (64, 128, fa.FA_KERNEL_ONE_TILE, fa.FA_ERR_UNSUPPORTED),
])
def test_block_kv_errors(block_kv, d, kernel, want):
    # rejected before any CUDA call
    assert _call(d=d, options=fa.FwdOptions(block_kv=block_kv, kernel=kernel)) == want
    assert fa.last_error() != ""

