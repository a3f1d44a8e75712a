"""Host-side checks of the launch planner (fa_fwd_plan), no GPU needed.

At head dims 32, 64 and 128 the library chooses per call between the two-tile kernel
(256-row units, optionally split along the keys) and the one-tile kernel (128-row
units) by replaying the kernels' static schedule on a cost model.  These tests pin that choice
to GB300 measurements: for every shape below one candidate was measured more than 2%
faster than the others (bf16, mean of 20 launches after 3 warm-ups, CUDA events; the
current kernels, with the row sum of the rounded P from the PV MMA and the next unit
decoded off the unit boundary; the d = 128 split launches with the merge kernel's
half-warp layout), and the planner, asked for 152 SMs, must pick it.
Candidates timed per head dim with `bench.py --d D --sweep out.json --kernel two|one
[--noncausal] [--splits S] --sweep-shapes ...` (S = 2, 3, 4, 5, 6, 8 on the shapes with
at most 152 two-tile or 304 one-tile units).  Near-ties (< 2%) are left out: either
choice is right there.  The tables key the shape as (1, B*H, N, causal): the planner
sees only B*H.
"""
import ctypes

import pytest

import tiled_online_softmax_fa_gb300 as fa

SMS = 152
TWO, ONE = fa.FA_KERNEL_TWO_TILE, fa.FA_KERNEL_ONE_TILE

# (B, H, N, causal) -> measured fastest of: "two" / "one" (the two-tile / one-tile kernel
# unsplit), "two-split" / "one-split" (that kernel split, the best count measured, where
# splits were timed)
MEASURED = {
    (1, 1, 4096, True): "one-split", (1, 1, 8192, True): "one-split",
    (1, 1, 12288, True): "one-split", (1, 1, 16384, True): "one-split",
    (1, 1, 24576, True): "two-split", (1, 1, 65536, True): "one",
    (1, 2, 8192, True): "one-split", (1, 2, 12288, True): "two-split",
    (1, 2, 16384, True): "one", (1, 2, 24576, True): "one", (1, 2, 32768, True): "one",
    (1, 3, 8192, True): "one", (1, 3, 12288, True): "one", (1, 3, 16384, True): "one",
    (1, 4, 4096, True): "one-split", (1, 4, 8192, False): "two", (1, 4, 8192, True): "one",
    (1, 4, 16384, True): "one", (1, 5, 6144, True): "one", (1, 6, 6144, True): "one",
    (1, 6, 8192, True): "one", (1, 8, 4096, False): "two", (1, 8, 4096, True): "one",
    (1, 10, 8192, True): "two", (1, 12, 4096, True): "one", (1, 16, 1024, True): "one",
    (1, 16, 2048, True): "one", (1, 16, 4096, False): "two", (1, 16, 4096, True): "two",
    (1, 24, 2048, True): "one", (1, 32, 256, True): "one", (1, 32, 512, True): "one",
    (1, 32, 1024, False): "two", (1, 32, 1024, True): "one", (1, 32, 2048, False): "two",
    (1, 32, 2048, True): "one", (1, 32, 4096, True): "two", (1, 40, 2048, True): "two",
    (1, 48, 1024, True): "one", (1, 48, 2048, False): "two", (1, 48, 2048, True): "one",
    (1, 64, 1024, True): "one", (1, 64, 2048, True): "one",
}

MEASURED_D64 = {
    (1, 1, 4096, True): "one-split", (1, 1, 8192, True): "one-split",
    (1, 1, 16384, True): "two-split", (1, 1, 24576, True): "two-split",
    (1, 1, 32768, True): "two-split", (1, 1, 65536, True): "two",
    (1, 2, 8192, True): "one-split", (1, 2, 12288, True): "two-split",
    (1, 2, 16384, True): "two-split", (1, 2, 24576, True): "one",
    (1, 2, 32768, True): "two", (1, 3, 12288, True): "one", (1, 3, 16384, True): "one",
    (1, 4, 8192, False): "two", (1, 4, 8192, True): "one", (1, 4, 16384, True): "two",
    (1, 5, 6144, True): "one", (1, 6, 6144, True): "one", (1, 6, 8192, True): "one",
    (1, 8, 4096, False): "two", (1, 8, 4096, True): "one", (1, 8, 8192, True): "two",
    (1, 10, 8192, True): "two", (1, 12, 4096, True): "one", (1, 16, 1024, True): "one",
    (1, 16, 2048, True): "one", (1, 16, 4096, False): "two", (1, 16, 4096, True): "two",
    (1, 20, 4096, True): "two", (1, 24, 2048, True): "two", (1, 32, 256, True): "one",
    (1, 32, 512, True): "one", (1, 32, 1024, False): "two", (1, 32, 1024, True): "one",
    (1, 32, 2048, False): "two", (1, 32, 4096, True): "two", (1, 40, 2048, True): "two",
    (1, 48, 2048, False): "two", (1, 64, 1024, True): "one", (1, 64, 2048, True): "two",
}

MEASURED_D32 = {
    (1, 1, 8192, True): "one-split", (1, 1, 12288, True): "two-split",
    (1, 1, 16384, True): "two-split", (1, 1, 24576, True): "two-split",
    (1, 1, 32768, True): "two-split", (1, 1, 65536, True): "two",
    (1, 2, 8192, True): "two-split", (1, 2, 12288, True): "two-split",
    (1, 2, 16384, True): "two-split", (1, 2, 32768, True): "two",
    (1, 3, 8192, True): "two-split", (1, 3, 12288, True): "one",
    (1, 4, 4096, True): "one-split", (1, 4, 8192, False): "two", (1, 4, 8192, True): "one",
    (1, 4, 16384, True): "two", (1, 5, 6144, True): "one", (1, 6, 6144, True): "one",
    (1, 8, 4096, False): "two", (1, 8, 4096, True): "one", (1, 8, 8192, True): "two",
    (1, 10, 8192, True): "two", (1, 16, 1024, True): "one", (1, 16, 2048, True): "one",
    (1, 16, 4096, False): "two", (1, 16, 4096, True): "two", (1, 20, 4096, True): "two",
    (1, 24, 2048, True): "two", (1, 32, 256, True): "one", (1, 32, 512, True): "one",
    (1, 32, 1024, False): "two", (1, 32, 1024, True): "one", (1, 32, 2048, False): "two",
    (1, 32, 4096, True): "two", (1, 40, 2048, True): "two", (1, 48, 1024, True): "one",
    (1, 48, 2048, False): "two", (1, 64, 1024, True): "one", (1, 64, 2048, True): "two",
}

MEASURED_D256 = {
    (1, 1, 4096, True): "one-split", (1, 1, 8192, True): "one-split",
    (1, 1, 12288, True): "one-split", (1, 1, 16384, True): "one-split",
    (1, 1, 24576, True): "one-split", (1, 1, 32768, True): "one",
    (1, 2, 8192, True): "one-split", (1, 2, 12288, True): "one", (1, 2, 16384, True): "one",
    (1, 3, 8192, True): "one", (1, 3, 12288, True): "one", (1, 4, 4096, True): "one-split",
    (1, 4, 8192, True): "one", (1, 5, 6144, True): "one", (1, 6, 6144, True): "one",
    (1, 8, 4096, True): "one",
}


def _label(kernel, splits):
    return ("one" if kernel == ONE else "two") + ("-split" if splits > 1 else "")


# Where the planner is known to pick wrong: (d, shape) -> measured loss of its launch.
#   d = 128, H40 N2048: the one-tile kernel (the two-tile one is 2.2 % faster);
#   d = 32, H3 N12288: the two-tile kernel split 2 ways (the one-tile kernel 5.9 % faster);
#   d = 256, H2 N12288: the one-tile kernel split 2 ways (unsplit 2.6 % faster).
KNOWN_MISSES = {(128, (1, 40, 2048, True)): 0.022, (32, (1, 3, 12288, True)): 0.059,
                (256, (1, 2, 12288, True)): 0.026}


def _cases():
    for d, table in ((128, MEASURED), (64, MEASURED_D64), (32, MEASURED_D32),
                     (256, MEASURED_D256)):
        for shape, want in sorted(table.items()):
            marks = ()
            if (d, shape) in KNOWN_MISSES:
                marks = pytest.mark.xfail(strict=True, reason="planner's pick measured "
                                          f"{KNOWN_MISSES[(d, shape)]:.0%} slower than the best")
            yield pytest.param(d, shape, want, marks=marks)


@pytest.mark.parametrize("d,shape,want", list(_cases()))
def test_plan_picks_the_measured_fastest(d, shape, want):
    B, H, N, causal = shape
    kernel, splits = fa.fwd_plan(B, H, N, d, causal, allow_split=True, num_sms=SMS)
    assert _label(kernel, splits) == want
    # without a workspace the split is not a candidate
    kernel1, splits1 = fa.fwd_plan(B, H, N, d, causal, allow_split=False, num_sms=SMS)
    assert splits1 == 1
    if not want.endswith("-split"):
        assert _label(kernel1, splits1) == want


def test_measured_two_vs_one_without_split():
    # where the split won, the unsplit choice is between the other two: measured
    # one-tile 590 vs two-tile 316 TFLOP/s (d128 H1 N16384), 905 vs 480 (H1 N24576)
    for N in (16384, 24576):
        assert fa.fwd_plan(1, 1, N, 128, True, num_sms=SMS) == (ONE, 1)


def test_head_dim_16_takes_the_two_tile_kernel():
    # the one-tile kernel writes each output row in 32-column chunks: head dim >= 32
    for H, N in [(1, 1024), (4, 8192), (1, 32768), (32, 8192)]:
        k, s = fa.fwd_plan(1, H, N, 16, True, allow_split=True, num_sms=SMS)
        assert k == TWO and s >= 1


def test_head_dim_256_takes_the_one_tile_kernel():
    for H, N in [(1, 1024), (4, 8192), (1, 32768), (32, 8192)]:
        assert fa.fwd_plan(1, H, N, 256, True, num_sms=SMS) == (ONE, 1)
        assert fa.fwd_plan(1, H, N, 256, True, allow_split=True, num_sms=SMS)[0] == ONE


def test_throughput_shape_takes_the_two_tile_kernel():
    # B8 H32 N8192: 8192 units of 256 rows, far beyond the modelled range
    assert fa.fwd_plan(8, 32, 8192, 128, True, allow_split=True, num_sms=SMS) == (TWO, 1)


def test_many_units_skip_the_model():
    # more than four 256-row units per SM: the two-tile kernel, whatever the mask
    for causal in (True, False):
        assert fa.fwd_plan(4, 160, 1024, 128, causal, num_sms=SMS)[0] == TWO


def test_fewer_sms_shift_the_choice():
    # 128 units of 256 rows: fewer than one per SM on 152 SMs (one-tile), but 16 per
    # SM on 8 SMs, where the schedule is even and the faster two-tile step wins
    assert fa.fwd_plan(1, 8, 4096, 128, True, num_sms=SMS)[0] == ONE
    assert fa.fwd_plan(1, 8, 4096, 128, True, num_sms=8)[0] == TWO


def test_batch_and_heads_enter_as_their_product():
    for B, H in [(1, 8), (2, 4), (8, 1)]:
        assert fa.fwd_plan(B, H, 4096, 128, True, num_sms=SMS) == (ONE, 1)


def test_empty_problem():
    assert fa.fwd_plan(0, 4, 128, 128, True, num_sms=SMS) == (TWO, 1)
    assert fa.fwd_plan(1, 4, 0, 64, True, num_sms=SMS) == (TWO, 1)
    assert fa.fwd_plan(1, 0, 128, 256, True, num_sms=SMS) == (ONE, 1)


@pytest.mark.parametrize("args,want", [
    ((-1, 1, 128, 128), fa.FA_ERR_INVALID_ARG),
    ((1, 1, -128, 128), fa.FA_ERR_INVALID_ARG),
    ((1, 1, 128, 48), fa.FA_ERR_UNSUPPORTED),
    ((1, 1, (1 << 30) + 1, 128), fa.FA_ERR_UNSUPPORTED),
])
def test_plan_rejects_bad_sizes(args, want):
    with pytest.raises(fa.FAError) as e:
        fa.fwd_plan(*args, True, num_sms=SMS)
    assert e.value.status == want


def test_plan_rejects_null_outputs_and_negative_sms():
    lib = fa.load_library()
    k = ctypes.c_int()
    s = ctypes.c_int()
    assert lib.fa_fwd_plan(1, 1, 128, 128, 1, 0, SMS, None, ctypes.byref(k), None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_fwd_plan(1, 1, 128, 128, 1, 0, SMS, ctypes.byref(k), None, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_fwd_plan(1, 1, 128, 128, 1, 0, -1, ctypes.byref(k), ctypes.byref(s),
                           None) == fa.FA_ERR_INVALID_ARG
    # the order output is optional
    assert lib.fa_fwd_plan(1, 1, 128, 128, 1, 0, SMS, ctypes.byref(k), ctypes.byref(s), None) == fa.FA_OK


# --- the kernel pin in fa_fwd_options: checked before any CUDA call -------------------
def _call_opts(d, **opt):
    return fa.fa_fwd_raw(0x10000, 0x20000, 0x30000, 0x40000, 0, 1, 1, 128, d, True, 0.1,
                         options=fa.FwdOptions(**opt))


def test_options_struct_layout():
    # the C struct: int64 budget, then five int32 fields (block_kv appended last, 0.3.0)
    assert ctypes.sizeof(fa.FwdOptions) == 32
    assert fa.FwdOptions.kernel.offset == 16 and fa.FwdOptions.order.offset == 20
    assert fa.FwdOptions.block_kv.offset == 24


@pytest.mark.parametrize("d,opt,want", [
    (128, dict(kernel=3), fa.FA_ERR_INVALID_ARG),
    (128, dict(kernel=-1), fa.FA_ERR_INVALID_ARG),
    (128, dict(order=4), fa.FA_ERR_INVALID_ARG),
    (128, dict(order=-1), fa.FA_ERR_INVALID_ARG),
    (16, dict(kernel=ONE), fa.FA_ERR_UNSUPPORTED),
    (256, dict(kernel=TWO), fa.FA_ERR_UNSUPPORTED),
])
def test_kernel_pin_rejected_before_cuda(d, opt, want):
    assert _call_opts(d, **opt) == want
    assert fa.last_error()


# --- unit order: one snake vs snakes per head group -----------------------------------
# (B, H, N, d) causal, two-tile kernel -> measured TFLOP/s with one snake, group snakes
# (odd groups mirrored) and shifted group snakes (profile `unit_order_d128`); the
# planner's order must be within 1 % of the best of the three.
MEASURED_ORDER = {
    (1, 32, 8192, 128): (1058, 1165, 1161),
    (4, 32, 8192, 128): (1112, 1193, 1203),
    (1, 16, 16384, 128): (1103, 1230, 1216),
    (2, 32, 8192, 128): (1169, 1183, 1188),
    (8, 32, 8192, 128): (1207, 1198, 1211),
    (8, 32, 4096, 128): (1035, 1095, 1101),
    (1, 8, 32768, 128): (1125, 1260, 1236),
    (1, 20, 8192, 128): (977, 962, 954),
    (1, 32, 16384, 128): (1218, 1235, 1235),
    (8, 32, 16384, 128): (1242, 1241, 1260),
    (4, 32, 2048, 128): (823, 855, 847),
    (2, 20, 8192, 64): (591, 683, 681),
    (4, 32, 8192, 64): (680, 697, 695),
    (1, 64, 8192, 64): (633, 691, 688),
}
ORDER_INDEX = {fa.FA_ORDER_ONE_SNAKE: 0, fa.FA_ORDER_GROUP_SNAKES: 1, fa.FA_ORDER_SHIFTED_SNAKES: 2}


@pytest.mark.parametrize("shape,tflops", sorted(MEASURED_ORDER.items()))
def test_order_is_within_one_percent_of_the_measured_best(shape, tflops):
    B, H, N, d = shape
    kernel, splits, order = fa.fwd_plan(B, H, N, d, True, with_order=True, num_sms=SMS)
    assert (kernel, splits) == (TWO, 1)
    assert tflops[ORDER_INDEX[order]] >= 0.99 * max(tflops)


def test_order_choice_where_the_orders_differ_most():
    # one snake over two groups of 3.4 rounds leaves the busiest CTA 14 % above average
    assert fa.fwd_plan(1, 32, 8192, 128, True, with_order=True, num_sms=SMS)[2] != \
        fa.FA_ORDER_ONE_SNAKE
    # a ragged last group of 4 heads (16 + 4) favours the one snake
    assert fa.fwd_plan(1, 20, 8192, 128, True, with_order=True, num_sms=SMS)[2] == \
        fa.FA_ORDER_ONE_SNAKE


def test_one_head_group_takes_the_one_snake():
    # K and V of all heads fit the ~64 MB L2 share: one group, the orders coincide
    for B, H, N, d in [(1, 4, 8192, 128), (1, 32, 1024, 128), (2, 16, 4096, 64), (1, 1, 65536, 128)]:
        assert fa.fwd_plan(B, H, N, d, True, with_order=True, num_sms=SMS)[2] == fa.FA_ORDER_ONE_SNAKE


def test_order_is_reported_for_every_plan():
    for d in (16, 32, 64, 128, 256):
        for B, H, N in [(1, 20, 8192), (8, 32, 2048), (1, 3, 100)]:
            k, s, o = fa.fwd_plan(B, H, N, d, False, allow_split=True, with_order=True, num_sms=SMS)
            assert o in (fa.FA_ORDER_ONE_SNAKE, fa.FA_ORDER_GROUP_SNAKES, fa.FA_ORDER_SHIFTED_SNAKES)


# --- invariants over many shapes --------------------------------------------------------
def _shapes(n=300, seed=2024):
    import random
    rng = random.Random(seed)
    for _ in range(n):
        B = rng.choice([1, 1, 1, 2, 4, 8])
        H = rng.choice([1, 2, 3, 4, 5, 8, 12, 16, 20, 32, 48, 64])
        N = rng.choice([1, 100, 128, 129, 255, 256, 300, 1000, 2048, 4096, 6000, 8192, 12288,
                        16384, 32768, 65536])
        d = rng.choice([16, 32, 64, 128, 256])
        yield B, H, N, d, rng.random() < 0.8


def test_every_plan_is_a_launch_the_library_can_run():
    orders = (fa.FA_ORDER_ONE_SNAKE, fa.FA_ORDER_GROUP_SNAKES, fa.FA_ORDER_SHIFTED_SNAKES)
    for B, H, N, d, causal in _shapes():
        for split in (False, True):
            kernel, splits, order = fa.fwd_plan(B, H, N, d, causal, allow_split=split,
                                                with_order=True, num_sms=SMS)
            assert kernel in (TWO, ONE)
            assert kernel != TWO or d <= 128, (B, H, N, d)   # the two-tile kernel: d <= 128
            assert kernel != ONE or d >= 32, (B, H, N, d)    # the one-tile kernel: d >= 32
            assert 1 <= splits <= 64 and (split or splits == 1)
            assert order in orders
            # the same answer again (the plan cache)
            assert fa.fwd_plan(B, H, N, d, causal, allow_split=split, with_order=True,
                               num_sms=SMS) == (kernel, splits, order)


def test_workspace_sizing_covers_both_kernels_split_layouts():
    # fa_splitkv_workspace_bytes sizes 256-row items (the two-tile kernel); the one-tile
    # kernel's items hold 128 rows over ceil(N / 128) query blocks.  The library puts the
    # partial outputs first and the partial lse after them, so both layouts must fit.
    for B, H, N, d, _ in _shapes():
        for splits in (2, 3, 8, 64):
            need = fa.splitkv_workspace_bytes(B, H, N, d, splits)
            one_tile = B * H * -(-N // 128) * splits * 128 * (d + 1) * 4
            assert one_tile <= need, (B, H, N, d, splits)
            if d <= 128:
                two_tile = B * H * -(-N // 256) * splits * 256 * (d + 1) * 4
                assert two_tile == need
