"""GPU parity of both kernels at head dims 32-128 and of the launch the planner picks.

At head dims 32, 64 and 128 a call runs either the two-tile kernel (256-row units) or
the one-tile kernel (128-row units), whichever fa_fwd_plan models as faster; small
problems go to the one-tile kernel.  Each kernel is pinned here through
fa_fwd_options.kernel and compared with the fp64 oracle on the same seeded inputs,
so both stay covered whatever the planner picks for the other tests' shapes.
"""
import numpy as np
import pytest
import torch

import _parity
import oracle
import tiled_online_softmax_fa_gb300 as fa
import workloads

pytestmark = pytest.mark.gpu
W = workloads.WORKLOADS
TWO, ONE = fa.FA_KERNEL_TWO_TILE, fa.FA_KERNEL_ONE_TILE
KERNELS = [pytest.param(TWO, id="two-tile"), pytest.param(ONE, id="one-tile")]


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.load_library()


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("N", [1, 2, 127, 128, 129, 255, 256, 257, 383, 700, 1000])
@pytest.mark.parametrize("causal", [True, False])
def test_pinned_ragged_and_small(kernel, N, causal):
    w = W["n1k"]
    rows = workloads.select_rows(w, B=2, H=3, N=N, seed=N + 128)
    _parity.check_case(w, causal, B=2, H=3, N=N, d=128, seed=N * 7 + 128, rows=rows,
                       kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
def test_pinned_n1k_full_tensor(kernel):
    """The B1 H32 N1024 workload, every row of every head."""
    w = W["n1k"]
    rows = np.array([(bh, i) for bh in range(32) for i in range(1024)], dtype=np.int64)
    _parity.check_case(w, True, rows=rows, kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
def test_pinned_large_logits(kernel):
    _parity.check_case(W["n32k"], True, B=1, H=4, N=1000, d=128, seed=205, kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("causal", [True, False])
def test_pinned_many_units_per_cta(kernel, causal):
    rows = workloads.select_rows(W["b8n8k"], B=4, H=40, N=1536, seed=6)
    _parity.check_case(W["n1k"], causal, B=4, H=40, N=1536, d=128, seed=6, rows=rows,
                       kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
def test_pinned_long_sequence_sampled(kernel):
    """One head at N = 16384: 128 (one-tile) or 64 (two-tile) units of very different
    lengths under the causal mask."""
    w = W["n32k"]
    rows = workloads.select_rows(w, B=1, H=1, N=16384, seed=207)
    _parity.check_case(w, True, B=1, H=1, N=16384, d=128, seed=207, rows=rows, kernel=kernel)


def test_one_tile_grid_cap_and_determinism():
    w = W["n1k"]
    q, k, v = (t.cuda() for t in workloads.make_inputs(w, B=2, H=8, N=1100, d=128, seed=12))
    opt = fa.FwdOptions(kernel=ONE)
    a, la = fa.fa_fwd(q, k, v, causal=True, options=opt)
    b, lb = fa.fa_fwd(q, k, v, causal=True, options=fa.FwdOptions(kernel=ONE, max_ctas=7))
    c, lc = fa.fa_fwd(q, k, v, causal=True, options=opt)
    assert fa.get_device_status() == fa.FA_OK
    assert torch.equal(a, b) and torch.equal(la, lb)
    assert torch.equal(a, c) and torch.equal(la, lc)


@pytest.mark.parametrize("d", [128, 64, 32])
@pytest.mark.parametrize("B,H,N", [(1, 4, 8192), (1, 32, 1024), (2, 16, 4096)])
def test_auto_equals_the_planned_kernel(d, B, H, N):
    q, k, v = (t.cuda() for t in workloads.make_inputs(W["n4k"], B=B, H=H, N=N, d=d, seed=N))
    kernel, splits = fa.fwd_plan(B, H, N, d, True)
    assert splits == 1
    a, la = fa.fa_fwd(q, k, v, causal=True)
    b, lb = fa.fa_fwd(q, k, v, causal=True, options=fa.FwdOptions(kernel=kernel))
    assert fa.get_device_status() == fa.FA_OK
    assert torch.equal(a, b) and torch.equal(la, lb)


def test_plan_uses_the_device_sm_count():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for H, N in [(1, 8192), (4, 8192), (1, 32768), (32, 8192)]:
        for split in (False, True):
            assert fa.fwd_plan(1, H, N, 128, True, allow_split=split) == \
                fa.fwd_plan(1, H, N, 128, True, allow_split=split, num_sms=sms)


@pytest.mark.parametrize("H,N", [(4, 8192), (1, 16384)])
def test_automatic_split_entry_points(H, N):
    """splits = 0 through both split entry points: the planned launch (one-tile at
    H4 N8192, a four-way split at H1 N16384 on 152 SMs) against the oracle."""
    w = W["n32k"]
    q, k, v = workloads.make_inputs(w, B=1, H=H, N=N, d=128, seed=H + N)
    rows = workloads.select_rows(w, B=1, H=H, N=N, seed=H + N)
    scale = float(np.float32(1.0 / np.sqrt(128)))
    o64, lse64 = oracle.attn_rows(q, k, v, rows, True, scale)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o, lse = fa.fa_fwd_splitkv(qd, kd, vd, causal=True, scale=scale, splits=0)
    assert fa.get_device_status() == fa.FA_OK
    _parity.compare(*_parity.gather_rows(o, lse, rows), o64, lse64)
    o2 = torch.empty_like(qd)
    lse2 = torch.empty((1, H, N), dtype=torch.float32, device="cuda")
    rc = fa.fa_fwd_splitkv_noalloc_raw(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o2.data_ptr(),
                                       lse2.data_ptr(), 1, H, N, 128, True, scale, 0,
                                       torch.cuda.current_stream().cuda_stream)
    assert rc == fa.FA_OK
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


@pytest.mark.parametrize("d", [32, 64])
@pytest.mark.parametrize("N", [1, 127, 128, 129, 257, 700])
@pytest.mark.parametrize("causal", [True, False])
def test_pinned_one_tile_small_head_dims(d, N, causal):
    """The one-tile kernel at head dims 32 and 64 (each output row written by two
    threads in 32-column chunks; at d = 32 the second thread writes none)."""
    w = W["n1k"]
    rows = workloads.select_rows(w, B=2, H=3, N=N, seed=N + d)
    _parity.check_case(w, causal, B=2, H=3, N=N, d=d, seed=N * 5 + d, rows=rows, kernel=ONE)


@pytest.mark.parametrize("d", [32, 64])
def test_pinned_one_tile_small_head_dims_large_logits_and_many_units(d):
    _parity.check_case(W["n32k"], True, B=1, H=4, N=1000, d=d, seed=300 + d, kernel=ONE)
    rows = workloads.select_rows(W["b8n8k"], B=4, H=40, N=1536, seed=d)
    _parity.check_case(W["n1k"], True, B=4, H=40, N=1536, d=d, seed=d, rows=rows, kernel=ONE)


def test_automatic_split_limited_by_the_workspace():
    """splits = 0 plans among the split counts the workspace holds: the plan for one head
    at N = 8192 takes several pieces; with room for two, or none, the call still runs
    (fewer pieces, or unsplit) and matches the oracle."""
    w = W["n32k"]
    B, H, N, d = 1, 1, 8192, 128
    q, k, v = workloads.make_inputs(w, B=B, H=H, N=N, d=d, seed=91)
    rows = workloads.select_rows(w, B=B, H=H, N=N, seed=92)
    scale = float(np.float32(1.0 / np.sqrt(d)))
    o64, lse64 = oracle.attn_rows(q, k, v, rows, True, scale)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    kernel, splits = fa.fwd_plan(B, H, N, d, True, allow_split=True)
    assert splits > 2
    for room in (splits, 2, 0):
        nbytes = fa.splitkv_workspace_bytes(B, H, N, d, room) if room > 1 else 0
        ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
        o = torch.empty_like(qd)
        lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
        rc = fa.fa_fwd_splitkv_raw(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), B, H, N, d, True, scale, 0,
                                   ws.data_ptr() if nbytes else 0, nbytes,
                                   torch.cuda.current_stream().cuda_stream)
        assert rc == fa.FA_OK, fa.last_error()
        torch.cuda.synchronize()
        assert fa.get_device_status() == fa.FA_OK
        _parity.compare(*_parity.gather_rows(o, lse, rows), o64, lse64)
