"""The allocation-free split-KV entry point (fa_fwd_splitkv_noalloc).

Some callers cannot allocate device memory while they run -- plug-ins whose host
framework owns every device buffer, loops that forbid allocator calls after start-up
-- so this entry point keeps its partial results in a fixed scratch array inside the
library instead of a caller-provided workspace.  These tests call it through the C
ABI and compare it with fa_fwd_splitkv (caller workspace) on the same inputs, for two
calls in a row with different inputs (the scratch keeps the previous call's data, so
stale contents must not leak into the next result).  With the same kernel and split
count both entry points run the same launches on the same inputs, so their outputs
must agree bit for bit; a d = 128 case is also checked against the fp64 oracle, and a
call is checked to leave the device's free memory unchanged.  This file is collected
last so a run that stops at the first failure has already run every other test; it
passes on its own in a fresh process as well.
"""
import numpy as np
import pytest
import torch

import _parity
import oracle
import tiled_online_softmax_fa_gb300 as fa
import workloads

pytestmark = pytest.mark.gpu

O_TOL = 8e-3     # the O tolerance the parity tests use
LSE_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.load_library()


def _inputs(seed, B, H, N, d, w="n1k"):
    q, k, v = workloads.make_inputs(workloads.WORKLOADS[w], B=B, H=H, N=N, d=d, seed=seed)
    return tuple(t.cuda() for t in (q, k, v))


def _noalloc(q, k, v, causal, splits):
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    scale = float(np.float32(1.0 / np.sqrt(d)))
    rc = fa.fa_fwd_splitkv_noalloc_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                       lse.data_ptr(), B, H, N, d, causal, scale, splits,
                                       torch.cuda.current_stream().cuda_stream)
    assert rc == fa.FA_OK, fa.last_error()
    assert fa.get_device_status() == fa.FA_OK
    return o, lse


def _with_workspace(q, k, v, causal, splits):
    d = q.shape[-1]
    scale = float(np.float32(1.0 / np.sqrt(d)))
    o, lse = fa.fa_fwd_splitkv(q, k, v, causal=causal, scale=scale, splits=splits)
    assert fa.get_device_status() == fa.FA_OK
    return o, lse


@pytest.mark.parametrize("splits,B,H,N,d,causal,w", [
    (2, 1, 2, 4096, 128, True, "n1k"),
    (3, 2, 3, 1000, 64, False, "n1k"),
    (4, 1, 4, 2048, 128, True, "n32k"),
])
def test_matches_workspace_entry_point_two_calls_in_a_row(splits, B, H, N, d, causal, w):
    for seed in (101, 202):  # two calls in a row, different inputs
        q, k, v = _inputs(seed, B, H, N, d, w)
        a, la = _noalloc(q, k, v, causal, splits)
        b, lb = _with_workspace(q, k, v, causal, splits)
        # same kernel, same pieces, same inputs: identical bits (a stale scratch value
        # leaking into the merge would show here, however small)
        assert torch.equal(a, b)
        assert torch.equal(la, lb)
        assert torch.isfinite(a.float()).all() and torch.isfinite(la).all()


def test_automatic_split_count():
    q, k, v = _inputs(303, 1, 1, 8192, 128)
    a, la = _noalloc(q, k, v, True, 0)
    b, lb = _with_workspace(q, k, v, True, 0)
    pieces = fa.fwd_plan(1, 1, 8192, 128, True, allow_split=True)[1]
    if fa.splitkv_workspace_bytes(1, 1, 8192, 128, pieces) <= fa.noalloc_scratch_bytes():
        # the scratch holds the plan's pieces, so both calls take the same launch
        assert torch.equal(a, b) and torch.equal(la, lb)
    assert (a.float() - b.float()).abs().max().item() <= O_TOL
    assert (la - lb).abs().max().item() <= LSE_TOL


@pytest.mark.parametrize("splits", [2, 5])
def test_matches_the_oracle_at_head_dim_128(splits):
    """Two calls in a row, each checked against the fp64 oracle with the parity gates."""
    w = workloads.WORKLOADS["n4k"]
    B, H, N, d = 1, 3, 1500, 128
    for seed in (404, 505):
        q, k, v = workloads.make_inputs(w, B=B, H=H, N=N, d=d, seed=seed)
        qd, kd, vd = (t.cuda() for t in (q, k, v))
        o, lse = _noalloc(qd, kd, vd, True, splits)
        rows = workloads.select_rows(w, B=B, H=H, N=N, seed=seed)
        og, lg = _parity.gather_rows(o, lse, rows)
        scale = float(np.float32(1.0 / np.sqrt(d)))
        o64, lse64 = oracle.attn_rows(q, k, v, rows, True, scale)
        _parity.compare(og, lg, o64, lse64)


def test_allocates_no_device_memory():
    """After a warm-up call (which loads the kernels), a split call leaves the device's
    free memory where it was: the partial results went to the built-in scratch."""
    q, k, v = _inputs(606, 1, 4, 4096, 128)
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    scale = float(np.float32(1.0 / np.sqrt(d)))
    stream = torch.cuda.current_stream().cuda_stream

    def call():
        rc = fa.fa_fwd_splitkv_noalloc_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                           lse.data_ptr(), B, H, N, d, True, scale, 4, stream)
        assert rc == fa.FA_OK, fa.last_error()
        torch.cuda.synchronize()

    call()
    need = fa.splitkv_workspace_bytes(B, H, N, d, 4)
    assert need > (4 << 20)   # a workspace allocation would show well above the slack
    free0 = torch.cuda.mem_get_info()[0]
    call()
    call()
    free1 = torch.cuda.mem_get_info()[0]
    assert abs(free0 - free1) <= (1 << 20), (free0, free1)
    assert fa.get_device_status() == fa.FA_OK


def test_sizes_beyond_the_scratch_are_rejected():
    cap = fa.noalloc_scratch_bytes()
    B, H, N, d, splits = 1, 64, 8192, 128, 8
    assert fa.splitkv_workspace_bytes(B, H, N, d, splits) > cap
    q = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    o = torch.full_like(q, 3.0)
    rc = fa.fa_fwd_splitkv_noalloc_raw(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), 0,
                                       B, H, N, d, True, 0.088, splits)
    assert rc == fa.FA_ERR_UNSUPPORTED
    assert "64 MiB" in fa.last_error()
    torch.cuda.synchronize()
    assert torch.all(o == 3.0)  # nothing was launched
