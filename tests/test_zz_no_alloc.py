"""The allocation-free split-KV entry point (fa_fwd_splitkv_noalloc).

Some callers cannot allocate device memory while they run -- plug-ins whose host
framework owns every device buffer, loops that forbid allocator calls after start-up
-- so this entry point keeps its partial results in a fixed scratch array inside the
library instead of a caller-provided workspace.  These tests call it through the C
ABI and compare it with fa_fwd_splitkv (caller workspace) on the same inputs, for two
calls in a row with different inputs (the scratch keeps the previous call's data, so
stale contents must not leak into the next result).  This file is collected last so a
run that stops at the first failure has already run every other test; it passes on
its own in a fresh process as well.
"""
import numpy as np
import pytest
import torch

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
        assert (a.float() - b.float()).abs().max().item() <= O_TOL
        assert (la - lb).abs().max().item() <= LSE_TOL
        assert torch.isfinite(a.float()).all() and torch.isfinite(la).all()


def test_automatic_split_count():
    q, k, v = _inputs(303, 1, 1, 8192, 128)
    a, la = _noalloc(q, k, v, True, 0)
    b, lb = _with_workspace(q, k, v, True, 0)
    assert (a.float() - b.float()).abs().max().item() <= O_TOL
    assert (la - lb).abs().max().item() <= LSE_TOL


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
