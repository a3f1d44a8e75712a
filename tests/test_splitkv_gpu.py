"""GPU parity of the split-KV forward (partial results per key range merged by lse)."""
import numpy as np
import pytest
import torch

import _parity
import oracle
import tiled_online_softmax_fa_gb300 as fa
import workloads

pytestmark = pytest.mark.gpu
W = workloads.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.load_library()


def _check(w, causal, splits, B, H, N, d, seed, rows=None):
    q, k, v = workloads.make_inputs(w, B=B, H=H, N=N, d=d, seed=seed)
    scale = float(np.float32(1.0 / np.sqrt(d)))
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o, lse = fa.fa_fwd_splitkv(qd, kd, vd, causal=causal, scale=scale, splits=splits)
    assert fa.get_device_status() == fa.FA_OK
    if rows is None:
        rows = workloads.select_rows(w, B=B, H=H, N=N, seed=seed)
    og, lg = _parity.gather_rows(o, lse, rows)
    o64, lse64 = oracle.attn_rows(q, k, v, rows, causal, scale)
    return _parity.compare(og, lg, o64, lse64), (qd, kd, vd, o, lse)


@pytest.mark.parametrize("splits", [2, 3, 4, 0])
def test_n1k_full_tensor(splits):
    _check(W["n1k"], True, splits, 1, 32, 1024, 128, 1002)


def test_n4k_noncausal_sampled():
    _check(W["n4k"], False, 3, 1, 32, 4096, 128, 1003)


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("N", [129, 300, 700])
@pytest.mark.parametrize("splits", [2, 4, 5])  # the merge: a half-warp per row up to 4 pieces
def test_ragged(d, N, splits):
    w = W["n1k"]
    rows = workloads.select_rows(w, B=2, H=3, N=N, seed=N + d)
    for causal in (True, False):
        _check(w, causal, splits, 2, 3, N, d, N * 11 + d, rows=rows)


def test_more_splits_than_key_tiles():
    """N = 200 has two key tiles: most of 8 ranges are empty and must be skipped."""
    w = W["n1k"]
    for causal in (True, False):
        _check(w, causal, 8, 1, 4, 200, 64, 31)


def test_large_logits():
    _check(W["n32k"], True, 3, 1, 4, 2048, 128, 41)


def test_one_split_equals_fa_fwd_bits():
    w = W["n1k"]
    q, k, v = (t.cuda() for t in workloads.make_inputs(w, B=1, H=4, N=777, d=128, seed=5))
    a, la = fa.fa_fwd(q, k, v, causal=True)
    b, lb = fa.fa_fwd_splitkv(q, k, v, causal=True, splits=1)
    assert torch.equal(a, b) and torch.equal(la, lb)


def test_split_is_deterministic_and_close_to_unsplit():
    w = W["n1k"]
    q, k, v = (t.cuda() for t in workloads.make_inputs(w, B=1, H=8, N=2048, d=128, seed=6))
    a, la = fa.fa_fwd(q, k, v, causal=True)
    b, lb = fa.fa_fwd_splitkv(q, k, v, causal=True, splits=4)
    c, lc = fa.fa_fwd_splitkv(q, k, v, causal=True, splits=4)
    assert torch.equal(b, c) and torch.equal(lb, lc)
    assert (a.float() - b.float()).abs().max() <= 8e-3
    assert (la - lb).abs().max() <= 1e-3


def test_workspace_guard_regions_untouched():
    w = W["n1k"]
    B, H, N, d, splits = 1, 3, 500, 64, 3
    q, k, v = (t.cuda() for t in workloads.make_inputs(w, B=B, H=H, N=N, d=d, seed=7))
    need = fa.splitkv_workspace_bytes(B, H, N, d, splits)
    pad = 4096
    buf = torch.full((pad + need + pad,), 0xA5, dtype=torch.uint8, device="cuda")
    ws = buf[pad:pad + need]
    o, lse = fa.fa_fwd_splitkv(q, k, v, causal=True, splits=splits, workspace=ws)
    assert fa.get_device_status() == fa.FA_OK
    assert torch.all(buf[:pad] == 0xA5) and torch.all(buf[-pad:] == 0xA5)
    ref, _ = fa.fa_fwd(q, k, v, causal=True)
    assert (o.float() - ref.float()).abs().max() <= 8e-3
