"""GPU parity of split-KV on the one-tile kernel (128-row units), head dims 32 to 256.

Each 128-row unit's key tiles are cut into pieces; every piece writes its normalised
partial output and the logsumexp of its scores, and the merge kernel combines them.
The kernel is pinned through fa_fwd_splitkv_opts and compared with the fp64 oracle.
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
ONE = fa.FA_KERNEL_ONE_TILE


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.load_library()


def _split_one(q, k, v, causal, scale, splits, **opt):
    o, lse = fa.fa_fwd_splitkv(q, k, v, causal=causal, scale=scale, splits=splits,
                               options=fa.FwdOptions(kernel=ONE, **opt))
    assert fa.get_device_status() == fa.FA_OK
    return o, lse


def _check(w, B, H, N, d, causal, splits, seed):
    q, k, v = workloads.make_inputs(w, B=B, H=H, N=N, d=d, seed=seed)
    scale = float(np.float32(1.0 / np.sqrt(d)))
    o, lse = _split_one(*(t.cuda() for t in (q, k, v)), causal, scale, splits)
    rows = workloads.select_rows(w, B=B, H=H, N=N, seed=seed + 1)
    o64, lse64 = oracle.attn_rows(q, k, v, rows, causal, scale)
    return _parity.compare(*_parity.gather_rows(o, lse, rows), o64, lse64)


@pytest.mark.parametrize("d", [32, 64, 128, 256])
@pytest.mark.parametrize("N", [127, 300, 1000])
@pytest.mark.parametrize("splits", [2, 3, 5])
@pytest.mark.parametrize("causal", [True, False])
def test_ragged(d, N, splits, causal):
    _check(W["n1k"], 2, 3, N, d, causal, splits, seed=N + 10 * splits + d)


@pytest.mark.parametrize("d", [128, 256])
def test_more_pieces_than_key_tiles(d):
    # N = 200: two key tiles per unit at most, eight pieces -> empty pieces
    _check(W["n1k"], 1, 4, 200, d, True, 8, seed=400 + d)


@pytest.mark.parametrize("d", [64, 256])
def test_large_logits(d):
    _check(W["n32k"], 1, 4, 1000, d, True, 3, seed=500 + d)


def test_long_sequence_sampled():
    _check(W["n32k"], 1, 2, 8192, 128, True, 4, seed=601)


@pytest.mark.parametrize("d", [128, 256])
def test_one_piece_equals_the_unsplit_kernel_bits(d):
    q, k, v = (t.cuda() for t in workloads.make_inputs(W["n4k"], B=1, H=3, N=1500, d=d, seed=7))
    scale = float(np.float32(1.0 / np.sqrt(d)))
    a, la = fa.fa_fwd(q, k, v, causal=True, scale=scale, options=fa.FwdOptions(kernel=ONE))
    b, lb = _split_one(q, k, v, True, scale, 1)
    assert torch.equal(a, b) and torch.equal(la, lb)


def test_orders_and_grid_cap_give_the_same_bits():
    q, k, v = (t.cuda() for t in workloads.make_inputs(W["n4k"], B=1, H=20, N=4096, d=128, seed=8))
    scale = float(np.float32(1.0 / np.sqrt(128)))
    a, la = _split_one(q, k, v, True, scale, 3, order=fa.FA_ORDER_ONE_SNAKE)
    b, lb = _split_one(q, k, v, True, scale, 3, order=fa.FA_ORDER_GROUP_SNAKES)
    c, lc = _split_one(q, k, v, True, scale, 3, max_ctas=9)
    e, le = _split_one(q, k, v, True, scale, 3, order=fa.FA_ORDER_SHIFTED_SNAKES, max_ctas=9)
    assert torch.equal(a, b) and torch.equal(la, lb)
    assert torch.equal(a, c) and torch.equal(la, lc)
    assert torch.equal(a, e) and torch.equal(la, le)


def test_head_dim_256_split_through_every_entry_point():
    """Explicit splits at d = 256 run the one-tile kernel; the allocation-free entry point
    gives the same bits as fa_fwd_splitkv with a workspace."""
    w = W["n1k"]
    q, k, v = workloads.make_inputs(w, B=1, H=2, N=2000, d=256, seed=9)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    scale = 0.0625
    a, la = fa.fa_fwd_splitkv(qd, kd, vd, causal=True, scale=scale, splits=3)
    assert fa.get_device_status() == fa.FA_OK
    b, lb = _split_one(qd, kd, vd, True, scale, 3)
    assert torch.equal(a, b) and torch.equal(la, lb)
    o3 = torch.empty_like(qd)
    l3 = torch.empty_like(la)
    rc = fa.fa_fwd_splitkv_noalloc_raw(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o3.data_ptr(),
                                       l3.data_ptr(), 1, 2, 2000, 256, True, scale, 3,
                                       torch.cuda.current_stream().cuda_stream)
    assert rc == fa.FA_OK
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    assert torch.equal(a, o3) and torch.equal(la, l3)
    rows = workloads.select_rows(w, B=1, H=2, N=2000, seed=10)
    o64, lse64 = oracle.attn_rows(q, k, v, rows, True, scale)
    _parity.compare(*_parity.gather_rows(a, la, rows), o64, lse64)


def test_pinned_kernel_needs_an_explicit_split_count():
    q = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.fa_fwd_splitkv(q, q, q, causal=True, splits=0, options=fa.FwdOptions(kernel=ONE),
                          workspace=torch.empty(1 << 20, dtype=torch.uint8, device="cuda"))
    assert e.value.status == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("d", [64, 256])
def test_guard_regions_untouched(d):
    """Canaries around o, lse and the workspace: the split kernel and the merge write
    exactly [B, H, N, d], [B, H, N] and the workspace the pieces need (one-tile items
    hold 128 rows, fewer than the 256-row sizing, so the tail of the sized workspace is
    not written either way, and the canary past it must survive)."""
    B, H, N, splits = 1, 3, 333, 3
    q, k, v = (t.cuda() for t in workloads.make_inputs(W["n1k"], B=B, H=H, N=N, d=d, seed=11))
    pad = 4096
    obuf = torch.full((pad + B * H * N * d + pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    lbuf = torch.full((pad + B * H * N + pad,), -3.0, dtype=torch.float32, device="cuda")
    need = fa.splitkv_workspace_bytes(B, H, N, d, splits)
    wbuf = torch.full((pad + need + pad,), 0xA5, dtype=torch.uint8, device="cuda")
    o = obuf[pad:pad + B * H * N * d].view(B, H, N, d)
    lse = lbuf[pad:pad + B * H * N].view(B, H, N)
    fa.fa_fwd_splitkv(q, k, v, o=o, lse=lse, causal=True, splits=splits,
                      workspace=wbuf[pad:pad + need], options=fa.FwdOptions(kernel=ONE))
    assert fa.get_device_status() == fa.FA_OK
    assert torch.all(obuf[:pad] == 7.0) and torch.all(obuf[-pad:] == 7.0)
    assert torch.all(lbuf[:pad] == -3.0) and torch.all(lbuf[-pad:] == -3.0)
    assert torch.all(wbuf[:pad] == 0xA5) and torch.all(wbuf[-pad:] == 0xA5)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    ref, lref = fa.fa_fwd(q, k, v, causal=True, options=fa.FwdOptions(kernel=ONE))
    assert (o.float() - ref.float()).abs().max() <= 8e-3
    assert (lse - lref).abs().max() <= 1e-3
