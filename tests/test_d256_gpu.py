"""GPU parity of head dim 256 (the one-query-tile kernel) against the fp64 oracle, plus
the cases that exercise what only that kernel does: 128-row work units, two score
buffers in tensor memory and the output rescale that waits for the previous P.V
product.  The ragged-shape grid in test_parity_gpu.py covers d = 256 as well."""
import numpy as np
import pytest
import torch

import _parity
import oracle
import tiled_online_softmax_fa_gb300 as fa
import workloads

pytestmark = pytest.mark.gpu
W = workloads.WORKLOADS
D = 256


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.load_library()


@pytest.mark.parametrize("causal", [True, False])
def test_sampled_rows_several_heads(causal):
    w = W["n4k"]
    rows = workloads.select_rows(w, B=2, H=6, N=2304, seed=31)
    _parity.check_case(w, causal, B=2, H=6, N=2304, d=D, seed=31, rows=rows)


def test_full_tensor_small():
    w = W["n1k"]
    B, H, N = 1, 2, 520
    rows = np.array([(bh, i) for bh in range(B * H) for i in range(N)], dtype=np.int64)
    _parity.check_case(w, True, B=B, H=H, N=N, d=D, seed=32, rows=rows)


def _ramp_inputs(B, H, N, d, seed, step):
    """Scores that grow along the keys by `step` (natural units) per 128-key tile on top
    of N(0, 1) noise, so the running maximum moves on almost every tile and the output
    is rescaled again and again (the lazy threshold is 8 in log2 units, ~5.5 natural)."""
    g = torch.Generator().manual_seed(seed)
    scale = 1.0 / np.sqrt(d)
    q = torch.randn((B, H, N, d), generator=g, dtype=torch.float32)
    k = torch.randn((B, H, N, d), generator=g, dtype=torch.float32)
    v = torch.randn((B, H, N, d), generator=g, dtype=torch.float32)
    # a shared direction u: q.u = 1, k_j.u = ramp_j, so s_ij gains scale * d * ramp_j / d
    q[..., 0] = 1.0
    ramp = torch.arange(N, dtype=torch.float32) * (step / 128.0) / scale
    k[..., 0] = ramp
    return (q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16),
            float(np.float32(scale)))


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [True, False])
def test_rescale_on_every_tile(d, causal):
    B, H, N = 1, 3, 1000
    q, k, v, scale = _ramp_inputs(B, H, N, d, seed=40 + d, step=9.0)
    rows = workloads.select_rows(W["n1k"], B=B, H=H, N=N, seed=41)
    o, lse = _parity.run_gpu(q, k, v, causal, scale)
    og, lg = _parity.gather_rows(o, lse, rows)
    import oracle
    o64, lse64 = oracle.attn_rows(q, k, v, rows, causal, scale)
    _parity.compare(og, lg, o64, lse64)


def test_many_units_and_grid_cap_same_bits():
    w = W["n1k"]
    q, k, v = (t.cuda() for t in workloads.make_inputs(w, B=2, H=20, N=1500, d=D, seed=33))
    a, la = fa.fa_fwd(q, k, v, causal=True)
    b, lb = fa.fa_fwd(q, k, v, causal=True, options=fa.FwdOptions(max_ctas=5))
    assert fa.get_device_status() == fa.FA_OK
    assert torch.equal(a, b) and torch.equal(la, lb)
    rows = workloads.select_rows(w, B=2, H=20, N=1500, seed=33)
    og, lg = _parity.gather_rows(a, la, rows)
    import oracle
    o64, lse64 = oracle.attn_rows(q.cpu(), k.cpu(), v.cpu(), rows, True,
                                  float(np.float32(1 / np.sqrt(D))))
    _parity.compare(og, lg, o64, lse64)


def test_scale_zero_gives_prefix_means():
    w = W["n1k"]
    q, k, v = workloads.make_inputs(w, B=1, H=2, N=300, d=D, seed=34)
    o, lse = _parity.run_gpu(q, k, v, True, 0.0)
    vv = v.double().reshape(2, 300, D)
    means = torch.cumsum(vv, dim=1) / torch.arange(1, 301, dtype=torch.float64)[None, :, None]
    assert (o.reshape(2, 300, D).double().cpu() - means).abs().max() <= 8e-3
    assert (lse.reshape(2, 300).double().cpu()
            - torch.log(torch.arange(1, 301, dtype=torch.float64))).abs().max() <= 1e-3


def test_guard_regions_and_determinism():
    B, H, N = 1, 3, 333
    q, k, v = (t.cuda() for t in workloads.make_inputs(W["n1k"], B=B, H=H, N=N, d=D, seed=35))
    pad = 4096
    obuf = torch.full((pad + B * H * N * D + pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    lbuf = torch.full((pad + B * H * N + pad,), -3.0, dtype=torch.float32, device="cuda")
    o = obuf[pad:pad + B * H * N * D].view(B, H, N, D)
    lse = lbuf[pad:pad + B * H * N].view(B, H, N)
    fa.fa_fwd(q, k, v, o=o, lse=lse, causal=True)
    o2, l2 = fa.fa_fwd(q, k, v, causal=True)
    assert fa.get_device_status() == fa.FA_OK
    assert torch.all(obuf[:pad] == 7.0) and torch.all(obuf[-pad:] == 7.0)
    assert torch.all(lbuf[:pad] == -3.0) and torch.all(lbuf[-pad:] == -3.0)
    assert torch.equal(o, o2) and torch.equal(lse, l2)


def test_split_entry_points():
    """splits = 0 plans the launch; an explicit split runs the one-tile kernel in pieces;
    the allocation-free entry point matches; all against the unsplit result's oracle."""
    w = W["n1k"]
    q, k, v = workloads.make_inputs(w, B=1, H=2, N=700, d=D, seed=36)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    scale = float(np.float32(1 / 16))
    rows = workloads.select_rows(w, B=1, H=2, N=700, seed=37)
    o64, lse64 = oracle.attn_rows(q, k, v, rows, True, scale)
    for splits in (0, 2):
        o, lse = fa.fa_fwd_splitkv(qd, kd, vd, causal=True, scale=scale, splits=splits)
        assert fa.get_device_status() == fa.FA_OK
        _parity.compare(*_parity.gather_rows(o, lse, rows), o64, lse64)
    o3 = torch.empty_like(qd)
    l3 = torch.empty((1, 2, 700), dtype=torch.float32, device="cuda")
    rc = fa.fa_fwd_splitkv_noalloc_raw(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o3.data_ptr(),
                                       l3.data_ptr(), 1, 2, 700, D, True, scale, 3)
    assert rc == fa.FA_OK
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    _parity.compare(*_parity.gather_rows(o3, l3, rows), o64, lse64)
