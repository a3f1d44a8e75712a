"""GPU parity: the C-ABI kernel path against the fp64 CPU oracle, element by element.

Every case draws its inputs from ``workloads`` (seeded), runs ``fa_fwd`` through the
C ABI on cuda:0 and compares O and lse with the oracle on the same bf16 bits.
"""
import json
import os

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


def _report(name, stats):
    print(name, json.dumps(stats))
    path = os.environ.get("FA_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": name, **stats}) + "\n")


# ---------------------------------------------------------------------------------------
# the five workloads at their stated sizes
# ---------------------------------------------------------------------------------------
def test_page_example_all_rows():
    """B1 H1 N64 d16 causal, the page's generator (seed 42) rounded to bf16, scale 1/4."""
    stats, (q, k, v, o, lse) = _parity.check_case(W["page"], True, scale=0.25)
    # row 0 has one admissible key: P = 1 exactly, so O row 0 is v[0] bit for bit
    assert torch.equal(o[0, 0, 0].cpu(), v[0, 0, 0])
    _report("page", stats)


def test_n1k_full_tensor():
    stats, _ = _parity.check_case(W["n1k"], True)
    _report("n1k", stats)


@pytest.mark.parametrize("causal", [True, False])
def test_n4k_heads_and_sampled_rows(causal):
    stats, _ = _parity.check_case(W["n4k"], causal)
    _report(f"n4k causal={causal}", stats)


def test_b8n8k_sampled_rows():
    """The throughput shape: 256 seeded rows per (b, h), rows 0 and N-1 included."""
    stats, _ = _parity.check_case(W["b8n8k"], True)
    _report("b8n8k", stats)


def test_n32k_large_logits():
    """Q,K ~ N(0, 9), V ~ N(0, 1): logits of std ~9 stress the max shift and rescale."""
    stats, _ = _parity.check_case(W["n32k"], True)
    _report("n32k", stats)


# ---------------------------------------------------------------------------------------
# shapes: ragged tails, tiny sequences, every head dim, several heads and batches
# ---------------------------------------------------------------------------------------
@pytest.mark.parametrize("d", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("N", [1, 2, 3, 127, 128, 129, 255, 256, 257, 383, 700])
@pytest.mark.parametrize("causal", [True, False])
def test_ragged_and_small(d, N, causal):
    w = W["n1k"]
    rows = workloads.select_rows(w, B=2, H=3, N=N, seed=N + d)
    _parity.check_case(w, causal, B=2, H=3, N=N, d=d, seed=N * 7 + d, rows=rows)


@pytest.mark.parametrize("d", [16, 64, 128, 256])
def test_large_logits_ragged(d):
    _parity.check_case(W["n32k"], True, B=1, H=4, N=1000, d=d, seed=77 + d)


def test_many_units_per_cta():
    """More work units than SMs on both the causal and the non-causal path."""
    w = W["n1k"]
    for causal in (True, False):
        rows = workloads.select_rows(W["b8n8k"], B=4, H=40, N=1536, seed=5)
        _parity.check_case(w, causal, B=4, H=40, N=1536, d=128, seed=5, rows=rows)


def _sampled(N, per_head, BH, seed):
    """Rows 0 and N-1 of every head plus `per_head` seeded random rows (unique, sorted)."""
    rng = np.random.default_rng(seed)
    rows = []
    for bh in range(BH):
        idx = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, per_head)]))
        rows.extend((bh, int(i)) for i in idx)
    return np.asarray(rows, dtype=np.int64)


def test_longest_sequence_sampled_rows():
    """N = 131072 (one head's K and V exceed the L2 share of a CTA group), unsplit and
    split by key ranges; rows near the end attend to 131072 keys."""
    w, N = W["n1k"], 131072
    rows = _sampled(N, 24, 2, seed=131)
    stats, (q, k, v, o, lse) = _parity.check_case(w, True, B=1, H=2, N=N, d=128, seed=131,
                                                  rows=rows)
    _report("N131072", stats)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    scale = float(np.float32(1.0 / np.sqrt(128)))
    o2, l2 = fa.fa_fwd_splitkv(qd, kd, vd, causal=True, scale=scale, splits=0)
    assert fa.get_device_status() == fa.FA_OK
    og, lg = _parity.gather_rows(o2, l2, rows)
    o64, lse64 = oracle.attn_rows(q, k, v, rows, True, scale)
    _parity.compare(og, lg, o64, lse64)


def test_many_short_heads():
    """B*H = 4096 one-tile units (far more units than CTAs, every unit a single block)."""
    w = W["n1k"]
    rows = _sampled(64, 2, 64 * 64, seed=9)[::7]
    _parity.check_case(w, True, B=64, H=64, N=64, d=64, seed=9, rows=rows)


# ---------------------------------------------------------------------------------------
# closed forms and special inputs
# ---------------------------------------------------------------------------------------
def test_scale_zero_gives_prefix_means():
    w = W["n1k"]
    q, k, v = workloads.make_inputs(w, B=1, H=2, N=300, d=64, seed=3)
    o, lse = _parity.run_gpu(q, k, v, True, 0.0)
    vv = v.double().reshape(2, 300, 64)
    means = torch.cumsum(vv, dim=1) / torch.arange(1, 301, dtype=torch.float64)[None, :, None]
    assert (o.reshape(2, 300, 64).double().cpu() - means).abs().max() <= 8e-3
    assert (lse.reshape(2, 300).double().cpu()
            - torch.log(torch.arange(1, 301, dtype=torch.float64))).abs().max() <= 1e-3


def test_constant_values():
    w = W["n32k"]
    q, k, _ = workloads.make_inputs(w, B=1, H=2, N=600, d=128, seed=4)
    v = torch.full_like(q, 0.375)
    o, _ = _parity.run_gpu(q, k, v, True, float(np.float32(1 / np.sqrt(128))))
    assert torch.all(o.cpu() == 0.375)


def test_without_lse_output():
    w = W["n1k"]
    q, k, v = workloads.make_inputs(w, B=1, H=2, N=200, d=64, seed=6)
    o1, _ = _parity.run_gpu(q, k, v, True, 0.125, want_lse=False)
    o2, _ = _parity.run_gpu(q, k, v, True, 0.125, want_lse=True)
    assert torch.equal(o1, o2)


def test_deterministic_bits():
    w = W["n4k"]
    q, k, v = workloads.make_inputs(w, B=1, H=8, N=2048, d=128, seed=9)
    a, la = _parity.run_gpu(q, k, v, True, 0.088)
    b, lb = _parity.run_gpu(q, k, v, True, 0.088)
    assert torch.equal(a, b) and torch.equal(la, lb)


def test_grid_cap_gives_same_bits():
    """Fewer persistent CTAs (more units each) must not change a single bit."""
    w = W["n1k"]
    q, k, v = (t.cuda() for t in workloads.make_inputs(w, B=2, H=8, N=1100, d=128, seed=12))
    a, la = fa.fa_fwd(q, k, v, causal=True)
    b, lb = fa.fa_fwd(q, k, v, causal=True, options=fa.FwdOptions(max_ctas=7))
    assert fa.get_device_status() == fa.FA_OK
    assert torch.equal(a, b) and torch.equal(la, lb)


def test_empty_is_noop():
    z = torch.empty((0, 4, 128, 64), dtype=torch.bfloat16, device="cuda")
    rc = fa.fa_fwd_raw(z.data_ptr(), z.data_ptr(), z.data_ptr(), z.data_ptr(), 0, 0, 4, 128, 64,
                       True, 0.125)
    assert rc == fa.FA_OK


def test_guard_regions_untouched():
    """Canaries around o and lse: the kernel writes exactly [B, H, N, d] and [B, H, N]."""
    B, H, N, d = 1, 3, 333, 128
    w = W["n1k"]
    q, k, v = (t.cuda() for t in workloads.make_inputs(w, B=B, H=H, N=N, d=d, seed=10))
    pad = 4096
    obuf = torch.full((pad + B * H * N * d + pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    lbuf = torch.full((pad + B * H * N + pad,), -3.0, dtype=torch.float32, device="cuda")
    o = obuf[pad:pad + B * H * N * d].view(B, H, N, d)
    lse = lbuf[pad:pad + B * H * N].view(B, H, N)
    fa.fa_fwd(q, k, v, o=o, lse=lse, causal=True)
    assert fa.get_device_status() == fa.FA_OK
    assert torch.all(obuf[:pad] == 7.0) and torch.all(obuf[-pad:] == 7.0)
    assert torch.all(lbuf[:pad] == -3.0) and torch.all(lbuf[-pad:] == -3.0)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


def test_bad_arguments_launch_nothing():
    q = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.full_like(q, 5.0)
    rc = fa.fa_fwd_raw(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), 0, 1, 1, 128, 48,
                       True, 0.1)
    assert rc == fa.FA_ERR_UNSUPPORTED
    rc = fa.fa_fwd_raw(q.data_ptr() + 2, q.data_ptr(), q.data_ptr(), o.data_ptr(), 0, 1, 1, 64,
                       64, True, 0.1)
    assert rc == fa.FA_ERR_MISALIGNED
    rc = fa.fa_fwd_raw(q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), 0, 1, 1, 128, 64,
                       True, 0.1)
    assert rc == fa.FA_ERR_INVALID_ARG  # o aliases the inputs
    torch.cuda.synchronize()
    assert torch.all(o == 5.0)
