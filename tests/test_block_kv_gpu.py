"""GPU parity of the key-tile width option (fa_fwd_options.block_kv).

aiml.sh "Speed up long contexts with FlashAttention" (lab.py `tiled_flash_attention`)
takes the query and key block sizes as arguments; the result does not depend on them.
Here block_kv = 64 runs the two-tile kernel with 64-key score tiles (half the keys per
online-softmax step and per S/PV MMA pair) and must meet the same oracle gates as the
default 128: every head dim it serves, ragged and tiny N, causal and not, the
large-logit workload that exercises the rescale, and split launches.
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


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.load_library()


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("N", [1, 2, 63, 64, 65, 127, 128, 129, 191, 257, 700])
@pytest.mark.parametrize("causal", [True, False])
def test_ragged_and_small(d, N, causal):
    w = W["n1k"]
    rows = workloads.select_rows(w, B=2, H=3, N=N, seed=N + d + 5)
    _parity.check_case(w, causal, B=2, H=3, N=N, d=d, seed=N * 13 + d, rows=rows, block_kv=64)


@pytest.mark.parametrize("d", [64, 128])
def test_large_logits(d):
    """Q, K ~ N(0, 9), V ~ N(0, 1): the running maximum moves often, O is rescaled."""
    _parity.check_case(W["n32k"], True, B=1, H=4, N=2048, d=d, seed=71, block_kv=64)


def test_n1k_full_tensor():
    _parity.check_case(W["n1k"], True, block_kv=64)


@pytest.mark.parametrize("causal", [True, False])
def test_n4k_sampled_rows(causal):
    _parity.check_case(W["n4k"], causal, block_kv=64)


def test_matches_128_key_tiles_closely():
    """Same inputs, 64- vs 128-key tiles: the same result up to accumulation order."""
    w = W["n1k"]
    q, k, v = (t.cuda() for t in workloads.make_inputs(w, B=1, H=8, N=1500, d=128, seed=5))
    a, la = fa.fa_fwd(q, k, v, causal=True, options=fa.FwdOptions(block_kv=64))
    b, lb = fa.fa_fwd(q, k, v, causal=True, options=fa.FwdOptions(block_kv=128))
    assert fa.get_device_status() == fa.FA_OK
    assert (a.float() - b.float()).abs().max().item() <= 8e-3
    assert (la - lb).abs().max().item() <= 1e-4


@pytest.mark.parametrize("splits", [2, 3, 0])
@pytest.mark.parametrize("d,N", [(128, 1024), (64, 700), (32, 2000)])
def test_split_launches(splits, d, N):
    w = W["n1k"]
    q, k, v = workloads.make_inputs(w, B=1, H=3, N=N, d=d, seed=N + splits)
    scale = float(np.float32(1.0 / np.sqrt(d)))
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o, lse = fa.fa_fwd_splitkv(qd, kd, vd, causal=True, scale=scale, splits=splits,
                               options=fa.FwdOptions(block_kv=64))
    assert fa.get_device_status() == fa.FA_OK
    rows = workloads.select_rows(w, B=1, H=3, N=N, seed=N)
    og, lg = _parity.gather_rows(o, lse, rows)
    o64, lse64 = oracle.attn_rows(q, k, v, rows, True, scale)
    _parity.compare(og, lg, o64, lse64)
