"""The C-ABI calls inside CUDA graphs: capture once, replay with new inputs.

Every forward entry point is asynchronous on the caller's stream and allocates nothing,
so after one warm-up call (the first call on a device sets the kernels' shared-memory
attribute and probes the device) it can be captured into a CUDA graph and replayed.
Each replay must give the same bits as an eager call on the same inputs, for the three
kinds of launch the planner picks: the two-tile kernel, the one-tile kernel and a split
launch with its merge kernel.
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


def _inputs(B, H, N, d, seed):
    return [t.cuda() for t in workloads.make_inputs(W["n4k"], B=B, H=H, N=N, d=d, seed=seed)]


@pytest.mark.parametrize("B,H,N,d,splitkv", [
    (2, 16, 4096, 128, False),   # two-tile kernel
    (1, 4, 8192, 128, False),    # one-tile kernel
    (1, 1, 8192, 128, True),     # key range split, partials merged by a second kernel
    (1, 8, 2048, 64, False),
])
def test_capture_and_replay(B, H, N, d, splitkv):
    q, k, v = _inputs(B, H, N, d, seed=1)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    scale = float(np.float32(1.0 / np.sqrt(d)))
    ws = None
    if splitkv:
        kernel, splits = fa.fwd_plan(B, H, N, d, True, allow_split=True)
        assert splits > 1
        ws = torch.empty(fa.splitkv_workspace_bytes(B, H, N, d, splits), dtype=torch.uint8,
                         device="cuda")

    def call():
        if splitkv:
            fa.fa_fwd_splitkv(q, k, v, o=o, lse=lse, causal=True, scale=scale, splits=0,
                              workspace=ws)
        else:
            fa.fa_fwd(q, k, v, o=o, lse=lse, causal=True, scale=scale)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()                       # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for seed in (2, 3):
        q2, k2, v2 = _inputs(B, H, N, d, seed)
        q.copy_(q2)
        k.copy_(k2)
        v.copy_(v2)
        g.replay()
        torch.cuda.synchronize()
        assert fa.get_device_status() == fa.FA_OK
        if splitkv:
            ref_o, ref_l = fa.fa_fwd_splitkv(q2, k2, v2, causal=True, scale=scale, splits=0)
        else:
            ref_o, ref_l = fa.fa_fwd(q2, k2, v2, causal=True, scale=scale)
        torch.cuda.synchronize()
        assert torch.equal(o, ref_o) and torch.equal(lse, ref_l)
    # and the last replay against the oracle
    rows = workloads.select_rows(W["n4k"], B=B, H=H, N=N, seed=4)
    o64, lse64 = oracle.attn_rows(q.cpu(), k.cpu(), v.cpu(), rows, True, scale)
    _parity.compare(*_parity.gather_rows(o, lse, rows), o64, lse64)


def test_one_graph_two_launches_on_shared_buffers():
    """Two forward calls of different shapes captured back to back in one graph."""
    qa, ka, va = _inputs(1, 32, 1024, 128, seed=5)
    qb, kb, vb = _inputs(4, 8, 2048, 64, seed=6)
    oa, ob = torch.empty_like(qa), torch.empty_like(qb)
    la = torch.empty((1, 32, 1024), dtype=torch.float32, device="cuda")
    lb = torch.empty((4, 8, 2048), dtype=torch.float32, device="cuda")

    def call():
        fa.fa_fwd(qa, ka, va, o=oa, lse=la, causal=True)
        fa.fa_fwd(qb, kb, vb, o=ob, lse=lb, causal=False)

    call()
    torch.cuda.synchronize()
    ea, eb, ela, elb = oa.clone(), ob.clone(), la.clone(), lb.clone()
    oa.zero_()
    ob.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    g.replay()
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    assert torch.equal(oa, ea) and torch.equal(ob, eb)
    assert torch.equal(la, ela) and torch.equal(lb, elb)
