"""Failure detection without a GPU fault: a K/V tile load that is never issued.

The test hook makes work unit 0 skip one TMA load, so the MMA issuer's bounded
wait on that ring slot runs out.  The kernel must wind down on its own (every role
sees the CTA's abort flag, in-flight copies and MMAs are drained, TMEM is freed),
the host must read FA_ERR_DEVICE_TIMEOUT from the status word, and the context
must stay usable: the next call computes the right answer and reports FA_OK.
"""
import numpy as np
import pytest
import torch

import _parity
import tiled_online_softmax_fa_gb300 as fa
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.load_library()


@pytest.mark.parametrize("d,kernel", [(128, fa.FA_KERNEL_TWO_TILE), (128, fa.FA_KERNEL_ONE_TILE),
                                      (256, fa.FA_KERNEL_ONE_TILE)])
def test_skipped_load_times_out_and_context_survives(d, kernel):
    """Both kernels (the one-tile kernel has its own ring order and, at d = 128, two Q
    buffers and four ring slots to drain)."""
    w = workloads.WORKLOADS["n1k"]
    q, k, v = workloads.make_inputs(w, B=1, H=2, N=1024, d=d, seed=21)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    assert fa.get_device_status() == fa.FA_OK  # clean start
    opts = fa.FwdOptions(wait_budget_cycles=20_000_000, inject_skip_kv_load=3, kernel=kernel)
    fa.fa_fwd(qd, kd, vd, causal=True, options=opts)
    assert fa.get_device_status() == fa.FA_ERR_DEVICE_TIMEOUT
    # the status word was cleared by the read, and the next call is correct
    stats, _ = _parity.check_case(w, True, B=1, H=2, N=1024, d=d, seed=21, kernel=kernel)
    assert fa.get_device_status() == fa.FA_OK
    assert stats["o_max_abs"] < 8e-3
