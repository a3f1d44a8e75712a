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


@pytest.mark.parametrize("fake_regs", [120, 96])
def test_register_split_mismatch_is_refused_before_launch(fake_regs):
    """The two-tile kernel's setmaxnreg split needs exactly 128 registers per thread at
    launch; a build with another allocation would wait forever in setmaxnreg.inc.  With
    the test hook standing in for such a build (no such kernel is compiled or run), the
    launch is refused on the host and nothing is written; with the hook cleared the same
    call runs and is correct."""
    w = workloads.WORKLOADS["n1k"]
    q, k, v = workloads.make_inputs(w, B=1, H=2, N=640, d=128, seed=23)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o = torch.full_like(qd, 7.0)
    lse = torch.full((1, 2, 640), 7.0, device="cuda")
    scale = float(np.float32(1.0 / np.sqrt(128)))
    two = fa.FwdOptions(kernel=fa.FA_KERNEL_TWO_TILE)
    try:
        fa.override_kernel_registers_for_test(fake_regs)
        rc = fa.fa_fwd_raw(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                           lse.data_ptr(), 1, 2, 640, 128, True, scale, options=two)
        assert rc == fa.FA_ERR_UNSUPPORTED
        assert "setmaxnreg" in fa.last_error() and str(fake_regs) in fa.last_error()
        torch.cuda.synchronize()
        assert torch.all(o == 7.0) and torch.all(lse == 7.0)   # nothing was launched
        # the one-tile kernel does not use setmaxnreg and still runs
        one = fa.FwdOptions(kernel=fa.FA_KERNEL_ONE_TILE)
        assert fa.fa_fwd_raw(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                             lse.data_ptr(), 1, 2, 640, 128, True, scale, options=one) == fa.FA_OK
    finally:
        fa.override_kernel_registers_for_test(0)
    assert fa.get_device_status() == fa.FA_OK
    stats, _ = _parity.check_case(w, True, B=1, H=2, N=640, d=128, seed=23,
                                  kernel=fa.FA_KERNEL_TWO_TILE)
    assert stats["o_max_abs"] < 8e-3
