"""Shared helpers for the GPU parity tests: run the C-ABI path, compare with the oracle.

Tolerances (fixed here, not tuned per case), each against the fp64 oracle run on
the same bf16 inputs:
  * O mean-abs <= 1e-3 over all checked elements;
  * lse max-abs <= 1e-3;
  * O max-abs <= 8e-3 on elements with |O| < 2, and within one bf16 ulp of the
    exact value on elements with |O| >= 2.
Why the split: a bf16 output is at best half a bf16 ulp from the exact value.  For
|O| in [2, 4) that floor reaches 7.8e-3, leaving 0.2e-3 for everything else (the P
matrix that feeds the tensor cores is itself bf16, a 2^-9 relative rounding per
weight), and for |O| >= 4 the floor alone exceeds 8e-3.  Below 2 the floor is at most
3.9e-3 and the stated 8e-3 applies as written.  Raw max-abs, the representability
floor and the count of elements above 8e-3 are reported with every comparison.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import tiled_online_softmax_fa_gb300 as fa
import workloads

O_MAX_ABS = 8e-3
O_MEAN_ABS = 1e-3
LSE_MAX_ABS = 1e-3
ULP_REGION = 2.0   # |O| at and above which the one-ulp gate applies


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    a = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def run_gpu(q, k, v, causal: bool, scale: float, want_lse: bool = True,
            kernel: int = fa.FA_KERNEL_AUTO, block_kv: int = 0):
    """fa_fwd on cuda:0; `kernel` pins FA_KERNEL_TWO_TILE or FA_KERNEL_ONE_TILE, `block_kv`
    the keys per K/V tile (0 = the library's choice)."""
    dev = torch.device("cuda:0")
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    opts = (fa.FwdOptions(kernel=kernel, block_kv=block_kv)
            if kernel != fa.FA_KERNEL_AUTO or block_kv else None)
    o, lse = fa.fa_fwd(qd, kd, vd, causal=causal, scale=scale, want_lse=want_lse, options=opts)
    status = fa.get_device_status()
    assert status == fa.FA_OK, fa.strerror(status)
    return o, lse


def gather_rows(o: torch.Tensor, lse: torch.Tensor | None, rows: np.ndarray):
    B, H, N, d = o.shape
    idx_bh = torch.as_tensor(rows[:, 0], device=o.device)
    idx_i = torch.as_tensor(rows[:, 1], device=o.device)
    og = o.reshape(B * H, N, d)[idx_bh, idx_i].double().cpu().numpy()
    lg = None
    if lse is not None:
        lg = lse.reshape(B * H, N)[idx_bh, idx_i].double().cpu().numpy()
    return og, lg


def compare(og: np.ndarray, lg, o64: np.ndarray, lse64: np.ndarray) -> dict:
    err = np.abs(og - o64)
    floor = np.abs(oracle.bf16_round(o64) - o64)
    big = np.abs(o64) >= ULP_REGION

    def mx(a):
        return float(a.max()) if a.size else 0.0

    stats = {
        "o_max_abs": mx(err), "o_mean_abs": float(err.mean()) if err.size else 0.0,
        "o_max_abs_below_2": mx(err[~big]), "o_max_abs_2_and_up": mx(err[big]),
        "o_floor_max": mx(floor), "o_floor_mean": float(floor.mean()) if floor.size else 0.0,
        "o_max_ulps_2_and_up": mx(err[big] / bf16_ulp(o64[big])) if big.any() else 0.0,
        "n_checked": int(err.size), "n_2_and_up": int(big.sum()),
        "n_over_8e-3": int((err > O_MAX_ABS).sum()),
    }
    assert np.all(np.isfinite(og)), "non-finite output"
    assert stats["o_max_abs_below_2"] <= O_MAX_ABS, stats
    assert np.all(err[big] <= bf16_ulp(o64[big])), stats
    assert stats["o_mean_abs"] <= O_MEAN_ABS, stats
    if lg is not None:
        lerr = np.abs(lg - lse64)
        stats["lse_max_abs"] = mx(lerr)
        assert np.all(np.isfinite(lg)), "non-finite lse"
        assert stats["lse_max_abs"] <= LSE_MAX_ABS, stats
    return stats


def check_case(w: workloads.Workload, causal: bool, B=None, H=None, N=None, d=None, seed=None,
               rows: np.ndarray | None = None, scale: float | None = None,
               kernel: int = fa.FA_KERNEL_AUTO, block_kv: int = 0):
    q, k, v = workloads.make_inputs(w, B=B, H=H, N=N, d=d, seed=seed)
    Bv, Hv, Nv, dv = q.shape
    if scale is None:
        scale = float(np.float32(1.0 / np.sqrt(dv)))
    if rows is None:
        rows = workloads.select_rows(w, B=Bv, H=Hv, N=Nv, seed=seed)
    o, lse = run_gpu(q, k, v, causal, scale, kernel=kernel, block_kv=block_kv)
    og, lg = gather_rows(o, lse, rows)
    o64, lse64 = oracle.attn_rows(q, k, v, rows, causal, scale)
    return compare(og, lg, o64, lse64), (q, k, v, o, lse)
