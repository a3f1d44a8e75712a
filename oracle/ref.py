"""fp64 restatements of what the source pages compute -- TEST INFRASTRUCTURE ONLY.

Sources (cited by page and by the function or JSON key on it):

* [lab.py]  aiml.sh "Speed up long contexts with FlashAttention", ``lab.py``:
  ``standard_attention`` (dense, materialised softmax), ``tiled_flash_attention``
  (block loop with a running max / running sum / rescaled accumulator),
  ``estimate_hbm_bytes`` (access-count traffic model).
* [run-output]  the same example's ``run-output.txt``: the JSON those functions
  print (``equivalence_check``, ``hbm_traffic_sweep``).
* [cfs-model]  chipfoundryservices.com "edge/flashattention": a reduced-order
  roofline / HBM model (``inputs``, ``outputs``, ``profile``).

The code is written from what the pages compute, vectorised with numpy where the
page loops over columns; the order of the algorithmic steps is the pages' order.
Nothing here is used by the CUDA path.
"""
from __future__ import annotations

import math

import numpy as np


def _as_f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


# --------------------------------------------------------------------------------------
# Dense attention: [lab.py] standard_attention
# --------------------------------------------------------------------------------------
def dense_attention(q, k, v, causal: bool = True, scale: float | None = None,
                    subtract_max: bool = True):
    """Materialised attention for one head, fp64.

    Scores S = scale * Q K^T, kept only for keys j <= i when causal (the page
    truncates row i to i+1 entries).  Each row is turned into probabilities by
    exp(s - m) / sum, with m the row maximum (or 0 when ``subtract_max`` is off,
    the page's textbook variant), and O = P V.

    Returns (O [N, d], lse [N], counters); ``lse`` is ln(sum_j exp(s_j)) of the
    scaled, masked scores (a plain definition; the pages do not compute it) and
    ``counters["materialized_nxn_elements"]`` counts the S and P entries the
    dense path holds, as the page does.
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    n, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.zeros((n, v.shape[1]))
    lse = np.zeros(n)
    held = 0
    for i in range(n):
        nkeys = i + 1 if causal else n
        s = (k[:nkeys] @ q[i]) * scale          # one materialised score row
        m = s.max() if subtract_max else 0.0
        e = np.exp(s - m)
        denom = e.sum()
        p = e / denom                           # one materialised probability row
        out[i] = p @ v[:nkeys]
        lse[i] = m + math.log(denom)
        held += 2 * nkeys
    return out, lse, {"materialized_nxn_elements": held}


# --------------------------------------------------------------------------------------
# Tiled online softmax: [lab.py] tiled_flash_attention
# --------------------------------------------------------------------------------------
def tiled_attention(q, k, v, block_q: int = 16, block_kv: int = 16, causal: bool = True,
                    scale: float | None = None, rescale_previous_acc: bool = True):
    """Blocked attention with an online softmax, fp64, in the page's step order.

    For each block of ``block_q`` query rows keep, per row, a running maximum m
    (initially -inf), a running sum l (0) and an accumulator acc (0).  Walk the
    key/value blocks in order, stopping at the first block that starts at or
    after the query block's end when causal.  For each row with at least one
    admissible key in the block (j <= i when causal):

      tile_max = max of the row's scaled scores in the block
      new_max  = max(m, tile_max)
      alpha    = exp(m - new_max), or 0 while m is still -inf
      l        = l * alpha + sum exp(s - new_max)
      acc      = acc * alpha + sum exp(s - new_max) v_j   (alpha replaced by 1 when
                 ``rescale_previous_acc`` is off: the page's broken variant)
      m        = new_max

    and finally O = acc / l.  Returns (O, lse, counters) where lse = m + ln l and
    the counters are the page's ``tiles_visited`` and ``max_sram_score_tile_elements``
    (plus ``materialized_nxn_elements`` = 0).
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    n, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.zeros((n, v.shape[1]))
    lse = np.zeros(n)
    tiles = 0
    for q0 in range(0, n, block_q):
        q1 = min(q0 + block_q, n)
        rows = q1 - q0
        run_max = np.full(rows, -np.inf)
        run_sum = np.zeros(rows)
        acc = np.zeros((rows, v.shape[1]))
        for k0 in range(0, n, block_kv):
            if causal and k0 >= q1:
                break
            k1 = min(k0 + block_kv, n)
            tiles += 1
            for r in range(rows):
                i = q0 + r
                hi = min(k1, i + 1) if causal else k1
                if hi <= k0:
                    continue                      # no admissible key in this block
                s = (k[k0:hi] @ q[i]) * scale
                tile_max = s.max()
                new_max = max(run_max[r], tile_max)
                alpha = math.exp(run_max[r] - new_max) if run_max[r] > -math.inf else 0.0
                ex = np.exp(s - new_max)
                run_sum[r] = run_sum[r] * alpha + ex.sum()
                acc_scale = alpha if rescale_previous_acc else 1.0
                acc[r] = acc[r] * acc_scale + ex @ v[k0:hi]
                run_max[r] = new_max
        out[q0:q1] = acc / run_sum[:, None]
        lse[q0:q1] = run_max + np.log(run_sum)
    return out, lse, {
        "materialized_nxn_elements": 0,
        "max_sram_score_tile_elements": block_q * block_kv,
        "tiles_visited": tiles,
    }


def max_abs_diff(a, b) -> float:
    """Largest elementwise |a - b| ([lab.py] max_abs_diff)."""
    return float(np.max(np.abs(_as_f64(a) - _as_f64(b))))


# --------------------------------------------------------------------------------------
# Traffic and roofline models: [lab.py] estimate_hbm_bytes, [cfs-model] outputs
# --------------------------------------------------------------------------------------
def hbm_access_model(seq_len: int, num_heads: int = 32, head_dim: int = 128,
                     bytes_per_elem: int = 2, block_q: int = 128, block_kv: int = 128) -> dict:
    """Logical HBM bytes of one multi-head attention layer ([lab.py] estimate_hbm_bytes).

    * q, k, v read and o written once:          4 H N d bytes_per_elem
    * the materialised path writes S, reads S, writes P, reads P (full N x N per head):
                                                 4 H N^2 bytes_per_elem
    * causal query-block tiling with no reuse between blocks: each query block of
      ``block_q`` rows starting at ``start`` reads min(N, start + block_q) key rows and
      as many value rows, on top of reading Q and writing O once:
                                                 (2 H N d + 2 H kv_rows d) bytes_per_elem
    Raw byte counts are returned beside the page's MB fields (rounded to 2 places).
    """
    n, h, dh, b = seq_len, num_heads, head_dim, bytes_per_elem
    qkvo = 4 * h * n * dh * b
    nxn = 4 * h * n * n * b
    q_blocks = -(-n // block_q)
    kv_rows = sum(min(n, s + block_q) for s in range(0, n, block_q))
    tiled = (2 * h * n * dh + 2 * h * kv_rows * dh) * b
    return {
        "seq_len": n, "num_heads": h, "head_dim": dh,
        "qkvo_bytes": qkvo, "nxn_bytes": nxn, "standard_total_bytes": qkvo + nxn,
        "tiled_no_reuse_bytes": tiled, "kv_rows_read": kv_rows,
        "standard_qkv_o_mb": round(qkvo / 1e6, 2),
        "standard_nxn_matrix_hbm_mb": round(nxn / 1e6, 2),
        "standard_total_hbm_mb": round((qkvo + nxn) / 1e6, 2),
        "tiled_logical_access_mb_no_cache_reuse": round(tiled / 1e6, 2),
        "qkvo_compulsory_bytes_mb": round(qkvo / 1e6, 2),
        "num_q_blocks": q_blocks,
    }


def reduced_order_model(batch: int = 8, heads: int = 32, seq: float = 8192, head_dim: int = 128,
                        elem_bytes: float = 2.0, sram_kb: float = 192.0, block: int = 128,
                        causal: bool = True, hbm_gb_s: float = 3350.0,
                        tflops: float = 990.0) -> dict:
    """The [cfs-model] roofline arithmetic for one attention forward.

    FLOPs are the two N x N x d products, 4 B H S^2 d, halved when causal.  The
    fused kernel moves Q, K, V, O once (4 B H S d elem_bytes); the naive one also
    writes and reads the score matrix (B H S^2 elem_bytes, halved when causal).
    Times are max(FLOPs / peak, bytes / bandwidth) on the assumed machine; SRAM
    need is four block x d tiles (my reading: Q, K, V and O tiles).
    """
    f = 0.5 if causal else 1.0
    flops = 4.0 * batch * heads * seq * seq * head_dim * f
    fa_bytes = 4.0 * batch * heads * seq * head_dim * elem_bytes
    scores = batch * heads * seq * seq * elem_bytes * f
    naive_bytes = fa_bytes + 2.0 * scores
    peak = tflops * 1e12
    bw = hbm_gb_s * 1e9
    compute_s = flops / peak
    fa_s = max(compute_s, fa_bytes / bw)
    naive_s = max(compute_s, naive_bytes / bw)
    sram_needed_kb = 4.0 * block * head_dim * elem_bytes / 1024.0
    max_block = int(sram_kb * 1024.0 // (4.0 * head_dim * elem_bytes))
    balance = peak / bw
    return {
        "flops_gflop": flops / 1e9,
        "fa_hbm_gb": fa_bytes / 1e9,
        "scores_matrix_gb": scores / 1e9,
        "naive_hbm_gb": naive_bytes / 1e9,
        "hbm_reduction_x": naive_bytes / fa_bytes,
        "machine_balance_flop_byte": balance,
        "arithmetic_intensity_fa": flops / fa_bytes,
        "arithmetic_intensity_naive": flops / naive_bytes,
        "fa_bottleneck": "compute" if flops / fa_bytes >= balance else "memory bandwidth",
        "naive_bottleneck": "compute" if flops / naive_bytes >= balance else "memory bandwidth",
        "compute_time_ms": compute_s * 1e3,
        "fa_time_ms": fa_s * 1e3,
        "naive_time_ms": naive_s * 1e3,
        "speedup_x": naive_s / fa_s,
        "sram_needed_kb": sram_needed_kb,
        "sram_fit": sram_needed_kb <= sram_kb,
        "max_block_sram": max_block,
        "q_blocks": int(math.ceil(seq / block)),
        "kv_blocks": int(math.ceil(seq / block)),
    }


def model_seq_points(lo: float = 512.0, hi: float = 131072.0, count: int = 48) -> list:
    """The [cfs-model] ``profile`` abscissae: ``count`` geometrically spaced lengths."""
    r = (hi / lo) ** (1.0 / (count - 1))
    return [lo * r ** i for i in range(count)]
