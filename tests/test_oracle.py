"""Pins for the CPU oracle: what the pages and the mathematics fix, independent of the oracle.

Page citations:
  [lab.py]     aiml.sh "Speed up long contexts with FlashAttention", lab.py
  [run-output] the same example's run-output.txt (JSON printed by lab.py)
  [cfs-model]  chipfoundryservices.com "edge/flashattention" reduced-order model
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import ref
import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _page_inputs():
    g = _golden("page_equivalence_check.json")
    q, k, v = workloads.make_qkv_page(g["seq_len"], g["head_dim"], g["seed"])
    return g, np.array(q), np.array(k), np.array(v)


def _c_oracle_head(q, k, v, causal, scale):
    """Run the C oracle on one fp64 head, every row."""
    o, lse = oracle.attn_full(q[None], k[None], v[None], causal, scale)
    return o[0], lse[0]


# ----------------------------------------------------------------------------------------
# 1. values the page prints for its worked example ([run-output] equivalence_check)
# ----------------------------------------------------------------------------------------
def test_page_sample_rows_all_three_implementations():
    g, q, k, v = _page_inputs()
    scale = 1.0 / math.sqrt(g["head_dim"])
    dense, _, _ = ref.dense_attention(q, k, v, causal=True)
    tiled, _, _ = ref.tiled_attention(q, k, v, g["block_q"], g["block_kv"], causal=True)
    c_o, _ = _c_oracle_head(q, k, v, True, scale)
    tol = 0.5 * 10 ** -g["samples_rounded_to_decimals"] + 1e-12
    for out in (dense, tiled, c_o):
        np.testing.assert_allclose(out[0, :4], g["sample_row0_first4"], rtol=0, atol=tol)
        np.testing.assert_allclose(out[-1, :4], g["sample_last_row_first4"], rtol=0, atol=tol)


def test_page_counters():
    g, q, k, v = _page_inputs()
    _, _, dmeta = ref.dense_attention(q, k, v, causal=True)
    _, _, tmeta = ref.tiled_attention(q, k, v, g["block_q"], g["block_kv"], causal=True)
    assert dmeta["materialized_nxn_elements"] == g["standard_materialized_elements"]
    assert tmeta["materialized_nxn_elements"] == g["flash_materialized_hbm_elements"]
    assert tmeta["max_sram_score_tile_elements"] == g["flash_sram_tile_elements"]
    assert tmeta["tiles_visited"] == g["flash_tiles_visited"]


def test_page_dense_equals_tiled_to_1e12():
    """The page finds 1.388e-16; summation order differs, so 1e-12 is the bound."""
    g, q, k, v = _page_inputs()
    dense, dlse, _ = ref.dense_attention(q, k, v, causal=True)
    tiled, tlse, _ = ref.tiled_attention(q, k, v, g["block_q"], g["block_kv"], causal=True)
    assert ref.max_abs_diff(dense, tiled) <= 1e-12
    assert ref.max_abs_diff(dlse, tlse) <= 1e-12
    assert ref.max_abs_diff(dense, tiled) < 100 * g["max_abs_diff"]


@pytest.mark.parametrize("bq,bkv", [(1, 1), (7, 13), (13, 7), (16, 64), (64, 16), (64, 64), (5, 3)])
@pytest.mark.parametrize("causal", [True, False])
def test_dense_equals_tiled_any_blocking(bq, bkv, causal):
    _, q, k, v = _page_inputs()
    dense, dlse, _ = ref.dense_attention(q, k, v, causal=causal)
    tiled, tlse, meta = ref.tiled_attention(q, k, v, bq, bkv, causal=causal)
    assert ref.max_abs_diff(dense, tiled) <= 1e-12
    assert ref.max_abs_diff(dlse, tlse) <= 1e-12
    n = q.shape[0]
    nq = -(-n // bq)
    if causal:
        expect = sum(min(-(-min(n, (b + 1) * bq) // bkv), -(-n // bkv)) for b in range(nq))
    else:
        expect = nq * (-(-n // bkv))
    assert meta["tiles_visited"] == expect


def test_negative_control_no_rescale_disagrees():
    """The page's rescale_previous_acc=False variant drops the alpha factor: it must fail."""
    g, q, k, v = _page_inputs()
    dense, _, _ = ref.dense_attention(q, k, v, causal=True)
    broken, _, _ = ref.tiled_attention(q, k, v, 16, 16, causal=True, rescale_previous_acc=False)
    assert ref.max_abs_diff(dense, broken) > 1e-3


# ----------------------------------------------------------------------------------------
# 2. special cases and closed forms
# ----------------------------------------------------------------------------------------
def test_causal_row0_is_v0_and_lse0_is_its_score():
    g, q, k, v = _page_inputs()
    scale = 0.25
    for qq, kk, vv in ((q, k, v),
                       tuple(t.double().reshape(64, 16).numpy()
                             for t in workloads.make_inputs(workloads.WORKLOADS["page"]))):
        o, lse = _c_oracle_head(qq, kk, vv, True, scale)
        assert np.array_equal(o[0], vv[0])          # a single admissible key: p = 1 exactly
        assert lse[0] == pytest.approx(scale * float(qq[0] @ kk[0]), abs=1e-15)
        d_o, d_lse, _ = ref.dense_attention(qq, kk, vv, causal=True, scale=scale)
        assert np.array_equal(d_o[0], vv[0])


@pytest.mark.parametrize("which", ["k_zero", "q_zero", "scale_zero"])
def test_uniform_weights_give_prefix_means(which):
    rng = np.random.default_rng(5)
    n, d = 37, 8
    q, k, v = rng.uniform(-1, 1, (3, n, d))
    scale = 0.3
    if which == "k_zero":
        k = np.zeros_like(k)
    elif which == "q_zero":
        q = np.zeros_like(q)
    else:
        scale = 0.0
    o, lse = _c_oracle_head(q, k, v, True, scale)
    means = np.cumsum(v, axis=0) / np.arange(1, n + 1)[:, None]
    np.testing.assert_allclose(o, means, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, np.log(np.arange(1, n + 1)), rtol=0, atol=1e-14)
    o2, lse2 = _c_oracle_head(q, k, v, False, scale)
    np.testing.assert_allclose(o2, np.broadcast_to(v.mean(0), o2.shape), rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse2, math.log(n), rtol=0, atol=1e-14)


def test_constant_values_and_probabilities_sum_to_one():
    rng = np.random.default_rng(6)
    n, d = 50, 16
    q, k = rng.normal(0, 3, (2, n, d))
    for causal in (True, False):
        v = np.full((n, d), 0.75)
        o, _ = _c_oracle_head(q, k, v, causal, 0.25)
        np.testing.assert_allclose(o, 0.75, rtol=0, atol=1e-14)
        # V = 1 reads back sum_j p_j: the probabilities of every row sum to one
        o1, _ = _c_oracle_head(q, k, np.ones((n, d)), causal, 0.25)
        np.testing.assert_allclose(o1, 1.0, rtol=0, atol=1e-14)


def test_output_in_convex_hull_of_values():
    rng = np.random.default_rng(7)
    n, d = 64, 16
    q, k, v = rng.normal(0, 2, (3, n, d))
    o, _ = _c_oracle_head(q, k, v, True, 0.25)
    for i in range(n):
        assert np.all(o[i] >= v[: i + 1].min(0) - 1e-14)
        assert np.all(o[i] <= v[: i + 1].max(0) + 1e-14)


def test_key_shift_invariance():
    """Adding a common vector u to every key moves each score row by scale*q_i.u:
    O is unchanged and lse moves by exactly that amount."""
    rng = np.random.default_rng(8)
    n, d = 40, 16
    q, k, v = rng.uniform(-1, 1, (3, n, d))
    u = rng.uniform(-1, 1, d)
    s = 0.25
    o, lse = _c_oracle_head(q, k, v, True, s)
    o2, lse2 = _c_oracle_head(q, k + u, v, True, s)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse2 - lse, s * (q @ u), rtol=0, atol=1e-13)


def test_noncausal_joint_key_value_permutation_invariance():
    rng = np.random.default_rng(9)
    n, d = 45, 16
    q, k, v = rng.uniform(-1, 1, (3, n, d))
    perm = rng.permutation(n)
    o, lse = _c_oracle_head(q, k, v, False, 0.25)
    o2, lse2 = _c_oracle_head(q, k[perm], v[perm], False, 0.25)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-13)
    # and a causal mask is NOT permutation invariant (sensitivity of the mask index)
    o3, _ = _c_oracle_head(q, k[perm], v[perm], True, 0.25)
    assert np.max(np.abs(o3 - _c_oracle_head(q, k, v, True, 0.25)[0])) > 1e-3


def test_heads_are_independent():
    rng = np.random.default_rng(10)
    H, n, d = 3, 20, 8
    q, k, v = rng.uniform(-1, 1, (3, H, n, d))
    o, lse = oracle.attn_full(q, k, v, True, 0.5)
    for h in range(H):
        oh, lh = _c_oracle_head(q[h], k[h], v[h], True, 0.5)
        assert np.array_equal(o[h], oh) and np.array_equal(lse[h], lh)
    k2 = k.copy()
    k2[1] += 1.0
    o2, _ = oracle.attn_full(q, k2, v, True, 0.5)
    assert np.array_equal(o2[0], o[0]) and np.array_equal(o2[2], o[2])
    assert not np.array_equal(o2[1], o[1])


# ----------------------------------------------------------------------------------------
# 3. brute force on tiny inputs: textbook softmax without the max shift, plain loops
# ----------------------------------------------------------------------------------------
def _brute(q, k, v, causal, scale):
    n, d = len(q), len(q[0])
    out, lses = [], []
    for i in range(n):
        keys = range(i + 1) if causal else range(n)
        w = {}
        for j in keys:
            t = 0.0
            for c in range(d):
                t += q[i][c] * k[j][c]
            w[j] = math.exp(t * scale)
        z = sum(w.values())
        out.append([sum(w[j] / z * v[j][c] for j in keys) for c in range(d)])
        lses.append(math.log(z))
    return np.array(out), np.array(lses)


@pytest.mark.parametrize("n,d,seed", [(1, 1, 0), (2, 3, 1), (5, 4, 2), (8, 4, 3), (7, 2, 4)])
@pytest.mark.parametrize("causal", [True, False])
def test_brute_force_tiny(n, d, seed, causal):
    rng = np.random.default_rng(seed)
    q, k, v = rng.uniform(-1.5, 1.5, (3, n, d))
    scale = 0.7
    bo, bl = _brute(q.tolist(), k.tolist(), v.tolist(), causal, scale)
    co, cl = _c_oracle_head(q, k, v, causal, scale)
    do, dl, _ = ref.dense_attention(q, k, v, causal=causal, scale=scale, subtract_max=False)
    to, tl, _ = ref.tiled_attention(q, k, v, 3, 2, causal=causal, scale=scale)
    for o, l in ((co, cl), (do, dl), (to, tl)):
        np.testing.assert_allclose(o, bo, rtol=0, atol=1e-14)
        np.testing.assert_allclose(l, bl, rtol=0, atol=1e-14)


def test_bf16_and_f64_inputs_agree():
    """The bf16 path of the C oracle widens the bits exactly."""
    q, k, v = workloads.make_inputs(workloads.WORKLOADS["n1k"], H=2, N=96, d=32)
    rows = workloads.select_rows(workloads.WORKLOADS["n1k"], H=2, N=96)
    o_b, l_b = oracle.attn_rows(q, k, v, rows, True, 0.125)
    o_f, l_f = oracle.attn_rows(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                rows, True, 0.125)
    assert np.array_equal(o_b, o_f) and np.array_equal(l_b, l_f)


def test_planted_mistakes_are_caught():
    """Each plausible slip in the dense definition fails one of the pins above."""
    g, q, k, v = _page_inputs()
    page0 = np.array(g["sample_row0_first4"])
    pageN = np.array(g["sample_last_row_first4"])

    def pins_hold(fn):
        o = fn(q, k, v)
        return (np.max(np.abs(o[0, :4] - page0)) < 1e-6 and np.max(np.abs(o[-1, :4] - pageN)) < 1e-6)

    def planted(mask_shift=0, scale_mult=1.0, transpose_qk=False, swap_kv=False):
        def fn(q, k, v):
            n, d = q.shape
            s = (k @ q.T).T if not transpose_qk else (q @ k.T).T
            s = s * scale_mult / math.sqrt(d)
            out = np.zeros_like(q)
            vv = k if swap_kv else v
            for i in range(n):
                hi = min(n, max(1, i + 1 + mask_shift))
                e = np.exp(s[i, :hi] - s[i, :hi].max())
                out[i] = (e / e.sum()) @ vv[:hi]
            return out
        return fn

    assert pins_hold(planted())                       # the correct definition passes
    assert not pins_hold(planted(mask_shift=-1))      # strict j < i mask
    assert not pins_hold(planted(mask_shift=+1))      # one key too many
    assert not pins_hold(planted(scale_mult=math.sqrt(16)))  # scale dropped
    assert not pins_hold(planted(transpose_qk=True))  # S transposed
    assert not pins_hold(planted(swap_kv=True))       # K and V swapped


# ----------------------------------------------------------------------------------------
# 4. traffic and roofline models ([lab.py] estimate_hbm_bytes, [cfs-model])
# ----------------------------------------------------------------------------------------
def test_hbm_access_model_reproduces_page_sweep():
    for row in _golden("page_hbm_traffic_sweep.json")["rows"]:
        got = ref.hbm_access_model(row["seq_len"], row["num_heads"], row["head_dim"], 2, 128, 128)
        for key, val in row.items():
            assert got[key] == val, (row["seq_len"], key, got[key], val)


def test_reduced_order_model_reproduces_page_outputs():
    g = _golden("cfs_reduced_order_model.json")
    i = g["inputs"]
    m = ref.reduced_order_model(i["batch_size"], i["num_heads"], i["seq_length"], i["head_dim"],
                                i["elem_bytes"], i["sram_kb"], i["block_size"], bool(i["causal"]),
                                i["hbm_bandwidth_gb_s"], i["compute_tops"])
    out = g["outputs"]
    for key, val in out.items():
        if isinstance(val, (bool, str)):
            assert m[key] == val, key
        elif isinstance(val, int):
            assert m[key] == val, key
        else:
            decimals = len(repr(val).split(".")[1]) if "." in repr(val) else 0
            assert round(m[key], decimals) == pytest.approx(val, abs=10 ** -decimals / 2 + 1e-9), key


def test_reduced_order_model_profile_points():
    g = _golden("cfs_reduced_order_model.json")
    i = g["inputs"]
    xs = ref.model_seq_points(count=g["profile_count"])
    assert len(xs) == 48 and xs[0] == 512.0 and xs[-1] == pytest.approx(131072.0)
    lookup = {round(x, 1): x for x in xs}
    for s, red in g["profile_points"]["reduction_vs_seq"]:
        m = ref.reduced_order_model(seq=lookup[s])
        assert round(m["hbm_reduction_x"], 3) == pytest.approx(red, abs=6e-4)
    for s, sp in g["profile_points"]["speedup_vs_seq"]:
        m = ref.reduced_order_model(seq=lookup[s])
        assert round(m["speedup_x"], 3) == pytest.approx(sp, abs=6e-4)


# ----------------------------------------------------------------------------------------
# 5. helpers: bf16 rounding floor, input generators
# ----------------------------------------------------------------------------------------
def test_bf16_round_matches_torch_on_fp32_values():
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.normal(0, 3, 20000), rng.uniform(-1e-3, 1e-3, 1000)]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    assert np.array_equal(oracle.bf16_round(x.astype(np.float64)), want)
    # ties go to even: 1 + 2^-8 sits halfway between 1 and 1 + 2^-7
    assert oracle.bf16_round(np.array([1.0 + 2.0 ** -8]))[0] == 1.0
    assert oracle.bf16_round(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 1.0 + 2 * 2.0 ** -7


def test_workload_generators_are_seeded_and_shaped():
    for name in ("page", "n1k"):
        w = workloads.WORKLOADS[name]
        kw = {} if name == "page" else dict(H=2, N=130)
        a = workloads.make_inputs(w, **kw)
        b = workloads.make_inputs(w, **kw)
        for x, y in zip(a, b):
            assert x.dtype == torch.bfloat16 and torch.equal(x, y)
        assert a[0].shape[-1] == w.d
    # the page generator rounds the page's own values
    q, _, _ = workloads.make_inputs(workloads.WORKLOADS["page"])
    q0, _, _ = workloads.make_qkv_page(64, 16, 42)
    assert torch.equal(q[0, 0], torch.tensor(q0, dtype=torch.float64).to(torch.bfloat16))
    n = workloads.make_inputs(workloads.WORKLOADS["n32k"], H=2, N=4096)
    assert 2.7 < float(n[0].float().std()) < 3.3 and 0.9 < float(n[2].float().std()) < 1.1


def test_row_selection():
    w = workloads.WORKLOADS["b8n8k"]
    rows = workloads.select_rows(w, B=1, H=3, N=1000)
    assert rows.shape == (3 * 256, 2)
    for bh in range(3):
        r = rows[rows[:, 0] == bh, 1]
        assert r[0] == 0 and r[-1] == 999 and np.all(np.diff(r) > 0)
    w3 = workloads.WORKLOADS["n4k"]
    rows3 = workloads.select_rows(w3, H=8, N=2048)
    counts = np.bincount(rows3[:, 0], minlength=8)
    assert sorted(counts.tolist()) == [512] * 4 + [2048] * 4
    assert np.array_equal(rows3, workloads.select_rows(w3, H=8, N=2048))
