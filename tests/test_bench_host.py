"""Host-side logic of bench.py, on CPU: multi-rank timing reduction (gloo, 2 ranks),
per-rank sharding of the weak-scaling workload, FLOP accounting and the
reference (CPU oracle) arm's JSON line."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    bench.dist_init(world, "gloo")
    bench.barrier(world)
    t = bench.max_over_ranks(float(rank) + 1.5, world, torch.device("cpu"))
    seed = bench.shard_seed(1004, rank)
    seeds = [None] * world
    torch.distributed.all_gather_object(seeds, seed)
    out[rank] = (t, seeds)
    torch.distributed.destroy_process_group()


def test_two_rank_max_and_distinct_shards():
    world = 2
    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True,
                       start_method="spawn")
    for r in range(world):
        t, seeds = out[r]
        assert t == 2.5                      # the slowest rank's time is reported
        assert len(set(seeds)) == world      # every rank owns an independent batch


def test_single_rank_helpers():
    assert bench.max_over_ranks(3.0, 1, torch.device("cpu")) == 3.0
    bench.barrier(1)
    assert bench.model_flops(8, 32, 8192, 128, True) == pytest.approx(4398.046511104e9)
    assert bench.model_flops(1, 1, 64, 16, False) == 4.0 * 64 * 64 * 16
    # causal FLOPs of all rows, counted per row, equal the closed form 2 d N (N+1)
    rows = np.stack([np.zeros(100, dtype=np.int64), np.arange(100)], axis=1)
    assert bench.oracle_rows_flops(rows, 100, 16, True) == 2 * 16 * 100 * 101


def test_reference_arm_json_line():
    args = bench.parse_args(["--impl", "reference", "--B", "1", "--H", "2", "--N", "256", "--d", "16",
                             "--steps", "2", "--warmup", "1", "--ref-seconds", "0.3"])
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(args) == 0
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["higher_is_better"] is True and line["metric"] == bench.METRIC


def test_page_traffic_models_match_the_page():
    """bench.py's statement of the page's traffic model reproduces the printed sweep."""
    with open(os.path.join(ROOT, "tests", "golden", "page_hbm_traffic_sweep.json")) as f:
        rows = json.load(f)["rows"]
    for r in rows:
        m = bench.page_traffic_models(1, r["num_heads"], r["seq_len"], r["head_dim"])
        assert round(m["qkvo_bytes"] / 1e6, 2) == r["qkvo_compulsory_bytes_mb"]
        assert round(m["materialised_bytes"] / 1e6, 2) == r["standard_total_hbm_mb"]
        assert round(m["tiled_no_reuse_bytes"] / 1e6, 2) == r["tiled_logical_access_mb_no_cache_reuse"]


def test_peak_follows_the_timed_region():
    """A timed region shorter than bench.SUSTAINED_S is measured against the burst bf16
    peak, a longer one (at the power cap) against the sustained peak, when the driver's
    measurements hold both."""
    path = os.path.join(bench.ROOT, "MEASURED_PEAKS.json")
    if not os.path.exists(path):
        pytest.skip("no MEASURED_PEAKS.json")
    with open(path) as f:
        pk = json.load(f)
    if not pk.get("bf16_tflops") or not pk.get("bf16_tflops_sustained"):
        pytest.skip("MEASURED_PEAKS.json lacks a bf16 figure")
    short, src_short = bench.load_peaks(0.05)
    long_, src_long = bench.load_peaks(bench.SUSTAINED_S + 0.5)
    assert short == pytest.approx(pk["bf16_tflops"]) and "burst" in src_short
    assert long_ == pytest.approx(pk["bf16_tflops_sustained"]) and "sustained" in src_long
