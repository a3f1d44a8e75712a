#!/usr/bin/env python3
"""Throughput benchmark of the sm_103a attention forward pass.

Workload (one step = one fa_fwd call = the whole hot path over one batch):
    B=8, H=32, N=8192, d=128, causal, bf16 inputs iid U(-0.8, 0.8) (seed 1004),
    the shape of the chipfoundryservices.com "edge/flashattention" model.
Metric: TFLOP/s with FLOPs = 2*B*H*N^2*d (causal; 4*B*H*N^2*d non-causal).

Prints ONE JSON line.  ``value`` is device-timed with inputs resident in HBM (1.6 GB,
larger than L2, so no flush between steps; smaller --B/--H/--N shapes write a buffer
of twice the L2 size before every timed step, outside its events); ``e2e`` is the same metric through the
same C-ABI call with pinned host buffers and the host<->device copies in the timed
region; ``roofline`` relates the kernel to the measured bf16 tensor peak;
``cpu_baseline`` times the fp64 CPU oracle on a bounded sample of the same workload.

``--impl reference`` times that oracle alone as the reference arm.
Multi-GPU (torchrun): every rank runs its own copy of the workload (weak scaling,
no data-path collective); the reported time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "FA fwd TFLOP/s (causal 2BHN²d) at b8 h32 S8192 d128 bf16; % of GB300 BF16 peak"
UNIT = "TFLOP/s"
FALLBACK_BF16_TFLOPS = 1900.0
SUSTAINED_S = 0.5  # timed regions this long run at the power cap: the sustained peak applies
# The device code of the kernel the bench line times (head dims 16-128): an ncu traffic
# record applies only while these files are unchanged.
SOURCES = ["tiled_online_softmax_fa_gb300/csrc/fa_fwd_kernel.cuh",
           "tiled_online_softmax_fa_gb300/csrc/ptx_sm103.cuh",
           "tiled_online_softmax_fa_gb300/csrc/fa_fwd_row_kernel.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "fa_fwd_traffic.json")


def model_flops(B, H, N, d, causal) -> float:
    return (2.0 if causal else 4.0) * B * H * N * N * d


def page_traffic_models(B, H, N, d, elem_bytes=2, block_q=128) -> dict:
    """HBM bytes of one attention forward as the aiml.sh lab.py page counts them
    (`estimate_hbm_bytes`), for B batches: Q,K,V read and O written once; the
    materialised path adding S and P written and read (4 H N^2 elements); causal
    query-block tiling with no reuse between blocks reading min(N, start + block_q)
    key and value rows per block."""
    qkvo = 4 * H * N * d * elem_bytes
    nxn = 4 * H * N * N * elem_bytes
    kv_rows = sum(min(N, s + block_q) for s in range(0, N, block_q))
    tiled = (2 * H * N * d + 2 * H * kv_rows * d) * elem_bytes
    return {"qkvo_bytes": B * qkvo, "materialised_bytes": B * (qkvo + nxn),
            "tiled_no_reuse_bytes": B * tiled}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks(timed_s=0.0):
    """The bf16 peak for a roofline fraction: the burst figure for a kernel timed alone,
    the sustained one (a seconds-long loop under the power cap) once the timed region
    lasts SUSTAINED_S or more."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        if timed_s >= SUSTAINED_S and pk.get("bf16_tflops_sustained"):
            return (float(pk["bf16_tflops_sustained"]),
                    f"measured (MEASURED_PEAKS.json bf16_tflops_sustained: timed region {timed_s:.2f} s)")
        if pk.get("bf16_tflops"):
            return (float(pk["bf16_tflops"]),
                    f"measured (MEASURED_PEAKS.json bf16_tflops, burst: timed region {timed_s:.2f} s)")
    return FALLBACK_BF16_TFLOPS, "fallback (1.9 PFLOP/s bf16 burst, earlier GB300 measurement)"


# --------------------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------------------
class _Nvml:
    """Read-only NVML queries through ctypes (libnvidia-ml ships with the driver): the SM
    clock, its maximum, the power draw and the active clock-event (throttle) reasons."""
    CLOCK_SM = 1
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_index: int):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.dev = ctypes.c_void_p()
        ok = False
        try:   # the GPU torch calls `torch_index`, found by UUID (NVML ignores CUDA_VISIBLE_DEVICES)
            uuid = "GPU-" + str(torch.cuda.get_device_properties(torch_index).uuid)
            ok = self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.dev)) == 0
        except Exception:  # noqa: BLE001 - an older torch without .uuid
            ok = False
        if not ok and self.lib.nvmlDeviceGetHandleByIndex_v2(torch_index, ctypes.byref(self.dev)) != 0:
            raise OSError("no NVML handle for the GPU")
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.reasons_fn = fn
        self.max_mhz = self._uint(self.lib.nvmlDeviceGetMaxClockInfo, self.CLOCK_SM)

    def _uint(self, fn, *args):
        v = self.ct.c_uint()
        if fn(self.dev, *args, self.ct.byref(v)) != 0:
            return None
        return int(v.value)

    def sample(self) -> dict:
        r = self.ct.c_ulonglong()
        reasons = int(r.value) if self.reasons_fn(self.dev, self.ct.byref(r)) == 0 else 0
        mw = self._uint(self.lib.nvmlDeviceGetPowerUsage)
        return {"sm": self._uint(self.lib.nvmlDeviceGetClockInfo, self.CLOCK_SM), "max": self.max_mhz,
                "power": mw / 1000.0 if mw is not None else None,
                "reasons": [name for bit, name in self.REASONS.items() if reasons & bit]}


class ClockSampler:
    """Clocks and throttle reasons while the timed region runs.  NVML is polled in-process
    every few milliseconds, so even a region of a few tens of milliseconds holds samples;
    where NVML cannot be loaded, nvidia-smi is polled every 20 ms instead."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_S = 0.004

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None
        self.active = False
        self.stopped = False
        self.source = None

    def start(self):
        try:
            nvml = _Nvml(self.gpu)
            self.source = f"NVML every {self.PERIOD_S * 1e3:.0f} ms"
            self.thread = threading.Thread(target=self._poll, args=(nvml,), daemon=True)
            self.thread.start()
            return
        except (OSError, AttributeError):
            pass
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.source = "nvidia-smi every 20 ms"
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _poll(self, nvml):
        while not self.stopped:
            rec = nvml.sample()
            rec["in_region"] = self.active
            self.samples.append(rec)
            time.sleep(self.PERIOD_S)

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rec = {"sm": float(parts[1]), "max": float(parts[2]),
                       "power": float(parts[3]) if parts[3] not in ("[N/A]", "N/A") else None,
                       "reasons": [name for key, name in ((5, "hw_slowdown"), (6, "hw_thermal_slowdown"),
                                                          (7, "sw_thermal_slowdown"), (8, "sw_power_cap"))
                                   if parts[key].lower() == "active"]}
            except ValueError:
                continue
            rec["in_region"] = self.active
            self.samples.append(rec)

    def stop(self):
        self.stopped = True
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self):
        region = [s for s in self.samples if s["in_region"] and s["sm"] is not None]
        if not region:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0,
                    "source": self.source}
        reasons = sorted({r for s in region for r in s["reasons"]})
        powers = [s["power"] for s in region if s["power"] is not None]
        return {"sm_mhz": statistics.median(s["sm"] for s in region),
                "sm_max_mhz": max(s["max"] or 0 for s in region) or None,
                "reasons": reasons, "samples": len(region),
                "power_w_max": max(powers) if powers else None, "source": self.source}


# --------------------------------------------------------------------------------------
# distributed plumbing (weak scaling: independent copies, max time over ranks)
# --------------------------------------------------------------------------------------
def dist_info():
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_init(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def shard_seed(base_seed: int, rank: int) -> int:
    """Each rank owns an independent batch of the workload (weak scaling)."""
    return base_seed + 1000 * rank


# --------------------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline)
# --------------------------------------------------------------------------------------
def oracle_rows_flops(rows: np.ndarray, N: int, d: int, causal: bool) -> float:
    keys = (rows[:, 1] + 1) if causal else np.full(len(rows), N)
    return float(4.0 * d * keys.sum())


def cpu_model() -> str:
    """The host CPU's model name (from /proc/cpuinfo; 'unknown' where it says none)."""
    try:
        with open("/proc/cpuinfo") as f:
            text = f.read()
    except OSError:
        return "unknown"
    for key in ("model name", "Model", "CPU part"):
        for line in text.splitlines():
            if line.startswith(key) and ":" in line:
                return f"{line.split(':', 1)[1].strip()} ({os.cpu_count()} cpus)"
    return f"unknown ({os.cpu_count()} cpus)"


def time_oracle(q, k, v, causal, scale, seconds: float, seed: int = 12345):
    """Run the oracle on seeded random query rows for about `seconds` of wall time.

    Returns (FLOP/s, rows done, seconds spent, threads used)."""
    import oracle
    BH = q.shape[0] * q.shape[1]
    N, d = q.shape[2], q.shape[3]
    rng = np.random.default_rng(seed)
    nthreads = oracle.default_threads()
    done_rows, flops, elapsed = 0, 0.0, 0.0
    chunk = max(nthreads * 2, 32)
    while elapsed < seconds:
        rows = np.stack([rng.integers(0, BH, chunk), rng.integers(0, N, chunk)], axis=1)
        rows = rows[np.lexsort((rows[:, 1], rows[:, 0]))]
        t0 = time.perf_counter()
        oracle.attn_rows(q, k, v, rows, causal, scale, nthreads)
        dt = time.perf_counter() - t0
        elapsed += dt
        flops += oracle_rows_flops(rows, N, d, causal)
        done_rows += chunk
        if dt < seconds / 8:
            chunk *= 2
    return flops / elapsed, done_rows, elapsed, nthreads


# --------------------------------------------------------------------------------------
def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--B", type=int, default=8)
    ap.add_argument("--H", type=int, default=32)
    ap.add_argument("--N", type=int, default=8192)
    ap.add_argument("--d", type=int, default=128)
    ap.add_argument("--noncausal", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=0, help="0 = min(--steps, 100)")
    ap.add_argument("--e2e-chunks", type=int, default=4, help="batch chunks pipelined per e2e step")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="CPU time budget of the whole --impl reference run")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--sweep", default="", help="write a sequence-length sweep (JSON) to this path "
                    "instead of the contract line")
    ap.add_argument("--sweep-n", default="512,1024,2048,4096,8192,16384,32768,65536,131072")
    ap.add_argument("--splits", type=int, default=1, help="sweep: key-range splits (0 = the "
                    "library's plan with splitting allowed, 1 = unsplit)")
    ap.add_argument("--kernel", choices=["auto", "two", "one"], default="auto",
                    help="sweep, unsplit: pin the two-tile or the one-tile kernel")
    ap.add_argument("--order", choices=["auto", "one", "group", "shifted"], default="auto",
                    help="sweep: pin the unit order (one snake / a snake per head group, odd "
                    "groups mirrored / shifted past the previous group's last round)")
    ap.add_argument("--block-kv", type=int, default=0, help="sweep: keys per K/V tile (0 = the "
                    "library's choice, 64 or 128)")
    ap.add_argument("--sweep-shapes", default="", help="sweep: 'B,H,N;B,H,N;...' (overrides "
                    "--B, --H and --sweep-n)")
    ap.add_argument("--sweep-launches", type=int, default=20, help="timed launches per length "
                    "(1 = a single untimed launch per length, for an ncu capture)")
    ap.add_argument("--materialised", action="store_true", help="sweep: time the materialised "
                    "baseline (S and P in device memory, cuBLAS GEMMs + row softmax) instead")
    return ap.parse_args(argv)


def workload_name(args):
    causal = not args.noncausal
    if (args.B, args.H, args.N, args.d, causal) == (8, 32, 8192, 128, True):
        return "b8 h32 S8192 d128 causal (b8n8k)", causal
    return f"b{args.B} h{args.H} S{args.N} d{args.d} {'causal' if causal else 'non-causal'}", causal


def run_reference(args):
    world, rank, _ = dist_info()
    if world > 1 and rank != 0:
        return 0
    w = workloads.WORKLOADS["b8n8k"]
    name, causal = workload_name(args)
    q, k, v = workloads.make_inputs(w, B=args.B, H=args.H, N=args.N, d=args.d)
    scale = float(np.float32(1.0 / np.sqrt(args.d)))
    # size each step so warm-up + steps take about --ref-seconds of CPU time
    per_step = max(0.05, args.ref_seconds / max(1, args.steps + args.warmup))
    time_oracle(q, k, v, causal, scale, per_step * max(1, args.warmup), seed=1)
    vals, times, rows_total, threads = [], [], 0, 0
    for s in range(args.steps):
        val, rows, el, threads = time_oracle(q, k, v, causal, scale, per_step, seed=100 + s)
        vals.append(val)
        times.append(el)
        rows_total += rows
    value = float(np.mean(vals)) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * float(np.mean(times)), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": name, "B": args.B, "H": args.H, "N": args.N, "d": args.d,
                   "causal": causal, "step": "fp64 CPU oracle over a bounded random-row sample"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{rows_total} random query rows over {args.steps} steps "
                                   f"(~{per_step:.2f} s each) of the {name} workload",
                         "cpu_model": cpu_model(),
                         "full_workload_s_extrapolated":
                             model_flops(args.B, args.H, args.N, args.d, causal) / (value * 1e12)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import tiled_online_softmax_fa_gb300 as fa

    world, rank, local = dist_info()
    if world == 1 and args.gpus > 1:
        raise SystemExit("--gpus > 1 needs torchrun (one process per GPU)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    fa.load_library()
    name, causal = workload_name(args)
    B, H, N, d = args.B, args.H, args.N, args.d
    w = workloads.WORKLOADS["b8n8k"]
    q, k, v = workloads.make_inputs(w, B=B, H=H, N=N, d=d, seed=shard_seed(w.seed, rank))
    scale = float(np.float32(1.0 / np.sqrt(d)))
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flops = model_flops(B, H, N, d, causal)

    def step():
        fa.fa_fwd(qd, kd, vd, o=o, lse=lse, causal=causal, scale=scale, stream=stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if fa.get_device_status(stream) != fa.FA_OK:
        raise SystemExit("device status reported a timeout during warm-up")

    sampler = None if args.no_clocks else ClockSampler(local)
    if sampler:
        sampler.start()
        time.sleep(0.5)
    # Inputs larger than L2 need no flush between steps; smaller ones get a buffer of
    # twice the L2 size written before every timed step, outside that step's events.
    l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (128 << 20))
    in_bytes = 3 * qd.numel() * qd.element_size()
    flush = None if in_bytes >= 2 * l2_bytes else torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev)
    l2_note = (f"inputs (3 x {in_bytes // 3 / 1e6:.0f} MB) larger than L2; no flush" if flush is None else
               f"inputs (3 x {in_bytes // 3 / 1e6:.1f} MB) smaller than L2: a {2 * l2_bytes >> 20} MB "
               "buffer is written before each timed step, outside its events")
    barrier(world)
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.active = True
    if flush is None:
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        ms_local = ev0.elapsed_time(ev1)
    else:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for e0, e1 in evs:
            flush.fill_(1)
            e0.record(stream)
            step()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        ms_local = sum(e0.elapsed_time(e1) for e0, e1 in evs)
    if sampler:
        sampler.active = False
    barrier(world)
    ms_total = max_over_ranks(ms_local, world, dev)
    status = fa.get_device_status(stream)
    if status != fa.FA_OK:
        raise SystemExit(f"device status after timing: {fa.strerror(status)}")
    ms_step = ms_total / args.steps
    value = flops * world / (ms_step * 1e-3) / 1e12
    kernel_tflops = flops / (ms_step * 1e-3) / 1e12

    # ---- end to end: pinned host buffers -> H2D -> fa_fwd -> D2H, every step ----
    # Each step moves its q, k, v in and its o, lse out.  The batch is cut into chunks
    # on three streams (copy in, compute, copy out) so copies of one chunk overlap the
    # kernel on another; a chunk's buffers are reused only after the previous step's
    # kernel (for inputs) and copy-out (for outputs) of that chunk finished.
    e2e = None
    if not args.no_e2e:
        hq, hk, hv = (t.pin_memory() for t in (q, k, v))
        ho = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
        hl = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
        n_e2e = args.e2e_steps or min(args.steps, 100)
        chunks = max(1, min(args.e2e_chunks, B))
        bounds = [(B * c // chunks, B * (c + 1) // chunks) for c in range(chunks)]
        s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = lambda: torch.cuda.Event()  # noqa: E731
        in_done = [ev() for _ in bounds]
        comp_done = [ev() for _ in bounds]
        out_done = [ev() for _ in bounds]
        first = [True]

        def e2e_step():
            for c, (b0, b1) in enumerate(bounds):
                with torch.cuda.stream(s_in):
                    if not first[0]:
                        s_in.wait_event(comp_done[c])      # inputs of chunk c are free
                    qd[b0:b1].copy_(hq[b0:b1], non_blocking=True)
                    kd[b0:b1].copy_(hk[b0:b1], non_blocking=True)
                    vd[b0:b1].copy_(hv[b0:b1], non_blocking=True)
                    in_done[c].record(s_in)
                s_comp.wait_event(in_done[c])
                if not first[0]:
                    s_comp.wait_event(out_done[c])         # outputs of chunk c were read
                fa.fa_fwd(qd[b0:b1], kd[b0:b1], vd[b0:b1], o=o[b0:b1], lse=lse[b0:b1],
                          causal=causal, scale=scale, stream=s_comp)
                comp_done[c].record(s_comp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(comp_done[c])
                    ho[b0:b1].copy_(o[b0:b1], non_blocking=True)
                    hl[b0:b1].copy_(lse[b0:b1], non_blocking=True)
                    out_done[c].record(s_out)
            first[0] = False

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize(dev)
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        s_comp.wait_event(e0)
        s_out.wait_event(e0)
        for _ in range(n_e2e):
            e2e_step()
        s_in.wait_stream(s_comp)
        s_in.wait_stream(s_out)
        e1.record(s_in)
        torch.cuda.synchronize(dev)
        barrier(world)
        ms_e2e = max_over_ranks(e0.elapsed_time(e1) / n_e2e, world, dev)
        h2d_bytes = 3 * q.numel() * 2
        d2h_bytes = o.numel() * 2 + lse.numel() * 4
        e2e = {"value": flops * world / (ms_e2e * 1e-3) / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
               "steps": n_e2e, "ms_per_step": ms_e2e, "chunks_per_step": chunks,
               "launches_per_step": chunks}
        if fa.get_device_status(stream) != fa.FA_OK:
            raise SystemExit("device status reported a timeout during the e2e leg")
        # the pipelined copies must return exactly what the device computed
        torch.cuda.synchronize(dev)
        if not (torch.equal(ho, o.cpu()) and torch.equal(hl, lse.cpu())):
            raise SystemExit("e2e outputs differ from the device outputs")
        # The host link on this machine, measured here with the step's own buffers: the
        # inputs copied in alone, the outputs copied out alone, and both at once.  The
        # step cannot beat moving its inputs in and its outputs out, so that time (with
        # both directions running at once) bounds the e2e rate.
        def timed_copies(h2d: bool, d2h: bool, reps: int = 3) -> float:
            best = float("inf")
            for _ in range(reps):
                t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                t0.record(s_in)
                s_out.wait_event(t0)
                if h2d:
                    with torch.cuda.stream(s_in):
                        for dst, src in ((qd, hq), (kd, hk), (vd, hv)):
                            dst.copy_(src, non_blocking=True)
                if d2h:
                    with torch.cuda.stream(s_out):
                        ho.copy_(o, non_blocking=True)
                        hl.copy_(lse, non_blocking=True)
                s_in.wait_stream(s_out)
                t1.record(s_in)
                torch.cuda.synchronize(dev)
                best = min(best, t0.elapsed_time(t1))
            return best
        ms_in, ms_out, ms_both = timed_copies(True, False), timed_copies(False, True), \
            timed_copies(True, True)
        e2e.update(link_h2d_gbs=h2d_bytes / (ms_in * 1e-3) / 1e9,
                   link_d2h_gbs=d2h_bytes / (ms_out * 1e-3) / 1e9,
                   link_both_ms=ms_both,
                   frac_of_link_bound=ms_both / ms_e2e,
                   link_note="copies of the step's own pinned buffers, best of 3; "
                             "frac_of_link_bound = (inputs in + outputs out, both at once) / e2e step")

    if sampler:
        sampler.stop()
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0

    peak, peak_src = load_peaks(ms_step * args.steps * 1e-3)
    traffic, traffic_note = None, "no ncu capture matching this kernel source"
    if os.path.exists(TRAFFIC_FILE):
        with open(TRAFFIC_FILE) as f:
            tr = json.load(f)
        if tr.get("kernel_source_hash") == kernel_source_hash() and \
                tr.get("shape") == [B, H, N, d, int(causal)]:
            traffic = tr.get("dram_bytes_per_launch")
            traffic_note = tr.get("note", "")
    roofline = {"bound": "tensor", "achieved": kernel_tflops, "peak": peak, "unit": "TFLOP/s",
                "frac": kernel_tflops / peak, "traffic": traffic, "traffic_note": traffic_note,
                "peak_source": peak_src, "algorithmic_flops_per_launch": flops,
                "qkvo_compulsory_bytes_per_launch": 4 * B * H * N * d * 2 + B * H * N * 4,
                "avg_launch_ms": ms_step,
                "kernel": ("fa_fwd_1tile_kernel" if fa.fwd_plan(B, H, N, d, causal)[0] ==
                           fa.FA_KERNEL_ONE_TILE else "fa_fwd_row_kernel") + f"<{d}>"}

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        val, rows, el, threads = time_oracle(q, k, v, causal, scale, args.cpu_seconds)
        cpu = {"value": val / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{rows} random query rows of the {name} workload, fp64, {el:.1f} s",
               "cpu_model": cpu_model(),
               "full_workload_s_extrapolated": flops / val}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": name, "B": B, "H": H, "N": N, "d": d, "causal": causal,
                   "global_batch": B * world, "seq_len": N, "parallelism": f"replicas{world}",
                   "l2": l2_note},
        "clocks": sampler.summary() if sampler else None, "e2e": e2e,
        "gpu_launches": args.steps, "roofline": roofline, "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_sweep(args):
    """Measured TFLOP/s per sequence length beside the pages' traffic models."""
    import tiled_online_softmax_fa_gb300 as fa

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fa.load_library()
    causal = not args.noncausal
    B, H, d = args.B, args.H, args.d
    w = workloads.WORKLOADS["b8n8k"]
    scale = float(np.float32(1.0 / np.sqrt(d)))
    stream = torch.cuda.current_stream(dev)
    results = []
    if args.sweep_shapes:
        shapes = [tuple(int(x) for x in t.split(",")) for t in args.sweep_shapes.split(";") if t]
    else:
        shapes = [(B, H, int(x)) for x in args.sweep_n.split(",")]
    pin = {"auto": fa.FA_KERNEL_AUTO, "two": fa.FA_KERNEL_TWO_TILE, "one": fa.FA_KERNEL_ONE_TILE}
    for B, H, N in shapes:
        q, k, v = (t.to(dev) for t in workloads.make_inputs(w, B=B, H=H, N=N, d=d, seed=7000 + N))
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        kernel = pin[args.kernel]
        if args.splits == 0:
            kernel, splits = fa.fwd_plan(B, H, N, d, causal, allow_split=True)
        else:
            splits = args.splits
            if splits == 1 and kernel == fa.FA_KERNEL_AUTO:
                kernel = fa.fwd_plan(B, H, N, d, causal)[0]
            elif splits > 1 and kernel == fa.FA_KERNEL_AUTO:
                kernel = fa.FA_KERNEL_ONE_TILE if d == 256 else fa.FA_KERNEL_TWO_TILE
        order = {"auto": fa.FA_ORDER_AUTO, "one": fa.FA_ORDER_ONE_SNAKE,
                 "group": fa.FA_ORDER_GROUP_SNAKES, "shifted": fa.FA_ORDER_SHIFTED_SNAKES}[args.order]
        opts = fa.FwdOptions(kernel=kernel, order=order, block_kv=args.block_kv) \
            if (splits == 1 or args.kernel != "auto" or args.block_kv) else None
        if args.materialised:
            splits = 1
            ws = torch.empty(fa.materialised_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
            run = lambda: fa.fa_fwd_materialised(q, k, v, o=o, lse=lse, causal=causal,  # noqa: E731
                                                 scale=scale, workspace=ws, stream=stream)
        elif splits > 1:
            ws = torch.empty(fa.splitkv_workspace_bytes(B, H, N, d, splits), dtype=torch.uint8,
                             device=dev)
            # with --splits 0 the library plans the launch itself (kernel, pieces, order);
            # the workspace is sized for the pieces its plan takes
            n_arg = 0 if args.splits == 0 else splits
            run = lambda: fa.fa_fwd_splitkv(q, k, v, o=o, lse=lse, causal=causal, scale=scale,  # noqa: E731
                                            splits=n_arg, workspace=ws, stream=stream,
                                            options=opts)
        else:
            run = lambda: fa.fa_fwd(q, k, v, o=o, lse=lse, causal=causal, scale=scale,  # noqa: E731
                                    stream=stream, options=opts)
        # the unit order the launch takes, where it is known here
        shown = None
        if args.materialised:
            pass
        elif order != fa.FA_ORDER_AUTO:
            shown = order
        elif args.kernel == "auto" and (splits == 1 or args.splits == 0):
            shown = fa.fwd_plan(B, H, N, d, causal, allow_split=args.splits == 0,
                                with_order=True)[2]
        rec = {"N": N, "B": B, "H": H, "d": d, "causal": causal, "splits": splits,
               "block_kv": args.block_kv or 128,
               "order": {fa.FA_ORDER_ONE_SNAKE: "one snake", fa.FA_ORDER_GROUP_SNAKES: "group snakes",
                         fa.FA_ORDER_SHIFTED_SNAKES: "shifted snakes", None: None}[shown],
               "kernel": None if args.materialised else
               {fa.FA_KERNEL_TWO_TILE: "two-tile", fa.FA_KERNEL_ONE_TILE: "one-tile"}[kernel],
               "path": "materialised" if args.materialised else "tiled",
               "flops": model_flops(B, H, N, d, causal)}
        if args.sweep_launches <= 1:
            run()
            torch.cuda.synchronize(dev)
        else:
            for _ in range(3):
                run()
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.sweep_launches):
                run()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ms = e0.elapsed_time(e1) / args.sweep_launches
            rec.update(ms=ms, tflops=rec["flops"] / (ms * 1e-3) / 1e12)
        if fa.get_device_status(stream) != fa.FA_OK:
            raise SystemExit(f"device status reported a timeout at N={N}")
        rec.update(page_traffic_models(B, H, N, d), lse_bytes=B * H * N * 4)
        results.append(rec)
        print(json.dumps(rec), flush=True)
        del q, k, v, o, lse
        ws = None
        torch.cuda.empty_cache()
    peak, peak_src = load_peaks()
    with open(args.sweep, "w") as f:
        json.dump({"peak_tflops": peak, "peak_source": peak_src, "results": results}, f, indent=1)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.sweep:
        return run_sweep(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
