"""Benchmark of the layout permute on GB300: one JSON line on stdout (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one ``tl_permute`` call over the whole workload (default: 65536 float16
tiles of 128x64, row-major -> column-major per tile, 1 GiB in + 1 GiB out).  The
metric is GB/s of algorithmic traffic (every element read once and written once,
2 * N * elem_bytes per step) and its fraction of the measured HBM copy bandwidth.

* ``value``: device-resident inputs; W warm-up steps, then K steps timed with CUDA
  events on the launching stream between barriers, max over ranks.  Inputs are
  larger than L2 (129 MB), so no flush is needed.
* ``e2e``: the same call with host buffers: every step copies the input from
  pinned host memory, permutes, and copies the result back, inside the timed
  region; consecutive steps alternate two buffer sets on two streams so that one
  step's device->host copy overlaps the next step's host->device copy.
* ``cpu_baseline``: the CPU oracle (test infrastructure) timed on this host's cores
  on a bounded sample of the same workload; the GPU output is checked against it
  on that sample (bit-exact).
* ``--impl reference``: the oracle alone, as the reference arm (rank 0 only).

Under ``torchrun`` each rank permutes its own copy of the workload on its own GPU
(independent batches, no collective on the data path; weak scaling) and rank 0
reports the whole-job throughput over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "permute GB/s (read+write bytes) and % of GB300 HBM peak, bit-exact vs oracle"
UNIT = "GB/s"
DEFAULT_WORKLOAD = "tile_transpose"
# Sources of the kernel the roofline line reports; a traffic figure recorded in
# profiles/ is only used while these files are unchanged.
KERNEL_SOURCES = {
    "tile": ["k_tile.cu", "tile_common.cuh", "tl_device.cuh"],
    "cluster": ["k_cluster.cu", "tile_common.cuh", "tl_device.cuh"],
    "rows": ["k_rows.cu", "tl_device.cuh"],
    "chunk": ["k_chunk.cu", "tl_device.cuh"],
    "panel": ["k_panel.cu", "tl_device.cuh"],
    "cols": ["k_cols.cu", "tl_device.cuh"],
    "block": ["k_block.cu", "tl_device.cuh"],
    "warp": ["k_warp.cu", "tl_device.cuh"],
    "generic": ["k_generic.cu", "tl_device.cuh"],
}
KERNEL_NAMES = {"tile": "k_tile", "cluster": "k_cluster", "rows": "k_rows", "chunk": "k_chunk",
                "panel": "k_panel", "cols": "k_cols", "block": "k_block",
                "warp": "k_warp", "generic": "k_generic"}
DTYPES = {"sf_transpose": "f32", "tile_transpose": "f16", "mx_sf": "u8", "attention": "bf16",
          "t2d_u8": "u8", "t2d_f16": "f16", "t2d_f32": "f32", "t2d_f64": "f64",
          "t2d_v16": "16-byte", "t2d_odd_f32": "f32", "t2d_odd_u8": "u8", "hwc_chw_u8": "u8", "nd6_f32": "f32",
          "nd8_f32": "f32", "nd8_u16": "u16"}


# ---------------------------------------------------------------------------
# multi-process helpers (also exercised by the CPU tests with gloo)
# ---------------------------------------------------------------------------
def dist_env():
    """(rank, local_rank, world_size) from the torchrun environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def reduce_max(value: float, device=None) -> float:
    """Maximum of a float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def whole_job_gbps(bytes_per_step_per_rank: int, steps: int, world: int, max_ms: float) -> float:
    """Aggregate GB/s of a weak-scaling run: every rank moves the same bytes."""
    return bytes_per_step_per_rank * steps * world / (max_ms * 1e-3) / 1e9


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    """SM clock and clock-event reasons of this rank's GPU, sampled in a thread.

    Uses NVML through ctypes (read-only queries of the driver's library), polled
    every ~2 ms so that even a few-millisecond timed region holds samples; falls
    back to `nvidia-smi -lms 50` when NVML cannot be loaded."""

    # NVML clock-event reason bits
    REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                   "hw_thermal_slowdown": 0x40}
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, local_rank: int, uuid: str | None = None):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        ids = [v.strip() for v in vis.split(",")] if vis else []
        self.gpu = ids[local_rank] if local_rank < len(ids) else str(local_rank)
        self.uuid = uuid
        self.samples = []          # (wall time, sm, max, power, {reason: active})
        self.proc = None
        self.thread = None
        self.stop_flag = threading.Event()
        self.source = None

    # -- NVML ---------------------------------------------------------------
    def _nvml_handle(self):
        import ctypes

        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            return None, None
        h = ctypes.c_void_p()
        ok = False
        if self.uuid:
            ok = lib.nvmlDeviceGetHandleByUUID(self.uuid.encode(), ctypes.byref(h)) == 0
        if not ok and self.gpu.startswith("GPU-"):
            ok = lib.nvmlDeviceGetHandleByUUID(self.gpu.encode(), ctypes.byref(h)) == 0
        if not ok and self.gpu.isdigit():
            ok = lib.nvmlDeviceGetHandleByIndex_v2(int(self.gpu), ctypes.byref(h)) == 0
        return (lib, h) if ok else (None, None)

    def _poll_nvml(self, lib, h):
        import ctypes

        sm, mx, pw = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint()
        reasons = ctypes.c_ulonglong()
        get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
        while not self.stop_flag.is_set():
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm)) == 0:
                r = reasons.value if get_reasons(h, ctypes.byref(reasons)) == 0 else 0
                p = pw.value / 1000.0 if lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw)) == 0 \
                    else None
                active = {k: bool(r & b) for k, b in self.REASON_BITS.items()}
                self.samples.append((time.time(), float(sm.value), float(mx.value), p, active))
            time.sleep(0.002)

    def start(self):
        try:
            lib, h = self._nvml_handle()
        except OSError:
            lib, h = None, None
        if lib is not None:
            self.source = "nvml"
            self.thread = threading.Thread(target=self._poll_nvml, args=(lib, h), daemon=True)
            self.thread.start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", self.gpu], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.source = "nvidia-smi"
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm, mx = float(parts[0]), float(parts[1])
                pw = float(parts[2]) if parts[2] not in ("[N/A]", "N/A") else None
            except ValueError:
                continue
            active = {r: ("Active" in p and "Not" not in p) for r, p in zip(self.REASONS, parts[3:7])}
            self.samples.append((time.time(), sm, mx, pw, active))

    def stop(self):
        self.stop_flag.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples_in_window": 0,
                    "note": "no clock samples (NVML and nvidia-smi unavailable)"}
        samples = list(self.samples)
        inside = [s for s in samples if t0 <= s[0] <= t1]
        n_in = len(inside)
        if not inside:   # window shorter than the sampling period: nearest samples
            mid = 0.5 * (t0 + t1)
            inside = sorted(samples, key=lambda s: abs(s[0] - mid))[:2]
        sms = sorted(s[1] for s in inside)
        reasons = sorted({r for s in inside for r, a in s[4].items() if a})
        powers = [s[3] for s in inside if s[3] is not None]
        return {"sm_mhz": sms[len(sms) // 2], "sm_max_mhz": max(s[2] for s in inside),
                "reasons": reasons, "samples_in_window": n_in, "source": self.source,
                "power_w_max": max(powers) if powers else None}


# ---------------------------------------------------------------------------
# roofline inputs
# ---------------------------------------------------------------------------
def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def kernel_source_hash(path_name: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES.get(path_name, []):
        with open(os.path.join(ROOT, "movement_tl_permute_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(path_name: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, or None when there is none or the kernel changed since."""
    fname = os.path.join(ROOT, "profiles", "%s_%s.md" % (KERNEL_NAMES.get(path_name, path_name),
                                                          workload))
    try:
        with open(fname) as f:
            text = f.read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256") != kernel_source_hash(path_name):
        return None
    try:
        return int(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------
def sample_layout(w, m):
    """The leading m indices of axis 0 of workload w (same strides)."""
    return (m,) + tuple(w.shape[1:])


def oracle_rate(w, src, dst, threads, budget_s):
    """Largest leading sample of axis 0 the oracle finishes in about budget_s.
    Returns (m, seconds for one run of it)."""
    import oracle

    m = max(1, min(w.shape[0], 8))
    while True:
        t0 = time.perf_counter()
        oracle.permute(src, dst, sample_layout(w, m), w.src_strides, w.dst_strides, w.elem_bytes,
                       nthreads=threads)
        dt = time.perf_counter() - t0
        if m >= w.shape[0] or dt >= 0.05 * budget_s:
            break
        m = min(w.shape[0], m * 4)
    if m < w.shape[0] and dt > 0:
        m = max(1, min(w.shape[0], int(m * budget_s / dt)))
        t0 = time.perf_counter()
        oracle.permute(src, dst, sample_layout(w, m), w.src_strides, w.dst_strides, w.elem_bytes,
                       nthreads=threads)
        dt = time.perf_counter() - t0
    return m, dt


def cpu_baseline(w, src, dst, budget_s=10.0):
    import oracle

    threads = max(1, min(len(os.sched_getaffinity(0)), oracle.max_threads()))
    m, dt = oracle_rate(w, src, dst, threads, budget_s)
    runs, total = 1, dt
    while total < 0.5 * budget_s and runs < 20:
        t0 = time.perf_counter()
        oracle.permute(src, dst, sample_layout(w, m), w.src_strides, w.dst_strides, w.elem_bytes,
                       nthreads=threads)
        total += time.perf_counter() - t0
        runs += 1
    per = total / runs
    n = m * (w.n_elems // w.shape[0])
    gbps = 2 * n * w.elem_bytes / per / 1e9
    return {"value": round(gbps, 3), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": "leading %d of %d along axis 0 (%d elements, %.1f MiB read+write), "
                      "%d run(s), %.2f s each" % (m, w.shape[0], n,
                                                  2 * n * w.elem_bytes / 2**20, runs, per)}, m


def sampled_parity(w, src, got, m, threads):
    """Bit-exact check of the GPU output ``got`` on the oracle's leading-m sample.

    The oracle writes the sample's image into two buffers filled with different
    canary bytes: the bytes where the two agree are exactly the ones the sample
    writes, and only those are compared (the rest of dst is not checked here).
    Returns (bit_exact, bytes compared)."""
    import numpy as np
    import oracle

    a = np.full(got.nbytes, 0xA5, dtype=np.uint8)
    b = np.full(got.nbytes, 0x5A, dtype=np.uint8)
    for buf in (a, b):
        oracle.permute(src, buf, sample_layout(w, m), w.src_strides, w.dst_strides,
                       w.elem_bytes, nthreads=threads)
    mask = a == b
    return bool(np.array_equal(got[mask], a[mask])), int(mask.sum())


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------
L2_BYTES = 129 * 1000 * 1000


def config_of(w, plan):
    return {"workload": "%s: %s" % (w.name, w.description), "shape": list(w.shape),
            "src_strides": list(w.src_strides), "dst_strides": list(w.dst_strides),
            "elem_bytes": w.elem_bytes, "bytes_per_step": w.algorithmic_bytes,
            "path": plan["path"] if plan else None,
            "grid": plan["grid"] if plan else None, "block": plan["block"] if plan else None,
            "l2": ("inputs larger than L2 (129 MB): no flush between steps"
                   if w.src_elems * w.elem_bytes > L2_BYTES else
                   "L2-resident working set: a latency measurement, not an HBM one"),
            "seed": w.seed}


def input_digest(buf) -> str:
    """SHA-256 of the input bytes (first 16 hex digits), logged with the seed."""
    return hashlib.sha256(memoryview(buf).cast("B")).hexdigest()[:16]


def run_reference(args, w):
    import numpy as np

    rank, _, world = dist_env()
    if rank != 0:
        return 0
    from movement_tl_permute_gb300 import workloads
    import oracle

    oracle.build()
    src = workloads.make_input(w)
    dst = np.zeros(w.dst_elems * w.elem_bytes, dtype=np.uint8)
    threads = max(1, min(len(os.sched_getaffinity(0)), oracle.max_threads()))
    per_step_budget = min(10.0, max(0.05, 90.0 / max(1, args.steps + args.warmup)))
    m, _ = oracle_rate(w, src, dst, threads, per_step_budget)
    shape = sample_layout(w, m)
    for _ in range(args.warmup):
        oracle.permute(src, dst, shape, w.src_strides, w.dst_strides, w.elem_bytes,
                       nthreads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.permute(src, dst, shape, w.src_strides, w.dst_strides, w.elem_bytes,
                       nthreads=threads)
    dt = time.perf_counter() - t0
    n = m * (w.n_elems // w.shape[0])
    per = dt / max(1, args.steps)
    gbps = 2 * n * w.elem_bytes / per / 1e9
    sample = ("leading %d of %d along axis 0 (%d elements, %.1f MiB read+write) per step"
              % (m, w.shape[0], n, 2 * n * w.elem_bytes / 2**20))
    peak, _ = measured_peak()
    line = {"impl": "reference", "metric": METRIC, "value": round(gbps, 3), "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(per * 1e3, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": DTYPES.get(w.name, "bits"), "data": "synthetic",
            "config": config_of(w, None), "pct_hbm_peak": round(100 * gbps / peak, 3),
            "cpu_baseline": {"value": round(gbps, 3), "unit": UNIT, "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(gbps, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# The five configurations of the headline metric, each measured in the same run:
# (entry name, workload, forced path).  The first is the one-warp latency case.
CONFIG_RUNS = [("tile_transpose", "tile_transpose", "auto"),
               ("tile_transpose_cluster", "tile_transpose", "cluster"),
               ("mx_sf", "mx_sf", "auto"), ("attention", "attention", "auto"),
               ("t2d_u8", "t2d_u8", "auto"), ("t2d_f16", "t2d_f16", "auto"),
               ("t2d_f32", "t2d_f32", "auto"), ("t2d_f64", "t2d_f64", "auto"),
               ("t2d_v16", "t2d_v16", "auto"), ("nd8_f32", "nd8_f32", "auto"),
               ("nd8_u16", "nd8_u16", "auto"), ("t2d_odd_u8", "t2d_odd_u8", "auto")]


def all_configs(args, tl, dev, stream, head_name, head_src):
    """Every configuration of the headline metric, one at a time (buffers freed in
    between): ``[GB/s, fraction of the measured HBM peak, bit_exact]`` per HBM
    workload (K back-to-back launches timed with CUDA events after 3 warm-ups;
    parity on an oracle sample of about a second), and the one-warp scale-factor
    transpose as microseconds per call, host launches and graph replay."""
    import numpy as np
    import torch

    import oracle
    from movement_tl_permute_gb300 import workloads

    peak, _ = measured_peak()
    sptr = stream.cuda_stream
    threads = max(1, min(len(os.sched_getaffinity(0)), oracle.max_threads()))
    steps = max(10, min(args.steps, 100))
    out = {}

    # config 1: the one-warp SF transpose (latency; L2-resident)
    w = workloads.get("sf_transpose")
    src_np = workloads.make_input(w)
    s_gpu = torch.from_numpy(src_np).to(dev)
    d_gpu = torch.zeros(w.dst_elems * w.elem_bytes, dtype=torch.uint8, device=dev)
    call = (w.shape, w.src_strides, w.dst_strides, w.elem_bytes)
    reps = 2000
    for _ in range(5):
        tl.tl_permute_ex(s_gpu.data_ptr(), d_gpu.data_ptr(), *call, sptr)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    h0 = time.perf_counter()
    for _ in range(reps):
        tl.tl_permute_ex(s_gpu.data_ptr(), d_gpu.data_ptr(), *call, sptr)
    host_us = (time.perf_counter() - h0) * 1e6 / reps
    e1.record(stream)
    torch.cuda.synchronize(dev)
    us_stream = e0.elapsed_time(e1) * 1e3 / reps
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cap = torch.cuda.current_stream(dev).cuda_stream
        for _ in range(reps):
            tl.tl_permute_ex(s_gpu.data_ptr(), d_gpu.data_ptr(), *call, cap)
    graph.replay()
    torch.cuda.synchronize(dev)
    e0.record(stream)
    graph.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    us_graph = e0.elapsed_time(e1) * 1e3 / reps
    want = np.zeros(w.dst_elems * w.elem_bytes, dtype=np.uint8)
    oracle.permute(src_np, want, *call)
    out["sf_transpose"] = {"us_per_call_stream": round(us_stream, 3),
                           "host_us_per_call": round(host_us, 3),
                           "us_per_call_graph": round(us_graph, 3),
                           "bit_exact": bool(np.array_equal(d_gpu.cpu().numpy(), want))}
    del graph, s_gpu, d_gpu

    # configs 2-5 (HBM-bound), then the two high-rank block-path workloads and the odd-pitch
    # u8 transpose
    for name, wname, path in CONFIG_RUNS:
        w = workloads.get(wname)
        src_np = head_src if wname == head_name else workloads.make_input(w)
        s_gpu = torch.from_numpy(src_np).to(dev)
        d_gpu = torch.empty(w.dst_elems * w.elem_bytes, dtype=torch.uint8, device=dev)
        call = (w.shape, w.src_strides, w.dst_strides, w.elem_bytes)

        def one():
            tl.tl_permute_ex(s_gpu.data_ptr(), d_gpu.data_ptr(), *call, sptr, path=path)

        for _ in range(3):
            one()
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(steps):
            one()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        gbps = w.algorithmic_bytes / (e0.elapsed_time(e1) / steps * 1e-3) / 1e9
        got = d_gpu.cpu().numpy()
        del s_gpu, d_gpu
        torch.cuda.empty_cache()
        m, _ = oracle_rate(w, src_np, np.empty_like(got), threads, 0.5)
        ok, _ = sampled_parity(w, src_np, got, m, threads)
        out[name] = [round(gbps, 1), round(gbps / peak, 4), ok]
        del got
    return out


def run_ours(args, w):
    import numpy as np
    import torch
    import torch.distributed as dist

    import movement_tl_permute_gb300 as tl
    from movement_tl_permute_gb300 import build as tl_build
    from movement_tl_permute_gb300 import workloads

    rank, local, world = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    tl_build.build()
    tl.load()
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream

    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None
    clocks = ClockSampler(local, uuid)
    clocks.start()
    src_np = workloads.make_input(w)
    nbytes_dst = w.dst_elems * w.elem_bytes
    s_gpu = torch.from_numpy(src_np).to(dev)
    d_gpu = torch.empty(nbytes_dst, dtype=torch.uint8, device=dev)
    args_call = (w.shape, w.src_strides, w.dst_strides, w.elem_bytes)
    plan = tl.tl_plan(s_gpu.data_ptr(), d_gpu.data_ptr(), *args_call, path=args.path)

    def step():
        tl.tl_permute_ex(s_gpu.data_ptr(), d_gpu.data_ptr(), *args_call, sptr, path=args.path)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    use_graph = args.launch == "graph" or (args.launch == "auto" and "small" in w.tags)
    graph = None
    if use_graph:
        # the K timed steps captured once; the replay launches every kernel again
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            cap = torch.cuda.current_stream(dev).cuda_stream
            for _ in range(args.steps):
                tl.tl_permute_ex(s_gpu.data_ptr(), d_gpu.data_ptr(), *args_call, cap,
                                 path=args.path)
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize(dev)

    # ------------------------------------------------ device-resident timing
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    launches0 = tl.tl_launch_count()
    t_wall0 = time.time()
    e0.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for _ in range(args.steps):
            step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    barrier()
    # a replayed graph launches the captured kernels without host calls
    launches = args.steps if graph is not None else tl.tl_launch_count() - launches0
    ms_local = e0.elapsed_time(e1)
    ms_max = reduce_max(ms_local, dev if world > 1 else None)

    # per-launch spread: a few steps timed one by one (outside the timed region)
    singles = []
    if graph is None:
        for _ in range(min(20, args.steps)):
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            step()
            s1.record(stream)
            s1.synchronize()
            singles.append(s0.elapsed_time(s1))
    singles.sort()

    # ------------------------------------------------ end to end, host buffers
    # Each step copies its input from pinned host memory, permutes and copies the
    # result back.  Consecutive steps alternate between two buffer sets on two
    # streams, so one step's device->host copy overlaps the next step's
    # host->device copy (the copy engines run both directions at once).
    src_pin = torch.from_numpy(src_np).pin_memory()
    dst_pins = [torch.empty(nbytes_dst, dtype=torch.uint8).pin_memory() for _ in range(2)]
    s_bufs = [s_gpu, torch.empty_like(s_gpu)]
    d_bufs = [d_gpu, torch.empty_like(d_gpu)]
    streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_step(i):
        k = i % 2
        with torch.cuda.stream(streams[k]):
            s_bufs[k].copy_(src_pin, non_blocking=True)
            tl.tl_permute_ex(s_bufs[k].data_ptr(), d_bufs[k].data_ptr(), *args_call,
                             streams[k].cuda_stream, path=args.path)
            dst_pins[k].copy_(d_bufs[k], non_blocking=True)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier()
    e0.record(stream)
    for st_k in streams:
        st_k.wait_event(e0)
    for i in range(e2e_steps):
        e2e_step(i)
    for st_k in streams:
        ev = torch.cuda.Event()
        ev.record(st_k)
        stream.wait_event(ev)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    e2e_ms = reduce_max(e0.elapsed_time(e1), dev if world > 1 else None)
    dst_pin = dst_pins[(e2e_steps - 1) % 2]
    clocks.stop()
    clock_summary = clocks.summary(t_wall0, t_wall1)

    if rank != 0:
        dist.destroy_process_group() if dist.is_initialized() else None
        return 0

    # ------------------------------------------------ CPU oracle + sampled parity
    got = dst_pin.numpy()                  # result of the last e2e step (same input)
    scratch = np.empty_like(got)
    base, m = cpu_baseline(w, src_np, scratch, budget_s=args.cpu_budget)
    del scratch
    parity, n_checked = sampled_parity(w, src_np, got, m, base["cores"])
    del got
    configs = (all_configs(args, tl, dev, stream, w.name, src_np)
               if args.configs == "all" or (args.configs == "auto" and w.name == DEFAULT_WORKLOAD
                                            and not args.leading and world == 1) else None)

    bytes_step = w.algorithmic_bytes
    value = whole_job_gbps(bytes_step, args.steps, world, ms_max)
    per_launch_gbps = bytes_step / (ms_local / max(1, args.steps) * 1e-3) / 1e9
    peak, peak_kind = measured_peak()
    traffic = recorded_traffic(plan["path"], w.name)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_max / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPES.get(w.name, "bits"),
        "data": "synthetic",
        "config": dict(config_of(w, plan), launch="cuda_graph" if graph is not None else "stream",
                       input_sha256=input_digest(src_np)),
        "pct_hbm_peak": round(100.0 * value / world / peak, 2),
        "parity": {"bit_exact": parity,
                   "checked": "GPU output vs oracle on the cpu_baseline sample: the %d dst "
                              "bytes it writes, of %d" % (n_checked, nbytes_dst)},
        "roofline": {"bound": "hbm", "achieved": round(per_launch_gbps, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(per_launch_gbps / peak, 4),
                     "traffic": traffic, "kernel": KERNEL_NAMES.get(plan["path"]),
                     "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs: copy, burst)" % peak_kind},
        "cpu_baseline": base,
        "e2e": {"value": round(whole_job_gbps(bytes_step, e2e_steps, world, e2e_ms), 2),
                "unit": UNIT, "h2d_bytes_per_step": int(src_np.nbytes),
                "d2h_bytes_per_step": int(nbytes_dst), "steps": e2e_steps},
        "gpu_launches": int(launches),
        "per_launch_ms": ({"median": round(singles[len(singles) // 2], 5),
                           "min": round(singles[0], 5), "n": len(singles),
                           "note": "steps timed one at a time after the timed region"}
                          if singles else None),
        "clocks": clock_summary,
    }
    if configs is not None:
        line["configs"] = configs
        parity = parity and all(v[2] for k, v in configs.items() if isinstance(v, list)) and \
            configs["sf_transpose"]["bit_exact"]
    print(json.dumps(line), flush=True)
    if dist.is_initialized():
        dist.destroy_process_group()
    return 0 if parity else 3


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--path", default="auto",
                    choices=["auto", "generic", "chunk", "tile", "warp", "rows", "cluster",
                             "panel", "cols", "block"],
                    help="force a kernel path (default: the planner's choice)")
    ap.add_argument("--leading", type=int, default=0,
                    help="override the outermost extent (smaller cases for profiling)")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle work for the CPU baseline")
    ap.add_argument("--launch", choices=["auto", "stream", "graph"], default="auto",
                    help="timed steps as stream launches, or replayed from one CUDA graph that "
                         "holds all of them (auto: graph for the one-warp workload, whose "
                         "step is shorter than a host-side launch)"),
    ap.add_argument("--configs", choices=["auto", "all", "none"], default="auto",
                    help="also measure every configuration of the metric and three layouts "
                         "outside them (auto: with the default workload at full size on one "
                         "GPU)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    from movement_tl_permute_gb300 import workloads

    w = workloads.get(args.workload)
    if args.leading:
        w = workloads.scaled(w, args.leading)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
