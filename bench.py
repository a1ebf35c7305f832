"""Benchmark of the fused ragged decode step (indexer -> top-512 -> gather -> sink attention).

Workload: 8 rows x 131072 keys (the long-context, bandwidth-bound decode case),
seeded synthetic bf16 inputs shaped like the DeepSeek-V4 decode rows.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line. `value` is decode rows/s over all ranks (each rank runs
its own 8 rows: rows are independent, so N GPUs are N replicas, weak scaling,
no data exchange), from K decode steps launched back to back as CUDA graph
replays and timed with CUDA events on the launching stream. The inputs (1.28 GB
of caches per step) are far larger than L2 and the queries rotate over four
seeded sets, so no step finds its data in L2. The latency of a single step
with L2 flushed first (a 512 MiB write, then a 512 MiB read, so that no dirty
flush lines are written back inside the step) is reported beside it.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# DRAM bytes (read + write) of one indexer launch on the 8 x 131072 workload, from an
# ncu capture of dram__bytes_read.sum and dram__bytes_write.sum (one pass) of the current kernel.
INDEXER_DRAM_BYTES_8x131072 = 268_619_008 + 2_567_936
CONFIG_INDEX = 3
METRIC = "decode rows/s (8 rows, 128K ctx) and achieved HBM GB/s vs GB300 peak"
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--config", type=int, default=CONFIG_INDEX)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="skip the other workloads' step latencies")
    ap.add_argument("--case", default="decode",
                    choices=["decode", "decode_steps", "topk", "indexer_topk", "indexer_queries", "decode_host",
                             "sparse_attn", "compressor"],
                    help="decode: the benchmark; any other: run only that entry point on the workload "
                         "(--warmup + --steps calls, no timing), for a profiler to capture its kernels")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def bf16_peak():
    """Dense bf16 tensor throughput (TFLOP/s): the measured burst figure, else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


REASON_NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


def clock_summary(samples, source):
    """Median SM clock under load, the maximum SM clock and every clock-event
    reason seen, from (sm_mhz, max_mhz, reasons) samples."""
    if not samples:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": source}
    reasons = set()
    for _, _, r in samples:
        reasons |= set(r)
    return {"sm_mhz": statistics.median(x[0] for x in samples), "sm_max_mhz": max(x[1] for x in samples),
            "reasons": sorted(reasons), "samples": len(samples), "source": source}


class NvmlClockSampler:
    """SM clock and clock-event reasons read through NVML (read-only queries)
    every `period_s` seconds by a thread while the timed region runs."""

    # nvmlClocksEventReason* bits
    BITS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown", 0x4: "sw_power_cap"}

    def __init__(self, device, period_s: float = 0.002, lib=None):
        import ctypes
        self.ct = ctypes
        self.period_s = period_s
        self.samples = []
        self.stop = threading.Event()
        self.nvml = lib if lib is not None else ctypes.CDLL("libnvidia-ml.so.1")
        if self.nvml.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.handle = self._handle(device)
        self.max_mhz = self._clock(self.nvml.nvmlDeviceGetMaxClockInfo)
        fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self.reasons_fn = fn if fn is not None else self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons

    def _handle(self, device):
        ct, h = self.ct, self.ct.c_void_p()
        uuid = None
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device).uuid)
        except Exception:
            pass
        if uuid:
            for u in (uuid, "GPU-" + uuid):
                if self.nvml.nvmlDeviceGetHandleByUUID(ct.c_char_p(u.encode()), ct.byref(h)) == 0:
                    return h
        index = device.index if getattr(device, "index", None) is not None else 0
        if self.nvml.nvmlDeviceGetHandleByIndex_v2(ct.c_uint(index), ct.byref(h)) != 0:
            raise OSError("no NVML handle for the device")
        return h

    def _clock(self, fn):
        v = self.ct.c_uint()
        if fn(self.handle, self.ct.c_int(1), self.ct.byref(v)) != 0:  # NVML_CLOCK_SM
            raise OSError("NVML clock query failed")
        return float(v.value)

    def _sample(self):
        r = self.ct.c_ulonglong()
        bits = r.value if self.reasons_fn(self.handle, self.ct.byref(r)) == 0 else 0
        sm = self._clock(self.nvml.nvmlDeviceGetClockInfo)
        self.samples.append((sm, self.max_mhz, [n for b, n in self.BITS.items() if bits & b]))

    def _run(self):
        while not self.stop.is_set():
            try:
                self._sample()
            except OSError:
                return
            self.stop.wait(self.period_s)

    def poll(self):
        """One more sample from the calling thread (a short timed region may
        end before the sampling thread is scheduled again)."""
        try:
            self._sample()
        except OSError:
            pass

    def __enter__(self):
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()
        return self

    def __exit__(self, *exc):
        self.stop.set()
        self.thread.join(timeout=5)
        self.nvml.nvmlShutdown()

    def summary(self):
        return clock_summary(self.samples, "nvml")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def poll(self):
        """nvidia-smi samples on its own period; nothing to add."""

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        samples = []
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm, mx = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            samples.append((sm, mx, [n for n, v in zip(REASON_NAMES, parts[2:6]) if v.lower() == "active"]))
        return clock_summary(samples, "nvidia-smi")


def clock_sampler(device):
    """NVML polling (every 0.2 ms) when the library loads, else nvidia-smi (every 100 ms)."""
    try:
        return NvmlClockSampler(device, period_s=0.0002)
    except (OSError, AttributeError):
        return ClockSampler(device.index or 0)


# ---------------------------------------------------------------------------
# CPU baseline: the oracle as it stands, single-threaded BLAS, bounded sample
# ---------------------------------------------------------------------------

_CPU_SNIPPET = r"""
import json, multiprocessing, os, sys, time
sys.path.insert(0, {root!r})
import numpy as np, oracle, workloads
wl = workloads.config({cfg})
budget = {budget}
# One thread: row decodes one after another, cycling over the rows.
t0 = time.perf_counter(); rows = 0
while True:
    oracle.decode(wl, entries=[rows % wl.num_rows]); rows += 1
    if time.perf_counter() - t0 > budget: break
dt = time.perf_counter() - t0
# Every core: one worker process per core, each decoding whole rows (one
# single-threaded BLAS each). Forked: this process never touches a GPU, and the
# workers share the workload's arrays instead of copying them.
def one(e):
    oracle.decode(wl, entries=[e])
    return e
cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
t1 = time.perf_counter(); prows = 0
with multiprocessing.get_context("fork").Pool(cores) as pool:
    while True:
        list(pool.imap_unordered(one, [(prows + i) % wl.num_rows for i in range(cores)]))
        prows += cores
        if time.perf_counter() - t1 > budget: break
pdt = time.perf_counter() - t1
print(json.dumps({{"rows": rows, "distinct": min(rows, wl.num_rows), "of": wl.num_rows,
                  "kv_lens": sorted({{int(r.kv_len) for r in wl.rows}}), "seconds": dt,
                  "par_rows": prows, "par_seconds": pdt, "cores": cores}}))
"""


def cpu_baseline(cfg: int, budget_s: float = 12.0):
    """The oracle as it stands on this host: rows/s with every core (one
    worker process per core) as the baseline, and with one thread beside it."""
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[v] = "1"
    env.pop("CUDA_VISIBLE_DEVICES", None)
    code = _CPU_SNIPPET.format(root=ROOT, cfg=cfg, budget=budget_s)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=900)
    if r.returncode != 0:
        return {"value": None, "unit": "rows/s", "cores": 1, "kind": "oracle", "error": r.stderr[-300:]}
    d = json.loads(r.stdout.strip().splitlines()[-1])
    lens = "/".join(map(str, d["kv_lens"]))
    return {"value": d["par_rows"] / d["par_seconds"], "unit": "rows/s", "cores": d["cores"], "kind": "oracle",
            "sample": f"{d['par_rows']} row decodes over {d['cores']} worker processes (one per core), cycling "
                      f"over the {d['of']} rows (kv_len {lens}), numpy float64 oracle, single-threaded BLAS "
                      f"per worker, {d['par_seconds']:.1f} s",
            "single_thread": {"value": d["rows"] / d["seconds"], "cores": 1,
                              "sample": f"{d['rows']} row decodes one after another, {d['seconds']:.1f} s"}}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    cb = cpu_baseline(args.config, budget_s=max(5.0, 20.0 / max(1, args.steps)))
    line = {
        "impl": "reference", "metric": METRIC, "value": cb["value"], "unit": "rows/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": (8 / cb["value"] * 1e3) if cb.get("value") else None,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "8 rows x 131072 keys (bounded sample of rows)", "rows": 8, "kv_len": 131072},
        "cpu_baseline": {k: cb.get(k) for k in ("value", "kind", "cores", "sample", "unit")},
        "e2e": {"value": cb["value"], "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# native arm
# ---------------------------------------------------------------------------

def percentiles(xs):
    """(p10, median, p90) of a list of numbers."""
    xs = sorted(xs)
    pick = lambda q: xs[min(len(xs) - 1, max(0, int(round(q * (len(xs) - 1)))))]
    return pick(0.1), pick(0.5), pick(0.9)


def graph_step_times(graph4, stream, graphs_timed, steps_per_graph=4):
    """Per-step device times (ms) of back-to-back replays of a graph of
    `steps_per_graph` consecutive steps: an event after every replay, the
    interval divided by the steps it holds."""
    import torch
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(graphs_timed + 1)]
    with torch.cuda.stream(stream):
        graph4.replay()
        ev[0].record(stream)
        for k in range(graphs_timed):
            graph4.replay()
            ev[k + 1].record(stream)
    torch.cuda.synchronize()
    return [ev[k].elapsed_time(ev[k + 1]) / steps_per_graph for k in range(graphs_timed)]


def other_configs(ds, workloads, to_device, device, stream, flush_l2, skip, steps=10, graphs_timed=40):
    """The decode on the other benchmark workloads: back to back from CUDA graphs
    of four consecutive steps (four query sets), as `value` is timed, with the
    p10 / median / p90 of the per-step times over graphs_timed x 4 steps; and
    the median latency of single steps with L2 flushed before each."""
    import torch
    from workloads.device import bf16_tensor
    res = {}
    for i in range(5):
        if i == skip:
            continue
        wl = workloads.config(i)
        dev = to_device(wl, device)
        nq = max(r.q_row for r in wl.rows) + 1
        out = torch.empty((nq, 64, 512), dtype=torch.bfloat16, device=device)
        idx = torch.empty((wl.index_elements,), dtype=torch.int32, device=device)
        ws = ds.workspace(wl.rows, device)
        qsets = [(dev.q_index, dev.w_index, dev.q_attn)]
        for k in range(3):
            qI, wI, qA = workloads.draw_queries(wl, 1000 + k)
            qsets.append((bf16_tensor(qI, device), torch.from_numpy(wI).to(device), bf16_tensor(qA, device)))

        def step(k=0):
            qI, wI, qA = qsets[k]
            ds.ds_rows_decode(dev.rows, qI, wI, dev.keys, qA, dev.kv, dev.sinks, dev.sinks_row_stride, dev.scale,
                              out, indices=idx, workspace_t=ws, stream=stream)

        with torch.cuda.stream(stream):
            for k in range(4):
                step(k)
        torch.cuda.synchronize(device)
        g4 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g4, stream=stream):
            for k in range(4):
                step(k)
        with torch.cuda.stream(stream):
            for _ in range(3):
                g4.replay()
        per_step = graph_step_times(g4, stream, graphs_timed)
        p10, p50, p90 = percentiles(per_step)
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        with torch.cuda.stream(stream):
            for k in range(steps):
                flush_l2(k)
                starts[k].record(stream)
                step(k % 4)
                ends[k].record(stream)
        torch.cuda.synchronize(device)
        ms = percentiles([s.elapsed_time(e) for s, e in zip(starts, ends)])[1]
        alg = wl.algorithmic_bytes()
        res[str(i)] = {"workload": wl.name, "rows": wl.num_rows,
                       "us_per_step": p50 * 1e3, "us_per_step_p10": p10 * 1e3, "us_per_step_p90": p90 * 1e3,
                       "steps_timed": 4 * graphs_timed,
                       "rows_per_s": wl.num_rows / (p50 / 1e3), "gbs": alg / (p50 / 1e3) / 1e9,
                       "us_per_step_flushed_median": ms * 1e3,
                       "launch": "back to back from CUDA graphs of 4 consecutive steps (as value); the flushed "
                                 "figure is single steps with L2 flushed before each"}
        del dev, out, idx, ws, g4, qsets
        torch.cuda.empty_cache()
    return res


def compressor_timings(ds, device, stream, calls=50):
    """ds_rows_compress_kv per supported shape, 8 rows, every row completing a
    block (the call that pools its window): microseconds per call and the bytes
    it must move (token inputs, the window read, the state row written, the
    overlap shift, ape, norm and the output)."""
    import torch
    res = {}
    g = torch.Generator(device="cpu").manual_seed(5)
    for ratio, head_dim in ((4, 128), (4, 512), (128, 512)):
        coff = 2 if ratio == 4 else 1
        P = coff * head_dim
        f = lambda *sh: torch.randn(*sh, generator=g).to(device)
        ks = [f(coff * ratio, P) for _ in range(8)]
        ss = [f(coff * ratio, P) for _ in range(8)]
        kv, sc, ape, norm = f(8, P), f(8, P), f(ratio, P), f(head_dim)
        out = torch.empty((8, head_dim), dtype=torch.bfloat16, device=device)
        pos = [ratio * (e + 1) - 1 for e in range(8)]
        with torch.cuda.stream(stream):
            for _ in range(3):
                ds.ds_rows_compress_kv(ks, ss, pos, kv, sc, ape, norm, ratio, head_dim, 1e-6, out, stream=stream)
        torch.cuda.synchronize(device)
        # One graph of `calls` calls: the GPU time per call, without the host's
        # per-call marshalling (longer than this kernel).
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(calls):
                ds.ds_rows_compress_kv(ks, ss, pos, kv, sc, ape, norm, ratio, head_dim, 1e-6, out, stream=stream)
        with torch.cuda.stream(stream):
            graph.replay()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            graph.replay()
            b.record(stream)
        torch.cuda.synchronize(device)
        us = a.elapsed_time(b) / calls * 1e3
        shift = 2 * 2 * ratio * P * 4 if ratio == 4 else 0
        per_row = 3 * P * 4 + 2 * coff * ratio * head_dim * 4 + 2 * P * 4 + shift + head_dim * 2
        nbytes = 8 * per_row + ratio * P * 4 + head_dim * 4
        res[f"{ratio}x{head_dim}"] = {"us_per_call": us, "bytes_per_call": nbytes, "gbs": nbytes / (us / 1e6) / 1e9}
    return res


def indexer_queries_timings(ds, workloads, wl, dev, device, stream, counts=(2, 4, 8), calls=10):
    """ds_rows_indexer_topk_queries on the same caches with Q consecutive queries
    per row (every key valid for the last query): microseconds per call, the
    algorithmic bytes (each key once, plus Q query rows, weights and 512 indices
    per row) and the indexer's tensor flops (2 x 64 x 128 per key and query)."""
    import torch
    from workloads.device import bf16_tensor
    R = len(wl.rows)
    keys_total = sum(r.kv_len for r in wl.rows)
    res = {}
    for Q in counts:
        qI, wI = workloads.draw_index_queries(wl, 900 + Q, R * Q)
        q = bf16_tensor(qI, device)
        w = torch.from_numpy(wI).to(device)
        rows = [ds.IndexerRow(r.kv_len, 4 * r.kv_len - Q, 0, e * Q, 512 * Q * e) for e, r in enumerate(wl.rows)]
        out = torch.empty((512 * Q * R,), dtype=torch.int32, device=device)
        ws = ds.indexer_topk_workspace(rows, device, Q)
        call = lambda: ds.ds_rows_indexer_topk_queries(rows, Q, q, w, dev.keys, out, workspace_t=ws, stream=stream)
        with torch.cuda.stream(stream):
            for _ in range(3):
                call()
        torch.cuda.synchronize(device)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(calls):
                call()
        with torch.cuda.stream(stream):
            graph.replay()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            graph.replay()
            b.record(stream)
        torch.cuda.synchronize(device)
        us = a.elapsed_time(b) / calls * 1e3
        nbytes = 256 * keys_total + R * Q * (16384 + 256 + 2048)
        flops = 2 * 64 * 128 * Q * keys_total
        res[str(Q)] = {"us_per_call": us, "us_per_query_row": us / Q, "bytes_per_call": nbytes,
                       "gbs": nbytes / (us / 1e6) / 1e9, "tflops": flops / (us / 1e6) / 1e12}
    return res


def run_case(args, ds, workloads, wl, dev, qsets, stream, device):
    """One entry point on the workload, --warmup + --steps calls back to back and
    no timing: the command a profiler wraps to capture that entry point's
    kernels on the benchmark workload (or on --config)."""
    import torch
    from workloads.device import bf16_tensor
    R = wl.num_rows
    calls = max(1, args.warmup) + max(1, args.steps)
    stride = max(r.kv_len for r in wl.rows)
    if args.case == "decode_steps":
        nq = max(r.q_row for r in wl.rows) + 1
        out = torch.empty((nq, 64, 512), dtype=torch.bfloat16, device=device)
        idx = torch.empty((wl.index_elements,), dtype=torch.int32, device=device)
        ws = ds.workspace(wl.rows, device)
        for k in range(calls):
            qI, wI, qA = qsets[k % 4]
            ds.ds_rows_decode(dev.rows, qI, wI, dev.keys, qA, dev.kv, dev.sinks, dev.sinks_row_stride, dev.scale,
                              out, indices=idx, workspace_t=ws, stream=stream)
    elif args.case in ("topk", "sparse_attn"):
        scores = torch.empty((R, stride), dtype=torch.float32, device=device)
        ds.ds_rows_indexer_score(dev.rows, dev.q_index, dev.w_index, dev.keys, scores, stride, stream=stream)
        idx = torch.empty((wl.index_elements,), dtype=torch.int32, device=device)
        ws = ds.workspace(wl.rows, device)
        ds.ds_rows_topk(dev.rows, scores, stride, idx, ws, stream=stream)
        nq = max(r.q_row for r in wl.rows) + 1
        out = torch.empty((nq, 64, 512), dtype=torch.bfloat16, device=device)
        for _ in range(calls):
            if args.case == "topk":
                ds.ds_rows_topk(dev.rows, scores, stride, idx, ws, stream=stream)
            else:
                ds.ds_rows_sparse_attn(dev.rows, dev.q_attn, dev.sinks, dev.sinks_row_stride, idx, dev.scale, out,
                                       dev.kv, workspace_t=ws, stream=stream)
    elif args.case == "indexer_topk":
        rows = [ds.IndexerRow(r.kv_len, 4 * r.kv_len - 1, 0, r.q_row, 512 * e) for e, r in enumerate(wl.rows)]
        pidx = torch.empty((512 * R,), dtype=torch.int32, device=device)
        pws = ds.indexer_topk_workspace(rows, device)
        for k in range(calls):
            ds.ds_rows_indexer_topk(rows, qsets[k % 4][0], qsets[k % 4][1], dev.keys, pidx, workspace_t=pws,
                                    stream=stream)
    elif args.case == "indexer_queries":
        Q = 4
        qI, wI = workloads.draw_index_queries(wl, 900 + Q, R * Q)
        q, w = bf16_tensor(qI, device), torch.from_numpy(wI).to(device)
        rows = [ds.IndexerRow(r.kv_len, 4 * r.kv_len - Q, 0, e * Q, 512 * Q * e) for e, r in enumerate(wl.rows)]
        qout = torch.empty((512 * Q * R,), dtype=torch.int32, device=device)
        qws = ds.indexer_topk_workspace(rows, device, Q)
        for _ in range(calls):
            ds.ds_rows_indexer_topk_queries(rows, Q, q, w, dev.keys, qout, workspace_t=qws, stream=stream)
    elif args.case == "compressor":
        # (ratio, head_dim) = (128, 512) for `calls` calls, then (4, 128): 8 rows that all
        # complete a block, so every call pools its window.
        g = torch.Generator(device="cpu").manual_seed(5)
        f = lambda *sh: torch.randn(*sh, generator=g).to(device)
        for ratio, head_dim in ((128, 512), (4, 128)):
            coff = 2 if ratio == 4 else 1
            P = coff * head_dim
            ks = [f(coff * ratio, P) for _ in range(8)]
            ss = [f(coff * ratio, P) for _ in range(8)]
            kv, sc, ape, norm = f(8, P), f(8, P), f(ratio, P), f(head_dim)
            out = torch.empty((8, head_dim), dtype=torch.bfloat16, device=device)
            pos = [ratio * (e + 1) - 1 for e in range(8)]
            for _ in range(calls):
                ds.ds_rows_compress_kv(ks, ss, pos, kv, sc, ape, norm, ratio, head_dim, 1e-6, out, stream=stream)
    elif args.case == "decode_host":
        h_sets = [tuple(t.cpu().pin_memory() for t in qs) for qs in qsets]
        h_sk = dev.sinks.cpu().pin_memory()
        nq = max(r.q_row for r in wl.rows) + 1
        h_out = torch.empty((nq, 64, 512), dtype=torch.bfloat16).pin_memory()
        hws = ds.host_workspace(wl.rows, dev.sinks_row_stride, device)
        for k in range(calls):
            qI, wI, qA = h_sets[k % 4]
            ds.ds_rows_decode_host(dev.rows, qI, wI, dev.keys, qA, dev.kv, h_sk, dev.sinks_row_stride, dev.scale,
                                   h_out, workspace_t=hws, stream=stream)
    torch.cuda.synchronize(device)
    print(json.dumps({"case": args.case, "calls": calls, "workload": wl.name}), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return

    import numpy as np
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", torch.cuda.current_device() if world == 1 else local)

    import deepseek_sparse_attention_ragged_gb300 as ds
    from deepseek_sparse_attention_ragged_gb300.replicas import job_rate, max_over_ranks
    import workloads
    from workloads.device import to_device

    ds.build()
    ds.load()

    wl = workloads.config(args.config)
    dev = to_device(wl, device)
    R = wl.num_rows
    nq = max(r.q_row for r in wl.rows) + 1
    out = torch.empty((nq, 64, 512), dtype=torch.bfloat16, device=device)
    idx = torch.empty((wl.index_elements,), dtype=torch.int32, device=device)
    ws = ds.workspace(wl.rows, device)
    stream = torch.cuda.Stream(device)

    # Four query sets for the same caches (the workload's own and three more drawn
    # with its recipe): consecutive steps select different KV rows, as real
    # decode steps do, so nothing selected by one step is still in L2 for the next.
    from workloads.device import bf16_tensor
    qsets = [(dev.q_index, dev.w_index, dev.q_attn)]
    for i in range(3):
        qI, wI, qA = workloads.draw_queries(wl, 1000 + i)
        qsets.append((bf16_tensor(qI, device), torch.from_numpy(wI).to(device), bf16_tensor(qA, device)))

    def step(i=0):
        qI, wI, qA = qsets[i]
        ds.ds_rows_decode(dev.rows, qI, wI, dev.keys, qA, dev.kv, dev.sinks, dev.sinks_row_stride, dev.scale, out,
                          indices=idx, workspace_t=ws, stream=stream)

    if args.case != "decode":
        run_case(args, ds, workloads, wl, dev, qsets, stream, device)
        return

    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=device)
    flush_read = torch.ones(128 * 2 ** 20, dtype=torch.int32, device=device)

    def flush_l2(k):
        # Write 512 MiB (evicts L2), then read 512 MiB so that the lines left in L2
        # are clean and no write-back of the flush lands in the timed step.
        flush.fill_(k & 0xFF)
        flush_read.max()

    def barrier():
        torch.cuda.synchronize(device)
        if world > 1:
            torch.distributed.barrier()

    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            step(i % 4)
    barrier()
    # A serving loop launches the fixed-shape decode step as a CUDA graph.
    graphs = []
    for i in range(4):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(i)
        graphs.append(g)
    # A decode loop captures consecutive steps in one graph: four steps (the four
    # query sets) per graph, each step ordered after the previous one completes
    # (its first kernel is an ordinary launch), so only launch gaps are saved.
    graph4 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph4, stream=stream):
        for i in range(4):
            step(i)
    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            graphs[i % 4].replay()
            graph4.replay()
    barrier()

    # Throughput: K steps back to back. The inputs (1.28 GB of caches a step)
    # are far larger than L2, and the queries rotate, so no flush is needed.
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with clock_sampler(device) as clocks:
        barrier()
        with torch.cuda.stream(stream):
            t_start.record(stream)
            for k in range(args.steps // 4):
                graph4.replay()
            for k in range(args.steps % 4):
                graphs[k].replay()
            t_end.record(stream)
        # While the timed work runs, this thread also samples the clocks, then
        # the barrier.
        while not t_end.query():
            clocks.poll()
            time.sleep(5e-5)
        barrier()
    total_ms = t_start.elapsed_time(t_end)
    # The spread of the step time: the same graphs again, an event after each
    # replay of four steps (outside the timed region above).
    s10, s50, s90 = percentiles(graph_step_times(graph4, stream, max(10, args.steps // 4)))

    def flushed(run_step):
        """Mean latency of single steps with L2 flushed before each (write, then read)."""
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        barrier()
        with torch.cuda.stream(stream):
            for k in range(args.steps):
                flush_l2(k)
                starts[k].record(stream)
                run_step(k % 4)
                ends[k].record(stream)
        barrier()
        return sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / args.steps

    latency_graph_ms = flushed(lambda i: graphs[i].replay())
    latency_eager_ms = flushed(step)
    total_ms = max_over_ranks(total_ms, device)
    ms_per_step = total_ms / args.steps
    value = job_rate(world, R, args.steps, total_ms)
    alg_bytes = wl.algorithmic_bytes()
    step_gbs = alg_bytes / (ms_per_step / 1e3) / 1e9

    # Dominant kernel (the indexer) alone: same kernel, same launch shape, through
    # its entry point; 20 launches back to back (keys larger than L2), timed as a batch.
    stride = max(r.kv_len for r in wl.rows)
    scores = torch.empty((R, stride), dtype=torch.float32, device=device)
    def graph_ms_per_call(call, reps=5):
        """Mean device time of call(i) for the four query sets i, captured in one
        CUDA graph and replayed `reps` times (no host marshalling in the timing)."""
        with torch.cuda.stream(stream):
            for i in range(4):
                call(i)
        torch.cuda.synchronize(device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(4):
                call(i)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()
            a.record(stream)
            for _ in range(reps):
                g.replay()
            b.record(stream)
        torch.cuda.synchronize(device)
        return a.elapsed_time(b) / (4 * reps)

    # The indexer alone, 20 launches back to back (keys larger than L2).
    idx_ms = graph_ms_per_call(lambda i: ds.ds_rows_indexer_score(dev.rows, qsets[i][0], qsets[i][1], dev.keys,
                                                                  scores, stride, stream=stream))
    idx_bytes = sum(256 * r.kv_len + 4 * r.kv_len + 16384 + 256 for r in wl.rows)
    # The step formula's share of the indexer: its keys and query (the score
    # write is the stand-alone stage's own output, the head weights are small).
    idx_bytes_alg = sum(256 * r.kv_len + 16384 for r in wl.rows)
    peak, peak_kind = peaks()
    idx_gbs = idx_bytes / (idx_ms / 1e3) / 1e9
    # DRAM bytes of one indexer launch on this workload, read + written, from an
    # ncu capture of the current kernel (dram__bytes_read.sum + dram__bytes_write.sum).
    idx_traffic = INDEXER_DRAM_BYTES_8x131072 if args.config == CONFIG_INDEX else None
    # The indexer's tensor work: 2 x 64 heads x 128 dims per key, against the
    # dense bf16 peak. The kernel is bound by HBM, so this fraction stays low.
    tpeak, tpeak_kind = bf16_peak()
    idx_tflops = sum(2 * 64 * 128 * r.kv_len for r in wl.rows) / (idx_ms / 1e3) / 1e12
    idx_tensor = {"achieved": idx_tflops, "peak": tpeak, "peak_kind": tpeak_kind, "unit": "TFLOP/s",
                  "frac": idx_tflops / tpeak, "flops_per_launch": sum(2 * 64 * 128 * r.kv_len for r in wl.rows)}

    # End to end through the C-ABI call with host buffers (ds_rows_decode_host):
    # per step the queries, head weights and sinks go host->device from pinned
    # memory and the output comes back, inside the call; the caches stay
    # resident (they are the decode state). The four query sets rotate as above.
    h_sets = [tuple(t.cpu().pin_memory() for t in qs) for qs in qsets]
    h_sk = dev.sinks.cpu().pin_memory()
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    hws = ds.host_workspace(wl.rows, dev.sinks_row_stride, device)
    h2d = sum(t.numel() * t.element_size() for t in (*h_sets[0], h_sk))
    d2h = h_out.numel() * h_out.element_size()

    def host_step(i):
        qI, wI, qA = h_sets[i % 4]
        ds.ds_rows_decode_host(dev.rows, qI, wI, dev.keys, qA, dev.kv, h_sk, dev.sinks_row_stride, dev.scale, h_out,
                               workspace_t=hws, stream=stream)

    # As for `value`, the calls are replayed from a CUDA graph of four
    # consecutive calls (the host's per-call marshalling is not the GPU's time);
    # each replayed call still copies its inputs in and its output back.
    with torch.cuda.stream(stream):
        for i in range(4):
            host_step(i)
    barrier()
    g_host = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_host, stream=stream):
        for i in range(4):
            host_step(i)
    e2e_graphs = max(2, args.steps // 8)
    with torch.cuda.stream(stream):
        g_host.replay()
    barrier()
    with torch.cuda.stream(stream):
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(e2e_graphs):
            g_host.replay()
        t1.record(stream)
    barrier()
    e2e_ms = t0.elapsed_time(t1) / (4 * e2e_graphs)
    e2e_ms = max_over_ranks(e2e_ms, device)

    # The positioned indexer with its causal top-512 (every key valid, offset 0)
    # on the same caches: 20 calls back to back.
    prow = [ds.IndexerRow(r.kv_len, 4 * r.kv_len - 1, 0, r.q_row, 512 * e) for e, r in enumerate(wl.rows)]
    pidx = torch.empty((512 * R,), dtype=torch.int32, device=device)
    pws = ds.indexer_topk_workspace(prow, device)
    pidx_ms = graph_ms_per_call(lambda i: ds.ds_rows_indexer_topk(prow, qsets[i][0], qsets[i][1], dev.keys, pidx,
                                                                  workspace_t=pws, stream=stream))
    pidx_bytes = sum(256 * r.kv_len + 16384 + 256 + 4 * 512 for r in wl.rows)

    per_config = None
    compressor = None
    queries = None
    if rank == 0 and world == 1 and not args.no_per_config:
        per_config = other_configs(ds, workloads, to_device, device, stream, flush_l2, skip=args.config)
        compressor = compressor_timings(ds, device, stream)
        queries = indexer_queries_timings(ds, workloads, wl, dev, device, stream)

    if rank == 0:
        cb = None
        if world == 1 and not args.no_cpu_baseline:
            cb = cpu_baseline(args.config)
        line = {
            "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"{R} rows x {stride} keys (indexer 64x128, attention 64x512, top-512)",
                       "rows": R, "kv_len": stride,
                       "l2": "inputs larger than L2 (1.28 GB of caches per step), no flush; queries rotate over "
                             "4 seeded sets so consecutive steps select different KV rows",
                       "launch": "K decode steps back to back from CUDA graphs of 4 consecutive steps; every step starts after the previous one completed",
                       "latency_ms_flushed_graph": latency_graph_ms, "latency_ms_flushed_eager": latency_eager_ms,
                       "parallelism": f"replicas{world}"},
            "step_gbs": step_gbs, "step_frac_of_peak": step_gbs / peak,
            "step_frac_of_nominal": step_gbs / NOMINAL_HBM_GBS, "nominal_hbm_gbs": NOMINAL_HBM_GBS,
            "algorithmic_bytes_per_step": alg_bytes,
            "roofline": {"kernel": "indexer_score_kernel", "bound": "hbm", "achieved": idx_gbs, "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": idx_gbs / peak, "traffic": idx_traffic,
                         "bytes_per_launch": idx_bytes, "ms_per_launch": idx_ms,
                         "bytes_per_launch_keys_and_query": idx_bytes_alg,
                         "frac_keys_and_query": idx_bytes_alg / (idx_ms / 1e3) / 1e9 / peak,
                         "tensor": idx_tensor},
            "spread": {"ms_per_step_p10": s10, "ms_per_step_median": s50, "ms_per_step_p90": s90,
                       "steps": 4 * max(10, args.steps // 4),
                       "how": "back-to-back replays of the 4-step graph, an event after each replay"},
            "e2e": {"value": job_rate(world, R, 1, e2e_ms), "unit": "rows/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": 3 * args.steps,
            "indexer_topk": {"entry": "ds_rows_indexer_topk", "workload": "same caches, every key valid, offset 0",
                             "ms_per_call": pidx_ms, "gbs": pidx_bytes / (pidx_ms / 1e3) / 1e9,
                             "frac": pidx_bytes / (pidx_ms / 1e3) / 1e9 / peak},
            "per_config": per_config,
            "compressor": compressor,
            "indexer_queries": queries,
            "clocks": clocks.summary(),
            "cpu_baseline": cb,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
