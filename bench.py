#!/usr/bin/env python3
"""Benchmark of the INT8 split-KV decode path on GB300.

Headline workload: sparse-candidate INT8 decode, S = 8 query rows, 24 query /
2 KV heads, head_dim 256, a 16384-token INT8 cache with per-channel scales,
2048 sorted unique candidates per row, softmax scale 1/16 (the shapes the
onnxruntime PR 33707 page measures).  One step is one decode pass over L
layers, each with its own cache, query rows and candidate lists (L = 32 by
default: 537 MB of caches, more than three times the L2), captured as one
CUDA graph of L dsa_decode calls (decode kernel + combine kernel each).

value = algorithmic bytes of all calls / device time (GB/s, whole job).  The
algorithmic bytes of one call are the gathered K and V rows, the query, the
index lists, the scales and the output; split-workspace traffic is not
counted.  The JSON line also carries us_per_call, the decode kernel's roofline
(its bytes / its own CUDA-event time from a graph of partials-only launches),
an end-to-end figure through the public API with host buffers, the FP64
oracle's CPU time, the SM clocks seen during the timed region, and the paged
decode, deep-context and prefill workloads measured the same way.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
For N > 1 run under torch.distributed.run: every rank decodes its own layers
(weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time
from typing import Optional

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

S_ROWS, HQ, HKV, D, N_CACHE, N_SEL, SIGMA = 8, 24, 2, 256, 16384, 2048, 1.0 / 16.0
WORKLOAD = ("sparse-candidate INT8 decode: S=8 rows, 24 query / 2 KV heads, head_dim 256, "
            "16384-token int8 cache per layer with per-channel scales, 2048 sorted unique "
            "candidates per row, softmax scale 1/16")
# H200 attention time incl. merge for this workload (onnxruntime PR 33707, Performance, 8 rows)
H200_US_PER_CALL = 13.2


def call_bytes(S=S_ROWS, Hq=HQ, Hkv=HKV, Dh=D, n_sel=N_SEL):
    kv = S * Hkv * n_sel * Dh * 2
    return dict(kv=kv, q=S * Hq * Dh * 2, idx=S * n_sel * 4, scales=2 * Hkv * Dh * 4,
                out=S * Hq * Dh * 2)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--layers", type=int, default=32)
    ap.add_argument("--extra", default="all",
                    choices=["all", "sparse", "paged", "variants", "fp8", "deep", "prefill",
                             "prefill_table", "quantize", "none"],
                    help="which other workloads to measure besides the headline")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing")
    ap.add_argument("--clock-sampler", default=None, help=argparse.SUPPRESS)
    return ap.parse_args()


# --------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline and the reference arm)
# --------------------------------------------------------------------------

def _oracle_worker(wid: int, nworkers: int, cmd_q, res_q):
    """One host core of the oracle pool: build the headline workload (seeded,
    the same in every worker), then on each command compute the requested
    number of query rows (both KV heads of a row) with the FP64 oracle.
    Worker w takes the rows w, w + nworkers, ... of the 8-row call, cycling."""
    import oracle
    import workloads as W
    c = W.sparse_decode(S_ROWS, seed=0)
    res_q.put(("ready", wid, 0))
    r = wid
    while True:
        n = cmd_q.get()
        if n is None:
            break
        for _ in range(n):
            k = r % S_ROWS
            oracle.sparse_attention(c.q[k:k + 1], c.k_codes, c.v_codes, c.k_scale, c.v_scale,
                                    c.scale_kind, c.idx[k:k + 1], c.sigma)
            r += nworkers
        res_q.put(("done", wid, n))


class OraclePool:
    """The FP64 oracle on every host core this process may use: one spawned
    worker per core, each with single-threaded BLAS, computing whole query rows
    of the headline workload.  A step sends every worker the same row count and
    ends when the last one is done (wall clock)."""

    def __init__(self, cores: int):
        import multiprocessing as mp
        self.cores = cores
        ctx = mp.get_context("spawn")  # never fork after CUDA has been touched
        saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS",
                                                 "MKL_NUM_THREADS", "CUDA_VISIBLE_DEVICES")}
        os.environ.update(OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
                          CUDA_VISIBLE_DEVICES="")
        try:
            self.cmd = [ctx.Queue() for _ in range(cores)]
            self.res = ctx.Queue()
            self.procs = [ctx.Process(target=_oracle_worker, args=(w, cores, self.cmd[w], self.res),
                                      daemon=True) for w in range(cores)]
            for p in self.procs:
                p.start()
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        for _ in range(cores):
            self._get()

    def _get(self):
        msg = self.res.get(timeout=600)
        return msg

    def step(self, rows_per_worker: int) -> float:
        """Wall seconds for every worker to compute rows_per_worker rows."""
        t0 = time.perf_counter()
        for q in self.cmd:
            q.put(rows_per_worker)
        for _ in range(self.cores):
            self._get()
        return time.perf_counter() - t0

    def close(self):
        for q in self.cmd:
            q.put(None)
        for p in self.procs:
            p.join(timeout=30)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_cpu_oracle(budget_s: float):
    """cpu_baseline: the oracle on all host cores for about budget_s seconds."""
    cores = host_cores()
    pool = OraclePool(cores)
    try:
        pool.step(1)  # warm-up: one row per worker
        t_row = pool.step(1)
        n = max(1, int(budget_s / max(t_row, 1e-6)))
        sec = pool.step(n)
    finally:
        pool.close()
    rows = n * cores
    row_bytes = sum(call_bytes().values()) / S_ROWS
    return dict(value=rows * row_bytes / sec / 1e9, unit="GB/s", cores=cores, kind="oracle",
                seconds=sec, rows=rows, seconds_per_call=sec / rows * S_ROWS,
                sample=f"{rows} query rows of the headline workload ({n} per core; a call is "
                       f"{S_ROWS} rows x 24 heads x 2048 candidates), FP64 NumPy oracle, one "
                       f"spawned process per host core ({cores}) with single-threaded BLAS, "
                       f"{sec:.1f} s wall")


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------

_NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                 0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


def clock_sampler(spec: str):
    """Child process: read the GPU's SM clock, its maximum and the clock event
    reasons through NVML (read only) every 2 ms and print one line per sample
    (wall time, MHz, max MHz, reason bits) until killed."""
    import ctypes
    a = json.loads(spec)
    nv = ctypes.CDLL("libnvidia-ml.so.1")
    if nv.nvmlInit_v2() != 0:
        raise SystemExit(2)
    h = ctypes.c_void_p()
    rc = -1
    if a.get("uuid"):  # the CUDA device's own UUID: right whatever CUDA_VISIBLE_DEVICES says
        rc = nv.nvmlDeviceGetHandleByUUID(a["uuid"].encode(), ctypes.byref(h))
    if rc != 0:
        rc = nv.nvmlDeviceGetHandleByIndex_v2(a["index"], ctypes.byref(h))
    if rc != 0:
        raise SystemExit(3)
    reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
        nv.nvmlDeviceGetCurrentClocksThrottleReasons
    mhz, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
    nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
    print("ready", flush=True)
    while True:
        nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz))
        reasons_fn(h, ctypes.byref(rs))
        print(f"{time.time():.6f} {mhz.value} {mx.value} {rs.value}", flush=True)
        time.sleep(0.002)


class ClockSampler:
    """SM clocks and clock event reasons sampled every 2 ms (NVML, in a child
    process) around the timed region; the samples inside it are kept."""

    def __init__(self, device_index: int, uuid: Optional[str]):
        self.spec = json.dumps(dict(index=device_index, uuid=uuid))
        self.proc = None
        self.t_start = self.t_stop = None

    def start(self):
        try:
            self.proc = subprocess.Popen([sys.executable, os.path.abspath(__file__),
                                          "--clock-sampler", self.spec],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
            line = self.proc.stdout.readline()
            if not line.startswith("ready"):
                self.proc.kill()
                self.proc = None
        except OSError:
            self.proc = None

    def mark(self, start: bool):
        if start:
            self.t_start = time.time()
        else:
            self.t_stop = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.01)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for ln in out.strip().splitlines():
            f = ln.split()
            if len(f) == 4:
                rows.append((float(f[0]), float(f[1]), float(f[2]), int(f[3])))
        inside = [r for r in rows if self.t_start is not None and
                  self.t_start <= r[0] <= (self.t_stop or 1e30)]
        window = "timed region" if inside else "around the timed region"
        rows = inside or rows[-20:]
        if not rows:
            return None
        reasons = sorted({name for r in rows for bit, name in _NVML_REASONS.items()
                          if r[3] & bit})
        return dict(sm_mhz=statistics.median(r[1] for r in rows),
                    sm_max_mhz=max(r[2] for r in rows), reasons=reasons, samples=len(rows),
                    window=window, source="NVML every 2 ms")


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, \
            "fallback"


def kernel_sources_digest(files=("decode_kernel.cuh", "device.cuh")):
    """Digest of a kernel's code (comments and blank lines dropped, so that only
    a change of the code itself retires a committed ncu figure); by default the
    decode kernel's."""
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "int8_kv_cache_gb300", "csrc", f)) as fh:
            for line in fh:
                code = line.split("//", 1)[0].strip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def ncu_traffic(name: str):
    """Per-launch DRAM bytes of a kernel from the committed ncu summary, or None
    when the kernel source changed since the capture."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            d = json.load(f)
    except OSError:
        return None
    e = d.get(name)
    files = PREFILL_SOURCES if name.startswith("sparse_prefill") else ("decode_kernel.cuh",
                                                                       "device.cuh")
    if not e or e.get("kernel_digest") != kernel_sources_digest(files):
        return None
    return e.get("dram_bytes_per_launch")


PREFILL_SOURCES = ("prefill_tc.cu", "tc.cuh", "device.cuh")


def time_graph(torch, graph, replays: int, stream):
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(replays):
            graph.replay()
        end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / 1e3


def capture(torch, fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()  # eager once (also sets kernel attributes) before capture
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def layer_seed(rank: int, layer: int) -> int:
    """Seed of one layer's synthetic inputs: every rank decodes layers of its
    own (replicas; weak scaling)."""
    return 1000 * rank + layer


def max_over_ranks(dist, value: float, device) -> float:
    """The largest of the ranks' values: the whole job ends with its slowest
    rank.  No process group: the value itself."""
    if dist is None:
        return value
    import torch
    tt = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def gpu_arm(args, rank, world, local_rank, dist):
    import numpy as np
    import torch

    import int8_kv_cache_gb300 as K
    import workloads as W

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.Stream()
    props = torch.cuda.get_device_properties(dev)
    peaks, peak_src = measured_peaks()
    l2 = int(getattr(props, "L2_cache_size", 0) or 0)
    L = args.layers

    # ---- inputs: L layers, each its own cache / rows / lists (seeded) ----
    layers = []
    for li in range(L):
        c = W.sparse_decode(S_ROWS, seed=layer_seed(rank, li))
        t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)
        layers.append(dict(q=t(c.q), k=t(c.k_codes), v=t(c.v_codes), ks=t(c.k_scale),
                           vs=t(c.v_scale), idx=t(c.idx), case=c if li == 0 else None,
                           out=torch.empty((S_ROWS, HQ, D), dtype=torch.float16, device=dev)))
    working_set = sum(x["k"].numel() + x["v"].numel() for x in layers)
    ns, chunk, wsb, wave = K.decode_plan(K.PATH_DSA, K.CACHE_INT8, N_SEL, S_ROWS, HQ, HKV, D,
                                         K.GEOM_POW2_TILES)
    ws = torch.empty(max(wsb // 4, 4), dtype=torch.float32, device=dev)
    kind = W.SCALE_PER_CHANNEL

    def step():
        for x in layers:
            K.dsa_decode(x["q"], x["k"], x["v"], x["ks"], x["vs"], kind, x["idx"], SIGMA,
                         num_splits=ns, chunk=chunk, workspace=ws, out=x["out"])

    def step_partials():
        for x in layers:
            K.dsa_decode(x["q"], x["k"], x["v"], x["ks"], x["vs"], kind, x["idx"], SIGMA,
                         num_splits=ns, chunk=chunk, workspace=ws, partials_only=True)

    g = capture(torch, step, stream)
    for _ in range(args.warmup):
        with torch.cuda.stream(stream):
            g.replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(local_rank, getattr(props, "uuid", None) and
                          "GPU-" + str(props.uuid).replace("GPU-", ""))
    clocks.start()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark(True)
    t = time_graph(torch, g, args.steps, stream)
    clocks.mark(False)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    t = max_over_ranks(dist, t, dev)

    b = call_bytes()
    bytes_call = sum(b.values())
    calls = args.steps * L * world
    value = calls * bytes_call / t / 1e9
    us_per_call = t / (args.steps * L) * 1e6
    launches = args.steps * L * (2 if ns > 1 else 1)

    # ---- the decode kernel alone: graph of partials-only launches ----
    gp = capture(torch, step_partials, stream)
    for _ in range(3):
        with torch.cuda.stream(stream):
            gp.replay()
    reps = max(20, min(args.steps, 500))
    tp = time_graph(torch, gp, reps, stream)
    t_kernel = tp / (reps * L)
    kernel_bytes = b["kv"] + b["q"] + b["idx"] + b["scales"]
    achieved = kernel_bytes / t_kernel / 1e9
    traffic = ncu_traffic("dsa_decode_S8")

    # ---- context: 7 rounds of the captured step, and uncaptured launches ----
    rounds = []
    for _ in range(7):
        rounds.append(time_graph(torch, g, max(20, min(args.steps, 200)), stream) /
                      (max(20, min(args.steps, 200)) * L) * 1e6)
    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        n_eager = max(3, min(args.steps, 50))
        for _ in range(n_eager):
            step()
        e1.record(stream)
    e1.synchronize()
    eager_us = e0.elapsed_time(e1) * 1e3 / (n_eager * L)
    attended = S_ROWS * N_SEL  # candidates per call (every list entry is valid)

    # ---- end to end through the public API with host buffers ----
    # Every step copies all layers' query rows and candidate lists from one
    # pinned host buffer (one copy each), calls dsa_decode per layer through
    # the Python binding, and copies all outputs back in one copy.
    dq_all = torch.stack([x["q"] for x in layers])
    didx_all = torch.stack([x["idx"] for x in layers])
    dout_all = torch.empty((L, S_ROWS, HQ, D), dtype=torch.float16, device=dev)
    hq_all = dq_all.cpu().pin_memory()
    hidx_all = didx_all.cpu().pin_memory()
    hout_all = torch.empty((L, S_ROWS, HQ, D), dtype=torch.float16).pin_memory()
    e2e_steps = max(3, min(args.steps, 100))

    views = [(dq_all[i], x["k"], x["v"], x["ks"], x["vs"], didx_all[i], dout_all[i])
             for i, x in enumerate(layers)]

    def e2e_step():
        dq_all.copy_(hq_all, non_blocking=True)
        didx_all.copy_(hidx_all, non_blocking=True)
        for q_, k_, v_, ks_, vs_, idx_, out_ in views:
            K.dsa_decode(q_, k_, v_, ks_, vs_, kind, idx_, SIGMA, num_splits=ns, chunk=chunk,
                         workspace=ws, out=out_)
        hout_all.copy_(dout_all, non_blocking=True)

    # (1) eager: the binding's calls issued from Python every step
    with torch.cuda.stream(stream):
        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        s1.record(stream)
    s1.synchronize()
    te_eager = max_over_ranks(dist, s0.elapsed_time(s1) / 1e3, dev)
    # (2) the same step (copies in, calls, copy out) captured once from the
    # binding and replayed every step, as a decode engine runs it
    ge = capture(torch, e2e_step, stream)
    for _ in range(3):
        with torch.cuda.stream(stream):
            ge.replay()
    torch.cuda.synchronize()
    te = max_over_ranks(dist, time_graph(torch, ge, e2e_steps, stream), dev)
    e2e = dict(value=e2e_steps * L * world * bytes_call / te / 1e9, unit="GB/s",
               h2d_bytes_per_step=L * (b["q"] + b["idx"]), d2h_bytes_per_step=L * b["out"],
               us_per_call=te / (e2e_steps * L) * 1e6, steps=e2e_steps,
               eager_us_per_call=te_eager / (e2e_steps * L) * 1e6,
               eager_value=e2e_steps * L * world * bytes_call / te_eager / 1e9,
               note="per step: one pinned-host copy of all layers' query rows and one of their "
                    "lists, the dsa_decode call of the Python binding per layer, one copy of "
                    "all outputs back; the step is captured once as a CUDA graph (copies "
                    "included) and replayed; eager_* issue the same step from Python every "
                    "time (host-bound by the binding's per-call overhead)")

    out = {
        "metric": "INT8 split-KV decode us/call and achieved HBM GB/s (% of GB300 peak)",
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 5),
        "us_per_call": round(us_per_call, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": round(H200_US_PER_CALL / us_per_call, 3),
        "vs_baseline_basis": "H200 attention time incl. merge for 8 rows, 13.2 us/call "
                             "(onnxruntime PR 33707, Performance; another machine: context)",
        "dtype": "int8 KV, fp16 MMA, fp32 accumulate", "data": "synthetic",
        "config": {"workload": WORKLOAD, "layers_per_step": L, "calls_per_step": L,
                   "num_splits": ns, "chunk": chunk, "wave_ctas": wave,
                   "geometry": "power-of-two tiles rule", "bytes_per_call": bytes_call,
                   "l2_policy": f"inputs larger than L2: {working_set / 1e6:.0f} MB of caches "
                                f"over the step vs L2 {l2 / 1e6:.0f} MB",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "gpu_launches": launches,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1),
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
                     "kernel": "decode_kernel<256,2,sparse,int8,hi+lo>",
                     "us_per_launch": round(t_kernel * 1e6, 3),
                     "bytes_per_launch": kernel_bytes, "peak_source": f"{peak_src} hbm_gbs"},
        "clocks": clk,
        "e2e": e2e,
        "context": {"rounds_us_per_call": [round(r, 3) for r in rounds],
                    "median_of_7_us_per_call": round(statistics.median(rounds), 3),
                    "attended_tokens_per_s": round(attended * calls / t),
                    "uncaptured_us_per_call": round(eager_us, 3),
                    "note": "rounds: the captured step re-timed 7 times after the timed "
                            "region; uncaptured: the same calls launched eagerly from Python"},
    }
    if args.extra != "none":
        out["other_configs"] = extra_configs(torch, K, W, np, dev, stream, peaks, args)
        if args.extra in ("all", "sparse"):
            out["other_configs"]["sparse_decode_rows"] = _sparse_rows(
                torch, K, W, layers, stream, peaks["hbm_gbs"], kernel_us_s8=t_kernel * 1e6,
                call_us_s8=us_per_call)
        deep = out["other_configs"].get("deep_context_int8")
        if deep is not None:
            a = deep["adaptive"]
            kb = deep["bytes_per_call"] - 16 * 16 * 128 * 2  # the kernel writes partials, not O
            out["roofline_deep"] = {
                "bound": "hbm", "achieved": round(kb / (a["kernel_us"] * 1e-6) / 1e9, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(kb / (a["kernel_us"] * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
                "traffic": ncu_traffic("deep_context_int8"),
                "kernel": "decode_kernel<128,1,paged,int8,hi+lo>", "us_per_launch": a["kernel_us"],
                "bytes_per_launch": kb, "us_per_call": a["us_per_call"],
                "workload": deep["workload"] + ", automatic geometry (wave rule, chunk on the CTA round of positions)",
                "peak_source": f"{peak_src} hbm_gbs"}
        pf = out["other_configs"].get("sparse_prefill")
        if pf is not None:
            # the tensor-core prefill against the tensor roofline: the selected
            # candidates' products per call (the algorithmic flops) over the
            # call's time, the executed (masked dense) products beside them
            out["roofline_prefill"] = {
                "bound": "tensor", "achieved": pf["tflops"], "peak": pf["tensor_peak"],
                "unit": "TFLOP/s", "frac": pf["frac_of_tensor"],
                "traffic": ncu_traffic("sparse_prefill_staged"),
                "kernel": "prefill_tc_kernel<256, staged> (+ prefill_stage_kernel<256>)",
                "ms_per_call": pf["ms_per_call"], "flops_per_call": pf["flops_per_call"],
                "executed_tflops": pf["executed_tflops"],
                "executed_frac": pf["executed_frac_of_tensor"],
                "workload": pf["workload"],
                "peak_source": f"{peak_src} bf16_tflops (burst; fp16 taken equal)"}
    return out


def _sparse_rows(torch, K, W, layers, stream, hbm, kernel_us_s8, call_us_s8):
    """The headline workload at S = 1, 2 and 4 query rows (the first S rows of
    each layer's S = 8 rows and lists, the same 32 caches): the call and the
    decode kernel alone, each as a graph of 32 calls."""
    res = {}
    for S in (1, 2, 4):
        ns, chunk, wsb, wave = K.decode_plan(K.PATH_DSA, K.CACHE_INT8, N_SEL, S, HQ, HKV, D,
                                             K.GEOM_POW2_TILES)
        ws = torch.empty(max(wsb // 4, 4), dtype=torch.float32, device=layers[0]["q"].device)
        views = [(x["q"][:S].contiguous(), x["k"], x["v"], x["ks"], x["vs"],
                  x["idx"][:S].contiguous(), torch.empty_like(x["q"][:S])) for x in layers]

        def fn(partials=False):
            for q_, k_, v_, ks_, vs_, idx_, out_ in views:
                K.dsa_decode(q_, k_, v_, ks_, vs_, W.SCALE_PER_CHANNEL, idx_, SIGMA,
                             num_splits=ns, chunk=chunk, workspace=ws,
                             out=None if partials else out_, partials_only=partials)
        b = call_bytes(S=S)
        sec = _graph_seconds(torch, fn, stream, len(views))
        row = dict(us_per_call=round(sec * 1e6, 3), gbs=round(sum(b.values()) / sec / 1e9, 1),
                   frac_of_hbm=round(sum(b.values()) / sec / 1e9 / hbm, 4), num_splits=ns,
                   chunk=chunk, wave_ctas=wave)
        if ns > 1:
            ksec = _graph_seconds(torch, lambda: fn(True), stream, len(views))
            kb = sum(b.values()) - b["out"]
            row.update(kernel_us=round(ksec * 1e6, 3),
                       kernel_frac_of_hbm=round(kb / ksec / 1e9 / hbm, 4))
        res[f"S{S}"] = row
    res["S8"] = dict(us_per_call=round(call_us_s8, 3), kernel_us=round(kernel_us_s8, 3),
                     note="the headline line above")
    return dict(workload=WORKLOAD.replace("S=8 rows", "S=1/2/4 rows") +
                "; 32 layers per graph (the headline's caches, its first S rows and lists)",
                **res)


def _graph_seconds(torch, fn, stream, calls, reps=50):
    g = capture(torch, fn, stream)
    for _ in range(3):
        with torch.cuda.stream(stream):
            g.replay()
    return time_graph(torch, g, reps, stream) / (reps * calls)


def extra_configs(torch, K, W, np, dev, stream, peaks, args):
    """Paged decode, deep-context split sweep and prefill, each as a CUDA graph
    of R calls over R distinct input copies (working set > L2 where the
    workload allows)."""
    res = {}
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    hbm = peaks["hbm_gbs"]

    def bench_graph(fn, R, reps=50):
        g = capture(torch, fn, stream)
        for _ in range(3):
            with torch.cuda.stream(stream):
                g.replay()
        return time_graph(torch, g, reps, stream) / (reps * R)

    if args.extra in ("all", "paged"):
        res["paged_decode"] = _paged(torch, K, W, np, t, dev, bench_graph, hbm)
        res["paged_decode_balanced"] = _paged(torch, K, W, np, t, dev, bench_graph, hbm,
                                              balanced=True)
    if args.extra in ("all", "paged", "variants"):
        res["paged_decode_softcap"] = _paged(torch, K, W, np, t, dev, bench_graph, hbm,
                                             softcap=30.0)
        res["paged_decode_window"] = _paged(torch, K, W, np, t, dev, bench_graph, hbm,
                                            window=1023)
    if args.extra in ("all", "paged", "fp8"):
        res["paged_decode_fp8"] = _paged(torch, K, W, np, t, dev, bench_graph, hbm, cache="fp8")
    if args.extra in ("all", "deep", "fp8"):
        for cache in (("fp8",) if args.extra == "fp8" else ("int8", "fp8", "fp16")):
            res[f"deep_context_{cache}"] = _deep(torch, K, W, np, t, dev, bench_graph, hbm, cache)
    if args.extra in ("all", "prefill"):
        res["sparse_prefill"] = _prefill(torch, K, W, np, t, bench_graph, peaks, dev, stream)
    if args.extra in ("all", "prefill_table"):
        res["sparse_prefill_table"] = _prefill_table(torch, K, W, np, t, bench_graph, peaks)
    if args.extra in ("all", "quantize", "fp8"):
        res["quantize_on_write"] = _quantize(torch, K, np, t, dev, bench_graph, hbm)
        res["quantize_on_write_fp8"] = _quantize(torch, K, np, t, dev, bench_graph, hbm, "fp8")
    return res


def _quantize(torch, K, np, t, dev, bench_graph, hbm, cache="int8"):
    """Quantize-on-write of one 8192-token prefill chunk (8 KV heads, D 128)
    into a paged INT8 or float8 e4m3fn cache with per-channel scales; R
    rotating sets of new rows, slot maps and destinations (inputs and outputs
    of a graph together exceed the L2 three times over)."""
    rng = np.random.default_rng(0)
    T, Hkv, Dh, bs = 8192, 8, 128, 16
    ks = t(np.exp(rng.uniform(-4, -2, size=(Hkv, Dh))).astype(np.float32))
    vs = t(np.exp(rng.uniform(-4, -2, size=(Hkv, Dh))).astype(np.float32))
    R = 8
    nb = T // bs
    cdt = torch.uint8 if cache == "fp8" else torch.int8
    sets = [dict(kn=t(rng.standard_normal((T, Hkv, Dh)).astype(np.float16)),
                 vn=t(rng.standard_normal((T, Hkv, Dh)).astype(np.float16)),
                 k=torch.zeros((nb, bs, Hkv, Dh), dtype=cdt, device=dev),
                 v=torch.zeros((nb, bs, Hkv, Dh), dtype=cdt, device=dev),
                 s=t(rng.permutation(nb * bs).astype(np.int32))) for _ in range(R)]

    def fn():
        for c in sets:
            K.reshape_and_cache(c["kn"], c["vn"], c["s"], c["k"], c["v"], ks, vs, 2)
    sec = bench_graph(fn, R, reps=50)
    byts = 2 * T * Hkv * Dh * 2 + 2 * T * Hkv * Dh + T * 4 + 2 * Hkv * Dh * 4
    name = "float8 e4m3fn" if cache == "fp8" else "INT8"
    return dict(workload=f"quantize-on-write: 8192 new tokens x 8 KV heads x head_dim 128 (fp16) "
                         f"into a paged {name} cache at a permuted slot mapping, per-channel "
                         f"scales",
                us_per_call=round(sec * 1e6, 2), gbs=round(byts / sec / 1e9, 1),
                frac_of_hbm=round(byts / sec / 1e9 / hbm, 4), bytes_per_call=byts,
                rotating_sets=R)


def _paged(torch, K, W, np, t, dev, bench_graph, hbm, softcap=0.0, window=-1, cache="int8",
           balanced=False):
    """Paged decode: 16 sequences, lengths U[512, 8192], 32/8 heads, D 128
    (optionally with a softcap and a sliding window, or a float8 e4m3fn cache;
    with ``balanced``, the balanced pieces instead of the wave rule's chunks)."""
    c = W.paged_decode(seed=0, cache=cache)
    dt = K.CACHE_FP8 if cache == "fp8" else K.CACHE_INT8
    B, Hq, Dh = c.q.shape
    nb, bs, Hkv, _ = c.k_cache.shape
    cap = c.block_table.shape[1] * bs
    R = 3
    copies = [dict(k=t(c.k_cache), v=t(c.v_cache)) for _ in range(R)]
    q, ks, vs = t(c.q), t(c.k_scale), t(c.v_scale)
    bt, lens, sink = t(c.block_table), t(c.seq_lens), t(c.sink)
    ns, chunk, wsb, wave = K.decode_plan(K.PATH_PAGED, dt, K.window_span(cap, window),
                                         B, Hq, Hkv, Dh,
                                         K.GEOM_BALANCED if balanced else K.GEOM_WAVE)
    ws = torch.empty(max(wsb // 4, 4), dtype=torch.float32, device=dev)
    out = torch.empty_like(q)
    live = np.minimum(c.seq_lens, window + 1) if window >= 0 else c.seq_lens
    tokens = int(live.sum())
    first = (c.seq_lens - live) // bs
    blocks = int(((c.seq_lens + bs - 1) // bs - first).sum())
    byts = tokens * Hkv * Dh * 2 + B * Hq * Dh * 4 + blocks * 4 + 2 * Hkv * Dh * 4

    def fn():
        for x in copies:
            K.paged_decode(q, x["k"], x["v"], ks, vs, c.scale_kind, bt, lens, c.sigma, sink,
                           num_splits=ns, chunk=chunk, workspace=ws, out=out, softcap=softcap,
                           window=window)
    sec = bench_graph(fn, R)
    opts = ""
    if balanced:
        opts += ", balanced pieces (device-cut, about one wave)"
    if softcap > 0:
        opts += f", softcap {softcap:g}"
    if window >= 0:
        opts += f", sliding window {window} (attended sum {tokens})"
    return dict(
        workload="paged %s decode: 16 sequences, lengths U[512,8192] (sum %d), block 16, "
                 "permuted block table, 32/8 heads, head_dim 128, per-channel scales, sink%s"
                 % ("float8 e4m3fn" if cache == "fp8" else "INT8", int(c.seq_lens.sum()), opts),
        us_per_call=round(sec * 1e6, 2), gbs=round(byts / sec / 1e9, 1),
        frac_of_hbm=round(byts / sec / 1e9 / hbm, 4), bytes_per_call=byts, num_splits=ns,
        chunk=chunk, wave_ctas=wave, rotating_copies=R)


def _deep(torch, K, W, np, t, dev, bench_graph, hbm, cache):
    """Deep-context split sweep: 16 rows, cap 4096, live 2600, 16/2 heads."""
    c = W.deep_context(seed=0, cache=cache)
    B, Hq, Dh = c.q.shape
    nb, bs, Hkv, _ = c.k_cache.shape
    esz = 2 if cache == "fp16" else 1
    R = 10 if cache == "fp16" else 20
    copies = [dict(k=t(c.k_cache), v=t(c.v_cache)) for _ in range(R)]
    q, ks, vs, bt, lens = t(c.q), t(c.k_scale), t(c.v_scale), t(c.block_table), t(c.seq_lens)
    byts = B * 2600 * Hkv * Dh * 2 * esz + B * Hq * Dh * 4 + B * (2600 // 16 + 1) * 4
    dt = {"int8": K.CACHE_INT8, "fp8": K.CACHE_FP8, "fp16": K.CACHE_FP16}[cache]
    row = {}
    for label, ovr in (("adaptive", 0), ("chunk128", 128), ("chunk256", 256), ("chunk512", 512)):
        ns, chunk, wsb, wave = K.decode_plan(K.PATH_PAGED, dt, 4096, B, Hq, Hkv, Dh,
                                             K.GEOM_WAVE, ovr)
        ws = torch.empty(max(wsb // 4, 4), dtype=torch.float32, device=dev)
        out = torch.empty_like(q)

        def fn(partials=False):
            for x in copies:
                K.paged_decode(q, x["k"], x["v"], ks, vs, c.scale_kind, bt, lens, c.sigma,
                               num_splits=ns, chunk=chunk, workspace=ws,
                               out=None if partials else out, partials_only=partials)
        sec = bench_graph(fn, R, reps=100)
        row[label] = dict(us_per_call=round(sec * 1e6, 2), gbs=round(byts / sec / 1e9, 1),
                          frac_of_hbm=round(byts / sec / 1e9 / hbm, 4), num_splits=ns,
                          chunk=chunk)
        if ns > 1:
            # the decode kernel alone (partials only, no combine); its bytes
            # exclude the output
            kb = byts - B * Hq * Dh * 2
            ks_ = bench_graph(lambda: fn(True), R, reps=100)
            row[label].update(kernel_us=round(ks_ * 1e6, 2),
                              kernel_frac_of_hbm=round(kb / ks_ / 1e9 / hbm, 4))
    return dict(workload=f"deep context: 16 rows, {cache} cache, live 2600 of cap 4096, 16/2 "
                         "heads, head_dim 128", bytes_per_call=byts, rotating_copies=R, **row)


def _prefill(torch, K, W, np, t, bench_graph, peaks, dev, stream):
    """Sparse prefill: 2048 rows over an 8192-token cache, 24/2 heads, D 256.
    The dense tensor-core kernel computes S and PV over every 128-token block
    some row of a 128-vector tile selects (rows' unselected positions get
    probability 0): `executed_tflops` counts those products, `tflops` only the
    selected candidates' (the algorithmic flops)."""
    c = W.sparse_prefill(seed=0)
    d = dict(q=t(c.q), k=t(c.k_codes), v=t(c.v_codes), ks=t(c.k_scale), vs=t(c.v_scale),
             idx=t(c.idx))
    out = torch.empty_like(d["q"])
    S, Hq, Dh = c.q.shape
    N, Hkv, _ = c.k_codes.shape
    # the staged form: the call converts the cache once into fp16 operand
    # images in this workspace (allocated once, like a decode's split workspace)
    ws = torch.empty(K.prefill_workspace_bytes(S, Hq, Hkv, Dh, N, c.idx.shape[1]),
                     dtype=torch.uint8, device=d["q"].device)

    def fn(staged=True):
        K.dsa_prefill(d["q"], d["k"], d["v"], d["ks"], d["vs"], c.scale_kind, d["idx"], c.sigma,
                      out=out, workspace=ws if staged else None)
    sec = bench_graph(fn, 1, reps=10)
    sec_conv = bench_graph(lambda: fn(False), 1, reps=10)
    # the SM clock while the staged form runs back to back for about 0.1 s
    # (dense tensor work at this rate runs into the board's power limit)
    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    sampler = ClockSampler(dev.index or 0, uuid and "GPU-" + str(uuid).replace("GPU-", ""))
    g = capture(torch, fn, stream)
    for _ in range(3):
        with torch.cuda.stream(stream):
            g.replay()
    torch.cuda.synchronize()
    sampler.start()
    sampler.mark(True)
    sec_long = time_graph(torch, g, 300, stream) / 300
    sampler.mark(False)
    clk = sampler.stop()
    G = Hq // Hkv
    n_att = int((c.idx >= 0).sum())
    flops = n_att * Hq * Dh * 4
    gathered = n_att * Hkv * 2 * Dh
    # blocks of 128 positions each 128-vector tile runs (the same for every KV
    # head: the tiles cover (row, head) pairs of one KV head)
    blk = np.where(c.idx >= 0, c.idx // 128, -1)
    nblk = (N + 127) // 128
    rowsel = np.zeros((S, nblk), bool)
    for r in range(S):
        b = blk[r][blk[r] >= 0]
        rowsel[r, b] = True
    tiles = (S * G + 127) // 128
    executed_blocks = 0
    for tt in range(tiles):
        r0, r1 = (tt * 128) // G, min(tt * 128 + 127, S * G - 1) // G
        executed_blocks += int(rowsel[r0:r1 + 1].any(axis=0).sum())
    executed = executed_blocks * Hkv * 128 * 128 * Dh * 4
    peak_tf = peaks["bf16_tflops"]
    return dict(
        workload="sparse prefill: 2048 rows at positions 6144+i over an 8192-token int8 cache, "
                 "2048 candidates per row, 24/2 heads, head_dim 256",
        kernel="prefill_stage_kernel<256> + prefill_tc_kernel<256, staged> (tcgen05, dense "
               "128-token blocks with row masks, fp16 operand images copied in by one thread)",
        ms_per_call=round(sec * 1e3, 4), tflops=round(flops / sec / 1e12, 2),
        converting_form_ms_per_call=round(sec_conv * 1e3, 4),
        workspace_bytes=int(ws.numel()),
        frac_of_tensor=round(flops / sec / 1e12 / peak_tf, 4), tensor_peak=peak_tf,
        executed_tflops=round(executed / sec / 1e12, 2),
        executed_frac_of_tensor=round(executed / sec / 1e12 / peak_tf, 4),
        gathered_gbs=round(gathered / sec / 1e9, 1), flops_per_call=flops,
        executed_flops_per_call=executed,
        back_to_back=dict(calls=300, ms_per_call=round(sec_long * 1e3, 4), clocks=clk))


def _prefill_table(torch, K, W, np, t, bench_graph, peaks):
    """Sparse prefill at the pages' row counts and contexts (128 / 2048 / 8192
    rows, the last rows of an 8192- or 32768-token cache, 2048 candidates per
    row, 24/2 heads, head_dim 256), and the literal reading of the configured
    workload (row i of 2048 at position i of an 8192-token cache, min(2048,
    i + 1) candidates).  Each call runs the path the library picks:
    the tensor-core kernel over dense blocks (staged form, with a workspace)
    where the lists cover at least a quarter of the cache, else the gathering
    kernel."""
    rows_out = []
    peak_tf = peaks["bf16_tflops"]
    shapes = [(rows, ctx, False) for ctx in (8192, 32768) for rows in (128, 2048, 8192)]
    shapes.append((2048, 8192, True))  # the literal reading: row i at position i
    for rows, ctx, literal in shapes:
        c = W.sparse_prefill(seed=0, rows=rows, N=ctx, literal=literal)
        d = dict(q=t(c.q), k=t(c.k_codes), v=t(c.v_codes), ks=t(c.k_scale),
                 vs=t(c.v_scale), idx=t(c.idx))
        out = torch.empty_like(d["q"])
        S, Hq, Dh = c.q.shape
        N, Hkv, _ = c.k_codes.shape
        wsb = K.prefill_workspace_bytes(S, Hq, Hkv, Dh, N, c.idx.shape[1])
        ws = torch.empty(wsb, dtype=torch.uint8, device=d["q"].device) if wsb else None

        def fn():
            K.dsa_prefill(d["q"], d["k"], d["v"], d["ks"], d["vs"], c.scale_kind, d["idx"],
                          c.sigma, out=out, workspace=ws)
        sec = bench_graph(fn, 1, reps=5 if rows > 2048 else 10)
        flops = int((c.idx >= 0).sum()) * Hq * Dh * 4
        # the automatic split count, from the workspace it asked for
        stage = Hkv * ((N + 127) // 128) * 2 * 128 * Dh * 2 + S * ((N + 127) // 128) * 16 + S * 4
        splits = 1 if wsb <= stage else \
            (wsb - (stage + 255) // 256 * 256) // (S * Hq * (Dh + 2) * 4)
        rows_out.append(dict(
            rows=rows, context=ctx, positions="i" if literal else f"{ctx - rows} + i",
            kernel=(f"prefill_tc_kernel<256, staged> (tcgen05), {splits} split(s)" +
                    (" + combine_kernel<256>" if splits > 1 else "")) if wsb else
                   "decode_kernel<256, sparse, int8, one probability tile> (mma.sync, "
                   "gathered rows, no splits)",
            ms_per_call=round(sec * 1e3, 4), tflops=round(flops / sec / 1e12, 2),
            frac_of_tensor=round(flops / sec / 1e12 / peak_tf, 4)))
        del d, out, ws
    return dict(workload="sparse prefill, rows at positions N - rows + i (and, last, row i at "
                         "position i) of an N-token int8 cache, min(2048, position + 1) sorted "
                         "unique candidates per row from [0, position], 24/2 heads, head_dim "
                         "256, per-channel scales, softmax scale 1/16",
                tensor_peak=peak_tf, cases=rows_out)


def reference_arm(args, rank, world):
    """The FP64 oracle on the host cores (one spawned process per core,
    single-threaded BLAS each), on the headline workload, metric and unit.
    Each step is a bounded sample: every core computes the same number of whole
    query rows, sized so the whole run stays near two minutes.  Under torchrun
    only rank 0 runs and prints."""
    if rank != 0:
        return None
    cores = host_cores()
    pool = OraclePool(cores)
    try:
        t_row = pool.step(1)
        n = max(1, int(120.0 / max(1, args.steps + args.warmup) / max(t_row, 1e-6)))
        for _ in range(args.warmup):
            pool.step(n)
        sec = sum(pool.step(n) for _ in range(args.steps))
    finally:
        pool.close()
    rows = n * cores * args.steps
    row_bytes = sum(call_bytes().values()) / S_ROWS
    v = rows * row_bytes / sec / 1e9
    sample = (f"{n * cores} query row(s) per step ({n} per core, both KV heads; a call is "
              f"{S_ROWS} rows) of the headline workload, {args.steps} timed step(s) after "
              f"{args.warmup} warm-up, FP64 NumPy oracle, one spawned process per host core "
              f"with single-threaded BLAS")
    return {"metric": "INT8 split-KV decode us/call and achieved HBM GB/s (% of GB300 peak)",
            "value": v, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": sec / args.steps * 1e3,
            "us_per_call": sec / rows * S_ROWS * 1e6,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD}, "impl": "reference",
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    if args.clock_sampler is not None:
        clock_sampler(args.clock_sampler)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if args.impl == "reference":
        res = reference_arm(args, rank, world)
        if res is not None:
            print(json.dumps(res))
        return
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(local_rank)
        tdist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        dist = tdist
    res = gpu_arm(args, rank, world, local_rank, dist)
    if rank == 0:
        try:
            res["cpu_baseline"] = None if args.no_cpu_baseline else run_cpu_oracle(10.0)
        except Exception as e:  # the GPU figure stands without it
            res["cpu_baseline"] = {"error": str(e)[:300]}
        print(json.dumps(res))
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
