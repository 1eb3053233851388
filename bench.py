"""Benchmark of the fused attention hot path on GB300.

One step = one pass of the attention forward (scores, scale, causal mask,
online softmax, P.V, normalisation and store) over the long-sequence causal
workload: batch 4, 16 heads, n_q = n_k = 8192, d_k = d_v = 128, bf16 Q/K/V =
0.5 N(0,1), lower-triangular mask, fp32 softmax statistics.  The metric is
attention forward TFLOP/s with 4 b h n_q n_k d_k FLOP per pass, halved for the
causal mask, whole job (all ranks).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload long_causal|restricted|decode|wide512|backward|
                                   backward512|tiny_f32|enc_base|enc_mha_base|dec_causal_base|
                                   cross_big|cross_mha_big]
Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(no data-path collective); the timed region is bracketed by a barrier and the
maximum over ranks is reported.  `--impl reference` times the CPU oracle on a
bounded sample of the same workload on the host cores (rank 0 only).

`--workload` other than the default measures one of the widened rows with the
same JSON line (value, roofline, e2e, clocks, an oracle baseline on a bounded
sample): restricted self-attention (r = 1024), one decoding step against
8192-token caches, Table 3's single 512-wide head, and the backward pass (at
d = 128 and at the 512-wide head); or
one of the smaller configurations of the base and big models: the fp32 tiny
case, the encoder's attention (core, and with its projections), the
decoder's causal self-attention, and the big model's cross-attention (core,
and with its projections).  These rotate over enough input sets that the
inputs exceed L2, and report their roofline in GB/s against the algorithmic
bytes (the multi-head lines: TFLOP/s of the whole call).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synthetic  # noqa: E402

WORKLOAD = "long_causal"
E2E_HEADS_PER_CHUNK = 8   # e2e pipeline granularity: (batch, 8 heads) per chunk
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
METRIC = "attention fwd TFLOP/s and % of GB300 BF16 tensor peak (1 GPU)"
KERNEL_SOURCE = os.path.join(ROOT, "transformer_scaled_dot_02_gb300", "csrc", "sdpa_tc.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")


def metric_flops(w: synthetic.Workload) -> float:
    f = 4.0 * w.b * w.h * w.n_q * w.n_k * w.d_k
    return f / 2 if w.causal else f


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_sha(source: str = KERNEL_SOURCE) -> str:
    """Hash of a kernel's code: comments and blank space are left out, so a
    comment edit keeps the recorded DRAM traffic valid; any code change voids it."""
    import re
    with open(source, encoding="utf-8") as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    code = " ".join(src.split())
    return hashlib.sha256(code.encode()).hexdigest()[:16]


def recorded_traffic(workload: str):
    """dram read+write bytes per launch from the committed ncu summary, or
    None when the kernel source changed since it was captured."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(workload)
    if not e:
        return None
    source = os.path.join(ROOT, "transformer_scaled_dot_02_gb300", "csrc",
                          e.get("source_file", "sdpa_tc.cu"))
    if e.get("kernel_sha") != kernel_sha(source):
        return None
    return e.get("bytes_per_launch")


# ------------------------------------------------------------------ clocks
_REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
            0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
            0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
            0x100: "display_clock_setting"}


class ClockSampler:
    """Reads the SM clock and the clock-event reasons through NVML (read only)
    on a background thread while the timed region runs."""

    def __init__(self, device_index: int, period_s: float = 0.002):
        self.samples = []
        self.max_mhz = None
        self.ok = False
        self._stop = threading.Event()
        self._period = period_s
        try:
            import ctypes
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            handle = ctypes.c_void_p()
            uuid = None
            vis = os.environ.get("CUDA_VISIBLE_DEVICES")
            idx = device_index
            if vis:
                parts = [p.strip() for p in vis.split(",") if p.strip()]
                if device_index < len(parts):
                    if parts[device_index].isdigit():
                        idx = int(parts[device_index])
                    else:
                        uuid = parts[device_index]
            if uuid is not None:
                rc = nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(handle))
            else:
                rc = nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(idx), ctypes.byref(handle))
            if rc != 0:
                return
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self._nv, self._h, self._ct = nv, handle, ctypes
            self.ok = True
        except OSError:
            return

    def _run(self):
        ct, nv, h = self._ct, self._nv, self._h
        clk = ct.c_uint()
        reasons = ct.c_ulonglong()
        while not self._stop.is_set():
            r1 = nv.nvmlDeviceGetClockInfo(h, 1, ct.byref(clk))
            r2 = nv.nvmlDeviceGetCurrentClocksEventReasons(h, ct.byref(reasons))
            if r1 == 0:
                self.samples.append((clk.value, reasons.value if r2 == 0 else 0))
            time.sleep(self._period)

    def __enter__(self):
        if self.ok:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *exc):
        if self.ok:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": "nvml" if self.ok else "unavailable"}
        mhz = [s[0] for s in self.samples]
        bits = 0
        for _, r in self.samples:
            bits |= r
        names = [n for b, n in _REASONS.items() if bits & b and n != "gpu_idle"]
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": self.max_mhz, "reasons": names,
                "samples": len(mhz), "source": "nvml"}


# ------------------------------------------------------------- distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value, pg, device):
    """The largest `value` of all ranks, on every rank (`value` itself with no
    process group): the job takes as long as its slowest replica."""
    if pg is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, flops_per_step, steps, ms):
    """Whole-job TFLOP/s: every replica's work over the slowest rank's time
    (weak scaling: each rank runs the full workload on its own GPU)."""
    return world * flops_per_step * steps / (ms * 1e-3) / 1e12


# ------------------------------------------------------------------- ours
def run_ours(args, world, rank, local):
    import torch
    import transformer_scaled_dot_02_gb300 as sd

    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist
    sd.load_library()

    w = synthetic.WORKLOADS[WORKLOAD]
    q, k, v, lens = synthetic.sdpa_inputs(w)
    dev = torch.device("cuda", local)
    qd = torch.from_numpy(q).to(torch.bfloat16).to(dev)
    kd = torch.from_numpy(k).to(torch.bfloat16).to(dev)
    vd = torch.from_numpy(v).to(torch.bfloat16).to(dev)
    od = torch.empty((w.b, w.h, w.n_q, w.d_v), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream

    def step():
        sd.sdpa_forward(qd, kd, vd, od, w.b, w.h, w.n_q, w.n_k, w.d_k, w.d_v, w.mask_kind,
                        None, 0.0, sp)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    sd.sdpa_device_check()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local)
    with sampler:
        t0.record(stream)
        for i in range(args.steps):
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        t1.record(stream)
        torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    sd.sdpa_device_check()
    total_ms = t0.elapsed_time(t1)
    launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = max_over_ranks(total_ms, pg, dev)

    # end to end through the C ABI: pinned host inputs -> device -> attention -> host
    e2e_steps = max(1, min(args.steps, 20))
    qh = torch.from_numpy(q).to(torch.bfloat16).pin_memory()
    kh = torch.from_numpy(k).to(torch.bfloat16).pin_memory()
    vh = torch.from_numpy(v).to(torch.bfloat16).pin_memory()
    oh = torch.empty(od.shape, dtype=torch.bfloat16).pin_memory()

    # The public host-buffer entry point (sdpa_forward_host in the C ABI): per
    # (batch, 8-head) chunk, the copy in, the attention and the copy out run on
    # the library's three streams, so the copies of one chunk overlap the
    # attention of another.
    def e2e_step():
        sd.attention_from_host(qh, kh, vh, oh, qd, kd, vd, od, w.mask_kind, None, 0.0,
                               heads_per_chunk=E2E_HEADS_PER_CHUNK, stream=stream)

    e2e_step()
    torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1)
    e2e_ms = max_over_ranks(e2e_ms, pg, dev)
    sd.sdpa_device_check()

    flops = metric_flops(w)
    value = job_throughput(world, flops, args.steps, total_ms)
    e2e_value = job_throughput(world, flops, e2e_steps, e2e_ms)
    peaks, peak_src = load_peaks()
    mean_launch_ms = float(np.mean(launch_ms))
    achieved = flops / (mean_launch_ms * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    traffic = recorded_traffic(WORKLOAD)

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "long-sequence causal self-attention b4 h16 n8192 d128 bf16",
                   "b": w.b, "h": w.h, "n_q": w.n_q, "n_k": w.n_k, "d_k": w.d_k, "d_v": w.d_v,
                   "mask": "causal", "values": "0.5*N(0,1) rounded to bf16",
                   "accumulate": "fp32", "parallelism": "replicas" if world > 1 else "single",
                   "l2": "inputs larger than L2 (Q+K+V 403 MB, O 134 MB vs 129 MB L2)"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "peak_source": "%s bf16_tflops (burst)" % peak_src,
                     "frac_of_sustained": round(achieved / peak_sus, 4),
                     "traffic": traffic, "kernel": "sdpa_fwd_bf16_tc<128, 128>",
                     "launch_ms_mean": round(mean_launch_ms, 4),
                     "launch_ms_min": round(float(np.min(launch_ms)), 4)},
        "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(qh.numel() * 2 + kh.numel() * 2 + vh.numel() * 2),
                "d2h_bytes_per_step": int(oh.numel() * 2), "steps": e2e_steps,
                "path": "sdpa_forward_host (C ABI): (batch, %d-head) chunks, copy in / "
                        "attention / copy out on the library's three streams"
                        % E2E_HEADS_PER_CHUNK},
        "gpu_launches": args.steps,
        "clocks": sampler.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_baseline(w, q, k, v, args.cpu_rows)
    if pg:
        pg.barrier()
        pg.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


# ------------------------------------------------ the widened rows (--workload)
ROW_WORKLOADS = ("restricted", "decode", "wide512", "backward", "backward512")


def _visible_restricted(w, rows):
    """Keys each query row i sees under the causal mask and window r."""
    i = rows % w.n_q
    left = (w.window - 1) // 2
    return np.minimum(i, left) + 1


def _time_steps(step, args, stream, pg, dev, local):
    """W warm-up steps, then K steps between a barrier and a synchronize on
    both sides, with an event pair around each step on the launching stream."""
    import torch
    import transformer_scaled_dot_02_gb300 as sd
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    sd.sdpa_device_check()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local)
    with sampler:
        t0.record(stream)
        for i in range(args.steps):
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        t1.record(stream)
        torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    sd.sdpa_device_check()
    total = max_over_ranks(t0.elapsed_time(t1), pg, dev)
    return total, [a.elapsed_time(b) for a, b in zip(starts, ends)], sampler.summary()


def _time_graph(step, args, pg, dev, local, cur):
    """The K steps captured into one CUDA graph (after a warm-up), then one
    replay timed between events on the replay stream, bracketed by a barrier
    and a synchronize.  `cur[0]` is the stream the steps launch on: the
    capture stream while capturing."""
    import torch
    import transformer_scaled_dot_02_gb300 as sd
    side = torch.cuda.Stream(dev)
    graph = torch.cuda.CUDAGraph()
    saved = cur[0]
    cur[0] = side.cuda_stream
    try:
        with torch.cuda.stream(side):
            for _ in range(args.warmup):
                step()
            torch.cuda.synchronize(dev)
            with torch.cuda.graph(graph, stream=side):
                for _ in range(args.steps):
                    step()
    finally:
        cur[0] = saved
    torch.cuda.synchronize(dev)
    sd.sdpa_device_check()
    replay = torch.cuda.current_stream(dev)
    graph.replay()      # one untimed replay
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local)
    with sampler:
        t0.record(replay)
        graph.replay()
        t1.record(replay)
        torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    sd.sdpa_device_check()
    return max_over_ranks(t0.elapsed_time(t1), pg, dev), sampler.summary()


def _time_e2e(e2e_step, args, stream, pg, dev):
    import torch
    import transformer_scaled_dot_02_gb300 as sd
    steps = max(1, min(args.steps, 20))
    e2e_step()
    torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    sd.sdpa_device_check()
    return max_over_ranks(e0.elapsed_time(e1), pg, dev), steps


def _pinned(a, dtype):
    import torch
    return torch.from_numpy(a).to(dtype).pin_memory()


def run_row(args, world, rank, local):
    """One of the widened rows: restricted, decode, wide512, backward or backward512."""
    import torch
    import transformer_scaled_dot_02_gb300 as sd

    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist
    sd.load_library()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    bf = torch.bfloat16
    kind = args.workload
    peaks, peak_src = load_peaks()

    if kind == "backward":
        w = synthetic.WORKLOADS["long_causal"]
    elif kind == "backward512":
        w = synthetic.WORKLOADS["wide_d512"]
    else:
        w = synthetic.WORKLOADS[{"restricted": "long_restricted", "decode": "decode_big",
                                 "wide512": "wide_d512"}[kind]]
    if kind == "decode" and args.decode_queries != w.n_q:
        import dataclasses
        w = dataclasses.replace(w, n_q=args.decode_queries)
    q, k, v, _ = synthetic.sdpa_inputs(w)
    hq, hk, hv = _pinned(q, bf), _pinned(k, bf), _pinned(v, bf)
    qd, kd, vd = hq.to(dev), hk.to(dev), hv.to(dev)
    od = torch.empty((w.b, w.h, w.n_q, w.d_v), dtype=bf, device=dev)
    ho = torch.empty(od.shape, dtype=bf).pin_memory()
    bh = w.b * w.h

    if kind in ("restricted", "wide512"):
        r = w.window

        def step():
            if r:
                sd.sdpa_forward_restricted(qd, kd, vd, od, w.b, w.h, w.n_q, w.n_k, w.d_k, w.d_v,
                                           w.mask_kind, None, r, 0.0, sp)
            else:
                sd.sdpa_forward(qd, kd, vd, od, w.b, w.h, w.n_q, w.n_k, w.d_k, w.d_v,
                                w.mask_kind, None, 0.0, sp)

        ins, outs = [(qd, hq), (kd, hk), (vd, hv)], [(ho, od)]
        if r:
            all_rows = np.arange(bh * w.n_q, dtype=np.int64)
            work = float(np.sum(4.0 * w.d_k * _visible_restricted(w, all_rows)))
            metric = "restricted self-attention fwd TFLOP/s over visible pairs (1 GPU)"
            desc = ("restricted causal self-attention b4 h16 n8192 d128 bf16, window r=%d "
                    "(keys i-(r-1)/2 .. i)" % r)
            kernel = "sdpa_fwd_one_tile<128>"
        else:
            work = metric_flops(w)
            metric = "attention fwd TFLOP/s, one 512-wide head (Table 3 row A) (1 GPU)"
            desc = "long causal self-attention b4 h1 n8192 d_k=d_v=512 bf16"
            kernel = "sdpa_fwd_one_tile<512>"
        unit, bound, peak = "TFLOP/s", "tensor", float(peaks["bf16_tflops"])
        launches = 1
        # every row of the workload: a few seconds of the fp64 oracle
        sample_rows = min(args.cpu_rows or bh * w.n_q, bh * w.n_q)

        def oracle_sample():
            import oracle
            threads = oracle.default_threads()
            rows = _sample_rows(w, sample_rows, 99)
            t = time.perf_counter()
            oracle.sdpa(q, k, v, w.mask_kind, None, rows=rows, threads=threads, window=r or None)
            dt = time.perf_counter() - t
            i = rows % w.n_q
            vis = _visible_restricted(w, rows) if r else (i + 1)
            return (float(np.sum(4.0 * w.d_k * vis)) / dt / 1e12, threads,
                    "%d of the %d query rows of the workload (fp64 C oracle, %.1f s)"
                    % (len(rows), bh * w.n_q, dt))
    elif kind == "decode":
        ws_bytes = sd.sdpa_decode_workspace_size(w.b, w.h, w.n_q, w.n_k, w.d_v)
        ws = torch.empty(max(1, ws_bytes), dtype=torch.uint8, device=dev)

        def step():
            sd.sdpa_decode(qd, kd, vd, od, ws, ws.numel(), w.b, w.h, w.n_q, w.n_k, w.d_k, w.d_v,
                           None, 0.0, sp)

        # a serving loop keeps the caches resident: each step brings in the new
        # queries and reads back their outputs
        ins, outs = [(qd, hq)], [(ho, od)]
        work = 2.0 * bh * w.n_k * (w.d_k + w.d_v)    # K and V caches, bf16, read once
        metric = "decode step: K/V cache read GB/s (1 GPU)"
        desc = ("one decoding step, b32 h16, %d quer%s against 8192-token K/V caches, d128 bf16"
                % (w.n_q, "y" if w.n_q == 1 else "ies"))
        kernel = "sdpa_decode_split + sdpa_decode_combine"
        unit, bound, peak = "GB/s", "hbm", float(peaks["hbm_gbs"])
        launches = 2
        sample_rows = min(args.cpu_rows or bh * w.n_q, bh * w.n_q)   # every (sequence, head)

        def oracle_sample():
            import oracle
            threads = oracle.default_threads()
            rows = np.sort(np.random.default_rng(99).choice(bh * w.n_q, size=sample_rows,
                                                            replace=False)).astype(np.int64)
            t = time.perf_counter()
            oracle.decode(q, k, v, None, rows=rows, threads=threads)
            dt = time.perf_counter() - t
            return (2.0 * len(rows) * w.n_k * (w.d_k + w.d_v) / dt / 1e9, threads,
                    "%d of the %d (sequence, head) decode rows (fp64 C oracle, %.1f s)"
                    % (len(rows), bh * w.n_q, dt))
    else:   # backward
        do = synthetic.dout_input(w)
        hdo = _pinned(do, bf)
        dod = hdo.to(dev)
        fwd_out, lse = sd.attention_with_lse(qd, kd, vd, w.mask_kind)
        hlse = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
        hlse.copy_(lse)
        hfo = torch.empty(fwd_out.shape, dtype=bf).pin_memory()
        hfo.copy_(fwd_out)
        grads = [torch.empty_like(x) for x in (qd, kd, vd)]
        hgrads = [torch.empty(x.shape, dtype=bf).pin_memory() for x in grads]
        ws = torch.empty(sd.sdpa_backward_workspace_size(w.b, w.h, w.n_q, w.d_k),
                         dtype=torch.uint8, device=dev)

        def step():
            sd.sdpa_backward(qd, kd, vd, fwd_out, dod, lse, *grads, ws, ws.numel(), w.b, w.h,
                             w.n_q, w.n_k, w.d_k, w.d_v, w.mask_kind, None, 0, 0.0, sp)

        ins = [(qd, hq), (kd, hk), (vd, hv), (fwd_out, hfo), (dod, hdo), (lse, hlse)]
        outs = list(zip(hgrads, grads))
        work = 2.0 * bh * w.n_q * w.n_k * (3 * w.d_k + 2 * w.d_v) / 2
        if kind == "backward":
            metric = "attention backward TFLOP/s (dQ, dK, dV: five products) (1 GPU)"
            desc = "backward of long causal self-attention b4 h16 n8192 d128 bf16"
            kernel = "sdpa_bwd_tc_n64<128, 128> (with its prep and convert kernels)"
        else:
            metric = ("attention backward TFLOP/s (dQ, dK, dV: five products), one 512-wide "
                      "head (Table 3 row A) (1 GPU)")
            desc = "backward of long causal self-attention b4 h1 n8192 d_k=d_v=512 bf16"
            kernel = "sdpa_bwd_tc_w512 (with its prep and convert kernels)"
        unit, bound, peak = "TFLOP/s", "tensor", float(peaks["bf16_tflops"])
        launches = 3
        # one whole head of the workload at d = 128 (about 12 s of the oracle);
        # at d = 512 its first 4096 query and key rows (about 12 s as well)
        default_rows = w.n_q if w.d_k <= 128 else w.n_q // 2
        prefix = min(args.cpu_rows or default_rows, w.n_q)

        def oracle_sample():
            import oracle
            threads = oracle.default_threads()
            sl = (slice(0, 1), slice(0, 1), slice(0, prefix))
            t = time.perf_counter()
            oracle.backward(q[sl], k[sl], v[sl], do[sl], w.mask_kind, threads=threads)
            dt = time.perf_counter() - t
            flops = 2.0 * prefix * prefix * (3 * w.d_k + 2 * w.d_v) / 2
            what = ("one whole head of the workload" if prefix == w.n_q else
                    "the first %d query and key rows of one head: itself a causal problem" % prefix)
            return flops / dt / 1e12, threads, "%s (fp64 C oracle, %.1f s)" % (what, dt)

    total_ms, launch_ms, clocks = _time_steps(step, args, stream, pg, dev, local)

    def e2e_step():
        for dst, src in ins:
            dst.copy_(src, non_blocking=True)
        step()
        for dst, src in outs:
            dst.copy_(src, non_blocking=True)

    e2e_ms, e2e_steps = _time_e2e(e2e_step, args, stream, pg, dev)
    scale = 1e12 if unit == "TFLOP/s" else 1e9
    value = world * work * args.steps / (total_ms * 1e-3) / scale
    mean_ms = float(np.mean(launch_ms))
    achieved = work / (mean_ms * 1e-3) / scale
    line = {
        "metric": metric, "value": round(value, 2), "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": desc, "b": w.b, "h": w.h, "n_q": w.n_q, "n_k": w.n_k,
                   "d_k": w.d_k, "d_v": w.d_v, "parallelism": "replicas" if world > 1 else "single",
                   "l2": "inputs larger than L2"},
        "roofline": {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
                     "frac": round(achieved / peak, 4),
                     "peak_source": "%s %s" % (peak_src, "hbm_gbs" if bound == "hbm"
                                               else "bf16_tflops (burst)"),
                     "traffic": recorded_traffic(kind), "kernel": kernel,
                     "launch_ms_mean": round(mean_ms, 4),
                     "launch_ms_min": round(float(np.min(launch_ms)), 4)},
        "e2e": {"value": round(world * work * e2e_steps / (e2e_ms * 1e-3) / scale, 3), "unit": unit,
                "h2d_bytes_per_step": int(sum(d.numel() * d.element_size() for d, _ in ins)),
                "d2h_bytes_per_step": int(sum(d.numel() * d.element_size() for d, _ in outs)),
                "steps": e2e_steps, "path": "pinned host inputs copied in, the C-ABI call, "
                                            "outputs copied back, one stream"},
        "gpu_launches": args.steps * launches,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        val, threads, sample = oracle_sample()
        line["cpu_baseline"] = {"value": val, "unit": unit, "cores": threads, "kind": "oracle",
                                "cpu": cpu_model(),
                                "sample": sample}
    if pg:
        pg.barrier()
        pg.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


# ------------------------------------ the smaller configurations (--workload)
# The base and big models' shapes ("Attention Is All You Need", section 3.2.2
# and Table 3): the fp32 tiny case, the encoder's attention (core and with its
# projections), the decoder's causal self-attention and the big model's
# cross-attention (core and with projections).
CONFIG_WORKLOADS = {
    "tiny_f32": "tiny_f32",
    "enc_base": "enc_mha_base",
    "enc_mha_base": "enc_mha_base",
    "dec_causal_base": "dec_causal_base",
    "cross_big": "cross_big",
    "cross_mha_big": "cross_big",
}
ROTATE_BYTES = 256 << 20   # input sets rotate over at least this many bytes (L2: 129 MB)


def sdpa_bytes(w) -> int:
    """Algorithmic HBM bytes of one attention pass: Q, K, V read once, O written once."""
    es = 4 if w.dtype == "f32" else 2
    return es * w.b * w.h * (w.n_q * w.d_k + w.n_k * w.d_k + w.n_k * w.d_v + w.n_q * w.d_v)


def mha_flops(w) -> float:
    """Multi-head forward FLOP: the Q, K, V and W^O products plus the attention."""
    dm = w.d_model
    proj = 2.0 * w.b * (w.n_q * dm * w.h * w.d_k + w.n_k * dm * w.h * (w.d_k + w.d_v)
                        + w.n_q * w.h * w.d_v * dm)
    return proj + metric_flops(w)


def run_config(args, world, rank, local):
    """One of the smaller configurations, through the same JSON contract.  Each
    step reads a different set of inputs, and the sets together exceed L2, so
    no step finds its inputs cached by an earlier one."""
    import torch
    import transformer_scaled_dot_02_gb300 as sd

    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist
    sd.load_library()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    cur = [stream.cuda_stream]   # the stream the calls go to (the capture stream while capturing)
    kind = args.workload
    w = synthetic.WORKLOADS[CONFIG_WORKLOADS[kind]]
    peaks, peak_src = load_peaks()
    mha = "_mha_" in kind
    f32 = w.dtype == "f32"
    tdt = torch.float32 if f32 else torch.bfloat16

    if mha:
        xq, xkv, wq, wk, wv, wo, lens = synthetic.mha_inputs(w)
        self_attn = xkv is xq
        per_set = (xq.size + (0 if self_attn else xkv.size) + w.b * w.n_q * w.d_model) * 2
        sets = max(2, -(-ROTATE_BYTES // per_set))
        hx = [_pinned(xq, tdt)] + ([] if self_attn else [_pinned(xkv, tdt)])
        xs = [torch.empty((sets,) + tuple(t.shape), dtype=tdt, device=dev) for t in hx]
        for x, h in zip(xs, hx):
            x[:] = h.to(dev)
        weights = [torch.from_numpy(a).to(tdt).to(dev) for a in (wq, wk, wv, wo)]
        ys = torch.empty((sets, w.b, w.n_q, w.d_model), dtype=tdt, device=dev)
        ld = None if lens is None else torch.from_numpy(lens).to(dev)
        ld_ptr = None if ld is None else ld.data_ptr()
        ws_bytes = sd.mha_workspace_size(w.b, w.n_q, w.n_k, w.h, w.d_k, w.d_v)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        w_ptrs = [t.data_ptr() for t in weights]
        # device addresses of every set, taken once: the timed loop makes no tensors
        ptrs = [(xs[0][i].data_ptr(), xs[0 if self_attn else 1][i].data_ptr(), ys[i].data_ptr())
                for i in range(sets)]
        counter = [0]

        def call(i):
            xq_p, xkv_p, y_p = ptrs[i]
            sd.mha_forward(xq_p, xkv_p, *w_ptrs, y_p, ws.data_ptr(), ws_bytes, w.b, w.n_q, w.n_k,
                           w.d_model, w.h, w.d_k, w.d_v, w.mask_kind, ld_ptr, 0.0, cur[0])

        def step():
            i = counter[0] % sets
            counter[0] += 1
            call(i)

        hy = torch.empty(ys.shape[1:], dtype=tdt).pin_memory()
        e2e_x = [x[0] for x in xs]

        def e2e_step():
            for dst, src in zip(e2e_x, hx):
                dst.copy_(src, non_blocking=True)
            call(0)
            hy.copy_(ys[0], non_blocking=True)

        h2d = sum(t.numel() * t.element_size() for t in hx)
        d2h = hy.numel() * hy.element_size()
        work, unit, launches = mha_flops(w), "TFLOP/s", 3
        metric = "multi-head attention fwd TFLOP/s (Q/K/V projections, attention, W^O) (1 GPU)"
        kernel = "gemm_bf16_tc (Q, K, V) + sdpa_fwd_one_tile + gemm_bf16_tc (W^O): one mha_forward"
        bound, peak = "tensor", float(peaks["bf16_tflops"])
        rot = "X and Y rotate over %d sets (%d MB); weights and workspace stay resident" % (
            sets, sets * per_set >> 20)
        desc = {"enc_mha_base": "base-model encoder multi-head self-attention: X [32,128,512], "
                                "h8 d64, key padding 64..128",
                "cross_mha_big": "big-model multi-head cross-attention: X_dec [32,256,1024], "
                                 "X_enc [32,384,1024], h16 d64, key padding 192..384"}[kind]
        sample_b = min(w.b, args.cpu_rows or (4 if w.d_model <= 512 else 2))

        def oracle_sample():
            import oracle
            threads = oracle.default_threads()
            rows = np.arange(sample_b * w.n_q, dtype=np.int64)
            t = time.perf_counter()
            oracle.mha(xq, xkv, wq, wk, wv, wo, w.h, w.d_k, w.d_v, w.mask_kind, lens, rows=rows,
                       threads=threads)
            dt = time.perf_counter() - t
            return (mha_flops(w) * sample_b / w.b / dt / 1e12, threads,
                    "every output row of the first %d of the %d batch entries (fp64 C oracle, %.1f s)"
                    % (sample_b, w.b, dt))
    else:
        q, k, v, lens = synthetic.sdpa_inputs(w)
        masks = [w.mask_kind] if not f32 else [synthetic.MASK_NONE, synthetic.MASK_CAUSAL]
        per_set = sdpa_bytes(w)
        step_bytes = per_set * len(masks)   # each call reads Q, K, V and writes O
        sets = max(2, -(-ROTATE_BYTES // per_set))
        hq, hk, hv = _pinned(q, tdt), _pinned(k, tdt), _pinned(v, tdt)
        qs, ks, vs = (torch.empty((sets,) + tuple(h.shape), dtype=tdt, device=dev)
                      for h in (hq, hk, hv))
        for x, h in ((qs, hq), (ks, hk), (vs, hv)):
            x[:] = h.to(dev)
        os_ = torch.empty((sets, w.b, w.h, w.n_q, w.d_v), dtype=tdt, device=dev)
        ld = None if lens is None else torch.from_numpy(lens).to(dev)
        ld_ptr = None if ld is None else ld.data_ptr()
        fwd = sd.sdpa_forward_f32 if f32 else sd.sdpa_forward
        # device addresses of every set, taken once: the timed loop makes no tensors
        ptrs = [(qs[i].data_ptr(), ks[i].data_ptr(), vs[i].data_ptr(), os_[i].data_ptr())
                for i in range(sets)]
        counter = [0]

        def call(i):
            for m in masks:
                fwd(*ptrs[i], w.b, w.h, w.n_q, w.n_k, w.d_k, w.d_v, m, ld_ptr, 0.0, cur[0])

        def step():
            i = counter[0] % sets
            counter[0] += 1
            call(i)

        ho = torch.empty(os_.shape[1:], dtype=tdt).pin_memory()

        def e2e_step():
            for dst, src in ((qs[0], hq), (ks[0], hk), (vs[0], hv)):
                dst.copy_(src, non_blocking=True)
            call(0)
            ho.copy_(os_[0], non_blocking=True)

        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
        d2h = ho.numel() * ho.element_size()
        import dataclasses
        work = sum(metric_flops(dataclasses.replace(w, mask_kind=m)) for m in masks)
        unit, launches = "TFLOP/s", len(masks)
        metric = METRIC if not f32 else "attention fwd TFLOP/s, fp32 (1 GPU)"
        kernel = ("sdpa_fwd_f32_simt (unmasked and causal)" if f32 else
                  "sdpa_fwd_one_tile<64, %d>" % (32 if kind == "cross_big" else 64))
        bound, peak = "hbm", float(peaks["hbm_gbs"])
        rot = "Q, K, V, O rotate over %d sets (%d MB)" % (sets, sets * per_set >> 20)
        desc = {"tiny_f32": "tiny fp32 attention b1 h1 n16 d64, unmasked and causal (two calls)",
                "enc_base": "base-model encoder attention core b32 h8 n128 d64 bf16, key padding "
                            "64..128",
                "dec_causal_base": "base-model decoder causal self-attention b16 h8 n512 d64 bf16",
                "cross_big": "big-model cross-attention core b32 h16 n_q256 n_k384 d64 bf16, key "
                             "padding 192..384"}[kind]
        n_rows = w.b * w.h * w.n_q

        def oracle_sample():
            import oracle
            threads = oracle.default_threads()
            reps = max(1, args.cpu_rows or (2000 if f32 else 1))
            t = time.perf_counter()
            for _ in range(reps):
                for m in masks:
                    oracle.sdpa(q, k, v, m, lens, threads=threads)
            dt = time.perf_counter() - t
            return (work * reps / dt / 1e12, threads,
                    "%severy one of the %d query rows of the workload (fp64 C oracle, %.1f s)"
                    % ("%d passes over " % reps if reps > 1 else "", n_rows, dt))

    # Eager: one C-ABI call per step from Python, an event pair around each.
    eager_ms, eager_launch_ms, _ = _time_steps(step, args, stream, pg, dev, local)
    # Timed: the same K steps captured once into a CUDA graph and replayed
    # between two events, so host launch gaps do not enter the device time.
    total_ms, clocks = _time_graph(step, args, pg, dev, local, cur)
    launch_ms = [total_ms / args.steps]
    e2e_ms, e2e_steps = _time_e2e(e2e_step, args, stream, pg, dev)
    value = world * work * args.steps / (total_ms * 1e-3) / 1e12
    mean_ms = float(np.mean(launch_ms))
    roof = {"bound": bound, "peak": peak, "kernel": kernel,
            "launch_ms_mean": round(mean_ms, 5), "launch_ms_min": round(float(np.min(launch_ms)), 5)}
    if bound == "hbm":
        gbs = step_bytes / (mean_ms * 1e-3) / 1e9
        roof.update({"achieved": round(gbs, 2), "unit": "GB/s", "frac": round(gbs / peak, 4),
                     "peak_source": "%s hbm_gbs" % peak_src,
                     "algorithmic_bytes": step_bytes,
                     "tflops": round(work / (mean_ms * 1e-3) / 1e12, 3),
                     "traffic": recorded_traffic(kind)})
    else:
        tf = work / (mean_ms * 1e-3) / 1e12
        roof.update({"achieved": round(tf, 2), "unit": "TFLOP/s", "frac": round(tf / peak, 4),
                     "peak_source": "%s bf16_tflops (burst)" % peak_src, "traffic": None})
    line = {
        "metric": metric, "value": round(value, 4), "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if f32 else "bf16", "data": "synthetic",
        "config": {"workload": desc, "b": w.b, "h": w.h, "n_q": w.n_q, "n_k": w.n_k,
                   "d_k": w.d_k, "d_v": w.d_v, "d_model": w.d_model if mha else None,
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "inputs larger than L2: " + rot},
        "roofline": roof,
        "e2e": {"value": round(world * work * e2e_steps / (e2e_ms * 1e-3) / 1e12, 4), "unit": unit,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "steps": e2e_steps, "path": "pinned host inputs copied in, the C-ABI call, "
                                            "the output copied back, one stream"},
        "gpu_launches": args.steps * launches,
        "timing": "K steps captured in one CUDA graph, replayed between two events; "
                  "eager (one call per step from Python): %.5f ms per step, %.5f ms per "
                  "step between its own events" % (eager_ms / args.steps,
                                                    float(np.mean(eager_launch_ms))),
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        val, threads, sample = oracle_sample()
        line["cpu_baseline"] = {"value": val, "unit": unit, "cores": threads, "kind": "oracle",
                                "cpu": cpu_model(), "sample": sample}
    if pg:
        pg.barrier()
        pg.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


# ----------------------------------------------------------- oracle timing
def _sample_rows(w, n_rows, seed):
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(w.b * w.h * w.n_q, size=n_rows, replace=False)).astype(np.int64)


def _rows_flops(w, rows):
    i = rows % w.n_q
    visible = (i + 1) if w.causal else np.full_like(i, w.n_k)
    return float(np.sum(4.0 * visible * w.d_k))


def cpu_model() -> str:
    """The host CPU's model name (x86 "model name"; on Arm, implementer/part
    codes when no name is given), for the oracle baseline's record."""
    import platform
    try:
        info = open("/proc/cpuinfo").read().splitlines()
    except OSError:
        return platform.machine()
    fields = {}
    for l in info:
        if ":" in l:
            key, val = (x.strip() for x in l.split(":", 1))
            fields.setdefault(key, val)
    if "model name" in fields:
        return fields["model name"]
    if "CPU part" in fields:
        # Arm Ltd (implementer 0x41) core part numbers
        arm_parts = {"0xd0c": "Neoverse-N1", "0xd40": "Neoverse-V1", "0xd49": "Neoverse-N2",
                     "0xd4f": "Neoverse-V2", "0xd84": "Neoverse-V3"}
        impl, part = fields.get("CPU implementer", "?"), fields["CPU part"]
        name = arm_parts.get(part) if impl == "0x41" else None
        return "%s %s (implementer %s, part %s)" % (platform.machine(), name or "core", impl, part)
    return platform.machine()


def oracle_baseline(w, q, k, v, n_rows):
    import oracle
    threads = oracle.default_threads()
    rows = _sample_rows(w, n_rows, 99)
    t = time.perf_counter()
    oracle.sdpa(q, k, v, w.mask_kind, None, rows=rows, threads=threads)
    dt = time.perf_counter() - t
    value = _rows_flops(w, rows) / dt / 1e12
    return {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": "%d query rows drawn uniformly from the %d rows of the workload "
                      "(fp64 C oracle, %.1f s)" % (len(rows), w.b * w.h * w.n_q, dt),
            "cpu": cpu_model()}


def run_reference(args, world, rank, local):
    """The reference arm: the CPU oracle as it stands, on the host cores."""
    if rank != 0:
        return
    import oracle
    w = synthetic.WORKLOADS[WORKLOAD]
    q, k, v, _ = synthetic.sdpa_inputs(w)
    threads = oracle.default_threads()
    rows_per_step = args.ref_rows
    for i in range(args.warmup):
        oracle.sdpa(q, k, v, w.mask_kind, None, rows=_sample_rows(w, rows_per_step, 1000 + i),
                    threads=threads)
    flops = 0.0
    t = time.perf_counter()
    for i in range(args.steps):
        rows = _sample_rows(w, rows_per_step, i)
        oracle.sdpa(q, k, v, w.mask_kind, None, rows=rows, threads=threads)
        flops += _rows_flops(w, rows)
    dt = time.perf_counter() - t
    value = flops / dt / 1e12
    sample = ("each step: %d query rows drawn uniformly from the %d rows of the workload "
              "(fp64 C oracle, %d threads)" % (rows_per_step, w.b * w.h * w.n_q, threads))
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": "long-sequence causal self-attention b4 h16 n8192 d128 bf16",
                   "b": w.b, "h": w.h, "n_q": w.n_q, "n_k": w.n_k, "d_k": w.d_k, "d_v": w.d_v,
                   "mask": "causal"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "cpu": cpu_model(),
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=("long_causal",) + ROW_WORKLOADS + tuple(CONFIG_WORKLOADS),
                    default="long_causal",
                    help="the headline workload, one of the widened rows, or one of the smaller "
                         "configurations")
    ap.add_argument("--cpu-rows", type=int, default=None,
                    help="size of the oracle's timed CPU sample (query rows; the backward: "
                         "a causal prefix length)")
    ap.add_argument("--ref-rows", type=int, default=2048,
                    help="query rows per step of the reference (oracle) arm")
    ap.add_argument("--decode-queries", type=int, default=1,
                    help="new queries per sequence and head of the decode workload (1 to 8)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    if args.impl == "reference" and args.workload != "long_causal":
        ap.error("the reference arm runs the default workload")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank, local)
    elif args.workload in CONFIG_WORKLOADS:
        run_config(args, world, rank, local)
    elif args.workload != "long_causal":
        run_row(args, world, rank, local)
    else:
        if args.cpu_rows is None:
            args.cpu_rows = 32768
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
