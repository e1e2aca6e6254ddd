#!/usr/bin/env python3
"""Benchmark of the batched-prefill projection over block-quantized weights.

One step = one transformer layer's seven projections (q, k, v, o, gate, up,
down) over one prompt, with the dequantization fused into each GEMM.  The
default workload is the Qwen3-8B-shaped layer with Q2_K weights (Q6_K down
projection) and an 8,192-token prompt; inputs are seeded synthetic tensors.
The line printed reports whole-job TFLOP/s (and tok/s, % of the dense fp16
tensor peak), the dominant kernel against its roofline, an end-to-end figure
through the C ABI with host buffers, the CPU oracle timed on the host cores,
and (rank 0 only) the remaining rows of the path: standalone dequant GB/s,
the Qwen3-1.7B-shaped layer and the 31,258-token chunked prefill in fused and
cached-f16 modes.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl qp|reference]

With N > 1 it runs under torch.distributed (one process per GPU): every rank
processes its own prompt with the same weights (weak scaling, no collective
on the data path); the step time is the max over ranks.
"""
import argparse
import ctypes
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402
from synth import workloads  # noqa: E402

METRIC = "fused dequant-GEMM prefill TFLOP/s & tok/s (% dense-FP16 peak); dequant HBM GB/s"
DEFAULT_WORKLOAD = "qwen3_8b_q2k_q6k_t8192"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic of the dominant kernel per launch (dram__bytes_read.sum +
# dram__bytes_write.sum), from one ncu capture of the kernel source whose hash
# is recorded; reported only while the source is unchanged.
NCU_TRAFFIC = {"source_sha": "8a84ee6a42054f95", "bytes_per_launch": 1559492864,
               "what": "fused Q2_K launch over q,k,v,o,gate,up on CTA pairs, T=8192 (read 469.54 MB + write "
                       "1089.96 MB); algorithmic 1321.9 MB (W 46.8 + X 134.2 + Y 1140.9): X_h is read again by "
                       "each projection that shares it, and part of Y is still in L2 at kernel end"}
KERNEL_SOURCES = ["block_quantized_weight_qp_gb300/csrc/qgemm.cu",
                  "block_quantized_weight_qp_gb300/csrc/qp_ptx.cuh",
                  "block_quantized_weight_qp_gb300/csrc/qp_sync.cuh",
                  "block_quantized_weight_qp_gb300/csrc/qp_decode.cuh"]


# ------------------------------------------------------------ distributed --

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value, world, device=None):
    """Max of a float over all ranks (the step time the job reports)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value, world, device=None):
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def job_throughput(units_per_rank, world, max_ms):
    """Units all ranks processed / the slowest rank's time (per second)."""
    return units_per_rank * world / (max_ms / 1e3)


# ------------------------------------------------------------------ peaks --

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_sha():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# ----------------------------------------------------------------- clocks --

class ClockSampler:
    """Samples SM clock, power and clock-event reasons through NVML (ctypes)
    every few milliseconds while running.  Reads only."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x2: "applications_clocks_setting"}

    def __init__(self, index, period_s=0.005):
        self.samples = []
        self.period = period_s
        self.ok = False
        self.max_mhz = None
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.handle = ctypes.c_void_p()
            if self.nvml.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(self.handle)) != 0:
                return
            m = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(m)) == 0:
                self.max_mhz = m.value
            self.ok = True
        except OSError:
            pass

    def _sample(self):
        c, r = ctypes.c_uint(), ctypes.c_ulonglong()
        if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(c)) != 0:
            return
        self.nvml.nvmlDeviceGetCurrentClocksEventReasons(self.handle, ctypes.byref(r))
        self.samples.append((c.value, r.value))

    def _run(self):
        while not self._stop.is_set():
            self._sample()
            time.sleep(self.period)

    def __enter__(self):
        if self.ok:
            self._stop = threading.Event()
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *exc):
        if self.ok:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0}
        mhz = [c for c, _ in self.samples]
        bits = 0
        for _, r in self.samples:
            bits |= r
        reasons = sorted(n for b, n in self.REASONS.items() if bits & b)
        return {"sm_mhz": float(statistics.median(mhz)), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(self.samples)}


# ------------------------------------------------------------- GPU arm ----

class Layer:
    """Weights and inputs of one workload on the device."""

    def __init__(self, wl, rank, device, need_f16=False, only=None):
        import torch
        self.wl = wl
        self.only = only
        self.T = wl["T"]
        dims = workloads.input_dims(wl)
        self.X_host = {k: synth.normal_f16((self.T, dims[k]), seed=wl["seed"] + 7919 * rank, tensor=1000 + i)
                       for i, k in enumerate(("h", "o", "f"))}
        self.X = {k: torch.from_numpy(v).to(device) for k, v in self.X_host.items()}
        self.W_host = [synth.blocks(qt, out_f, in_f, seed=wl["seed"], tensor=i)
                       for i, (_, out_f, in_f, _, qt) in enumerate(wl["projections"])]
        self.W = [torch.from_numpy(w).to(device) for w in self.W_host]
        self.Y = [torch.empty((self.T, out_f), dtype=torch.float32, device=device)
                  for (_, out_f, _, _, _) in wl["projections"]]
        self.W16 = None
        if need_f16:
            import block_quantized_weight_qp_gb300 as qp
            self.W16 = []
            for w, (_, out_f, in_f, _, qt) in zip(self.W, wl["projections"]):
                h = torch.empty((out_f, in_f), dtype=torch.float16, device=device)
                qp.qp_dequant_f16(qt, w, out_f, in_f, h)
                self.W16.append(h)

    def flops(self, T=None, idx=None):
        T = self.T if T is None else T
        return sum(2 * T * out_f * in_f for i, (name, out_f, in_f, _, _) in enumerate(self.wl["projections"])
                   if (not self.only or name == self.only) and (idx is None or i in idx))

    def launches(self, grouped=True):
        """The step's launches as (block type, [projection indices]): with
        grouping, each run of consecutive projections of one type is one
        qp_prefill_gemm_group launch; without, one launch per projection."""
        if grouped and not self.only:
            return workloads.type_runs(self.wl["projections"])
        return [(qt, [i]) for i, (name, _, _, _, qt) in enumerate(self.wl["projections"])
                if not self.only or name == self.only]


def run_layer(qp, layer, stream, events=None, mode="fused", chunk=None, X=None, Y=None, grouped=True):
    """Launch the seven projections (or the one named by layer.only) through
    the grouped entry points; events[k] = (start, end) recorded around
    launch k of layer.launches(grouped) when given."""
    for k, (qt, idx) in enumerate(layer.launches(grouped)):
        descs = []
        for i in idx:
            _, out_f, in_f, src, _ = layer.wl["projections"][i]
            w = layer.W[i] if mode == "fused" else layer.W16[i]
            descs.append((w, out_f, in_f, layer.X[src] if X is None else X[src],
                          layer.Y[i] if Y is None else Y[i]))
        ty = qt if mode == "fused" else 0
        if events is not None:
            events[k][0].record(stream)
        if chunk:
            qp.qp_prefill_chunked_group(ty, descs, layer.T, chunk, stream)
        else:
            qp.qp_prefill_gemm_group(ty, descs, layer.T, stream)
        if events is not None:
            events[k][1].record(stream)


def time_layer(qp, layer, stream, steps, warmup, mode="fused", chunk=None):
    """Mean ms per layer pass over `steps` passes (one timed region)."""
    import torch
    for _ in range(warmup):
        run_layer(qp, layer, stream, mode=mode, chunk=chunk)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        run_layer(qp, layer, stream, mode=mode, chunk=chunk)
    e1.record(stream)
    torch.cuda.synchronize()
    qp.qp_check(stream)
    return e0.elapsed_time(e1) / steps


def bench_dequant(qp, stream, device, launches=64, only=None):
    """Standalone dequant throughput: GB/s of quantized bytes read + output
    bytes written.  `launches` launches run back to back over rotating
    input/output buffer sets whose total is at least 4x the L2 size, so every
    launch finds its data in HBM.  They are captured once in a CUDA graph and
    the replay is timed with one CUDA-event pair (`gbs`, `us`: the device
    time per launch without the host's launch overhead); the same launches
    made eagerly from Python are timed beside it (`eager_gbs`).  Reference:
    a device-to-device copy moving the same bytes (half read, half written)
    over the same rotating buffers, also replayed from a graph."""
    import torch
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    cases = [("Q4_K", qp.Q4_K, 4096, 4096, 12), ("Q8_0", qp.Q8_0, 4096, 4096, 13),
             ("Q2_K", qp.Q2_K, 4096, 4096, 14), ("Q6_K", qp.Q6_K, 4096, 12288, 15),
             ("Q5_K", qp.Q5_K, 4096, 4096, 16), ("F16", qp.F16, 4096, 4096, 17)]
    side = torch.cuda.Stream(device)

    def timed(fn, graph):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if graph is None:
            for i in range(launches):
                fn(i, stream)
        else:
            graph.replay()
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / launches

    def captured(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                for i in range(launches):
                    fn(i, side)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        return g

    out = {}
    for name, qt, rows, cols, tid in cases:
        if only and not any(o.startswith(name) for o in only):
            continue
        w0 = torch.from_numpy(synth.blocks(qt, rows, cols, seed=1, tensor=tid)).to(device)
        for f16 in (False, True):
            if only and "%s_%s" % (name, "f16" if f16 else "f32") not in only:
                continue
            esize = 2 if f16 else 4
            nbytes = w0.numel() + rows * cols * esize
            nsets = max(2, -(-4 * l2 // nbytes))
            ws = [w0.clone() for _ in range(nsets)]
            ys = [torch.empty((rows, cols), dtype=torch.float16 if f16 else torch.float32, device=device)
                  for _ in range(nsets)]
            deq = qp.qp_dequant_f16 if f16 else qp.qp_dequant_f32

            def fn(i, st):
                deq(qt, ws[i % nsets], rows, cols, ys[i % nsets], st)

            for i in range(nsets):
                fn(i, stream)
            ms_eager = timed(fn, None)
            g = captured(fn)
            ms = timed(fn, g)
            del g
            srcs = [y.view(torch.uint8).view(-1)[: nbytes // 2] for y in ys]
            dsts = [torch.empty(nbytes // 2, dtype=torch.uint8, device=device) for _ in range(nsets)]

            def cp(i, st):
                with torch.cuda.stream(st):
                    dsts[i % nsets].copy_(srcs[(i + 1) % nsets])

            for i in range(nsets):
                cp(i, stream)
            gc = captured(cp)
            copy_ms = timed(cp, gc)
            del gc
            out["%s_%dx%d_%s" % (name, rows, cols, "f16" if f16 else "f32")] = {
                "gbs": round(nbytes / (ms / 1e3) / 1e9, 1), "us": round(ms * 1e3, 2), "bytes": nbytes,
                "eager_gbs": round(nbytes / (ms_eager / 1e3) / 1e9, 1), "buffer_sets": nsets,
                "same_bytes_copy_gbs": round(nbytes / (copy_ms / 1e3) / 1e9, 1)}
            del ws, ys, srcs, dsts
    qp.qp_check(stream)
    return out


def bench_gemv(qp, layer, stream, device, peaks, steps=20, ts=(1, 8)):
    """The decode GEMV over the layer's seven weights for T = 1 and 8 token
    rows, as one grouped launch per block type (qp_decode_gemv_group; for the
    Q2_K layer the six Q2_K projections, then the Q6_K down projection),
    captured in a CUDA graph as a decode loop would run it.  Also timed: the
    same launches made eagerly, and the seven projections launched one at a
    time (graph).  The weights (88 MB for the Q2_K layer, 108.5 and 132.6 MB for
    the Q4_K and Q5_K ones) fit in L2 or nearly, so before every timed step a 256 MB
    buffer is written (outside the timed region: events bracket the GEMV
    launches of each step only).  GB/s counts the weight bytes plus the X and
    Y bytes of a step.

    Also timed, as a decode loop runs layer after layer: STACK copies of the
    layer (each its own copy of the weights, so four layers hold 353 MB for
    the Q2_K one, more than L2) launched back to back in one graph; reported
    per layer.  There each launch's ring prefill overlaps the previous
    launch's tail, which a single layer timed alone cannot show.

    L2 flush: the 256 MB write evicts the weights, and the following read of
    another 256 MB buffer leaves the L2 holding only clean lines, as it does
    when a decode step streams a layer's weights after the previous layer's
    (a flush left dirty would make the timed GEMV pay for writing 129 MB of
    someone else's data back to HBM)."""
    import torch
    wl = layer.wl
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    flush_rd = torch.ones(64 << 20, dtype=torch.int32, device=device)

    def flush_l2():
        flush.fill_(1)
        flush_rd.sum()
    wbytes = sum(w.numel() for w in layer.W)
    out = {}
    for T in ts:
        dims = workloads.input_dims(wl)
        X = {k: torch.from_numpy(synth.normal_f16((T, d), seed=wl["seed"], tensor=3000 + i)).to(device)
             for i, (k, d) in enumerate(dims.items())}
        Y = [torch.empty((T, o), dtype=torch.float32, device=device) for _, o, _, _, _ in wl["projections"]]

        def grouped(st):
            for qt, idx in layer.launches(True):
                descs = [(layer.W[i], wl["projections"][i][1], wl["projections"][i][2],
                          X[wl["projections"][i][3]], Y[i]) for i in idx]
                qp.qp_decode_gemv_group(qt, descs, T, st)

        def single(st):
            for i, (_, o, n, src, qt) in enumerate(wl["projections"]):
                qp.qp_decode_gemv(qt, layer.W[i], o, n, X[src], T, Y[i], st)

        grouped(stream)
        single(stream)
        torch.cuda.synchronize()
        cap = torch.cuda.Stream(device)
        graphs = {}
        for name, fn in (("grouped", grouped), ("single", single)):
            graphs[name] = torch.cuda.CUDAGraph()
            with torch.cuda.stream(cap):
                with torch.cuda.graph(graphs[name], stream=cap):
                    fn(cap)
        torch.cuda.synchronize()
        # each grouped launch on its own (eager, L2 flushed before each step)
        per_launch = {}
        nl = len(layer.launches(True))
        evl = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nl)]
               for _ in range(steps)]
        for _ in range(3):                       # untimed warm-up
            flush_l2()
            grouped(stream)
        for s_ev in evl:
            flush_l2()
            for k, (qt, idx) in enumerate(layer.launches(True)):
                descs = [(layer.W[i], wl["projections"][i][1], wl["projections"][i][2],
                          X[wl["projections"][i][3]], Y[i]) for i in idx]
                s_ev[k][0].record(stream)
                qp.qp_decode_gemv_group(qt, descs, T, stream)
                s_ev[k][1].record(stream)
        torch.cuda.synchronize()
        for k, (qt, idx) in enumerate(layer.launches(True)):
            wb = sum(layer.W[i].numel() for i in idx)
            us = statistics.mean(e[k][0].elapsed_time(e[k][1]) for e in evl) * 1e3
            per_launch["%s:%s" % (synth.NAMES[qt], ",".join(wl["projections"][i][0] for i in idx))] = {
                "us": round(us, 2), "weight_bytes": wb, "weight_gbs": round(wb / (us / 1e6) / 1e9, 1)}
        # STACK layers back to back, each with its own copy of the weights and Y
        STACK = 4
        Wst = [layer.W] + [[w.clone() for w in layer.W] for _ in range(STACK - 1)]
        Yst = [Y] + [[torch.empty_like(y) for y in Y] for _ in range(STACK - 1)]

        def stacked(st):
            for li in range(STACK):
                for qt, idx in layer.launches(True):
                    descs = [(Wst[li][i], wl["projections"][i][1], wl["projections"][i][2],
                              X[wl["projections"][i][3]], Yst[li][i]) for i in idx]
                    qp.qp_decode_gemv_group(qt, descs, T, st)
        stacked(stream)
        torch.cuda.synchronize()
        graphs["stacked"] = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(graphs["stacked"], stream=cap):
                stacked(cap)
        torch.cuda.synchronize()
        res = {}
        for how in ("grouped", "single", "eager", "stacked"):
            for _ in range(3):                   # untimed warm-up of this way of launching
                flush_l2()
                if how == "eager":
                    grouped(stream)
                else:
                    graphs[how].replay()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
            for e0, e1 in ev:
                flush_l2()
                e0.record(stream)
                if how == "eager":
                    grouped(stream)
                else:
                    graphs[how].replay()
                e1.record(stream)
            torch.cuda.synchronize()
            res[how] = statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev)
        qp.qp_check(stream)
        del graphs, Wst, Yst
        ms = res["grouped"]
        nbytes = wbytes + sum(x.numel() * 2 for x in X.values()) + sum(y.numel() * 4 for y in Y)
        gbs = nbytes / (ms / 1e3) / 1e9
        ms_l = res["stacked"] / STACK
        gbs_l = nbytes / (ms_l / 1e3) / 1e9
        out["T%d" % T] = {"ms": round(ms, 4), "bytes": nbytes, "gbs": round(gbs, 1),
                          "pct_hbm": round(100.0 * gbs / peaks["hbm_gbs"], 1),
                          "tok_per_s": round(T / (ms / 1e3), 1), "eager_ms": round(res["eager"], 4),
                          "one_launch_per_projection_ms": round(res["single"], 4), "per_launch_eager": per_launch,
                          "layers_back_to_back": {"layers": STACK, "ms_per_layer": round(ms_l, 4),
                                                  "gbs": round(gbs_l, 1),
                                                  "pct_hbm": round(100.0 * gbs_l / peaks["hbm_gbs"], 1)}}
    del flush, flush_rd
    return out


def cpu_oracle_sample(wl, seconds=10.0, rows_max=4096):
    """The CPU oracle as it stands on a bounded sample of the workload: it
    dequantizes all seven weights to f32 and computes the fp64 projection for
    a sample of token rows; the time is extrapolated linearly in rows to the
    full prompt.  Returns the cpu_baseline object."""
    import oracle
    t0 = time.perf_counter()
    Ws = [oracle.dequant_f32(qt, synth.blocks(qt, out_f, in_f, seed=wl["seed"], tensor=i), out_f, in_f)
          for i, (_, out_f, in_f, _, qt) in enumerate(wl["projections"])]
    t_deq = time.perf_counter() - t0
    dims = workloads.input_dims(wl)
    X = {k: synth.normal_f16((64, dims[k]), seed=wl["seed"], tensor=1000 + i) for i, k in enumerate(("h", "o", "f"))}

    def gemm_rows(n):
        rows = np.arange(n, dtype=np.int64)
        t = time.perf_counter()
        for W, (_, _, _, src, _) in zip(Ws, wl["projections"]):
            Xs = X[src] if n <= 64 else np.resize(X[src], (n, X[src].shape[1]))
            oracle.gemm_f64(Xs, W, rows)
        return time.perf_counter() - t

    probe = 4
    t_probe = gemm_rows(probe)
    n = int(min(rows_max, max(probe, (seconds - t_deq) / max(t_probe / probe, 1e-9))))
    t_rows = gemm_rows(n) if n > probe else t_probe
    per_row = t_rows / n
    T = wl["T"]
    t_full = t_deq + per_row * T
    flops = workloads.flops(wl)
    return {"value": round(flops / t_full / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": "scalar-C oracle: f32 dequant of all 7 weights (%.2f s) + fp64 GEMM of %d token rows "
                      "(%.2f s), extrapolated linearly to T=%d" % (t_deq, n, t_rows, T)}


def cpu_dequant_rows(seconds_per_case=0.2):
    """The CPU oracle's dequant throughput per block type (the same weights as
    the GPU dequant rows), on one core and on every core of the process's
    affinity mask: GB/s of quantized bytes read + output bytes written."""
    import oracle
    cores = len(os.sched_getaffinity(0))
    cases = [("Q4_K", synth.Q4_K, 4096, 4096, 12), ("Q8_0", synth.Q8_0, 4096, 4096, 13),
             ("Q2_K", synth.Q2_K, 4096, 4096, 14), ("Q6_K", synth.Q6_K, 4096, 12288, 15),
             ("Q5_K", synth.Q5_K, 4096, 4096, 16), ("F16", synth.F16, 4096, 4096, 17)]
    out = {"cores": cores}
    try:
        for name, qt, rows, cols, tid in cases:
            w = synth.blocks(qt, rows, cols, seed=1, tensor=tid)
            for f16 in (False, True):
                fn = oracle.dequant_f16 if f16 else oracle.dequant_f32
                nbytes = w.size + rows * cols * (2 if f16 else 4)
                res = {}
                for label, n in (("one_core", 1), ("all_cores", cores)):
                    oracle.set_num_threads(n)
                    reps, t0 = 0, time.perf_counter()
                    while True:
                        fn(qt, w, rows, cols)
                        reps += 1
                        dt = time.perf_counter() - t0
                        if dt >= seconds_per_case:
                            break
                    res[label + "_gbs"] = round(nbytes * reps / dt / 1e9, 3)
                out["%s_%dx%d_%s" % (name, rows, cols, "f16" if f16 else "f32")] = res
    finally:
        oracle.set_num_threads(cores)
    return out


def measure_matmul_peaks(device, n=8192, reps=10):
    """Dense tensor-core reference: torch.matmul of two n x n matrices in fp16
    and in bf16, best of `reps` (burst), 2 n^3 flops."""
    import torch
    out = {}
    for name, dt in (("fp16", torch.float16), ("bf16", torch.bfloat16)):
        a = torch.randn((n, n), device=device).to(dt)
        b = torch.randn((n, n), device=device).to(dt)
        for _ in range(3):
            torch.matmul(a, b)
        best = None
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch.matmul(a, b)
            e1.record()
            e1.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        out[name + "_tflops"] = round(2.0 * n ** 3 / (best / 1e3) / 1e12, 1)
        del a, b
    return out


def main_dequant_only(args):
    """Standalone dequant rows only (profiling runs)."""
    import torch

    import block_quantized_weight_qp_gb300 as qp
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    qp.load()
    stream = torch.cuda.current_stream(device)
    only = args.dequant_cases.split(",") if args.dequant_cases else None
    rows = bench_dequant(qp, stream, device, launches=args.steps, only=only)
    print(json.dumps({"dequant": rows}))


def main_gemv_only(args):
    """Decode GEMV row only (profiling runs): the workload's weights, T = 1 and 8."""
    import torch

    import block_quantized_weight_qp_gb300 as qp
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    qp.load()
    peaks, _ = load_peaks()
    stream = torch.cuda.current_stream(device)
    layer = Layer(workloads.WORKLOADS[args.workload], 0, device)
    ts = (args.gemv_t,) if args.gemv_t else (1, 8)
    print(json.dumps({"decode_gemv": bench_gemv(qp, layer, stream, device, peaks, steps=args.steps, ts=ts)}))


def main_qp(args):
    import torch

    import block_quantized_weight_qp_gb300 as qp
    if args.dequant_only:
        return main_dequant_only(args)
    if args.gemv_only:
        return main_gemv_only(args)
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    qp.load()
    qp.qp_set_gemm_cta_pairs(args.cta_pairs)
    peaks, peak_src = load_peaks()
    wl = workloads.WORKLOADS[args.workload]
    stream = torch.cuda.current_stream(device)
    layer = Layer(wl, rank, device, need_f16=args.mode == "cached", only=args.only_proj)
    T = layer.T
    flops = layer.flops()
    grouped = not args.no_group
    launches = layer.launches(grouped)
    nlaunch = len(launches)

    # ---- timed region: K steps, per-launch events on the launch stream
    for _ in range(args.warmup):
        run_layer(qp, layer, stream, mode=args.mode, grouped=grouped)
    torch.cuda.synchronize()
    qp.qp_check(stream)
    events = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in range(nlaunch)]
              for _ in range(args.steps)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    with sampler:
        e0.record(stream)
        for s in range(args.steps):
            run_layer(qp, layer, stream, events=events[s], mode=args.mode, grouped=grouped)
        e1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    qp.qp_check(stream)
    ms = e0.elapsed_time(e1) / args.steps
    max_ms = max_over_ranks(ms, world, device)
    value = job_throughput(flops, world, max_ms) / 1e12
    tok_s = job_throughput(T, world, max_ms)
    per_launch = []
    for k, (qt, idx) in enumerate(launches):
        t_ms = statistics.mean(events[s][k][0].elapsed_time(events[s][k][1]) for s in range(args.steps))
        f = layer.flops(idx=idx)
        per_launch.append({"type": synth.NAMES[qt], "projections": [wl["projections"][i][0] for i in idx],
                           "ms": round(t_ms, 4), "tflops": round(f / (t_ms / 1e3) / 1e12, 1), "flops": f})
    # dominant kernel: the launch with the most time (mean over the timed steps)
    dom_launch = max(per_launch, key=lambda d: d["ms"])
    dom = dom_launch["type"]
    achieved = dom_launch["flops"] / (dom_launch["ms"] / 1e3) / 1e12
    # breakdown by projection: the same projections launched one at a time
    per_proj = []
    single = layer.launches(grouped=False)
    ev1 = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in single]
           for _ in range(args.steps)]
    run_layer(qp, layer, stream, mode=args.mode, grouped=False)
    for s in range(args.steps):
        run_layer(qp, layer, stream, events=ev1[s], mode=args.mode, grouped=False)
    torch.cuda.synchronize()
    qp.qp_check(stream)
    for k, (qt, (i,)) in enumerate(single):
        name, out_f, in_f, _, _ = wl["projections"][i]
        t_ms = statistics.mean(ev1[s][k][0].elapsed_time(ev1[s][k][1]) for s in range(args.steps))
        per_proj.append({"proj": name, "type": synth.NAMES[qt], "out": out_f, "in": in_f, "ms": round(t_ms, 4),
                         "tflops": round(2.0 * T * out_f * in_f / (t_ms / 1e3) / 1e12, 1)})
    peak = peaks["bf16_tflops"]
    traffic = None
    if NCU_TRAFFIC["source_sha"] and NCU_TRAFFIC["source_sha"] == kernel_source_sha():
        traffic = NCU_TRAFFIC["bytes_per_launch"]
    kname = (("pair_fused_kernel", " cta_group::2 on CTA pairs", "pair_gemm_kernel") if args.cta_pairs
             else ("prefill_gemm_kernel", " on one CTA per tile", "prefill_gemm_kernel"))
    roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "traffic_what": NCU_TRAFFIC["what"] if traffic else None,
                "kernel": ("%s<%s> (fused dequant, tcgen05%s; one launch over %s)"
                           % (kname[0], dom, kname[1], ",".join(dom_launch["projections"])) if args.mode == "fused"
                           else "%s<f16 weight> (cached mode, tcgen05%s; one launch over %s)"
                           % (kname[2], kname[1], ",".join(dom_launch["projections"]))),
                "peak_source": "%s dense bf16 burst (fp16 runs at the bf16 rate)" % peak_src}

    # ---- end to end through the C ABI with host buffers
    Xh = {k: torch.from_numpy(v).pin_memory() for k, v in layer.X_host.items()}
    Yh = [torch.empty(y.shape, dtype=y.dtype, pin_memory=True) for y in layer.Y]
    h2d = sum(v.numel() * v.element_size() for v in Xh.values())
    d2h = sum(y.numel() * y.element_size() for y in Yh)

    # Every step copies its X in from pinned host memory on one copy stream
    # and reads each projection's Y back on another as soon as that
    # projection is done, so both directions overlap the GEMMs.  The host link
    # is full duplex and the read-back of Y bounds this path, so consecutive
    # steps overlap as well: the device-side X and Y are double-buffered, and
    # step i + 1's X moves in while step i's Y moves out.  Each step's copies
    # all fall inside the timed region.  Here every projection is its own
    # launch, so that its Y starts moving as soon as it is written.
    Xd2 = [layer.X] + [{k: torch.empty_like(v) for k, v in layer.X.items()}]
    Yd2 = [layer.Y] + [[torch.empty_like(y) for y in layer.Y]]
    h2d_s = torch.cuda.Stream(device)
    d2h_streams = [torch.cuda.Stream(device) for _ in range(max(1, args.d2h_streams))]
    x_free = [None, None]     # the GEMMs of the step that last read buffer set b are done
    y_free = [None, None]     # the read-back of the step that last wrote buffer set b is done
    step_no = [0]

    def e2e_step():
        bset = step_no[0] % 2
        step_no[0] += 1
        Xd, Yd = Xd2[bset], Yd2[bset]
        if x_free[bset] is not None:
            h2d_s.wait_event(x_free[bset])
        ready = {}
        with torch.cuda.stream(h2d_s):
            for k in ("h", "o", "f"):
                Xd[k].copy_(Xh[k], non_blocking=True)
                ready[k] = torch.cuda.Event()
                ready[k].record(h2d_s)
        if y_free[bset] is not None:
            stream.wait_event(y_free[bset])
        for qt, idx in layer.launches(grouped=False):
            descs = []
            for i in idx:
                _, out_f, in_f, src, _ = wl["projections"][i]
                stream.wait_event(ready[src])
                descs.append((layer.W[i], out_f, in_f, Xd[src], Yd[i]))
            qp.qp_prefill_gemm_group(qt, descs, T, stream)
            done = torch.cuda.Event()
            done.record(stream)
            # the read-back of each Y is split row-wise over the copy streams
            parts = len(d2h_streams)
            rows = -(-T // parts)
            for i in idx:
                for j, ds in enumerate(d2h_streams):
                    ds.wait_event(done)
                    with torch.cuda.stream(ds):
                        Yh[i][j * rows:(j + 1) * rows].copy_(Yd[i][j * rows:(j + 1) * rows], non_blocking=True)
        x_free[bset] = torch.cuda.Event()
        x_free[bset].record(stream)
        # one event after every copy stream's read-back of this step
        y_done = torch.cuda.Event()
        with torch.cuda.stream(d2h_streams[0]):
            for ds in d2h_streams[1:]:
                d2h_streams[0].wait_stream(ds)
            y_done.record(d2h_streams[0])
        y_free[bset] = y_done

    def e2e_drain():
        # the timed region ends when the last step's Y is on the host
        for ds in d2h_streams:
            stream.wait_stream(ds)
        stream.wait_stream(h2d_s)

    e2e = None
    if not args.no_e2e and args.mode == "fused":
        e2e_steps = max(3, min(args.steps, 10))
        for _ in range(2):
            e2e_step()
        e2e_drain()
        torch.cuda.synchronize()
        barrier(world)
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        h2d_s.wait_event(f0)
        for ds in d2h_streams:
            ds.wait_event(f0)
        for _ in range(e2e_steps):
            e2e_step()
        e2e_drain()
        f1.record(stream)
        torch.cuda.synchronize()
        qp.qp_check(stream)
        e2e_ms = max_over_ranks(f0.elapsed_time(f1) / e2e_steps, world, device)
        e2e = {"value": round(job_throughput(flops, world, e2e_ms) / 1e12, 2), "unit": "TFLOP/s",
               "d2h_streams": len(d2h_streams), "steps_overlap": "double-buffered X and Y on the device",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 3),
               "tok_per_s": round(job_throughput(T, world, e2e_ms), 1)}
    del Xh, Yh, Xd2, Yd2

    rows = None
    cpu = None
    if rank == 0 and world == 1:
        if not args.no_rows:
            rows = {"dequant": bench_dequant(qp, stream, device)}
            l17 = Layer(workloads.WORKLOADS["qwen3_1p7b_q4k_t2048"], rank, device)
            ms17 = time_layer(qp, l17, stream, max(5, args.steps), 3)
            rows["qwen3_1p7b_q4k_t2048"] = {"ms": round(ms17, 4), "tflops": round(l17.flops() / ms17 / 1e9, 1),
                                            "tok_per_s": round(l17.T / ms17 * 1e3, 1)}
            del l17
            # The decode GEMV rows run before the seconds-long GEMM rows of
            # their layer: right after those, the GPU measured slower for a
            # few dozen microsecond-long steps.
            rows["decode_gemv_" + args.workload] = bench_gemv(qp, layer, stream, device, peaks)
            l5k = Layer(workloads.WORKLOADS["qwen3_8b_q5k_t8192"], rank, device)
            rows["decode_gemv_qwen3_8b_q5k"] = bench_gemv(qp, l5k, stream, device, peaks)
            ms5k = time_layer(qp, l5k, stream, max(5, args.steps // 2), 3)
            rows["qwen3_8b_q5k_t8192"] = {"ms": round(ms5k, 4), "tflops": round(l5k.flops() / ms5k / 1e9, 1),
                                          "tok_per_s": round(l5k.T / ms5k * 1e3, 1)}
            del l5k
            wl5 = workloads.WORKLOADS["qwen3_8b_q4k_t31258_chunk4864"]
            l5 = Layer(wl5, rank, device, need_f16=True)
            rows["decode_gemv_qwen3_8b_q4k"] = bench_gemv(qp, l5, stream, device, peaks)
            ms_f = time_layer(qp, l5, stream, 3, 1, mode="fused", chunk=wl5["chunk"])
            ms_c = time_layer(qp, l5, stream, 3, 1, mode="cached", chunk=wl5["chunk"])
            rows["qwen3_8b_q4k_t31258_chunk4864"] = {
                "fused": {"ms": round(ms_f, 3), "tok_per_s": round(l5.T / ms_f * 1e3, 1),
                          "tflops": round(l5.flops() / ms_f / 1e9, 1)},
                "cached_f16": {"ms": round(ms_c, 3), "tok_per_s": round(l5.T / ms_c * 1e3, 1),
                               "tflops": round(l5.flops() / ms_c / 1e9, 1),
                               "note": "excludes the one-time f16 weight build"}}
            del l5
            rows["matmul_peaks_8192"] = measure_matmul_peaks(device)
        if not args.no_cpu_baseline:
            cpu = cpu_oracle_sample(wl, seconds=args.cpu_seconds)
            if rows is not None:
                rows["cpu_oracle_dequant"] = cpu_dequant_rows()

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(max_ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
            "data": "synthetic (seeded; weights and activations drawn as the workload states)",
            "config": {"workload": args.workload, "T": T, "tokens_per_rank": T, "mode": args.mode,
                       "tiling": "cta_pairs" if args.cta_pairs else "one_cta",
                       "projections": "q,k,v,o,gate,up (Q2_K) + down (Q6_K); hidden 4096, kv 1024, ffn 12288",
                       "accumulate": "f32", "parallelism": "replicas x%d (weak scaling, no collective)" % world,
                       "l2": "inputs larger than L2: each step streams %.2f GB of X, W and Y" % (
                           (sum(v.numel() * 2 for v in layer.X.values()) + sum(w.numel() for w in layer.W)
                            + sum(y.numel() * 4 for y in layer.Y)) / 1e9)},
            "tok_per_s": round(tok_s, 1),
            "pct_dense_fp16_peak": round(100.0 * value / (peak * world), 2),
            "per_launch": [{k: v for k, v in d.items() if k != "flops"} for d in per_launch],
            "per_projection": per_proj,
            "roofline": roofline,
            "e2e": e2e,
            "gpu_launches": args.steps * nlaunch,
            "clocks": sampler.summary(),
            "cpu_baseline": cpu,
            "rows": rows,
        }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------- reference arm ----

def main_reference(args):
    """The CPU oracle timed on this host's cores on the same workload and
    metric; each step dequantizes all seven weights (f32) and computes the
    fp64 projection for a bounded sample of token rows."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    wl = workloads.WORKLOADS[args.workload]
    dims = workloads.input_dims(wl)
    n_rows = args.reference_rows
    X = {k: synth.normal_f16((n_rows, dims[k]), seed=wl["seed"], tensor=1000 + i)
         for i, k in enumerate(("h", "o", "f"))}
    W_q = [synth.blocks(qt, out_f, in_f, seed=wl["seed"], tensor=i)
           for i, (_, out_f, in_f, _, qt) in enumerate(wl["projections"])]
    rows = np.arange(n_rows, dtype=np.int64)

    def step():
        for w, (_, out_f, in_f, src, qt) in zip(W_q, wl["projections"]):
            W = oracle.dequant_f32(qt, w, out_f, in_f)
            oracle.gemm_f64(X[src], W, rows)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    flops = workloads.flops(wl, n_rows)
    value = flops / dt / 1e12
    sample = ("each step: f32 dequant of all 7 weights + fp64 GEMM of %d of the %d token rows" % (n_rows, wl["T"]))
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)", "config": {"workload": args.workload, "T": wl["T"],
                                                     "sampled_rows_per_step": n_rows},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line))


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["qp", "reference"], default="qp")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads.WORKLOADS))
    p.add_argument("--no-rows", action="store_true", help="skip the other rows of the path")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffer) measurement")
    p.add_argument("--only-proj", default=None, help="time only this projection (profiling runs)")
    p.add_argument("--no-group", action="store_true",
                   help="launch the step's projections one at a time instead of one grouped launch per type")
    p.add_argument("--d2h-streams", type=int, default=1, help="copy streams for the e2e read-back of Y")
    p.add_argument("--cta-pairs", type=int, choices=[0, 1], default=1,
                   help="GEMM tiling: 1 = 256-row tiles on CTA pairs (default), 0 = 128-row tiles on one CTA")
    p.add_argument("--mode", choices=["fused", "cached"], default="fused",
                   help="cached: the same step over f16 weights made once by qp_dequant_f16")
    p.add_argument("--dequant-only", action="store_true", help="only the standalone dequant rows")
    p.add_argument("--gemv-only", action="store_true", help="only the decode GEMV row")
    p.add_argument("--gemv-t", type=int, default=0, choices=range(0, 9),
                   help="with --gemv-only: time this token count only (default: 1 and 8)")
    p.add_argument("--dequant-cases", default=None, help="e.g. Q4_K_f16,Q2_K_f32 (with --dequant-only)")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--reference-rows", type=int, default=8)
    a = p.parse_args(argv)
    if a.warmup < 3:
        p.error("--warmup must be >= 3")
    return a


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        main_reference(args)
    else:
        main_qp(args)


if __name__ == "__main__":
    main()
