#!/usr/bin/env python3
"""Benchmark: quantized GEMV effective HBM GB/s (and % of peak) on GB300.

Step = one fused dual Q4_0 projection (two weights N = K = 4096, x f32
[1, 4096]) through the C ABI, the workload the headline metric is quoted on.
The same line also reports M = 8, and a sweep over every workload of the
hot path (single Q4_0, Q4_K, affine u8/packed at M = 1/8/512, the decode-layer
chain and the QKV split).

Timing: W eager warm-up steps, then K steps replayed from CUDA graphs and
bracketed by CUDA events on the launching stream (barrier + synchronize on
both sides, max over ranks). Every step reads a different weight set out of
a rotation whose total size is several times the 129 MB L2, so each call
streams its weights from HBM. Effective bytes per call = quantized weight
bytes (codes + scales) + x + y.

--impl reference times the plain CPU oracle on the host cores instead (each
step: a bounded sample of rows of the same workload).
"""
from __future__ import annotations

import argparse
import hashlib
import itertools
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("quantized GEMV effective HBM GB/s and % of GB300 peak at M=1/8; µs/call")
L2_BYTES = 129 * 1024 * 1024
NOMINAL_HBM_GBS = 8000.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured", d
    except Exception:
        return FALLBACK_HBM_GBS, "fallback", {}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampled every 50 ms in the background; keeps timestamps."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return

        def reader():
            for line in self.proc.stdout:
                self.samples.append((time.time(), line.strip()))

        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = []
        for ts, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            rows.append((ts, parts))
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        inside = [r for r in rows if t0 <= r[0] <= t1]
        if not inside:  # timed region shorter than the sampling period
            inside = sorted(rows, key=lambda r: abs(r[0] - 0.5 * (t0 + t1)))[:3]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[0]) for _, p in inside if num(p[0]) is not None]
        mx = [num(p[1]) for _, p in inside if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, p in inside for i in range(4)
                          if p[4 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside)}


# ---------------------------------------------------------------- workloads
def q4_0_row_bytes(K):
    return K // 32 * 18


def q4_k_row_bytes(K):
    return K // 256 * 144


def n_sets(bytes_per_call: int, factor: float = 4.0, lo: int = 2, hi: int = 64) -> int:
    return int(min(hi, max(lo, math.ceil(factor * L2_BYTES / max(1, bytes_per_call)))))


class Runner:
    """A workload bound to rotating device buffer sets: call(i) runs set i."""

    def __init__(self, name, et_bytes, flops, call, nsets, launches_per_call=1):
        self.name, self.et_bytes, self.flops = name, et_bytes, flops
        self.call, self.nsets, self.launches = call, nsets, launches_per_call


_CASES = {}


def cached(kind, case, N, K, M, **kw):
    """synth workload with the weights drawn once per (kind, case, N, K)."""
    from bit_quantized_gemv_dequant_gb300 import synth
    key = (kind, case, N, K, tuple(sorted(kw.items())))
    if key not in _CASES:
        if kind == "q4_0":
            _CASES[key] = synth.q4_0_case(case, N, K, 1, **kw)
        elif kind == "q4_k":
            _CASES[key] = synth.q4_k_case(case, N, K, 1)
        else:
            _CASES[key] = synth.affine_case(case, N, K, 1, kw["gs"])
    c = dict(_CASES[key])
    c["x"] = synth.normal(1000 * case + synth.T_X, (M, K))
    return c


def replicate(t, nsets):
    """nsets copies of a device tensor at distinct addresses."""
    import torch
    return [t] + [t.clone() for _ in range(nsets - 1)]


def make_dual_q4_0(M, N=4096, K=4096, case=1, nsets=None):
    import torch
    import bit_quantized_gemv_dequant_gb300 as qg
    from bit_quantized_gemv_dequant_gb300 import synth
    c = cached("q4_0", case, N, K, M, dual=True)
    wb = 2 * N * q4_0_row_bytes(K)
    et = wb + 4 * M * K + 2 * 4 * M * N
    ns = nsets or n_sets(et)
    dev = torch.device("cuda", torch.cuda.current_device())
    wa = replicate(torch.from_numpy(c["w"]).to(dev), ns)
    wbt = replicate(torch.from_numpy(c["w_b"]).to(dev), ns)
    xs = replicate(torch.from_numpy(c["x"]).to(dev), ns)
    ya = [torch.empty((M, N), device=dev) for _ in range(ns)]
    yb = [torch.empty((M, N), device=dev) for _ in range(ns)]
    ws_need = qg.workspace_size(qg.QG_OP_DUAL_Q4_0, M, N, K)
    ws = torch.empty(max(ws_need, 16), dtype=torch.uint8, device=dev)
    L = qg.lib()
    ptr = [(wa[i].data_ptr(), wbt[i].data_ptr(), xs[i].data_ptr(), ya[i].data_ptr(),
            yb[i].data_ptr()) for i in range(ns)]

    def call(i, stream):
        p = ptr[i % ns]
        rc = L.qgemv_dual_q4_0(p[0], p[1], p[2], p[3], p[4], M, N, K, ws.data_ptr(),
                               ws.numel(), stream)
        if rc:
            raise RuntimeError(f"qgemv_dual_q4_0 failed: {qg.status_string(rc)}")

    r = Runner(f"dual_q4_0 M={M} N={N} K={K}", et, 2 * 2 * M * N * K, call, ns,
               1 + (1 if ws_need else 0))
    r.host = {"c": c, "M": M, "N": N, "K": K, "xs": xs, "ya": ya, "yb": yb, "wa": wa, "wb": wbt,
              "ws": ws}
    return r


def make_single(fmt, M, N, K, case, gs=64, packed=0):
    import torch
    import bit_quantized_gemv_dequant_gb300 as qg
    from bit_quantized_gemv_dequant_gb300 import synth
    dev = torch.device("cuda", torch.cuda.current_device())
    L = qg.lib()
    if fmt == "q4_0":
        c = cached("q4_0", case, N, K, M)
        wbytes, op = N * q4_0_row_bytes(K), qg.QG_OP_Q4_0
    elif fmt == "q4_k":
        c = cached("q4_k", case, N, K, M)
        wbytes, op = N * q4_k_row_bytes(K), qg.QG_OP_Q4_K
    else:
        c = cached("affine", case, N, K, M, gs=gs)
        c["w"] = c["q_packed"] if packed else c["q"]
        wbytes = N * (K // 2 if packed else K) + 2 * 4 * N * (K // gs)
        op = qg.QG_OP_AFFINE
    et = wbytes + 4 * M * K + 4 * M * N
    ns = n_sets(et)
    w = replicate(torch.from_numpy(np.ascontiguousarray(c["w"])).to(dev), ns)
    xs = replicate(torch.from_numpy(c["x"]).to(dev), ns)
    ys = [torch.empty((M, N), device=dev) for _ in range(ns)]
    ws_need = qg.workspace_size(op, M, N, K, gs, packed)
    ws = torch.empty(max(ws_need, 16), dtype=torch.uint8, device=dev)
    if fmt == "affine":
        s = replicate(torch.from_numpy(c["s"]).to(dev), ns)
        b = replicate(torch.from_numpy(c["b"]).to(dev), ns)

    def call(i, stream):
        j = i % ns
        if fmt == "q4_0":
            rc = L.qgemv_q4_0(w[j].data_ptr(), xs[j].data_ptr(), ys[j].data_ptr(), M, N, K,
                              ws.data_ptr(), ws.numel(), stream)
        elif fmt == "q4_k":
            rc = L.qgemv_q4_k(w[j].data_ptr(), xs[j].data_ptr(), ys[j].data_ptr(), M, N, K,
                              ws.data_ptr(), ws.numel(), stream)
        else:
            rc = L.qmm_affine(xs[j].data_ptr(), w[j].data_ptr(), s[j].data_ptr(),
                              b[j].data_ptr(), ys[j].data_ptr(), M, N, K, gs, packed,
                              ws.data_ptr(), ws.numel(), stream)
        if rc:
            raise RuntimeError(f"{fmt} failed: {qg.status_string(rc)}")

    name = f"{fmt}{'/packed' if packed else ('/u8' if fmt == 'affine' else '')} M={M} N={N} K={K}"
    return Runner(name, et, 2 * M * N * K, call, ns)


def make_af4(M, N=4096, K=4096, case=90):
    """qmm_af4_g64 on the prepared layout (prepared once, outside the timing):
    one kernel reads the prepared words directly."""
    import torch
    import bit_quantized_gemv_dequant_gb300 as qg
    from bit_quantized_gemv_dequant_gb300 import synth
    dev = torch.device("cuda", torch.cuda.current_device())
    c = synth.af4_case(case, N, K, M)
    bf = lambda b: torch.from_numpy(b.view(np.int16)).to(dev).view(torch.bfloat16)
    plane, meta = qg.prepare_af4_g64(torch.from_numpy(c["q"]).to(dev), bf(c["s_bits"]),
                                     bf(c["b_bits"]))
    et = N * K // 2 + 4 * N * (K // 64) + 4 * M * K + 4 * M * N
    ns = n_sets(et)
    planes, metas = replicate(plane, ns), replicate(meta, ns)
    xs = replicate(torch.from_numpy(c["x"]).to(dev), ns)
    ys = [torch.empty((M, N), device=dev) for _ in range(ns)]
    L = qg.lib()

    def call(i, stream):
        j = i % ns
        rc = L.qmm_af4_g64(xs[j].data_ptr(), planes[j].data_ptr(), metas[j].data_ptr(),
                           ys[j].data_ptr(), M, N, K, None, 0, stream)
        if rc:
            raise RuntimeError(f"qmm_af4_g64 failed: {qg.status_string(rc)}")

    return Runner(f"af4_g64 M={M} N={N} K={K}", et, 2 * M * N * K, call, ns, 1)


def make_qkv(seq=4096, qs=2048, ks=2048, vs=4096, case=4):
    import torch
    import bit_quantized_gemv_dequant_gb300 as qg
    from bit_quantized_gemv_dequant_gb300 import synth
    dev = torch.device("cuda", torch.cuda.current_device())
    src = torch.from_numpy(synth.qkv_case(case, seq, qs, ks, vs)).to(dev)
    q = torch.empty((seq, qs), device=dev)
    k = torch.empty((seq, ks), device=dev)
    v = torch.empty((seq, vs), device=dev)
    L = qg.lib()
    et = 2 * 4 * seq * (qs + ks + vs)

    def call(i, stream):
        rc = L.qkv_split(src.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), seq, qs, ks,
                         vs, stream)
        if rc:
            raise RuntimeError(f"qkv_split failed: {qg.status_string(rc)}")

    return Runner(f"qkv_split seq={seq} spans={qs}/{ks}/{vs}", et, 0, call, 1)


def make_layer(M, hidden=4096, ffn=12288):
    """One decode layer of projections as a single step: Q+gate dual Q4_0
    (N = hidden), K+V dual Q4_0 (N = hidden / 4), FFN up Q4_K (N = ffn) and
    FFN down Q4_K (K = ffn), launched back to back (under a CUDA graph with
    programmatic dependent launch each call's weight stream overlaps the
    previous call's tail)."""
    parts = [make_dual_q4_0(M, hidden, hidden, 40), make_dual_q4_0(M, hidden // 4, hidden, 50),
             make_single("q4_k", M, ffn, hidden, 60), make_single("q4_k", M, hidden, ffn, 70)]
    ns = max(p.nsets for p in parts)

    def call(i, stream):
        for p in parts:
            p.call(i, stream)

    r = Runner(f"decode layer M={M}", sum(p.et_bytes for p in parts),
               sum(p.flops for p in parts), call, ns, sum(p.launches for p in parts))
    return r


# ------------------------------------------------------------------ timing
def sweep_specs():
    """(name, runner factory) for every configuration the sweep times."""
    specs = [
        ("cfg0 q4_0", lambda: make_single("q4_0", 1, 1024, 1024, 0)),
        ("cfg2 q4_k N=4096", lambda: make_single("q4_k", 1, 4096, 4096, 2)),
        ("cfg2 q4_k N=12288", lambda: make_single("q4_k", 1, 12288, 4096, 2)),
        ("cfg3 affine u8 M=1", lambda: make_single("affine", 1, 4096, 4096, 3, 64, 0)),
        ("cfg3 affine packed M=1", lambda: make_single("affine", 1, 4096, 4096, 3, 64, 1)),
        ("cfg3 affine u8 M=8", lambda: make_single("affine", 8, 4096, 4096, 3, 64, 0)),
        ("cfg3 affine packed M=8", lambda: make_single("affine", 8, 4096, 4096, 3, 64, 1)),
        ("cfg3 affine u8 M=512", lambda: make_single("affine", 512, 4096, 4096, 3, 64, 0)),
        ("cfg3 affine packed M=512", lambda: make_single("affine", 512, 4096, 4096, 3, 64, 1)),
        ("cfg4 qkv_split", lambda: make_qkv()),
        ("af4_g64 M=1", lambda: make_af4(1)),
        ("af4_g64 M=8", lambda: make_af4(8)),
        ("af4_g64 M=32", lambda: make_af4(32)),
        # Q4_0 / Q4_K prefill: repacked to affine codes (group 32), tcgen05 MMAs.
        ("prefill dual q4_0 N=K=4096 M=512", lambda: make_dual_q4_0(512, 4096, 4096, 80)),
        ("prefill q4_k N=K=4096 M=512", lambda: make_single("q4_k", 512, 4096, 4096, 81)),
        # The same prefill calls with the folded-weight kernel (QG_OPT_PREFILL_FOLD).
        ("cfg3 affine u8 M=512 folded", lambda: make_single("affine", 512, 4096, 4096, 3, 64, 0)),
        ("cfg3 affine packed M=512 folded", lambda: make_single("affine", 512, 4096, 4096, 3, 64, 1)),
        ("prefill dual q4_0 N=K=4096 M=512 folded", lambda: make_dual_q4_0(512, 4096, 4096, 80)),
        ("prefill q4_k N=K=4096 M=512 folded", lambda: make_single("q4_k", 512, 4096, 4096, 81)),
        # 8 < M < 64 on the CUDA cores (f32 bar), against the f32 FMA roofline.
        ("mid-M dual q4_0 N=K=4096 M=16", lambda: make_dual_q4_0(16, 4096, 4096, 85)),
        ("mid-M dual q4_0 N=K=4096 M=32", lambda: make_dual_q4_0(32, 4096, 4096, 85)),
    ]
    for M in (1, 2, 4, 8):
        specs += [
            (f"cfg4 M={M} q+gate dual", lambda M=M: make_dual_q4_0(M, 4096, 4096, 40)),
            (f"cfg4 M={M} k+v dual", lambda M=M: make_dual_q4_0(M, 1024, 4096, 50)),
            (f"cfg4 M={M} ffn up q4_k", lambda M=M: make_single("q4_k", M, 12288, 4096, 60)),
            (f"cfg4 M={M} ffn down q4_k", lambda M=M: make_single("q4_k", M, 4096, 12288, 70)),
            (f"cfg4 M={M} decode layer (4 calls, one graph)", lambda M=M: make_layer(M)),
        ]
    return specs


def time_runner(r: Runner, steps: int, warmup: int, chunk: int = 1000):
    """Warm up eagerly, then replay `steps` calls from CUDA graphs (chunks of
    at most `chunk` calls), timed with events on the capture stream. Returns
    (total_ms, t0_wall, t1_wall)."""
    import torch
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        h = stream.cuda_stream
        for i in range(warmup):
            r.call(i, h)
    torch.cuda.synchronize()
    graphs = []
    done = 0
    while done < steps:
        n = min(chunk, steps - done)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            h = stream.cuda_stream
            for i in range(n):
                r.call(done + i, h)
        graphs.append(g)
        done += n
    # One untimed replay of the first graph so that graph upload is excluded.
    with torch.cuda.stream(stream):
        graphs[0].replay()
    torch.cuda.synchronize()
    return graphs, stream


# A bounded sleep kernel (fixed cycle count, no flag) queued ahead of the start
# event: the host enqueues the graphs while it runs, so the timed region starts
# with the work already queued and measures the calls, not the host's graph
# launch latency (which matters for short runs such as 20 steps).
QUEUE_AHEAD_US = 100.0


def replay_timed(graphs, stream, barrier=None):
    import torch
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if barrier:
        barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    with torch.cuda.stream(stream):  # replay() launches on the current stream
        torch.cuda._sleep(int(QUEUE_AHEAD_US * 2.1e3))  # ~100 us at up to 2.1 GHz
        e0.record(stream)
        for g in graphs:
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if barrier:
        barrier()
    return e0.elapsed_time(e1), t0, t1


def measure(r: Runner, steps: int, warmup: int, repeats: int = 1):
    """µs per call: the median over `repeats` timed replays of `steps` calls."""
    graphs, stream = time_runner(r, steps, warmup)
    runs = [1000.0 * replay_timed(graphs, stream)[0] / steps for _ in range(repeats)]
    us = float(np.median(runs))
    out = {"us_per_call": us, "gbs": r.et_bytes / (us * 1e3), "et_bytes": r.et_bytes,
           "sets": r.nsets}
    if repeats > 1:
        out["repeats"] = repeats
        out["us_min_max"] = [min(runs), max(runs)]
    return out


# --------------------------------------------------------------- e2e
def e2e_dual(steps: int, warmup: int, M: int = 1, N: int = 4096, K: int = 4096):
    """The headline workload end to end, through the public C ABI with host
    buffers: every step is one qgemv_dual_q4_0_host call with x, y_a and y_b
    in page-locked host memory. The call moves x to the GPU (a fetch kernel),
    runs the dual projection (which stores y_a and y_b straight into host
    memory) and returns once the outputs hold the result. Also reported: the
    same call on pageable buffers (one cudaMemcpyAsync per buffer through
    device staging), and the device-resident call followed by a stream
    synchronize (the launch and the host round trip alone). Steps rotate
    over the same weight sets as the headline (more than 4x the L2), so
    every step streams its weights from HBM."""
    import torch
    import bit_quantized_gemv_dequant_gb300 as qg
    from bit_quantized_gemv_dequant_gb300 import synth
    dev = torch.device("cuda", torch.cuda.current_device())
    c = synth.q4_0_case(1, N, K, M, dual=True)
    et = 2 * N * q4_0_row_bytes(K) + 4 * M * K + 2 * 4 * M * N
    ns = n_sets(et)
    wa = replicate(torch.from_numpy(c["w"]).to(dev), ns)
    wb = replicate(torch.from_numpy(c["w_b"]).to(dev), ns)
    x_pin = torch.from_numpy(c["x"]).pin_memory()
    y_pin = [torch.empty((M, N), dtype=torch.float32).pin_memory() for _ in range(2)]
    x_page = torch.from_numpy(c["x"]).clone()
    y_page = [torch.empty((M, N), dtype=torch.float32) for _ in range(2)]
    x_dev = x_pin.to(dev)
    y_dev = [torch.empty((M, N), device=dev) for _ in range(2)]
    L = qg.lib()
    stream = torch.cuda.Stream()
    h = stream.cuda_stream
    need = qg.workspace_size(qg.QG_OP_DUAL_Q4_0_HOST, M, N, K)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    pws = ws.data_ptr()
    wp = [(wa[i].data_ptr(), wb[i].data_ptr()) for i in range(ns)]

    def host_call(x, ya, yb):
        args = [(pa, pb, x.data_ptr(), ya.data_ptr(), yb.data_ptr(), M, N, K, pws, need, h)
                for pa, pb in wp]
        it = itertools.count()

        def step():
            rc = L.qgemv_dual_q4_0_host(*args[next(it) % ns])
            if rc:
                raise RuntimeError(f"qgemv_dual_q4_0_host failed: {qg.status_string(rc)}")
        return step

    dargs = [(pa, pb, x_dev.data_ptr(), y_dev[0].data_ptr(), y_dev[1].data_ptr(), M, N, K, None,
              0, h) for pa, pb in wp]
    dit = itertools.count()

    def device_call():
        rc = L.qgemv_dual_q4_0(*dargs[next(dit) % ns])
        if rc:
            raise RuntimeError(f"qgemv_dual_q4_0 failed: {qg.status_string(rc)}")
        stream.synchronize()

    out = {}
    pdl_old = qg.get_option(qg.QG_OPT_PDL)
    for name, step in (("pinned", host_call(x_pin, *y_pin)),
                       ("pageable", host_call(x_page, *y_page)),
                       ("device", device_call)):
        # The device route is one call followed by a synchronize: a lone
        # call, launched plainly (not declared to overlap its neighbours).
        qg.set_option(qg.QG_OPT_PDL, 0 if name == "device" else pdl_old)
        try:
            for _ in range(warmup):
                step()
            t0 = time.perf_counter()
            for _ in range(steps):
                step()
            t1 = time.perf_counter()
        finally:
            qg.set_option(qg.QG_OPT_PDL, pdl_old)
        out[name] = 1e6 * (t1 - t0) / steps
    # The three routes give the same bits.
    for i in range(2):
        ref = y_dev[i].cpu().numpy().view(np.uint32)
        for got in (y_pin[i], y_page[i]):
            if not np.array_equal(got.numpy().view(np.uint32), ref):
                raise RuntimeError("e2e: host-buffer result differs from the device call")
    us = out["pinned"]
    return {"value": et / (us * 1e3), "unit": "GB/s", "us_per_step": us, "steps": steps,
            "h2d_bytes_per_step": 4 * M * K, "d2h_bytes_per_step": 2 * 4 * M * N,
            "breakdown_us": {
                "step: qgemv_dual_q4_0_host, page-locked buffers (zero-copy)": out["pinned"],
                "same call, pageable buffers (cudaMemcpyAsync through device staging)":
                    out["pageable"],
                "device-resident call (plain launch) + stream synchronize (no host data)":
                    out["device"]},
            "weight_sets": ns,
            "how": "one qgemv_dual_q4_0_host call per step through ctypes: a fetch kernel "
                   "copies x from page-locked host memory into the workspace, the GEMV follows "
                   "as its programmatic dependent and stores y_a and y_b into page-locked host "
                   "memory; the call synchronizes the stream before it returns"}


# -------------------------------------------------------------- traffic
TRAFFIC_SOURCES = ("bit_quantized_gemv_dequant_gb300/csrc/gemv_xreg.cuh",
                   "bit_quantized_gemv_dequant_gb300/csrc/gemv.cu",
                   "bit_quantized_gemv_dequant_gb300/csrc/gemv_xreg_q4_0.cu",
                   "bit_quantized_gemv_dequant_gb300/csrc/qg_internal.cuh")


def source_hash():
    """sha256 over the sources of the dual Q4_0 GEMV kernel and its planner."""
    h = hashlib.sha256()
    for rel in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def recorded_traffic(kernel_key: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)
    except Exception:
        return None
    e = d.get(kernel_key)
    if not e or e.get("source_sha256") != source_hash():
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------ CPU oracle
def oracle_dual_sample(M, N, K, budget_s, rows_per_call=None):
    """Time the oracle's dual projection on the host. Returns (GB/s, rows,
    calls, seconds). Effective bytes are scaled to the rows computed."""
    import oracle
    from bit_quantized_gemv_dequant_gb300 import synth
    c = synth.q4_0_case(1, N, K, M, dual=True)
    rows_per_call = rows_per_call or N
    rng = np.random.default_rng(0)
    calls, rows_done = 0, 0
    t0 = time.perf_counter()
    while True:
        start = int(rng.integers(0, max(1, N - rows_per_call + 1)))
        rows = np.arange(start, start + rows_per_call)
        oracle.gemv_dual_q4_0(c["w"], c["w_b"], c["x"], M, N, K, rows=rows)
        calls += 1
        rows_done += rows_per_call
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    per_row = 2 * q4_0_row_bytes(K) + 2 * 4 * M
    bytes_done = rows_done * per_row + calls * 4 * M * K
    return bytes_done / dt / 1e9, rows_done, calls, dt


def oracle_dual_sample_threads(M, N, K, budget_s, threads):
    """The same oracle call on `threads` host threads at once, each on its own
    row range (the C oracle releases the GIL). Returns (GB/s, rows, seconds)."""
    import concurrent.futures as cf
    import oracle
    from bit_quantized_gemv_dequant_gb300 import synth
    c = synth.q4_0_case(1, N, K, M, dual=True)
    chunk = max(1, N // threads)
    t0 = time.perf_counter()

    def worker(tid):
        rows_done, calls = 0, 0
        start = (tid * chunk) % N
        rows = np.arange(start, min(N, start + chunk))
        while time.perf_counter() - t0 < budget_s:
            oracle.gemv_dual_q4_0(c["w"], c["w_b"], c["x"], M, N, K, rows=rows)
            rows_done += len(rows)
            calls += 1
        return rows_done, calls

    with cf.ThreadPoolExecutor(threads) as ex:
        res = list(ex.map(worker, range(threads)))
    dt = time.perf_counter() - t0
    rows_done = sum(r for r, _ in res)
    calls = sum(n for _, n in res)
    per_row = 2 * q4_0_row_bytes(K) + 2 * 4 * M
    return (rows_done * per_row + calls * 4 * M * K) / dt / 1e9, rows_done, dt


def reference_arm(args, rank, world):
    """--impl reference: the oracle as it stands, timed on the host cores."""
    if rank != 0:
        return
    M, N, K = 1, 4096, 4096
    # Size each step so the whole run takes about a minute at most.
    import oracle
    from bit_quantized_gemv_dequant_gb300 import synth
    c = synth.q4_0_case(1, 64, K, M, dual=True)
    t0 = time.perf_counter()
    oracle.gemv_dual_q4_0(c["w"], c["w_b"], c["x"], M, 64, K)
    per_row = (time.perf_counter() - t0) / 64
    total_steps = args.steps + args.warmup
    rows = int(max(1, min(N, 60.0 / max(1, total_steps) / max(per_row, 1e-9))))
    c = synth.q4_0_case(1, N, K, M, dual=True)
    for i in range(args.warmup):
        oracle.gemv_dual_q4_0(c["w"], c["w_b"], c["x"], M, N, K, rows=np.arange(rows))
    t0 = time.perf_counter()
    for i in range(args.steps):
        start = (i * rows) % (N - rows + 1)
        oracle.gemv_dual_q4_0(c["w"], c["w_b"], c["x"], M, N, K,
                              rows=np.arange(start, start + rows))
    dt = time.perf_counter() - t0
    per_row_bytes = 2 * q4_0_row_bytes(K) + 2 * 4 * M
    step_bytes = rows * per_row_bytes + 4 * M * K
    gbs = step_bytes * args.steps / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000 * dt / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(M),
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"each step: rows [s, s+{rows}) of both weights of the "
                                       f"dual Q4_0 projection N=K=4096, M=1"},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def max_over_ranks(value: float) -> float:
    """Maximum of a host-side float over all ranks (gloo process group)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload_config(M):
    return {"workload": "fused dual Q4_0 projection: two Q4_0 weights N=K=4096 "
                        "(W ~ N(0,0.02^2)), shared x f32 [M,4096] ~ N(0,1)",
            "M": M, "N": 4096, "K": 4096,
            "l2": "inputs larger than L2: rotation of weight sets totalling >= 4x the 129 MB L2",
            "parallelism": "replicas (one independent problem per GPU)"}


# ------------------------------------------------------------------ main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200000)
    ap.add_argument("--warmup", type=int, default=100)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--sweep-steps", type=int, default=400)
    ap.add_argument("--only", default=None, metavar="NAME",
                    help="time one sweep configuration (e.g. 'cfg3 affine u8 M=512') for "
                         "--steps calls and print its line; for profiling runs")
    ap.add_argument("--pdl", type=int, default=2, choices=[0, 1, 2],
                    help="QG_OPT_PDL for the headline: 2 = independent back-to-back calls "
                         "(default), 1 = each call waits for the previous one, 0 = plain launches")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")

    if args.impl == "reference":
        reference_arm(args, rank, world)
        if dist:
            dist.destroy_process_group()
        return

    import torch
    import bit_quantized_gemv_dequant_gb300 as qg
    torch.cuda.set_device(local)
    qg.lib()

    barrier = dist.barrier if dist else None
    hbm_peak, peak_src, peak_doc = peaks()
    tensor_peak = float(peak_doc.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
    qg.set_option(qg.QG_OPT_PDL, args.pdl)

    if args.only is not None:
        specs = dict(sweep_specs())
        if args.only not in specs:
            ap.error(f"--only: unknown configuration {args.only!r}; one of {sorted(specs)}")
        qg.set_option(qg.QG_OPT_PREFILL_FOLD, 1 if args.only.endswith("folded") else 0)
        r = specs[args.only]()
        res = measure(r, args.steps, args.warmup)
        res["tflops"] = r.flops / (res["us_per_call"] * 1e6)
        if qg.device_error():
            raise RuntimeError("device error word set")
        print(json.dumps({"only": args.only, **res}), flush=True)
        return

    # Headline: dual Q4_0, M = 1.
    r1 = make_dual_q4_0(1)
    graphs, stream = time_runner(r1, args.steps, args.warmup)
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    ms, t0, t1 = replay_timed(graphs, stream, barrier)
    if sampler:
        time.sleep(0.2)
        sampler.stop()
    del graphs
    if dist:
        ms = max_over_ranks(ms)
    us = 1000.0 * ms / args.steps
    value = world * r1.et_bytes * args.steps / (ms * 1e-3) / 1e9
    achieved = r1.et_bytes / (us * 1e3)
    err = qg.device_error()
    if err:
        raise RuntimeError(f"device error word {err:#x} after the timed region")

    if rank != 0:
        if dist:
            dist.barrier()
            dist.destroy_process_group()
        return

    clocks = sampler.summary(t0, t1)
    out = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
           "data": "synthetic (seeded; weights replicated at distinct addresses for the L2 "
                   "rotation)",
           "config": workload_config(1),
           "us_per_call": us, "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
           "gpu_launches": args.steps * r1.launches,
           "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak,
                        "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                        if peak_src == "measured" else "fallback 6.8 TB/s",
                        "unit": "GB/s", "frac": achieved / hbm_peak,
                        "traffic": recorded_traffic("dual_q4_0_m1_n4096_k4096")},
           "clocks": clocks}

    out["launch_mode"] = {
        2: "CUDA graph of back-to-back independent calls (QG_OPT_PDL = 2: each call reads "
           "and writes only its own buffers, so consecutive calls overlap)",
        1: "CUDA graph of back-to-back calls, each waiting for the previous one "
           "(QG_OPT_PDL = 1, programmatic dependent launch)",
        0: "CUDA graph of back-to-back calls, plain launches"}[args.pdl]
    out["queue_ahead"] = (f"graphs queued behind a {QUEUE_AHEAD_US:.0f} us sleep kernel before "
                          "the start event")
    # The same workload in the other launch modes, for reference: a chain in
    # which every call waits for the previous one (a decode chain whose x is
    # the previous y), and plain launches.
    for mode, key in ((1, "dependent_chain"), (0, "no_pdl")):
        if mode == args.pdl:
            continue
        qg.set_option(qg.QG_OPT_PDL, mode)
        res = measure(r1, min(args.steps, 20000), args.warmup)
        res["frac_of_hbm_peak"] = res["gbs"] / hbm_peak
        out[key] = res
    qg.set_option(qg.QG_OPT_PDL, args.pdl)

    # Hot L2 (labelled as such, not the headline): one weight set reused by
    # every call, so the 18.9 MB of weights stay in the 129 MB L2.
    rh = make_dual_q4_0(1, nsets=1)
    hot = measure(rh, min(args.steps, 20000), args.warmup)
    hot["note"] = "hot L2: the same weight set every call (not HBM-bound; for reference only)"
    out["hot_l2"] = hot
    del rh

    # M = 8 on the same weights (FP32-FMA bound; reported against the ALU peak).
    r8 = make_dual_q4_0(8)
    m8 = measure(r8, min(args.steps, 20000), args.warmup)
    sm_mhz = clocks.get("sm_max_mhz") or peak_doc.get("sm_max_mhz") or 2070.0
    n_sm = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    alu_peak = n_sm * 128 * 2 * sm_mhz * 1e6 / 1e12  # TFLOP/s f32 FMA
    tflops = r8.flops / (m8["us_per_call"] * 1e-6) / 1e12
    m8.update({"frac_of_hbm_peak": m8["gbs"] / hbm_peak,
               "roofline": {"bound": "alu", "achieved": tflops, "peak": alu_peak,
                            "unit": "TFLOP/s", "frac": tflops / alu_peak,
                            "peak_source": f"{n_sm} SMs x 128 f32 FMA/clk x 2 x max SM clock"}})
    out["m8"] = m8

    out["e2e"] = e2e_dual(2000, 50)

    if not args.no_cpu:
        gbs1, rows1, calls1, dt1 = oracle_dual_sample(1, 4096, 4096, budget_s=6.0)
        nthr = os.cpu_count() or 1
        gbsn, rowsn, dtn = oracle_dual_sample_threads(1, 4096, 4096, 6.0, nthr)
        out["cpu_baseline"] = {
            "value": gbsn, "unit": "GB/s", "cores": nthr, "kind": "oracle",
            "sample": f"dual Q4_0 N=K=4096 M=1, {nthr} host threads on disjoint row ranges: "
                      f"{rowsn} rows per weight in {dtn:.1f} s",
            "single_thread": {"value": gbs1, "unit": "GB/s", "cores": 1,
                              "sample": f"{calls1} full projections ({rows1} rows per weight) "
                                        f"in {dt1:.1f} s"}}

    if not args.no_sweep:
        sweep = {}
        del r1, r8
        torch.cuda.empty_cache()
        specs = sweep_specs()
        for name, mk in specs:
            fold_old = qg.get_option(qg.QG_OPT_PREFILL_FOLD)
            try:
                qg.set_option(qg.QG_OPT_PREFILL_FOLD, 1 if name.endswith("folded") else 0)
                r = mk()
                steps = args.sweep_steps if "512" not in name else max(20, args.sweep_steps // 20)
                res = measure(r, steps, 5, repeats=20)
                res["frac_of_hbm_peak"] = res["gbs"] / hbm_peak
                if "decode layer" in name and args.pdl != 1:
                    # The same four projections when each waits for the one
                    # before it (a decode chain whose inputs are outputs).
                    qg.set_option(qg.QG_OPT_PDL, 1)
                    dep = measure(r, steps, 5, repeats=20)
                    qg.set_option(qg.QG_OPT_PDL, args.pdl)
                    res["dependent_chain"] = {"us_per_call": dep["us_per_call"],
                                              "gbs": dep["gbs"],
                                              "frac_of_hbm_peak": dep["gbs"] / hbm_peak}
                if r.flops and "512" not in name:
                    # CUDA-core f32 FMAs: against the same ALU peak as the M = 8 line
                    res["alu_tflops"] = r.flops / (res["us_per_call"] * 1e6)
                    res["frac_of_alu_peak"] = res["alu_tflops"] / alu_peak
                if "512" in name:
                    # tensor-core prefill: fp16 MMAs, compared with the measured dense
                    # bf16 peak (fp16 and bf16 share one tensor-core rate)
                    res["tflops"] = r.flops / (res["us_per_call"] * 1e6)
                    res["frac_of_tensor_peak"] = res["tflops"] / tensor_peak
                    res["tensor_peak_tflops"] = tensor_peak
                sweep[name] = res
                del r
                torch.cuda.empty_cache()
            except Exception as e:  # report, keep going
                sweep[name] = {"error": str(e)[:200]}
            finally:
                qg.set_option(qg.QG_OPT_PREFILL_FOLD, fold_old)
        out["sweep"] = sweep
        if qg.device_error():
            raise RuntimeError("device error word set during the sweep")

    print(json.dumps(out), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
