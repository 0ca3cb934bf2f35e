#!/usr/bin/env python3
"""Benchmark of the PARO W4A8 linear layer (prologue + GEMM) on GB300.

One step = one forward of the layer's hot path over one batch of synthetic
input: pq_rotate_quant (fused rotate + quantise prologue) followed by pq_gemm
(the uint4 x e4m3 group GEMM; CUDA-core kernel at M <= 16, tcgen05 above).
Weights, tables and activations are resident in HBM when the timed region
starts; every step uses the next of several input copies whose total size is
more than twice the L2, so no step is served from L2.

Headline (the JSON line's value): the decode gate_up layer, M=1, K=5120,
N=17408, one partition -- microseconds per step (lower is better).  The other
workloads (M=4, 16, prefill M=2048, down-projection M=8192 K=8704 N=5120,
merged QKV M=512 with three rotations) are timed the same way and reported
under "workloads".

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl pq|reference]
For N > 1 launch with torchrun; ranks run independent replicas (the layer does
not shard across GPUs in this build) and rank 0 prints the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import pqgen  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
METRIC = "pq prologue+GEMM µs, TFLOP/s & HBM GB/s vs roofline at M=1/2048/8192"
HEADLINE = ("decode", 1)
EXTRA = [("decode", 4), ("decode", 16), ("prefill", None), ("down", None), ("qkv", None)]


def describe(name, M=None):
    c = dict(pqgen.CONFIGS[name])
    if M is not None:
        c["M"] = M
    labels = {"decode": "decode gate_up", "prefill": "prefill gate_up", "down": "down-proj",
              "qkv": "merged QKV", "tiny": "tiny"}
    return c, "%s M=%d K=%d N=%d P=%d" % (labels[name], c["M"], c["K"], c["N"], c["P"])


def algorithmic(c):
    """Bytes each kernel must move and the GEMM's flops (per step)."""
    M, K, N, P = c["M"], c["K"], c["N"], c["P"]
    G = K // 128
    gemm_bytes = N * K // 2 + 4 * G * N + P * M * K + 8 * P * M * G + 2 * M * N
    pro_bytes = 2 * M * K + 2 * P * K + P * 8 * (K // 2) * 8 + P * M * K + 8 * P * M * G
    return gemm_bytes, pro_bytes, 2.0 * M * N * K


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return dict(hbm=pk["hbm_gbs"], bf16=pk["bf16_tflops"],
                    bf16_sus=pk.get("bf16_tflops_sustained", pk["bf16_tflops"]), src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- our path
class Workload:
    def __init__(self, pq, torch, name, M, dev):
        self.c, self.label = describe(name, M)
        self.name = name if M is None else "%s:%d" % (name, M)
        c = self.c
        prob = pqgen.make_problem(**c)
        self.prob = prob
        rec, sz, w = pq.pq_pack(prob.qweight, prob.qzeros, prob.scales, prob.pairs, prob.theta)
        gemm_bytes, pro_bytes, flops = algorithmic(c)
        per_copy = w.nbytes + sz.nbytes + rec.nbytes + prob.x.nbytes + 2 * prob.cs.nbytes + \
            2 * c["M"] * c["N"] + c["P"] * c["M"] * c["K"]
        self.copies = max(2, min(16, -(-2 * L2_BYTES // per_copy) + 1))
        t = torch

        def u16(a):
            return t.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)

        self.w = [t.from_numpy(w).to(dev) for _ in range(self.copies)]
        self.sz = [u16(sz) for _ in range(self.copies)]
        self.rec = [t.from_numpy(rec).to(dev) for _ in range(self.copies)]
        self.cs = [u16(prob.cs) for _ in range(self.copies)]
        self.x = [u16(prob.x).view(t.bfloat16) for _ in range(self.copies)]
        P, M, K, N, G = c["P"], c["M"], c["K"], c["N"], c["K"] // 128
        self.a = [t.empty((P, M, K), dtype=t.uint8, device=dev) for _ in range(self.copies)]
        self.asg = [t.empty((P, G, M), dtype=t.float32, device=dev) for _ in range(self.copies)]
        self.rs = [t.empty((P, G, M), dtype=t.float32, device=dev) for _ in range(self.copies)]
        self.y = [t.empty((M, N), dtype=t.bfloat16, device=dev) for _ in range(self.copies)]
        self.pb1, self.pb2 = prob.pb1, prob.pb2
        self.gemm_bytes, self.pro_bytes, self.flops = gemm_bytes, pro_bytes, flops
        sms = torch_sms(t)
        if M_of(c) == 1 or (M_of(c) <= pq.pq_gemm_skinny_max_m() and 2 * (c["N"] // 128) < sms):
            self.gemm_kernel = "skinny"          # the kernel pq_gemm dispatches to
        elif M_of(c) <= pq.pq_gemm_skinny_max_m():
            self.gemm_kernel = "tcn"
        else:
            self.gemm_kernel = "tcgen05"

    def prologue(self, pq, i, stream):
        j = i % self.copies
        pq.pq_rotate_quant(self.x[j], self.rec[j], self.cs[j], a=self.a[j], asg=self.asg[j],
                           rs=self.rs[j], stream=stream)

    def producer_buffers(self, torch, dev):
        """Inputs and outputs of the fused producer (residual add + RMSNorm +
        rotate + quant), one set per input copy, allocated on first use."""
        if getattr(self, "res", None) is not None:
            return
        c, t = self.c, torch
        M, K = c["M"], c["K"]
        rng = np.random.default_rng(17)
        r = t.from_numpy(rng.standard_normal((M, K)).astype(np.float32) * np.float32(0.7)).to(t.bfloat16)
        g = t.from_numpy(rng.standard_normal(K).astype(np.float32) * np.float32(0.2)).to(t.bfloat16)
        self.res = [r.to(dev) for _ in range(self.copies)]
        self.gamma = [g.to(dev) for _ in range(self.copies)]
        self.res_out = [t.empty((M, K), dtype=t.bfloat16, device=dev) for _ in range(self.copies)]
        self.h = [t.empty((M, K), dtype=t.bfloat16, device=dev) for _ in range(self.copies)]
        # the silu-mul producer's merged gate/up input, for I = K
        yv = rng.standard_normal((M, 2 * K)).astype(np.float32) * np.float32(3.0)
        self.ygu = [t.from_numpy(yv).to(t.bfloat16).to(dev) for _ in range(self.copies)]
        self.act = [t.empty((M, K), dtype=t.bfloat16, device=dev) for _ in range(self.copies)]
        P, G = c["P"], K // 128
        # bytes the producer must move: x, residual, gamma, cs, records in;
        # new residual, normed rows, codes, scales and row-sums out
        self.prod_bytes = 2 * M * K * 2 + K * 2 + P * K * 2 + P * 8 * G * 64 * 8 + \
            2 * M * K * 2 + P * M * K + 2 * P * G * M * 4

    def producer(self, pq, i, stream):
        j = i % self.copies
        pq.pq_add_rms_rotate_quant(self.x[j], self.res[j], self.gamma[j], 1e-6, self.rec[j], self.cs[j],
                                   residual_out=self.res_out[j], h=self.h[j], a=self.a[j], asg=self.asg[j],
                                   rs=self.rs[j], stream=stream)

    def silu_producer(self, pq, i, stream):
        j = i % self.copies
        pq.pq_silu_mul_rotate_quant(self.ygu[j], self.rec[j], self.cs[j], act=self.act[j], a=self.a[j],
                                    asg=self.asg[j], rs=self.rs[j], stream=stream)

    def ptok_buffers(self, torch, dev):
        """The per-token path's bf16 rotated rows and token scales, one set per
        input copy, allocated on first use."""
        if getattr(self, "xr", None) is not None:
            return
        P, M, K = self.c["P"], self.c["M"], self.c["K"]
        self.xr = [torch.empty((P, M, K), dtype=torch.bfloat16, device=dev) for _ in range(self.copies)]
        self.As = [torch.empty((P, M), dtype=torch.float32, device=dev) for _ in range(self.copies)]

    def ptok_prologue(self, pq, i, stream):
        j = i % self.copies
        pq.pq_rotate_tokquant(self.x[j], self.rec[j], self.cs[j], xr=self.xr[j], a=self.a[j], As=self.As[j],
                              rs=self.rs[j], stream=stream)

    def ptok_gemm(self, pq, i, stream):
        j = i % self.copies
        pq.pq_gemm_ptok(self.a[j], self.As[j], self.rs[j], self.w[j], self.sz[j], self.pb1, self.pb2,
                        y=self.y[j], stream=stream)

    def int5_buffers(self, pq, torch, dev):
        """The same layer with int5 weights (same seed: the same activations
        and rotations), packed by pq_pack5, one set per input copy."""
        if getattr(self, "w5", None) is not None:
            return
        p5 = pqgen.make_problem(**self.c, bits=5)
        _, sz, w, whi = pq.pq_pack5(p5.qweight, p5.qzeros, p5.qweight_hi, p5.qzeros_hi, p5.scales, p5.pairs,
                                    p5.theta)
        u16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)
        self.w5 = [torch.from_numpy(w).to(dev) for _ in range(self.copies)]
        self.whi5 = [torch.from_numpy(whi).to(dev) for _ in range(self.copies)]
        self.sz5 = [u16(sz) for _ in range(self.copies)]
        self.gemm5_bytes = self.gemm_bytes + whi.nbytes

    def gemm5(self, pq, i, stream, fn=None):
        j = i % self.copies
        (fn or pq.pq_gemm5)(self.a[j], self.asg[j], self.rs[j], self.w5[j], self.whi5[j], self.sz5[j], self.pb1,
                            self.pb2, y=self.y[j], stream=stream)

    def gemm(self, pq, i, stream, fn=None):
        j = i % self.copies
        (fn or pq.pq_gemm)(self.a[j], self.asg[j], self.rs[j], self.w[j], self.sz[j], self.pb1,
                           self.pb2, y=self.y[j], stream=stream)

    def step(self, pq, i, stream):
        self.prologue(pq, i, stream)
        self.gemm(pq, i, stream)


def torch_sms(torch):
    return torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count


def M_of(c):
    return c["M"]


def _capture(torch, fn):
    """A CUDA graph of fn() (the library launches on torch's current stream,
    which is the capture stream inside the context)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def time_graph(torch, g, calls_per_replay, stream, min_ms=150.0, min_reps=5, max_reps=2000):
    """Replays graph g (already warm) back to back, one CUDA-event pair per
    replay on `stream`, for at least min_ms of device time and min_reps
    replays (the count is set from one probe replay).  Returns ms per call:
    (mean, median, best)."""
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    g.replay()
    b.record(stream)
    b.synchronize()
    n = int(min(max_reps, max(min_reps, min_ms / max(a.elapsed_time(b), 1e-3) + 1)))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for e0, e1 in ev:
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    per = [e0.elapsed_time(e1) / calls_per_replay for e0, e1 in ev]
    return float(np.mean(per)), float(np.median(per)), float(np.min(per))


def time_workload(pq, torch, wl, steps, warmup, stream, barrier=None, sampler=None):
    """Times exactly `steps` steps replayed from CUDA graphs (one graph holds one
    step per input copy, so consecutive steps never share inputs), then the two
    kernels on their own from graphs of the same shape.  Returns ms totals."""
    for i in range(max(warmup, wl.copies)):
        wl.step(pq, i, None)
    torch.cuda.synchronize()
    C = wl.copies
    g_full = _capture(torch, lambda: [wl.step(pq, j, None) for j in range(C)])
    rem = steps % C
    g_rem = _capture(torch, lambda: [wl.step(pq, j, None) for j in range(rem)]) if rem else None
    g_pro = _capture(torch, lambda: [wl.prologue(pq, j, None) for j in range(C)])
    g_gem = _capture(torch, lambda: [wl.gemm(pq, j, None) for j in range(C)])
    for _ in range(2):
        g_full.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if barrier:
        barrier()
    torch.cuda.synchronize()
    ctx = sampler if sampler is not None else _Null()
    with ctx:
        t0 = time.perf_counter()
        e0.record(stream)
        for _ in range(steps // C):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    if barrier:
        barrier()
    total_ms = e0.elapsed_time(e1)
    per, stats = {}, {}
    for key, g in (("pro", g_pro), ("gemm", g_gem)):
        g.replay()
        torch.cuda.synchronize()
        mean, med, best = time_graph(torch, g, C, stream)
        per[key] = mean
        stats[key] = (mean, med, best)

    def time_each(call):
        """ms per call of call(pq, j, None), from a graph of one call per copy"""
        for j in range(C):
            call(pq, j, None)
        torch.cuda.synchronize()
        g = _capture(torch, lambda: [call(pq, j, None) for j in range(C)])
        g.replay()
        torch.cuda.synchronize()
        return time_graph(torch, g, C, stream, min_ms=60.0)[0]

    # the fused producer (residual add + RMSNorm + rotate + quant) on its own
    wl.producer_buffers(torch, wl.x[0].device)
    per["prod"] = time_each(wl.producer)
    # the silu-mul producer on its own
    per["silu"] = time_each(wl.silu_producer)
    paths = time_gemm_paths(pq, torch, wl, stream) if wl.c["M"] <= 16 else {}
    out = dict(total_ms=total_ms, wall_s=wall, pro_ms=per["pro"], gemm_ms=per["gemm"], paths=paths,
               prod_ms=per["prod"], silu_ms=per["silu"], stats=stats)
    # the same GEMM on int5 weights
    wl.int5_buffers(pq, torch, wl.x[0].device)
    out["int5_gemm_ms"] = time_each(wl.gemm5)
    if wl.c["M"] <= 16:
        # the two int5 decode kernels on their own (pq_gemm5 takes one of them)
        out["int5_paths"] = {
            "tcn": time_each(lambda pq_, j, s: wl.gemm5(pq_, j, s, fn=pq_.pq_gemm5_tcn)),
            "skinny": time_each(lambda pq_, j, s: wl.gemm5(pq_, j, s, fn=pq_.pq_gemm5_skinny)),
        }
    if wl.c["M"] > 16:
        # the per-token activation-scale path: its two-pass prologue, then its GEMM
        wl.ptok_buffers(torch, wl.x[0].device)
        out["ptok_pro_ms"] = time_each(wl.ptok_prologue)
        out["ptok_gemm_ms"] = time_each(wl.ptok_gemm)
    return out


def time_gemm_paths(pq, torch, wl, stream):
    """GEMM-only time per launch (ms) of every kernel that accepts this M,
    each from a graph of one launch per input copy, replayed for at least
    60 ms."""
    M = wl.c["M"]
    paths = [("tc", pq.pq_gemm_tc)]
    if M <= pq.pq_gemm_skinny_max_m():
        paths += [("skinny", pq.pq_gemm_skinny), ("tcn", pq.pq_gemm_tcn)]
    out = {}
    for name, fn in paths:
        C = wl.copies
        g = _capture(torch, lambda: [wl.gemm(pq, j, None, fn) for j in range(C)])
        g.replay()
        torch.cuda.synchronize()
        out[name] = time_graph(torch, g, C, stream, min_ms=60.0)[0]
    return out


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        pass


def e2e_workload(pq, torch, wl, steps, warmup, stream, dev):
    """Same step through the public API from pinned host buffers: H2D of x,
    prologue + GEMM, D2H of y, all inside the timed region."""
    c = wl.c
    xh = torch.from_numpy(wl.prob.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    yh = torch.empty((c["M"], c["N"]), dtype=torch.bfloat16).pin_memory()

    def one(i):
        j = i % wl.copies
        wl.x[j].copy_(xh, non_blocking=True)
        wl.step(pq, i, stream)
        yh.copy_(wl.y[j], non_blocking=True)

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        one(i)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps, xh.numel() * 2, yh.numel() * 2


def e2e_graph_workload(pq, torch, wl, steps, warmup, stream, zero_copy=True):
    """The same step through the public graph API (PQLinear.make_graph): each
    replay moves x from pinned host memory to the GPU, runs the prologue and
    the GEMM, and moves y back to pinned host memory.  zero_copy: the prologue
    reads x from, and the GEMM writes y to, the pinned host buffers directly;
    otherwise two copy operations.  One layer and graph per weight copy,
    replayed round robin, so the weights stream from HBM as in the timed
    region."""
    c = wl.c
    xh = torch.from_numpy(wl.prob.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    yh = torch.empty((c["M"], c["N"]), dtype=torch.bfloat16).pin_memory()
    steps_fns = [pq.PQLinear.from_tables(wl.rec[j], wl.sz[j], wl.w[j], wl.cs[j], (wl.pb1, wl.pb2))
                 .make_graph(xh, yh, zero_copy=zero_copy) for j in range(wl.copies)]
    for i in range(max(warmup, wl.copies)):
        steps_fns[i % wl.copies]()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        steps_fns[i % wl.copies]()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one
# ncu capture of the kernel on the workload, with the SHA-256 of the kernel's
# sources (concatenated in the listed order, comments removed) at capture time.  The figure is
# reported only while those sources are unchanged; otherwise traffic is null.
_CSRC = "w4a8_rotated_int4_gb300/csrc/"
NCU_TRAFFIC = {
    ("pq_gemm_skinny", "decode:1"): dict(
        bytes=47382528 + 0,
        src=[_CSRC + "pq_gemm_skinny.cu", _CSRC + "pq_device.cuh"],
        sha256="8ae33f144b01316d9ba3ed44a5a901a7adf157283aa932cb99984aba391671e7"),
    ("pq_gemm_tc", "prefill"): dict(
        bytes=72359936 + 38439168,
        src=[_CSRC + "pq_gemm_tc.cu", _CSRC + "pq_tcgen05.cuh", _CSRC + "pq_device.cuh"],
        sha256="8ddafd2a536289b0a8ed5973aaf82ef1ef18b8b88f9c1915bad3b72b25c01b08"),
    ("pq_gemm_tc", "down"): dict(
        bytes=99625472 + 54697728,
        src=[_CSRC + "pq_gemm_tc.cu", _CSRC + "pq_tcgen05.cuh", _CSRC + "pq_device.cuh"],
        sha256="8ddafd2a536289b0a8ed5973aaf82ef1ef18b8b88f9c1915bad3b72b25c01b08"),
    ("pq_gemm_tc", "qkv"): dict(
        bytes=30699520 + 768,
        src=[_CSRC + "pq_gemm_tc.cu", _CSRC + "pq_tcgen05.cuh", _CSRC + "pq_device.cuh"],
        sha256="8ddafd2a536289b0a8ed5973aaf82ef1ef18b8b88f9c1915bad3b72b25c01b08"),
    ("pq_gemm_tcn", "decode:16"): dict(
        bytes=47479552 + 512,
        src=[_CSRC + "pq_gemm_tcn.cu", _CSRC + "pq_tcgen05.cuh", _CSRC + "pq_device.cuh"],
        sha256="2d7ff27b4dafff28166a5aa77267241f542efa9f11d7e8942924852fa83fd60a"),
}


def sources_sha256(files):
    """SHA-256 of the listed sources with their comments and blank lines
    removed, so a comment-only edit keeps the captured traffic valid while any
    change to the code voids it."""
    import hashlib
    import re
    m = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "r", encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        lines = [ln.rstrip() for ln in text.splitlines() if ln.strip()]
        m.update("\n".join(lines).encode())
    return m.hexdigest()


def ncu_traffic(kernel, workload):
    e = NCU_TRAFFIC.get((kernel, workload))
    if e is None:
        return None
    if sources_sha256(e["src"]) != e["sha256"]:
        return None
    return e["bytes"]


KERNEL_NAMES = {"skinny": "pq_gemm_skinny", "tcn": "pq_gemm_tcn", "tcgen05": "pq_gemm_tc"}


# Dense FP8 MMA throughput per SM and clock: an isolated probe kernel issued
# tcgen05 m128n128k32 e4m3 MMAs back to back at one per 64 cycles
# (2 * 128 * 128 * 32 / 64 = 16384 FLOP per cycle per SM).
FP8_FLOP_PER_CLK_SM = 16384


def roofline(wl, r, peaks, traffic=None, sm_mhz=None, sms=None):
    if wl.gemm_kernel in ("skinny", "tcn"):      # decode band: weights streamed once
        achieved = wl.gemm_bytes / (r["gemm_ms"] * 1e-3) / 1e9
        return {"kernel": KERNEL_NAMES[wl.gemm_kernel], "bound": "hbm", "achieved": round(achieved, 1),
                "peak": peaks["hbm"], "unit": "GB/s", "frac": round(achieved / peaks["hbm"], 4),
                "peak_source": peaks["src"] + " (hbm_gbs)", "traffic": traffic}
    fp8_peak = 2.0 * peaks["bf16"]
    achieved = wl.flops / (r["gemm_ms"] * 1e-3) / 1e12
    out = {"kernel": "pq_gemm_tc", "bound": "tensor", "achieved": round(achieved, 1),
           "peak": round(fp8_peak, 1), "unit": "TFLOP/s", "frac": round(achieved / fp8_peak, 4),
           "peak_source": peaks["src"] + " bf16_tflops x 2 (dense fp8 : bf16 nominal ratio)",
           "traffic": traffic}
    if sm_mhz and sms:
        # the same against the FP8 rate the tensor cores reach at the SM clock
        # sampled during this workload's timing
        clk_peak = FP8_FLOP_PER_CLK_SM * sms * sm_mhz * 1e6 / 1e12
        out["peak_at_sampled_clock"] = round(clk_peak, 1)
        out["frac_at_sampled_clock"] = round(achieved / clk_peak, 4)
    return out


def summarize(wl, r, steps, peaks, clocks=None, sms=None):
    step_us = r["total_ms"] * 1e3 / steps
    st = r.get("stats", {})
    return {
        "workload": wl.label, "us_per_step": round(step_us, 3),
        "prologue_us": round(r["pro_ms"] * 1e3, 3), "gemm_us": round(r["gemm_ms"] * 1e3, 3),
        # per-launch times over the replays: mean (used above), median, best
        "prologue_us_median_best": [round(v * 1e3, 3) for v in st["pro"][1:]] if "pro" in st else None,
        "gemm_us_median_best": [round(v * 1e3, 3) for v in st["gemm"][1:]] if "gemm" in st else None,
        "gemm_kernel": wl.gemm_kernel,
        "gemm_tflops": round(wl.flops / (r["gemm_ms"] * 1e-3) / 1e12, 2),
        "gemm_gbs": round(wl.gemm_bytes / (r["gemm_ms"] * 1e-3) / 1e9, 1),
        "prologue_gbs": round(wl.pro_bytes / (r["pro_ms"] * 1e-3) / 1e9, 1),
        # the fused producer (residual add + RMSNorm + rotate + quant) alone
        "producer_us": round(r["prod_ms"] * 1e3, 3),
        "producer_gbs": round(wl.prod_bytes / (r["prod_ms"] * 1e-3) / 1e9, 1),
        # the silu-mul producer (silu(gate) * up + rotate + quant, I = K) alone
        "silu_producer_us": round(r["silu_ms"] * 1e3, 3),
        "roofline": roofline(wl, r, peaks, ncu_traffic(KERNEL_NAMES[wl.gemm_kernel], wl.name),
                             (clocks or {}).get("sm_mhz"), sms),
        "clocks": clocks,
        # per-token activation scales (M > 16): prologue (two passes) and GEMM
        "ptok": ({"prologue_us": round(r["ptok_pro_ms"] * 1e3, 3), "gemm_us": round(r["ptok_gemm_ms"] * 1e3, 3),
                  "gemm_tflops": round(wl.flops / (r["ptok_gemm_ms"] * 1e-3) / 1e12, 2),
                  "gemm_frac_fp8": round(wl.flops / (r["ptok_gemm_ms"] * 1e-3) / 1e12 / (2 * peaks["bf16"]), 4),
                  "step_us": round((r["ptok_pro_ms"] + r["ptok_gemm_ms"]) * 1e3, 3)}
                 if "ptok_pro_ms" in r else None),
        # int5 weights (W5A8): the GEMM alone, bytes incl. the fifth-bit planes
        "int5": {"gemm_us": round(r["int5_gemm_ms"] * 1e3, 3),
                 "gemm_gbs": round(wl.gemm5_bytes / (r["int5_gemm_ms"] * 1e-3) / 1e9, 1),
                 "gemm_tflops": round(wl.flops / (r["int5_gemm_ms"] * 1e-3) / 1e12, 2),
                 "vs_int4_time": round(r["int5_gemm_ms"] / r["gemm_ms"], 3),
                 "gemm_us_by_kernel": {k: round(v * 1e3, 3) for k, v in r.get("int5_paths", {}).items()}},
        "copies": wl.copies,
        "gemm_us_by_kernel": {k: round(v * 1e3, 3) for k, v in r.get("paths", {}).items()},
    }


# ---------------------------------------------------------------- oracle timing
class OracleSample:
    """The CPU oracle (as it stands) on a bounded sample of the workload: the
    prologue for a slice of the tokens and the fp64 GEMM for a slice of the
    output columns, both scaled to the whole workload.  The slices are sized
    so one step takes about `step_budget_s`.  Inputs are generated and packed
    once."""

    def __init__(self, name, M=None, step_budget_s=1.0, threads=None):
        import oracle
        self.oracle = oracle
        self.threads = threads
        self._use_threads()
        c, self.label = describe(name, M)
        self.c = c
        self.prob = pqgen.make_problem(**c)
        self.tab = oracle.pack(self.prob)
        N, Mt = c["N"], c["M"]
        # token slice for the prologue: halve until it fits half the budget
        self.mtok = Mt
        while True:
            t = self._time_prologue()
            if t <= step_budget_s / 2 or self.mtok == 1:
                break
            self.mtok = max(1, self.mtok // 2)
        self.a, self.asg, self.rs = self.oracle.rotate_quant(self.prob.x, self.prob.cs, self.tab["rec"])
        # column slice for the GEMM (all tokens, codes from the full prologue)
        self.ncols = 8
        while True:
            self._slice()
            t = self._gemm()
            if t > step_budget_s / 4 or self.ncols >= N:
                break
            self.ncols = min(N, self.ncols * 2)
        while self.ncols > 8 and t > step_budget_s / 2:
            self.ncols //= 2
            self._slice()
            t = self._gemm()

    def _time_prologue(self):
        x = np.ascontiguousarray(self.prob.x[:self.mtok])
        t0 = time.perf_counter()
        self.oracle.rotate_quant(x, self.prob.cs, self.tab["rec"])
        return time.perf_counter() - t0

    def _slice(self):
        self.codes = np.ascontiguousarray(self.tab["codes"][:, :self.ncols])
        self.sz = np.ascontiguousarray(self.tab["sz"][:, :self.ncols])

    def _gemm(self):
        pb = min(self.prob.pb1, self.ncols), min(self.prob.pb2, self.ncols)
        t0 = time.perf_counter()
        self.oracle.gemm_f64(self.a, self.asg, self.rs, self.codes, self.sz, pb[0], pb[1])
        return time.perf_counter() - t0

    def _use_threads(self):
        if self.threads is not None:
            self.oracle.set_num_threads(self.threads)

    def step_us(self):
        self._use_threads()
        t_pro = self._time_prologue() * (self.c["M"] / self.mtok)
        t_g = self._gemm() * (self.c["N"] / self.ncols)
        return (t_pro + t_g) * 1e6

    def describe(self):
        return ("prologue on %d of %d tokens + fp64 GEMM on %d of %d output columns per step, "
                "both scaled to the whole workload" % (self.mtok, self.c["M"], self.ncols, self.c["N"]))

    def cores(self):
        """Threads the sample actually keeps busy: the oracle's loops are
        parallel over tokens (the prologue over partitions x tokens), so a
        decode workload of one token runs on one thread whatever the pool."""
        self._use_threads()
        P = 1 + (self.prob.pb1 < self.c["N"]) + (self.prob.pb2 < self.c["N"])
        width = max(self.c["M"], P * self.mtok)
        return min(self.oracle.num_threads(), width)


def cpu_model():
    """The host CPU's model from /proc/cpuinfo (Arm cores report implementer
    and part numbers instead of a model name)."""
    try:
        info = open("/proc/cpuinfo").read()
    except OSError:
        return "unknown"
    fields = {}
    for line in info.splitlines():
        k, _, v = line.partition(":")
        fields.setdefault(k.strip(), v.strip())
    if fields.get("model name"):
        return fields["model name"]
    parts = {("0x41", "0xd4f"): "Arm Neoverse-V2", ("0x41", "0xd40"): "Arm Neoverse-V1",
             ("0x41", "0xd0c"): "Arm Neoverse-N1"}
    imp, part = fields.get("CPU implementer"), fields.get("CPU part")
    if imp and part:
        return parts.get((imp, part), "Arm implementer %s part %s" % (imp, part))
    return "unknown"


def cpu_baseline(name, M, budget_s=4.0, reps=3):
    """The oracle on the host cores: all hardware threads (OpenMP) and one
    thread, each on a bounded sample of the workload scaled to the whole
    workload; median and best of `reps` steps."""
    import oracle
    n_all = oracle.num_threads()
    out = {}
    for key, threads, budget in (("all", n_all, budget_s), ("single", 1, budget_s / 2)):
        orc = OracleSample(name, M, step_budget_s=budget, threads=threads)
        v = [orc.step_us() for _ in range(reps)]
        out[key] = dict(median=float(np.median(v)), best=float(np.min(v)), cores=orc.cores(),
                        sample=orc.describe())
    oracle.set_num_threads(n_all)
    a, one = out["all"], out["single"]
    return {"value": round(a["median"], 1), "unit": "us", "cores": a["cores"], "threads_in_pool": n_all,
            "kind": "oracle",
            "sample": a["sample"] + ", median of %d" % reps, "best": round(a["best"], 1),
            "cpu_model": cpu_model(),
            "single_thread": {"value": round(one["median"], 1), "best": round(one["best"], 1), "cores": 1,
                              "sample": one["sample"] + ", median of %d" % reps}}


# ---------------------------------------------------------------- main
def dist_init(backend="nccl"):
    """(rank, world size, torch.distributed or None).  Ranks are replicas:
    the layer needs no exchange, so the only collectives are the barriers
    around the timed region and the max of the per-rank times."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, None
    import torch.distributed as dist
    rank = int(os.environ.get("RANK", "0"))
    dist.init_process_group(backend=backend)
    return rank, ws, dist


def combine_ranks(total_ms, steps, ws, dist, device):
    """The job's time for `steps` steps is the slowest rank's; the reported
    value is that time per step divided by the number of replicas (each ran
    `steps` steps, so the whole job finished ws * steps of them)."""
    if dist:
        import torch
        t = torch.tensor([total_ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    step_us = total_ms * 1e3 / steps
    return total_ms, step_us / ws


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["pq", "reference"], default="pq")
    ap.add_argument("--extra-steps", type=int, default=50)
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--workload", default="decode:1",
                    help="headline workload NAME[:M], NAME in %s" % ", ".join(pqgen.CONFIGS))
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    rank, ws, dist = dist_init()
    name, _, m_txt = args.workload.partition(":")
    M = int(m_txt) if m_txt else None
    if name not in pqgen.CONFIGS:
        raise SystemExit("unknown workload %r" % name)

    if args.impl == "reference":
        if rank != 0:
            return
        # the whole --warmup W --steps K run stays near 90 s of host time
        orc = OracleSample(name, M, step_budget_s=min(1.0, 90.0 / max(1, args.steps + args.warmup)))
        per_step = []
        for i in range(args.warmup + args.steps):
            us = orc.step_us()
            if i >= args.warmup:
                per_step.append(us)
        v = float(np.mean(per_step))
        cores, desc, label = orc.cores(), orc.describe(), orc.label
        line = {"impl": "reference", "metric": METRIC, "value": round(v, 1), "unit": "us",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(v / 1e3, 3), "higher_is_better": False, "scaling": "weak",
                "vs_baseline": None, "dtype": "f32 prologue, f64 GEMM (CPU oracle)",
                "data": "synthetic", "config": {"workload": label},
                "cpu_baseline": {"value": round(v, 1), "unit": "us", "cores": cores,
                                 "kind": "oracle", "sample": desc, "cpu_model": cpu_model()},
                "e2e": {"value": round(v, 1), "unit": "us", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import torch
    import w4a8_rotated_int4_gb300 as pq
    import __graft_entry__
    __graft_entry__.build_library()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    peaks = load_peaks()
    barrier = (lambda: dist.barrier()) if dist else None

    wl = Workload(pq, torch, name, M, dev)
    sms = torch_sms(torch)
    sampler = ClockSampler(local) if rank == 0 else None
    r = time_workload(pq, torch, wl, args.steps, args.warmup, stream, barrier, sampler)
    total_ms, value = combine_ranks(r["total_ms"], args.steps, ws, dist, dev)
    step_us = total_ms * 1e3 / args.steps
    e2e_ms, h2d, d2h = (None, 0, 0) if args.no_e2e else e2e_workload(
        pq, torch, wl, max(50, args.steps // 10), args.warmup, stream, dev)
    e2e_graph_ms = None if args.no_e2e else e2e_graph_workload(
        pq, torch, wl, max(50, args.steps // 10), args.warmup, stream, zero_copy=True)
    e2e_copy_ms = None if args.no_e2e else e2e_graph_workload(
        pq, torch, wl, max(50, args.steps // 10), args.warmup, stream, zero_copy=False)
    clocks = sampler.summary() if sampler else {}
    head = summarize(wl, dict(r, total_ms=total_ms), args.steps, peaks, clocks, sms)

    extra = []
    if not args.no_extra:
        for en, em in EXTRA:
            if (en, em) == (name, M):
                continue
            w2 = Workload(pq, torch, en, em, dev)
            # clocks sampled over this workload's whole timing (steps and kernels)
            s2 = ClockSampler(local) if rank == 0 else None
            with (s2 if s2 is not None else _Null()):
                r2 = time_workload(pq, torch, w2, args.extra_steps, args.warmup, stream, barrier)
            extra.append(summarize(w2, r2, args.extra_steps, peaks, s2.summary() if s2 else None, sms))
            del w2
            torch.cuda.empty_cache()

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "us", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_us / 1e3, 6),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32 prologue; e4m3 x u4 tensor/CUDA-core MMA, f32 accumulate; bf16 out",
        "data": "synthetic",
        "config": {"workload": wl.label, "M": wl.c["M"], "K": wl.c["K"], "N": wl.c["N"],
                   "P": wl.c["P"], "parallelism": "replicas" if ws > 1 else "single GPU",
                   "l2": "%d rotating input copies (> 2x L2)" % wl.copies},
        "prologue_us": head["prologue_us"], "gemm_us": head["gemm_us"],
        "producer_us": head["producer_us"], "silu_producer_us": head["silu_producer_us"],
        "roofline": head["roofline"],
        "gemm_us_by_kernel": head["gemm_us_by_kernel"],
        "int5": head["int5"],
        "e2e": None if e2e_ms is None else {
            "value": round(e2e_graph_ms * 1e3, 3), "unit": "us", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "how": "public API PQLinear.make_graph(zero_copy=True): one CUDA "
            "graph replay per step = pq_rotate_quant reading x from pinned host memory + pq_gemm "
            "writing y to pinned host memory (the bytes cross the host link inside the kernels); "
            "one graph per weight copy, round robin",
            "copy_graph_value": round(e2e_copy_ms * 1e3, 3),
            "copy_graph_how": "make_graph(zero_copy=False): the same graph with a pinned H2D copy of x "
            "before the prologue and a D2H copy of y after the GEMM",
            "eager_value": round(e2e_ms * 1e3, 3),
            "eager_how": "public API per step, host-driven: pinned H2D of x, pq_rotate_quant + "
            "pq_gemm, D2H of y"},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "workloads": extra,
        "peaks": peaks,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(name, M)
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
