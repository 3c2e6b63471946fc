"""Benchmark of the MXFP8 MoE layer training step on GB300.

One step = the whole hot path over one batch of the full-layer workload
(T=16384 tokens, H=5120, E=16 experts, FFN F=8192, top-1 softmax router on
N(0,1) logits): MXFP8 weight quantization (both layouts of W1|W3 and W2),
router, grouping map, fused quantize+permute, GEMM1 with fused SwiGLU, GEMM2,
combine, and the backward (gate gradient, gradient shuffle+quantize, dgrad2,
SwiGLU backward+quantize, wgrad2, dgrad1, input column quantize, wgrad1,
combine).  Metric: MoE layer fwd+bwd TFLOP/s (algorithmic GEMM FLOPs of the
real routed rows) and, on its own workload, MXFP8 quantize GB/s.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun (N > 1) every rank runs the same single-GPU step on its own
GPU (replicas: the path has no exchange step), timed between barriers, and
rank 0 prints one JSON line with the max time over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "MoE layer fwd+bwd TFLOP/s (MXFP8 grouped GEMM) and quantize GB/s, 1 GB300"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_PER_BF16 = 2.0   # nominal dense fp8 / bf16 tensor rate (4.5 / 2.25 PFLOP/s)


# DRAM traffic of the six grouped-GEMM launches of one full-layer step
# (dram__bytes_read.sum + dram__bytes_write.sum per launch, summed), from an
# ncu capture of those launches alone.  Valid only for the GEMM sources it was
# taken on (checked by hash); reported as null otherwise.
GEMM_TRAFFIC_BYTES_PER_STEP = 15727732480
GEMM_TRAFFIC_HOW = ("ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum -k regex:k_grouped_gemm_pair "
                    "-s 6 -c 6 on this full-size layer step (T=16384, H=5120, E=16, F=8192, top-1): "
                    "1.053x the algorithmic bytes")
GEMM_TRAFFIC_SOURCES = ("gemm_pair.cu", "gemm_shared.cuh", "common.cuh")
GEMM_TRAFFIC_SHA256 = "9961f9c43be866eea696926fe680ac362a578d4e6b27b747c1435e25eb015bfb"


def _gemm_sources_sha256():
    import hashlib
    h = hashlib.sha256()
    for f in GEMM_TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, "mxfp8_mixture_experts_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            return d, "measured"
        except Exception:
            pass
    return FALLBACK, "fallback"


def _peak_val(d, *keys):
    for k in keys:
        if k in d and isinstance(d[k], (int, float)):
            return float(d[k])
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,enforced.power.limit")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.first = 0

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def begin(self):
        """Mark the start of the timed region: only later samples count."""
        self.first = len(self.lines)

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, power, limit, reasons = [], [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        timed = self.lines[self.first:] or self.lines
        for ln in timed:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            try:
                power.append(float(parts[3]))
            except ValueError:
                pass
            if len(parts) > 9:
                try:
                    limit.append(float(parts[9]))
                except ValueError:
                    pass
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w": statistics.median(power) if power else None,
                "power_limit_w": max(limit) if limit else None, "reasons": sorted(reasons),
                "samples": len(sm), "interval_ms": 50}


# ----------------------------------------------------------------------------
# the step, launch by launch (the same C-ABI calls moe_layer_fwd/bwd make), on
# preallocated buffers, with CUDA events between launches
# ----------------------------------------------------------------------------
class LayerStep:
    def __init__(self, d, inp, dev, grad_elem=0, wgrad_bf16=False):
        import mxfp8_mixture_experts_gb300 as m
        self.grad_elem = grad_elem  # element format of the backward's gradient operands (0 E4M3, 1 E5M2)
        self.wgrad_cd = 0 if wgrad_bf16 else 1  # weight-gradient output: MX_OUT_BF16 or MX_OUT_F32
        wdt = torch.bfloat16 if wgrad_bf16 else torch.float32
        self.m = m
        self.L = m.lib()
        self.d = d
        self.dev = dev
        T, H, F, E, k = d.T, d.H, d.F, d.E, d.k
        R = m.moe_rows_cap(T, k, E)
        self.R = R
        sb = lambda r, c: m.mx_scale_bytes(r, c, 1)
        u8 = lambda n: torch.empty(int(n), dtype=torch.uint8, device=dev)
        self.inp = inp
        self.W13 = torch.cat([inp["W1"], inp["W3"]], dim=2).contiguous()
        self.W2 = inp["W2"]
        b = {}
        b["w13_rq"], b["w13_rs"] = u8(E * H * 2 * F), u8(sb(E * H, 2 * F))
        b["w13_cq"], b["w13_cs"] = u8(E * 2 * F * H), u8(sb(E * 2 * F, H))
        b["w2_rq"], b["w2_rs"] = u8(E * F * H), u8(sb(E * F, H))
        b["w2_cq"], b["w2_cs"] = u8(E * H * F), u8(sb(E * H, F))
        self.routed = inp.get("logits") is not None
        if self.routed:
            b["ids"] = torch.empty((T, k), dtype=torch.int32, device=dev)
            b["gate"] = torch.empty((T, k), dtype=torch.float32, device=dev)
        else:  # ids and gates given (no router launch)
            b["ids"] = inp["ids"].to(dev, torch.int32).contiguous()
            b["gate"] = inp["gate"].to(dev, torch.float32).contiguous()
        b["counts"] = torch.empty(E, dtype=torch.int32, device=dev)
        b["off"] = torch.empty(E + 1, dtype=torch.int32, device=dev)
        b["dst"] = torch.empty(T * k, dtype=torch.int32, device=dev)
        b["src"] = torch.empty(R, dtype=torch.int32, device=dev)
        self.map_ws_bytes = int(self.L.moe_permute_map_workspace_size(T, k, E))
        b["map_ws"] = u8(max(self.map_ws_bytes, 16))
        b["xq"], b["xs"] = u8(R * H), u8(sb(R, H))
        b["ab"] = torch.empty((R, 2 * F), dtype=torch.bfloat16, device=dev)
        b["hq"], b["hs"] = u8(R * F), u8(sb(R, F))
        b["y"] = torch.empty((R, H), dtype=torch.bfloat16, device=dev)
        b["out"] = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        b["d_gate"] = torch.empty((T, k), dtype=torch.float32, device=dev)
        b["dy_rq"], b["dy_rs"] = u8(R * H), u8(sb(R, H))
        b["dy_cq"], b["dy_cs"] = u8(H * R), u8(sb(H, R))
        b["dh"] = torch.empty((R, F), dtype=torch.float32, device=dev)
        b["dab_rq"], b["dab_rs"] = u8(R * 2 * F), u8(sb(R, 2 * F))
        b["dab_cq"], b["dab_cs"] = u8(2 * F * R), u8(sb(2 * F, R))
        b["h_cq"], b["h_cs"] = u8(F * R), u8(sb(F, R))
        b["dW2"] = torch.empty((E, F, H), dtype=wdt, device=dev)
        b["dxp"] = torch.empty((R, H), dtype=torch.bfloat16, device=dev)
        b["xp_cq"], b["xp_cs"] = u8(H * R), u8(sb(H, R))
        b["dW13"] = torch.empty((E, H, 2 * F), dtype=wdt, device=dev)
        b["dX"] = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        b["status"] = torch.zeros(1, dtype=torch.int32, device=dev)
        self.b = b
        self.p = {n: t.data_ptr() for n, t in b.items()}
        # (name, kind, algorithmic work) of every launch, in order
        self.launches = []

    def run(self, stream, events=None):
        """Enqueue one step; if ``events`` is a list, record an event after
        every launch (events[0] before the first)."""
        L, p, d, m = self.L, self.p, self.d, self.m
        T, H, F, E, k, R = d.T, d.H, d.F, d.E, d.k, self.R
        s = stream.cuda_stream
        x = self.inp["x"].data_ptr()
        dOut = self.inp["dOut"].data_ptr()
        logits = self.inp["logits"].data_ptr() if self.routed else None
        st = p["status"]
        ev = events

        def mark():
            if ev is not None:
                e = torch.cuda.Event(enable_timing=True)
                e.record(stream)
                ev.append(e)

        def chk(code, what):
            if code != 0:
                raise RuntimeError(f"{what}: {L.mx_status_string(code).decode()}")

        mark()
        chk(L.mx_quantize(self.W13.data_ptr(), E, H, 2 * F, 3, 1, 0, p["w13_rq"], p["w13_rs"], p["w13_cq"], p["w13_cs"], s), "q W13"); mark()
        chk(L.mx_quantize(self.W2.data_ptr(), E, F, H, 3, 1, 0, p["w2_rq"], p["w2_rs"], p["w2_cq"], p["w2_cs"], s), "q W2"); mark()
        if self.routed:
            chk(L.moe_route(logits, T, E, k, p["ids"], p["gate"], s), "route")
        mark()
        chk(L.moe_permute_map(p["ids"], T, k, E, R, p["counts"], p["off"], p["dst"], p["src"], p["map_ws"],
                              self.map_ws_bytes, st, s), "map"); mark()
        chk(L.moe_permute(2, x, None, T, H, k, p["dst"], p["src"], R, p["xq"], p["xs"], 1, s), "permute"); mark()
        chk(L.moe_gemm1_swiglu(p["xq"], p["xs"], p["w13_cq"], p["w13_cs"], p["off"], E, R, F, H, p["ab"], p["hq"],
                               p["hs"], st, s), "gemm1"); mark()
        ge = self.grad_elem
        chk(L.mx_grouped_gemm(0, p["hq"], p["hs"], p["w2_cq"], p["w2_cs"], p["off"], E, R, H, F, p["y"], 0, 0, 0, st, s),
            "gemm2"); mark()
        chk(L.moe_unpermute(p["y"], p["dst"], p["gate"], T, H, k, p["out"], s), "combine"); mark()
        chk(L.moe_gate_grad(dOut, p["y"], p["dst"], T, H, k, p["d_gate"], s), "gate grad"); mark()
        lim = p["off"] + 4 * E  # offsets[E]: the routed rows end there
        chk(L.moe_gather_quant(dOut, p["gate"], p["src"], T, H, k, R, 3, ge, p["dy_rq"], p["dy_rs"], p["dy_cq"],
                               p["dy_cs"], lim, s), "dY quant"); mark()
        chk(L.mx_grouped_gemm(1, p["dy_rq"], p["dy_rs"], p["w2_rq"], p["w2_rs"], p["off"], E, R, F, H, p["dh"], 1, ge, 0, st,
                              s), "dgrad2"); mark()
        chk(L.moe_swiglu_bwd(p["dh"], p["ab"], R, F, ge, p["dab_rq"], p["dab_rs"], p["dab_cq"], p["dab_cs"], p["h_cq"],
                             p["h_cs"], lim, s), "swiglu bwd"); mark()
        chk(L.mx_grouped_gemm(2, p["h_cq"], p["h_cs"], p["dy_cq"], p["dy_cs"], p["off"], E, R, F, H, p["dW2"], self.wgrad_cd, 0, ge, st,
                              s), "wgrad2"); mark()
        chk(L.mx_grouped_gemm(1, p["dab_rq"], p["dab_rs"], p["w13_rq"], p["w13_rs"], p["off"], E, R, H, 2 * F,
                              p["dxp"], 0, ge, 0, st, s), "dgrad1"); mark()
        chk(L.moe_gather_quant(x, None, p["src"], T, H, k, R, 2, 0, None, None, p["xp_cq"], p["xp_cs"], lim, s),
            "x col quant"); mark()
        chk(L.mx_grouped_gemm(2, p["xp_cq"], p["xp_cs"], p["dab_cq"], p["dab_cs"], p["off"], E, R, H, 2 * F,
                              p["dW13"], self.wgrad_cd, 0, ge, st, s), "wgrad1"); mark()
        chk(L.moe_unpermute(p["dxp"], p["dst"], None, T, H, k, p["dX"], s), "combine dX"); mark()

    NAMES = ["quantize W13", "quantize W2", "route", "map", "permute+quant", "gemm1+swiglu", "gemm2", "combine",
             "gate grad", "dY gather+quant", "dgrad2", "swiglu bwd", "wgrad2", "dgrad1", "x col quant", "wgrad1",
             "combine dX"]
    # our kernel launches per entry (the map is three kernels)
    KERNELS = [1, 1, 1, 3, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1]


def _gemm_flops(d, routed):
    T, H, F = routed, d.H, d.F
    g1 = 2 * T * H * 2 * F
    g2 = 2 * T * F * H
    return {"gemm1+swiglu": g1, "gemm2": g2, "dgrad2": g2, "wgrad2": g2, "dgrad1": g1, "wgrad1": g1}


def _gemm_alg_bytes(d, R):
    """Operands read once plus outputs written once, over the 6 GEMM launches
    of one step (R routed rows, fp8 data with 1/32 scale bytes)."""
    T, H, F, E = R, d.H, d.F, d.E
    q = 1 + 1 / 32
    g1 = (T * H + E * 2 * F * H) * q + T * 2 * F * 2 + T * F * q
    g2 = (T * F + E * H * F) * q + T * H * 2
    dg2 = (T * H + E * F * H) * q + T * F * 4
    wg2 = (F * T + H * T) * q + E * F * H * 4
    dg1 = (T * 2 * F + E * H * 2 * F) * q + T * H * 2
    wg1 = (H * T + 2 * F * T) * q + E * H * 2 * F * 4
    return int(g1 + g2 + dg2 + wg2 + dg1 + wg1)


def _quant_bench(dev, iters=20):
    """MXFP8 quantize, BOTH mode, bf16 [16384, 7168] with swizzled scales."""
    import mxfp8_mixture_experts_gb300 as m
    R, C = workloads.QUANTIZE_SHAPE
    x = workloads.quantize_input(R, C, seed=0, device=dev)
    outs = [torch.empty(R * C, dtype=torch.uint8, device=dev) for _ in range(2)]
    sc = [torch.empty(m.mx_scale_bytes(R, C, 1), dtype=torch.uint8, device=dev) for _ in range(2)]
    L = m.lib()
    s = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    times = []
    for i in range(iters + 3):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        code = L.mx_quantize(x.data_ptr(), 1, R, C, 3, 1, 0, outs[0].data_ptr(), sc[0].data_ptr(), outs[1].data_ptr(),
                             sc[1].data_ptr(), s.cuda_stream)
        e1.record(s)
        assert code == 0
        torch.cuda.synchronize()
        if i >= 3:
            times.append(e0.elapsed_time(e1) * 1e-3)
    t = statistics.median(times)
    nbytes = R * C * 2 + 2 * (R * C + R * C // 32)
    return {"GB/s": nbytes / t / 1e9, "us": t * 1e6, "bytes": nbytes, "l2": "flushed (256 MiB write) before each launch"}


def _dequant_bench(dev, iters=20):
    """MXFP8 dequantize of the quantize workload's ROW output (E4M3 [16384,
    7168] + swizzled scales) to bf16, each launch timed after an L2 flush."""
    import mxfp8_mixture_experts_gb300 as m
    R, C = workloads.QUANTIZE_SHAPE
    x = workloads.quantize_input(R, C, seed=0, device=dev)
    q, sc, _, _ = m.mx_quantize(x, m.MX_MODE_ROW, m.MX_SCALE_SWIZZLED)
    out = torch.empty((R, C), dtype=torch.bfloat16, device=dev)
    L = m.lib()
    s = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    times = []
    for i in range(iters + 3):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        code = L.mx_dequantize(q.data_ptr(), sc.data_ptr(), 1, R, C, 1, 0, 0, out.data_ptr(), s.cuda_stream)
        e1.record(s)
        assert code == 0
        torch.cuda.synchronize()
        if i >= 3:
            times.append(e0.elapsed_time(e1) * 1e-3)
    t = statistics.median(times)
    nbytes = R * C + R * C // 32 + 2 * R * C
    return {"GB/s": nbytes / t / 1e9, "us": t * 1e6, "bytes": nbytes, "out": "bf16",
            "l2": "flushed (256 MiB write) before each launch"}


def _rowmax_bench(dev, iters=20):
    """Row-max-scaled FP8 on the quantize workload (bf16 [16384, 7168]): the
    quantize kernel's GB/s after an L2 flush, and the accuracy of both schemes
    on the same data as SQNR of the decoded values against the bf16 input
    (MX: 32-element blocks with E8M0 scales, decoded by mx_dequantize; row
    max: E4M3 times the row's fp32 scale, decoded with torch for the
    comparison only)."""
    import mxfp8_mixture_experts_gb300 as m
    R, C = workloads.QUANTIZE_SHAPE
    x = workloads.quantize_input(R, C, seed=0, device=dev)
    L = m.lib()
    q = torch.empty((R, C), dtype=torch.uint8, device=dev)
    sc = torch.empty(R, dtype=torch.float32, device=dev)
    s = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    times = []
    for i in range(iters + 3):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        code = L.fp8_quantize_rowmax(x.data_ptr(), R, C, q.data_ptr(), sc.data_ptr(), s.cuda_stream)
        e1.record(s)
        assert code == 0
        torch.cuda.synchronize()
        if i >= 3:
            times.append(e0.elapsed_time(e1) * 1e-3)
    t = statistics.median(times)
    nbytes = R * C * 2 + R * C + R * 4
    xf = x.float()
    sig = (xf.double() ** 2).sum()
    rm = q.view(torch.float8_e4m3fn).float() * sc[:, None]
    mq, ms, _, _ = m.mx_quantize(x, m.MX_MODE_ROW, m.MX_SCALE_PLAIN)
    mxd = torch.empty((R, C), dtype=torch.float32, device=dev)
    assert L.mx_dequantize(mq.data_ptr(), ms.data_ptr(), 1, R, C, 0, 0, 1, mxd.data_ptr(), s.cuda_stream) == 0
    torch.cuda.synchronize()
    sqnr = lambda d: float(10 * torch.log10(sig / ((xf - d).double() ** 2).sum()))
    return {"GB/s": nbytes / t / 1e9, "us": t * 1e6, "bytes": nbytes, "sqnr_db_rowmax": sqnr(rm),
            "sqnr_db_mx": sqnr(mxd), "l2": "flushed (256 MiB write) before each launch",
            "what": "one fp32 scale per row (amax / 448), E4M3 elements; SQNR of decoded values vs the bf16 input, "
                    "beside MXFP8's on the same data"}


def _permute_bench(dev, iters=10):
    """Token permute / unpermute workload: T=32768 tokens, H=5120, E=16
    experts, top-4 Zipf(1.1) expert choice over 14 live experts (two empty).
    MXFP8 rows (E4M3 + plain scales) are scattered into 128-row-padded expert
    groups (swizzled scales out); the combine reads k bf16 rows per token and
    writes one.  Each launch timed with CUDA events after an L2 flush."""
    import mxfp8_mixture_experts_gb300 as m
    d = workloads.PERMUTE_DIMS
    T, H, E, k = d["T"], d["H"], d["E"], d["k"]
    inp = workloads.permute_inputs(T, H, E, k, seed=0, device=dev)
    xq, xs, _, _ = m.mx_quantize(inp["x"], m.MX_MODE_ROW, m.MX_SCALE_PLAIN)
    L = m.lib()
    counts, off, dst, src = m.moe_permute_map(inp["ids"], E)
    R = src.numel()
    out = torch.empty((R, H), dtype=torch.uint8, device=dev)
    out_s = torch.empty(m.mx_scale_bytes(R, H, m.MX_SCALE_SWIZZLED), dtype=torch.uint8, device=dev)
    y = workloads.randn_bf16((R, H), 1.0, workloads.generator(1, dev), dev)
    comb = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    s = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def timed(fn):
        ts = []
        for i in range(iters + 3):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            fn()
            e1.record(s)
            torch.cuda.synchronize()
            if i >= 3:
                ts.append(e0.elapsed_time(e1) * 1e-3)
        return statistics.median(ts)

    def perm():
        code = L.moe_permute(m.MX_PERMUTE_FP8, xq.data_ptr(), xs.data_ptr(), T, H, k, dst.data_ptr(), src.data_ptr(),
                             R, out.data_ptr(), out_s.data_ptr(), m.MX_SCALE_SWIZZLED, s.cuda_stream)
        assert code == 0

    def unperm():
        code = L.moe_unpermute(y.data_ptr(), dst.data_ptr(), inp["gate"].data_ptr(), T, H, k, comb.data_ptr(),
                               s.cuda_stream)
        assert code == 0

    t_p, t_u = timed(perm), timed(unperm)
    padded = int(off[E].item())
    row_b = H + H // 32
    pb = T * row_b + padded * row_b            # read each token once, write every padded group row
    ub = T * k * H * 2 + T * H * 2             # read k routed rows per token, write one
    return {"permute": {"GB/s": pb / t_p / 1e9, "us": t_p * 1e6, "bytes": pb, "padded_rows": padded},
            "unpermute": {"GB/s": ub / t_u / 1e9, "us": t_u * 1e6, "bytes": ub},
            "workload": f"T={T}, H={H}, E={E}, top-{k} Zipf(1.1) over {E - 2} live experts; MXFP8 rows in, "
                        f"128-row-padded groups out; combine of k bf16 rows per token",
            "l2": "flushed (256 MiB write) before each launch"}


def _gemm_bench(dev, args):
    """Grouped GEMM workload: E=8, 32768 routed rows in Zipf-sized groups (one
    empty), K=7168, N=2048; forward (bf16 out), dgrad (bf16 out) and wgrad
    (fp32 out), each timed with CUDA events after warm-up, L2 flushed before
    each launch."""
    import mxfp8_mixture_experts_gb300 as m
    d = workloads.GEMM_DIMS
    E, M, K, N = d["E"], d["M"], d["K"], d["N"]
    sizes = workloads.gemm_group_sizes(E, M, seed=0)
    inp = workloads.gemm_inputs(E, M, K, N, sizes, seed=0, device=dev)
    off = torch.tensor(np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32), device=dev)
    a_rq, a_rs, a_cq, a_cs = m.mx_quantize(inp["A"], m.MX_MODE_BOTH, m.MX_SCALE_SWIZZLED)
    w_rq, w_rs, w_cq, w_cs = m.mx_quantize(inp["W"], m.MX_MODE_BOTH, m.MX_SCALE_SWIZZLED)
    c_rq, c_rs, c_cq, c_cs = m.mx_quantize(inp["dC"], m.MX_MODE_BOTH, m.MX_SCALE_SWIZZLED)
    del inp
    C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    dA = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    dW = torch.empty((E, N, K), dtype=torch.float32, device=dev)
    ops = {
        "fwd": lambda: m.mx_grouped_gemm(m.MX_GEMM_FWD, a_rq, a_rs, w_cq, w_cs, off, E, M, N, K, m.MX_OUT_BF16, out=C),
        "dgrad": lambda: m.mx_grouped_gemm(m.MX_GEMM_DGRAD, c_rq, c_rs, w_rq, w_rs, off, E, M, K, N, m.MX_OUT_BF16,
                                           out=dA),
        "wgrad": lambda: m.mx_grouped_gemm(m.MX_GEMM_WGRAD, c_cq, c_cs, a_cq, a_cs, off, E, M, N, K, m.MX_OUT_F32,
                                           out=dW),
    }
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    s = torch.cuda.current_stream(dev)
    flops = 2 * M * N * K
    res = {}
    for name, fn in ops.items():
        times = []
        for i in range(max(args.warmup, 1) + max(args.steps, 1)):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            fn()
            e1.record(s)
            torch.cuda.synchronize()
            if i >= max(args.warmup, 1):
                times.append(e0.elapsed_time(e1) * 1e-3)
        t = statistics.median(times)
        res[name] = {"TFLOP/s": flops / t / 1e12, "us": t * 1e6}
    res["sizes"] = sizes
    res["flops_per_op"] = flops
    res["workload"] = (f"grouped GEMM: E={E}, {M} routed rows in Zipf(1.1) groups {sizes}, K={K}, N={N}; fwd and "
                       f"dgrad bf16 out, wgrad fp32 out")
    res["l2"] = "flushed (256 MiB write) before each launch"
    del a_rq, a_rs, a_cq, a_cs, w_rq, w_rs, w_cq, w_cs, c_rq, c_rs, c_cq, c_cs, C, dA, dW
    res["wgrad_splitk"] = _splitk_bench(dev, args)
    return res


def _tiny_layer_bench(dev, iters=20):
    """Tiny MoE layer workload (T=512, H=256, E=4, F=512, top-1 ids uniform
    over experts, gate 1): one fwd+bwd step of the same launches as the full
    layer (no router: the ids are given), each step timed with CUDA events
    after an L2 flush.  Launch- and latency-bound at this size, so the step
    is also captured once into a CUDA graph and timed as graph replays (the
    library makes no host synchronisation, so the whole step captures); the
    eager time is reported beside it."""
    import mxfp8_mixture_experts_gb300 as m
    dims = workloads.TINY_LAYER
    d = m.MoELayerDims(T=dims.T, H=dims.H, F=dims.F, E=dims.E, k=dims.k)
    inp = workloads.layer_inputs(dims, seed=0, device=dev, router="uniform")
    step = LayerStep(d, inp, dev)
    s = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def timed(fn):
        times = []
        for i in range(iters + 3):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            fn()
            e1.record(s)
            torch.cuda.synchronize()
            if i >= 3:
                times.append(e0.elapsed_time(e1) * 1e-3)
        return statistics.median(times)

    t_eager = timed(lambda: step.run(s))
    assert int(step.b["status"].item()) == 0
    side = torch.cuda.Stream(dev)
    side.wait_stream(s)
    with torch.cuda.stream(side):
        step.run(side)
    s.wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step.run(torch.cuda.current_stream(dev))
    t = timed(graph.replay)
    assert int(step.b["status"].item()) == 0
    flops = sum(_gemm_flops(d, dims.T * dims.k).values())
    return {"us_per_step": t * 1e6, "TFLOP/s": flops / t / 1e12, "flops": flops,
            "us_per_step_eager": t_eager * 1e6,
            "how": "CUDA graph of the step's launches, replayed (eager launches beside it)",
            "workload": f"tiny MoE layer fwd+bwd: T={dims.T}, H={dims.H}, E={dims.E}, F={dims.F}, top-1 ids "
                        f"uniform, gate 1", "launches": sum(LayerStep.KERNELS) - 1,
            "l2": "flushed (256 MiB write) before each step"}


def _bf16_layer_bench(dev, d, inp, steps, warmup):
    """Context for the pages' MoE-layer speedup claim: the same layer step
    (T, H, E, F, top-k from the same logits and inputs) in bf16 with plain
    PyTorch eager ops -- torch.mm per expert (cuBLAS bf16 GEMMs, fp32
    accumulation, bf16 outputs including the weight gradients), torch
    elementwise SwiGLU, index-based permute and combine.  Not part of the
    library; timed with CUDA events over the same number of steps."""
    T, H, F, E, k = d.T, d.H, d.F, d.E, d.k
    W13 = torch.cat([inp["W1"], inp["W3"]], dim=2).contiguous()       # [E, H, 2F]
    W2 = inp["W2"]                                                      # [E, F, H]
    x, dOut, logits = inp["x"], inp["dOut"], inp["logits"]
    dW13 = torch.empty_like(W13)
    dW2 = torch.empty_like(W2)

    def step():
        top = logits.topk(k, dim=1)
        ids = top.indices
        gate = torch.softmax(logits, dim=1).gather(1, ids)
        flat = ids.reshape(-1)
        order = torch.argsort(flat, stable=True)
        counts = torch.bincount(flat, minlength=E).tolist()
        tok = order // k
        xp = x.index_select(0, tok)
        g = gate.reshape(-1).index_select(0, order).to(torch.bfloat16).unsqueeze(1)
        dY = dOut.index_select(0, tok) * g
        out = torch.zeros_like(x)
        dX = torch.zeros_like(x)
        start = 0
        ys, dxps = [], []
        for e in range(E):
            n = counts[e]
            if n == 0:
                dW13[e].zero_()
                dW2[e].zero_()
                continue
            sl = slice(start, start + n)
            start += n
            ab = xp[sl] @ W13[e]
            a, b = ab[:, :F], ab[:, F:]
            sa = torch.sigmoid(a.float())
            h = (a.float() * sa * b.float()).to(torch.bfloat16)
            y = h @ W2[e]
            ys.append(y)
            dh = (dY[sl] @ W2[e].t()).float()
            dW2[e] = h.t() @ dY[sl]
            da = dh * b.float() * sa * (1 + a.float() * (1 - sa))
            db = dh * a.float() * sa
            dab = torch.cat([da, db], dim=1).to(torch.bfloat16)
            dxps.append(dab @ W13[e].t())
            dW13[e] = xp[sl].t() @ dab
        y = torch.cat(ys)
        out.index_add_(0, tok, y * g)
        dX.index_add_(0, tok, torch.cat(dxps))
        return out, dX

    s = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(steps):
        step()
    e1.record(s)
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) * 1e-3 / steps
    flops = sum(_gemm_flops(d, T * k).values())
    return {"ms_per_step": t * 1e3, "TFLOP/s": flops / t / 1e12,
            "what": "bf16 layer in plain PyTorch eager: torch.mm per expert (cuBLAS bf16, fp32 accumulation, bf16 "
                    "outputs incl. weight gradients), elementwise SwiGLU in fp32, index-based permute/combine; "
                    "context only, not part of the library"}


def _splitk_bench(dev, args):
    """Split-K wgrad (mx_grouped_gemm_wgrad_splitk) against the plain wgrad:
    on the grouped-GEMM workload (E=8, 32768 tokens in Zipf groups, N=2048,
    K=7168: 1792 output tiles, plenty for 74 CTA pairs) and on a few-tile
    case (E=2, tokens 30720 + 2048, N=K=1024: 32 output tiles), each launch
    after an L2 flush."""
    import mxfp8_mixture_experts_gb300 as m
    res = {}
    cases = {"grouped_gemm_workload": (workloads.gemm_group_sizes(8, 32768, seed=0), 2048, 7168),
             "few_tiles_E2_N1024_K1024": ([30720, 2048], 1024, 1024)}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    s = torch.cuda.current_stream(dev)
    g = workloads.generator(11, dev)
    for name, (sizes, N, K) in cases.items():
        E, M = len(sizes), sum(sizes)
        off = torch.tensor(np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32), device=dev)
        _, _, xq, xs = m.mx_quantize(workloads.randn_bf16((M, N), 1.0, g, dev), m.MX_MODE_COL, m.MX_SCALE_SWIZZLED)
        _, _, yq, ys = m.mx_quantize(workloads.randn_bf16((M, K), 1.0, g, dev), m.MX_MODE_COL, m.MX_SCALE_SWIZZLED)
        C = torch.empty((E, N, K), dtype=torch.float32, device=dev)
        ws = torch.empty(int(m.lib().mx_wgrad_splitk_workspace_size(E, N, K, 4)), dtype=torch.uint8, device=dev)
        flops = 2 * M * N * K
        row = {}
        for splits in (0, 1, 2, 4):
            def fn():
                if splits == 0:
                    m.mx_grouped_gemm(m.MX_GEMM_WGRAD, xq, xs, yq, ys, off, E, M, N, K, m.MX_OUT_F32, out=C)
                else:
                    m.mx_grouped_gemm_wgrad_splitk(xq, xs, yq, ys, off, E, M, N, K, splits, out=C, ws=ws)
            times = []
            for i in range(max(args.warmup, 1) + max(args.steps, 1)):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(s)
                fn()
                e1.record(s)
                torch.cuda.synchronize()
                if i >= max(args.warmup, 1):
                    times.append(e0.elapsed_time(e1) * 1e-3)
            t = statistics.median(times)
            row["plain" if splits == 0 else f"splits={splits}"] = {"us": t * 1e6, "TFLOP/s": flops / t / 1e12}
        row["sizes"] = sizes
        res[name] = row
    return res


def _cpu_baseline(d_full, seconds_hint=20.0):
    """The oracle (numpy, fp64) on a bounded sample of the full-layer workload:
    one expert at the full hidden size H, a 512-wide slice of its FFN width
    (W1/W3 columns and W2 rows, quantized both ways as a step does) and 128
    routed tokens, through forward and backward.  Returns TFLOP/s over the
    GEMM FLOPs of the sample."""
    from oracle import moe
    n, f_s = 256, 1024
    d = workloads.LayerDims(T=n, H=d_full.H, E=1, F=f_s, k=1)
    g = workloads.generator(0, "cpu")
    x = workloads.randn_bf16((n, d.H), 1.0, g, "cpu")
    W1 = workloads.randn_bf16((1, d.H, d.F), 0.02, g, "cpu")
    W3 = workloads.randn_bf16((1, d.H, d.F), 0.02, g, "cpu")
    W2 = workloads.randn_bf16((1, d.F, d.H), 0.02, g, "cpu")
    dOut = workloads.randn_bf16((n, d.H), 1.0, g, "cpu")
    ids = np.zeros((n, 1), np.int32)
    gate = np.ones((n, 1), np.float32)
    bits = {k_: workloads.bf16_bits(v) for k_, v in dict(x=x, W1=W1, W3=W3, W2=W2, dOut=dOut).items()}
    t0 = time.perf_counter()
    f = moe.layer_forward(bits["x"], bits["W1"], bits["W3"], bits["W2"], ids, gate, quant=True)
    moe.layer_backward(f, bits["x"], bits["W1"], bits["W3"], bits["W2"], bits["dOut"])
    t = time.perf_counter() - t0
    flops = moe.layer_flops(n, d.H, d.F)["total"]
    cores = len(os.sched_getaffinity(0))
    return {"value": flops / t / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"oracle layer fwd+bwd (numpy fp64, MXFP8 semantics): one expert, H={d.H}, a {f_s}-wide "
                      f"slice of F={d_full.F} (weights quantized both ways), {n} routed tokens; {t:.1f} s",
            "seconds": t}


def _fp8_peaks(peaks, clk):
    """Dense fp8 tensor peaks (2 x the measured cuBLAS bf16 rates, the nominal
    fp8/bf16 ratio) and the one this run is held to: the burst figure when
    the clock record of the timed region shows the SM clock at its maximum
    with no power cap, the sustained (power-capped) figure otherwise."""
    burst = (_peak_val(peaks, "bf16_tflops") or FALLBACK["bf16_tflops"]) * FP8_PER_BF16
    sust = (_peak_val(peaks, "bf16_tflops_sustained") or FALLBACK["bf16_tflops_sustained"]) * FP8_PER_BF16
    sm, smax = clk.get("sm_mhz"), clk.get("sm_max_mhz")
    capped = "sw_power_cap" in clk.get("reasons", [])
    at_max = sm is not None and smax and sm >= 0.97 * smax
    kind = "burst" if at_max and not capped else "sustained"
    return {"burst": burst, "sustained": sust, "kind": kind,
            "chosen": burst if kind == "burst" else sust, "other": sust if kind == "burst" else burst,
            "rule": "burst when the timed region's median SM clock is >= 97% of max and no sw_power_cap sample; "
                    "sustained otherwise"}


def _reduce_max(value: float, device) -> float:
    """The slowest rank's value (replicas: the job's time is the max over
    ranks); the value itself without an initialised process group."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-quant", action="store_true",
                    help="skip the per-workload kernel lines (quantize, permute, dequantize, grouped GEMM, tiny layer)")
    ap.add_argument("--no-bf16", action="store_true", help="skip the bf16 PyTorch layer timing (context)")
    ap.add_argument("--T", type=int, default=None, help="override the token count (profiling of small cases)")
    ap.add_argument("--E", type=int, default=None, help="override the expert count (profiling of small cases)")
    ap.add_argument("--k", type=int, default=None, help="override top-k (a variant; the bench line is top-1)")
    ap.add_argument("--grad-format", default="e4m3", choices=["e4m3", "e5m2"],
                    help="element format of the backward's gradient operands (a variant; the bench line is e4m3)")
    ap.add_argument("--wgrad-dtype", default="f32", choices=["f32", "bf16"],
                    help="weight gradients in fp32 or bf16 (a variant; the bench line is fp32)")
    ap.add_argument("--workload", default="layer",
                    choices=["layer", "gemm", "quantize", "dequantize", "permute", "rowmax"],
                    help="layer: the full training step (the bench line); gemm / quantize / dequantize / "
                         "permute: one kernel family on its own workload, for profiling")
    args = ap.parse_args()
    rank, world, local = _dist()
    if args.workload != "layer":
        dev = torch.device("cuda", local)
        torch.cuda.set_device(dev)
        if args.workload == "gemm":
            r = _gemm_bench(dev, args)
        elif args.workload == "permute":
            r = _permute_bench(dev, max(args.steps, 1))
        elif args.workload == "dequantize":
            r = _dequant_bench(dev, max(args.steps, 1))
        elif args.workload == "rowmax":
            r = _rowmax_bench(dev, max(args.steps, 1))
        else:
            r = _quant_bench(dev, max(args.steps, 1))
        print(json.dumps({"workload": args.workload, **r}))
        return

    dims = workloads.FULL_LAYER
    if args.T or args.E or args.k:
        dims = workloads.LayerDims(T=args.T or dims.T, H=dims.H, E=args.E or dims.E, F=dims.F, k=args.k or dims.k)
    config = {"workload": f"full MoE SwiGLU layer fwd+bwd: T={dims.T} tokens, H={dims.H}, E={dims.E} experts, "
                          f"F={dims.F}, top-{dims.k} softmax router on N(0,1) logits, MXFP8 on all expert GEMMs",
              "T": dims.T, "H": dims.H, "E": dims.E, "F": dims.F, "k": dims.k,
              "l2": "inputs larger than L2 (weights 4 GB, activations 168 MB per tensor); no flush",
              "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"}
    if args.grad_format != "e4m3":
        config["grad_format"] = args.grad_format
    if args.wgrad_dtype != "f32":
        config["wgrad_dtype"] = args.wgrad_dtype

    if args.impl == "reference":
        if rank != 0:
            return
        vals = []
        for i in range(args.warmup + args.steps):
            r = _cpu_baseline(dims)
            if i >= args.warmup:
                vals.append(r)
        v = statistics.median([r["value"] for r in vals])
        secs = sum(r["seconds"] for r in vals)
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": 1,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / len(vals),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic (seeded)", "config": config,
                "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": vals[0]["cores"], "kind": "oracle",
                                 "sample": vals[0]["sample"]},
                "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import mxfp8_mixture_experts_gb300 as m
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    d = m.MoELayerDims(T=dims.T, H=dims.H, F=dims.F, E=dims.E, k=dims.k)
    inp = workloads.layer_inputs(dims, seed=rank, device=dev, router="logits")
    step = LayerStep(d, inp, dev, grad_elem=1 if args.grad_format == "e5m2" else 0, wgrad_bf16=args.wgrad_dtype == "bf16")
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    for _ in range(args.warmup):
        step.run(stream)
    torch.cuda.synchronize()
    assert int(step.b["status"].item()) == 0, "device status set during warm-up"

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    all_events = []
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks.begin()
    t0.record(stream)
    for _ in range(args.steps):
        evs = []
        step.run(stream, evs)
        all_events.append(evs)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    elapsed = t0.elapsed_time(t1) * 1e-3
    elapsed = _reduce_max(elapsed, dev)
    assert int(step.b["status"].item()) == 0, "device status set during the timed steps"

    # the same step captured once into a CUDA graph and replayed: how much of
    # the step is launch overhead (context; the line's value is the eager run)
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step.run(side)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step.run(torch.cuda.current_stream(dev))
    graph.replay()
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    graph_ms = g0.elapsed_time(g1) / args.steps
    assert int(step.b["status"].item()) == 0, "device status set during the graph replays"
    del graph

    per = {n: [] for n in LayerStep.NAMES}
    for evs in all_events:
        for i, n in enumerate(LayerStep.NAMES):
            per[n].append(evs[i].elapsed_time(evs[i + 1]) * 1e-3)
    avg = {n: sum(v) / len(v) for n, v in per.items()}
    routed = int(step.b["counts"].sum().item())
    gf = _gemm_flops(d, routed)
    total_flops = sum(gf.values())
    ms = elapsed / args.steps * 1e3
    value = world * total_flops * args.steps / elapsed / 1e12

    peaks, src = _peaks()
    hbm = _peak_val(peaks, "hbm_gbs") or FALLBACK["hbm_gbs"]
    pk = _fp8_peaks(peaks, clk)
    gemm_time = sum(avg[n] for n in gf)
    gemm_tflops = total_flops / gemm_time / 1e12

    quant = perm = deq = gemm = tiny = bf16 = rowmax = None
    if not args.no_quant:
        quant = _quant_bench(dev)
        quant["frac"] = quant["GB/s"] / hbm
        quant["peak"] = hbm
        quant["peak_source"] = f"{src} hbm_gbs"
        perm = _permute_bench(dev)
        for key in ("permute", "unpermute"):
            perm[key]["frac"] = perm[key]["GB/s"] / hbm
        deq = _dequant_bench(dev)
        deq["frac"] = deq["GB/s"] / hbm
        rowmax = _rowmax_bench(dev)
        rowmax["frac"] = rowmax["GB/s"] / hbm
        gemm = _gemm_bench(dev, args)
        for op in ("fwd", "dgrad", "wgrad"):
            gemm[op]["frac_burst"] = gemm[op]["TFLOP/s"] / pk["burst"]
        gemm["peak"] = pk["burst"]
        gemm["peak_source"] = f"{src} bf16_tflops (burst: each launch timed alone) x {FP8_PER_BF16}"
        tiny = _tiny_layer_bench(dev)
    if not args.no_bf16:
        bf16 = _bf16_layer_bench(dev, d, inp, steps=min(args.steps, 10), warmup=2)
        bf16["mxfp8_speedup"] = bf16["ms_per_step"] / ms

    # the capture is of the default workload only: full sizes, top-1, E4M3 gradients
    default_work = (args.T is None and args.E is None and args.k in (None, 1) and args.grad_format == "e4m3"
                    and args.wgrad_dtype == "f32")
    traffic = (GEMM_TRAFFIC_BYTES_PER_STEP if default_work and GEMM_TRAFFIC_SHA256 == _gemm_sources_sha256()
               else None)
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp8",
            "dtype_detail": "E4M3 x E4M3 block-scaled (E8M0, 32-element blocks) MMAs accumulating in fp32",
            "data": "synthetic (seeded, random-init weights)", "config": config,
            "gpu_launches": args.steps * (sum(LayerStep.KERNELS) - (0 if step.routed else 1)),
            "clocks": clk,
            "roofline": {"bound": "tensor", "kernel": "k_grouped_gemm_pair (6 launches per step)",
                         "achieved": gemm_tflops, "peak": pk["chosen"], "unit": "TFLOP/s",
                         "frac": gemm_tflops / pk["chosen"], "peak_kind": pk["kind"],
                         "peak_other": pk["other"], "frac_vs_other": gemm_tflops / pk["other"],
                         "peak_rule": pk["rule"],
                         "traffic": traffic,
                         "traffic_unit": "DRAM bytes per step of the 6 GEMM launches",
                         "traffic_how": GEMM_TRAFFIC_HOW if traffic is not None else
                         "null: no ncu capture of the current GEMM sources on this workload",
                         "algorithmic_bytes": _gemm_alg_bytes(d, R=routed),
                         "peak_source": f"{src} bf16_tflops / bf16_tflops_sustained x {FP8_PER_BF16} (nominal "
                                        f"dense fp8/bf16 ratio)"},
            "value_excl_weight_prep": total_flops / (ms * 1e-3 - avg['quantize W13'] - avg['quantize W2']) / 1e12,
            "ms_per_step_cuda_graph": graph_ms,
            "kernels_ms": {n: round(v * 1e3, 4) for n, v in avg.items()},
            "gemm_tflops": {n: round(gf[n] / avg[n] / 1e12, 1) for n in gf},
            "gemm_frac": {n: round(gf[n] / avg[n] / 1e12 / pk["chosen"], 3) for n in gf},
            "quantize": quant,
            "permute": perm,
            "dequantize": deq,
            "rowmax_fp8": rowmax,
            "grouped_gemm": gemm,
            "tiny_layer": tiny,
            "bf16_layer_context": bf16,
            "routed_rows": routed}

    if not args.no_e2e:
        line["e2e"] = _e2e(m, d, dims, inp, dev, args, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = {k_: v for k_, v in _cpu_baseline(dims).items() if k_ != "seconds"}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def _e2e(m, d, dims, inp, dev, args, world):
    """The same step through the layer entry points (moe_layer_prep_weights,
    moe_layer_fwd, moe_layer_bwd), with every step's inputs (x, logits, dOut)
    copied in from pinned host memory and its results (out, dX, d_gate) read
    back to pinned host memory inside the timed region.  Host-to-device and
    device-to-host copies run on two streams of their own (the two directions
    overlap each other and the compute) into double-buffered device tensors:
    step i+1's inputs and step i-1's results move while step i computes.  The
    timed region ends when the last result has reached the host.  The weight
    gradients stay on the device (an optimizer would consume them there)."""
    W13 = torch.cat([inp["W1"], inp["W3"]], dim=2).contiguous()
    W2 = inp["W2"]
    wq = torch.empty(m.moe_layer_weights_size(d.H, d.F, d.E), dtype=torch.uint8, device=dev)
    ws = torch.empty(m.moe_layer_workspace_size(d), dtype=torch.uint8, device=dev)
    h_in = {"x": inp["x"].cpu().pin_memory(), "lg": inp["logits"].cpu().pin_memory(),
            "dO": inp["dOut"].cpu().pin_memory()}
    wdt = torch.bfloat16 if args.wgrad_dtype == "bf16" else torch.float32
    wcd = m.MX_OUT_BF16 if args.wgrad_dtype == "bf16" else m.MX_OUT_F32
    dW13 = torch.empty((d.E, d.H, 2 * d.F), dtype=wdt, device=dev)
    dW2 = torch.empty((d.E, d.F, d.H), dtype=wdt, device=dev)
    ids = torch.empty((d.T, d.k), dtype=torch.int32, device=dev)
    gate = torch.empty((d.T, d.k), dtype=torch.float32, device=dev)
    bufs = []
    for _ in range(2):
        b = {n: torch.empty_like(t, device=dev) for n, t in h_in.items()}
        b["out"] = torch.empty((d.T, d.H), dtype=torch.bfloat16, device=dev)
        b["dX"] = torch.empty_like(b["out"])
        b["dg"] = torch.empty((d.T, d.k), dtype=torch.float32, device=dev)
        bufs.append(b)
    h_out = [{n: torch.empty(bufs[0][n].shape, dtype=bufs[0][n].dtype).pin_memory() for n in ("out", "dX", "dg")}
             for _ in range(2)]
    s = torch.cuda.current_stream(dev)
    hs, ds = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    tev = lambda: torch.cuda.Event(enable_timing=True)
    # Each copy is split at the forward/backward boundary, so the pipeline
    # fills and drains with as little exposed copy time as the data allow:
    # the weight prep needs no step input and runs while x and logits arrive,
    # dOut arrives while the forward runs, and out leaves while the backward
    # runs; only dX and d_gate follow the last backward.
    in_fwd = [tev(), tev()]        # x, logits of the buffer copied in
    in_bwd = [tev(), tev()]        # dOut of the buffer copied in
    fwd_done = [tev(), tev()]      # forward on the buffer finished
    done = [tev(), tev()]          # backward on the buffer finished
    out_read = [tev(), tev()]      # results of the buffer copied out
    marks = []                     # per step: h2d (start, end), d2h out (start, end), d2h rest (start, end)

    def h2d(i, mk):
        b = bufs[i % 2]
        if i >= 2:
            hs.wait_event(done[i % 2])         # step i-2 no longer reads this buffer
        mk[0].record(hs)
        with torch.cuda.stream(hs):
            b["x"].copy_(h_in["x"], non_blocking=True)
            b["lg"].copy_(h_in["lg"], non_blocking=True)
            in_fwd[i % 2].record(hs)
            b["dO"].copy_(h_in["dO"], non_blocking=True)
        in_bwd[i % 2].record(hs)
        mk[1].record(hs)

    def compute(i):
        b = bufs[i % 2]
        if i >= 2:
            s.wait_event(out_read[i % 2])      # step i-2's results have left this buffer
        m.moe_layer_prep_weights(W13, W2, wq)
        s.wait_event(in_fwd[i % 2])
        m.moe_layer_fwd(b["x"], wq, d, ws, logits=b["lg"], ids=ids, gate=gate, out=b["out"])
        fwd_done[i % 2].record(s)
        s.wait_event(in_bwd[i % 2])
        m.moe_layer_bwd(b["x"], b["dO"], gate, wq, d, ws, dX=b["dX"], dW13=dW13, dW2=dW2, d_gate=b["dg"],
                        grad_elem=1 if args.grad_format == "e5m2" else 0, wgrad_dtype=wcd)
        done[i % 2].record(s)

    def d2h(i, mk):
        b, h = bufs[i % 2], h_out[i % 2]
        ds.wait_event(fwd_done[i % 2])
        mk[2].record(ds)
        with torch.cuda.stream(ds):
            h["out"].copy_(b["out"], non_blocking=True)
        mk[3].record(ds)
        ds.wait_event(done[i % 2])
        mk[4].record(ds)
        with torch.cuda.stream(ds):
            h["dX"].copy_(b["dX"], non_blocking=True)
            h["dg"].copy_(b["dg"], non_blocking=True)
        out_read[i % 2].record(ds)
        mk[5].record(ds)

    def run(k, start, record):
        hs.wait_event(start)
        ds.wait_event(start)
        mks = [[tev() for _ in range(6)] for _ in range(k)]
        h2d(0, mks[0])
        if k > 1:
            h2d(1, mks[1])
        for i in range(k):
            compute(i)
            d2h(i, mks[i])
            if i + 2 < k:
                h2d(i + 2, mks[i + 2])
        fin_h, fin_d = tev(), tev()
        fin_h.record(hs)
        fin_d.record(ds)
        s.wait_event(fin_h)
        s.wait_event(fin_d)
        if record:
            marks.extend(mks)

    st = tev()
    st.record(s)
    run(max(args.warmup, 1), st, False)
    torch.cuda.synchronize()
    e0, e1 = tev(), tev()
    e0.record(s)
    run(args.steps, e0, True)
    e1.record(s)
    torch.cuda.synchronize()
    el = e0.elapsed_time(e1) * 1e-3
    routed = d.T * d.k
    flops = sum(_gemm_flops(d, routed).values())
    h2d_b = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h_b = sum(t.numel() * t.element_size() for t in h_out[0].values())
    h2d_ms = statistics.mean(mk[0].elapsed_time(mk[1]) for mk in marks)
    d2h_ms = statistics.mean(mk[2].elapsed_time(mk[3]) + mk[4].elapsed_time(mk[5]) for mk in marks)
    return {"value": world * flops * args.steps / el / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d_b,
            "d2h_bytes_per_step": d2h_b, "ms_per_step": el / args.steps * 1e3,
            "h2d_ms_per_step": h2d_ms, "d2h_ms_per_step": d2h_ms,
            "h2d_GBps": h2d_b / h2d_ms / 1e6, "d2h_GBps": d2h_b / d2h_ms / 1e6,
            "copies": "pinned host <-> device, H2D and D2H on two streams of their own, double-buffered, inside "
                      "the timed region, each split at the fwd/bwd boundary (dOut in while the forward runs, out "
                      "back while the backward runs); weight gradients stay on the device"}


if __name__ == "__main__":
    main()
