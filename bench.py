"""Benchmark of the FP8 SwiGLU FFN block on GB300.

One step = one pass of the whole prefill chain (fused residual + RMSNorm +
abs-max, quantisation, gate|up GEMM with the SwiGLU epilogue, requantisation,
down GEMM) over the Llama-3-8B FFN workload: N = 8 x 2048 = 16384 tokens,
C = 4096, H = 14336, seeded synthetic data.  The metric is GEMM TFLOP/s
(2*N*C*2H + 2*N*H*C FLOP per step).  The same line carries the single-token
decode FFN (GB/s of weights + scales + x + out streamed per call) under
"decode".

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Multi-GPU runs (torchrun) are independent replicas: every rank runs the whole
workload on its own GPU, no data crosses ranks, value = all ranks' work / the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from ffn_inputs import DECODE, PREFILL, decode_inputs, prefill_inputs  # noqa: E402

PREFILL_CFG = PREFILL["llama3-8b"]
DECODE_LAYERS = 32      # decoder layers of Llama-3-8B: one decode token runs 32 FFNs
DECODE_CFG = DECODE["llama3-8b-decode"]
METRIC = "FP8 SwiGLU-FFN fwd TFLOP/s (8B shape, 16k tok)"
DECODE_METRIC = "M=1 decode FFN HBM GB/s"
L2_BYTES = 129 * 1024 * 1024
FP8_PER_BF16 = 2.0          # nominal dense FP8 / BF16 tensor rate ratio
# DRAM bytes (read + write) per launch of the dominant kernels, from one ncu
# capture of this benchmark's full-size workload (dram__bytes_read.sum +
# dram__bytes_write.sum).  Set to None whenever the kernel changes until it
# is captured again.
TRAFFIC_GATE_UP_BYTES = (553.4 + 443.9) * 1e6
TRAFFIC_DUAL_GEMV_BYTES = (117.6 + 0.0) * 1e6


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "sm_max_mhz": float(p.get("sm_max_mhz", 0.0)) or None, "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


# ---------------------------------------------------------------- distributed plumbing
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        return rank, local, world, dist
    return rank, local, world, None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def job_throughput(units_per_rank: float, world: int, ms_slowest: float, scale: float = 1e12):
    """Whole-job throughput of `world` replicas: every rank's units / the slowest rank's time."""
    return units_per_rank * world / (ms_slowest * 1e-3) / scale


def max_over_ranks(dist, v: float) -> float:
    if dist is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        with open(self.file.name) as f:
            lines = [l.strip() for l in f if l.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in lines:
            p = [x.strip() for x in l.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                smax.append(float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        under_load = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(under_load), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- device helpers
def to_dev(a, torch, device):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.int16)
    return t.to(device)


def prefill_setup(q, torch, device, cfg=None):
    cfg = cfg or PREFILL_CFG
    inp = prefill_inputs(cfg)
    N, C, H = cfg.N, cfg.C, cfg.H
    d = {}
    d["res"] = to_dev(inp["res"], torch, device)
    d["x"] = to_dev(inp["x"], torch, device)
    d["gain"] = to_dev(inp["gain"], torch, device)
    wstats = torch.zeros(4, dtype=torch.float32, device=device)
    d["w1"] = torch.empty(2 * H, C, dtype=torch.uint8, device=device)
    d["w2"] = torch.empty(C, H, dtype=torch.uint8, device=device)
    for w, src, st in ((d["w1"], inp["w1"], wstats[0:2]), (d["w2"], inp["w2"], wstats[2:4])):
        wb = to_dev(src, torch, device)
        q.qffn_absmax(st, wb, src.size)
        q.qffn_quantize(w, st, wb, src.size)
        del wb
    d["w1_scale"], d["w2_scale"] = wstats[1:2], wstats[3:4]
    d["res_out"] = torch.empty(N, C, dtype=torch.int16, device=device)
    d["out"] = torch.empty(N, C, dtype=torch.int16, device=device)
    d["rstd"] = torch.empty(N, dtype=torch.float32, device=device)
    d["stats"] = torch.zeros(4, dtype=torch.float32, device=device)
    d["ws"] = torch.empty(q.qffn_forward_workspace_size(cfg.B, cfg.T, C, H), dtype=torch.uint8,
                          device=device)
    off = q.qffn_forward_workspace_offsets(cfg.B, cfg.T, C, H)
    d["y"] = d["ws"][off[0]:].view(torch.int16)
    d["yq"] = d["ws"][off[1]:]
    d["h"] = d["ws"][off[2]:].view(torch.int16)
    d["hq"] = d["ws"][off[3]:]
    d["host_res"], d["host_x"] = inp["res"], inp["x"]
    torch.cuda.synchronize()
    return d


def forward(q, d, stream, cfg=None):
    cfg = cfg or PREFILL_CFG
    q.qffn_forward(d["res_out"], d["out"], d["rstd"], d["stats"][0:2], d["stats"][2:4], d["res"],
                   d["x"], d["gain"], cfg.eps, d["w1"], d["w1_scale"], d["w2"], d["w2_scale"],
                   cfg.B, cfg.T, cfg.C, cfg.H, d["ws"], stream=stream)


def staged_forward(q, d, stream, ev, cfg=None):
    """The launches of qffn_forward, issued stage by stage with events between them."""
    cfg = cfg or PREFILL_CFG
    N, C, H = cfg.N, cfg.C, cfg.H
    st = d["stats"]
    ev[0].record(stream)
    q.qffn_rmsnorm_absmax(d["res_out"], d["y"], d["rstd"], st[0:2], d["res"], d["x"], d["gain"],
                          cfg.eps, N, C, stream=stream)
    ev[1].record(stream)
    q.qffn_quantize(d["yq"], st[0:2], d["y"], N * C, stream=stream)
    ev[2].record(stream)
    q.qffn_gate_up_swiglu(d["h"], st[2:4], d["yq"], st[1:2], d["w1"], d["w1_scale"], N, C, H,
                          stream=stream)
    ev[3].record(stream)
    q.qffn_quantize(d["hq"], st[2:4], d["h"], N * H, stream=stream)
    ev[4].record(stream)
    q.qffn_fp8_gemm_scaled(d["out"], d["hq"], st[3:4], d["w2"], d["w2_scale"], N, C, H,
                           stream=stream)
    ev[5].record(stream)


def gemm_clock_mhz(q, d, stream, steps):
    """Mean SM clock (MHz) of the gate|up and of the down GEMM at the end of `steps`
    back-to-back forwards (the power state of the timed region), from each GEMM's own
    clock sample: %clock64 cycles over %globaltimer ns of its first CTA."""
    cfg = PREFILL_CFG
    N, C, H = cfg.N, cfg.C, cfg.H
    st = d["stats"]
    for _ in range(steps):
        forward(q, d, stream)
    cyc, ns = q.qffn_gemm_clock_sample(stream)        # the last down GEMM
    down = cyc / ns * 1e3
    for _ in range(steps - 1):
        forward(q, d, stream)
    q.qffn_rmsnorm_absmax(d["res_out"], d["y"], d["rstd"], st[0:2], d["res"], d["x"], d["gain"],
                          cfg.eps, N, C, stream=stream)
    q.qffn_quantize(d["yq"], st[0:2], d["y"], N * C, stream=stream)
    q.qffn_gate_up_swiglu(d["h"], st[2:4], d["yq"], st[1:2], d["w1"], d["w1_scale"], N, C, H,
                          stream=stream)
    cyc, ns = q.qffn_gemm_clock_sample(stream)
    return cyc / ns * 1e3, down


def bench_prefill(q, torch, device, steps, warmup, dist, peaks):
    cfg = PREFILL_CFG
    N, C, H = cfg.N, cfg.C, cfg.H
    d = prefill_setup(q, torch, device)
    stream = torch.cuda.Stream(device)
    flop = cfg.gemm_flop
    gate_up_flop = 2 * N * C * 2 * H
    # warm-up
    for _ in range(warmup):
        forward(q, d, stream)
    torch.cuda.synchronize()
    q.qffn_check_status(stream)

    # ---- timed region 1: whole chain through qffn_forward, inputs resident in HBM
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        barrier(dist)
        torch.cuda.synchronize()
        t0.record(stream)
        for _ in range(steps):
            forward(q, d, stream)
        t1.record(stream)
        torch.cuda.synchronize()
        barrier(dist)
        ms_total = t0.elapsed_time(t1)
        # ---- timed region 2: the same launches stage by stage, per-kernel events
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(steps)]
        for i in range(steps):
            staged_forward(q, d, stream, evs[i])
        torch.cuda.synchronize()
    q.qffn_check_status(stream)
    stage_ms = [statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs) for j in range(5)]
    staged_total = statistics.mean(e[0].elapsed_time(e[5]) for e in evs)
    gu_mhz, down_mhz = gemm_clock_mhz(q, d, stream, steps)
    q.qffn_check_status(stream)
    ms_total = max_over_ranks(dist, ms_total)
    ms_step = ms_total / steps

    # ---- end to end through the public API with host buffers (pinned), copies timed.
    # Steps are pipelined over three streams with two device buffer sets: the
    # host->device copy of step i+1 and the device->host copy of step i-1 run on
    # the copy engines while step i computes.  Every step still copies its own
    # inputs in and its result out inside the timed region.
    pin_res = torch.from_numpy(d["host_res"]).view(torch.int16).pin_memory()
    pin_x = torch.from_numpy(d["host_x"]).view(torch.int16).pin_memory()
    bufs = []
    for b in range(2):
        bufs.append({
            "res": d["res"] if b == 0 else torch.empty_like(d["res"]),
            "x": d["x"] if b == 0 else torch.empty_like(d["x"]),
            "out": d["out"] if b == 0 else torch.empty_like(d["out"]),
            "res_out": d["res_out"] if b == 0 else torch.empty_like(d["res_out"]),
            "pin_out": torch.empty((N, C), dtype=torch.int16).pin_memory(),
            "pin_rout": torch.empty((N, C), dtype=torch.int16).pin_memory(),
            "h2d": torch.cuda.Event(), "comp": torch.cuda.Event(), "d2h": torch.cuda.Event(),
        })
    s_in = torch.cuda.Stream(device)
    s_out = torch.cuda.Stream(device)
    e_steps = max(4, steps)

    def e2e_step(i):
        b = bufs[i % 2]
        dd = dict(d, res=b["res"], x=b["x"], out=b["out"], res_out=b["res_out"])
        s_in.wait_event(b["comp"])            # step i-2 finished reading this buffer set
        with torch.cuda.stream(s_in):
            b["res"].copy_(pin_res, non_blocking=True)
            b["x"].copy_(pin_x, non_blocking=True)
        b["h2d"].record(s_in)
        stream.wait_event(b["h2d"])
        stream.wait_event(b["d2h"])            # step i-2's result has left this buffer set
        forward(q, dd, stream)
        b["comp"].record(stream)
        s_out.wait_event(b["comp"])
        with torch.cuda.stream(s_out):
            b["pin_out"].copy_(b["out"], non_blocking=True)
            b["pin_rout"].copy_(b["res_out"], non_blocking=True)
        b["d2h"].record(s_out)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(dist)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(e_steps):
        e2e_step(i)
    e1.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(dist, e0.elapsed_time(e1)) / e_steps
    # the last result really came back: compare with the device copy
    last = bufs[(e_steps - 1) % 2]
    assert torch.equal(last["pin_out"], last["out"].cpu())
    fp8_peak = peaks["bf16_tflops"] * FP8_PER_BF16
    gate_up_ms = stage_ms[2]
    achieved = gate_up_flop / (gate_up_ms * 1e-3) / 1e12
    res = {
        "ms_per_step": ms_step,
        "value_per_rank": flop / (ms_step * 1e-3) / 1e12,
        "e2e_ms": e2e_ms,
        "e2e_bytes": (2 * N * C * 2, 2 * N * C * 2),
        "stage_ms": {"rmsnorm_absmax": stage_ms[0], "quantize_y": stage_ms[1],
                     "gate_up_swiglu_gemm": stage_ms[2], "quantize_h": stage_ms[3],
                     "down_gemm": stage_ms[4], "staged_total": staged_total},
        "roofline": {"bound": "tensor", "kernel": "gemm_fp8_kernel<swiglu> (gate|up GEMM + SwiGLU)",
                     "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                     "frac": achieved / fp8_peak, "traffic": TRAFFIC_GATE_UP_BYTES,
                     "traffic_unit": "bytes per launch",
                     "peak_note": f"{peaks['source']} bf16 burst x {FP8_PER_BF16:g} (nominal FP8/BF16 ratio)"},
        "clocks": clk.summary(),
        "launches_per_step": 5,
    }
    # the tensor cores' rate per clock at the clock the GEMMs themselves ran at
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    per_clock_peak = sms * gu_mhz * 1e6 * FP8_FLOP_PER_CLK_PER_SM / 1e12
    res["gemm_clock"] = {
        "gate_up_sm_mhz": gu_mhz, "down_sm_mhz": down_mhz,
        "source": "each GEMM's first CTA: %clock64 cycles / %globaltimer ns from its start to its end "
                  "(qffn_gemm_clock_sample), after back-to-back forwards",
        "gate_up_per_clock_peak_tflops": per_clock_peak,
        "gate_up_frac_of_per_clock_peak": achieved / per_clock_peak,
    }
    # HBM-side fractions of the elementwise stages (algorithmic bytes / time)
    hbm = peaks["hbm_gbs"]
    bytes_rms = 4 * N * C * 2 + C * 2 + 4 * N
    bytes_qy = N * C * 3
    bytes_qh = N * H * 3
    res["elementwise_gbs"] = {
        "rmsnorm_absmax": bytes_rms / (stage_ms[0] * 1e-3) / 1e9,
        "quantize_y": bytes_qy / (stage_ms[1] * 1e-3) / 1e9,
        "quantize_h": bytes_qh / (stage_ms[3] * 1e-3) / 1e9,
        "hbm_peak_gbs": hbm,
    }
    res["down_gemm_tflops"] = 2 * N * H * C / (stage_ms[4] * 1e-3) / 1e12

    # ---- the recompute form: the same chain re-run with the abs-maxes the
    # forward recorded (4 launches; the gate|up epilogue writes E4M3 h directly)
    st_rec = d["stats"].clone()

    def recompute():
        q.qffn_forward_recompute(d["res_out"], d["out"], d["rstd"], st_rec[0:2], st_rec[2:4],
                                 d["res"], d["x"], d["gain"], cfg.eps, d["w1"], d["w1_scale"],
                                 d["w2"], d["w2_scale"], cfg.B, cfg.T, C, H, d["ws"], stream=stream)

    for _ in range(warmup):
        recompute()
    torch.cuda.synchronize()
    r0 = torch.cuda.Event(enable_timing=True)
    r1 = torch.cuda.Event(enable_timing=True)
    r0.record(stream)
    for _ in range(steps):
        recompute()
    r1.record(stream)
    torch.cuda.synchronize()
    ms_rec = r0.elapsed_time(r1) / steps
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(steps):
        q.qffn_gate_up_swiglu_quant(d["hq"], st_rec[2:4], d["yq"], st_rec[1:2], d["w1"],
                                    d["w1_scale"], N, C, H, stream=stream)
    g1.record(stream)
    torch.cuda.synchronize()
    q.qffn_check_status(stream)
    ms_gq = g0.elapsed_time(g1) / steps
    res["recompute"] = {
        "what": "qffn_forward_recompute: the chain with the recorded abs-maxes given "
                "(no bf16 h, no requantisation pass)",
        "ms_per_step": ms_rec, "tflops": flop / (ms_rec * 1e-3) / 1e12, "launches_per_step": 4,
        "gate_up_swiglu_e4m3_gemm_ms": ms_gq,
        "gate_up_swiglu_e4m3_gemm_tflops": gate_up_flop / (ms_gq * 1e-3) / 1e12,
    }
    return res


def bench_workload(q, torch, device, cfg, steps, warmup, peaks):
    """The prefill chain on another of the pages' workload shapes: whole-chain time through
    qffn_forward and the gate|up GEMM's own time from a staged pass."""
    d = prefill_setup(q, torch, device, cfg)
    stream = torch.cuda.Stream(device)
    N, C, H = cfg.N, cfg.C, cfg.H
    for _ in range(warmup):
        forward(q, d, stream, cfg)
    torch.cuda.synchronize()
    q.qffn_check_status(stream)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    # small workloads run in microseconds: more steps for a stable figure
    reps = steps if cfg.gemm_flop >= 1e11 else max(steps, 500)
    t0.record(stream)
    for _ in range(reps):
        forward(q, d, stream, cfg)
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / reps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(steps)]
    for i in range(steps):
        staged_forward(q, d, stream, evs[i], cfg)
    torch.cuda.synchronize()
    q.qffn_check_status(stream)
    stage_ms = [statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs) for j in range(5)]
    gate_up = 2 * N * C * 2 * H / (stage_ms[2] * 1e-3) / 1e12
    peak = peaks["bf16_tflops"] * FP8_PER_BF16
    ws_bytes = 8 * N * C + 2 * C + 3 * H * C + 4 * N            # inputs, weights and outputs once
    res = {"workload": f"{cfg.name}: B={cfg.B}, T={cfg.T} (N={N}), C={C}, H={H}",
           "ms_per_step": ms, "tflops": cfg.gemm_flop / (ms * 1e-3) / 1e12, "steps": reps,
           "gate_up_ms": stage_ms[2], "gate_up_tflops": gate_up,
           "gate_up_roofline_frac": gate_up / peak,
           "stages_ms": dict(zip(["rmsnorm_absmax", "quantize_y", "gate_up_swiglu", "quantize_h",
                                  "down_gemm"], stage_ms)),
           "l2": "working set larger than L2" if ws_bytes > L2_BYTES
           else "working set fits in L2 (resident across steps)"}
    del d
    torch.cuda.empty_cache()
    return res


def bench_attention_projections(q, torch, device, steps, warmup):
    """The attention-side uses of the same primitives at the Llama-3-8B shape:
    LN1 (fused residual + RMSNorm + abs-max) into the QKV projection
    (N x 4096 -> N x 6144, forward_qmm), and the abs-max of the attention output
    into the output projection (N x 4096 -> N x 4096).  The attention output is
    a synthetic N(0,1) stand-in; weights are N(0, 0.02) quantised on the GPU."""
    from ffn_inputs import random_bf16
    cfg = PREFILL_CFG
    N, C = cfg.N, cfg.C
    nqkv = C + 2 * 1024                      # 32 query heads + 2 x 8 key/value heads of 128
    inp = prefill_inputs(cfg)
    res, x, gain = (to_dev(inp[k], torch, device) for k in ("res", "x", "gain"))
    att = to_dev(random_bf16((N, C), seed=301), torch, device)
    wst = torch.zeros(4, dtype=torch.float32, device=device)
    wqkv = torch.empty(nqkv, C, dtype=torch.uint8, device=device)
    wo = torch.empty(C, C, dtype=torch.uint8, device=device)
    for w, seed, st in ((wqkv, 302, wst[0:2]), (wo, 303, wst[2:4])):
        wb = to_dev(random_bf16(tuple(w.shape), seed=seed, std=0.02), torch, device)
        q.qffn_absmax(st, wb, wb.numel())
        q.qffn_quantize(w, st, wb, wb.numel())
        del wb
    r = torch.empty(N, C, dtype=torch.int16, device=device)
    y = torch.empty(N, C, dtype=torch.int16, device=device)
    rstd = torch.empty(N, dtype=torch.float32, device=device)
    st = torch.zeros(4, dtype=torch.float32, device=device)
    qbuf = torch.empty(N, C, dtype=torch.uint8, device=device)
    qkv = torch.empty(N, nqkv, dtype=torch.int16, device=device)
    atto = torch.empty(N, C, dtype=torch.int16, device=device)
    stream = torch.cuda.Stream(device)

    def ln1():
        q.qffn_rmsnorm_absmax(r, y, rstd, st[0:2], res, x, gain, cfg.eps, N, C, stream=stream)

    def qkv_proj():
        q.qffn_qmm(qkv, qbuf, st[0:2], y, None, wqkv, wst[1:2], N, nqkv, C, stream=stream)

    def out_proj():
        q.qffn_absmax(st[2:4], att, N * C, stream=stream)
        q.qffn_qmm(atto, qbuf, st[2:4], att, None, wo, wst[3:4], N, C, C, stream=stream)

    out = {}
    for name, fn in (("ln1", ln1), ("qkv_qmm", qkv_proj), ("out_proj", out_proj)):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        out[name] = a.elapsed_time(b) / steps
    q.qffn_check_status(stream)
    f_qkv = 2.0 * N * nqkv * C
    f_o = 2.0 * N * C * C
    return {
        "workload": f"llama3-8b attention projections: N={N}, C={C}, QKV out {nqkv}",
        "ln1_ms": out["ln1"], "qkv_qmm_ms": out["qkv_qmm"], "out_proj_ms": out["out_proj"],
        "qkv_tflops": f_qkv / (out["qkv_qmm"] * 1e-3) / 1e12,
        "out_proj_tflops": f_o / (out["out_proj"] * 1e-3) / 1e12,
        "ln1_plus_qkv_tflops": f_qkv / ((out["ln1"] + out["qkv_qmm"]) * 1e-3) / 1e12,
    }


def bench_backward(q, torch, device, steps, warmup, peaks):
    """The FP8 FFN backward (qffn_ffn_backward) at the Llama-3-8B shape, fed the
    forward's quantised activations and a synthetic N(0, 1e-3) output gradient.
    FLOPs: dgrad and wgrad of both projections (12 N C H) plus the recomputed
    up projection (4 N C H)."""
    from ffn_inputs import random_bf16
    cfg = PREFILL_CFG
    N, C, H = cfg.N, cfg.C, cfg.H
    d = prefill_setup(q, torch, device)
    stream = torch.cuda.Stream(device)
    forward(q, d, stream)
    torch.cuda.synchronize()
    dout = to_dev(random_bf16((N, C), seed=401, std=1e-3), torch, device)
    st = torch.zeros(4, dtype=torch.float32, device=device)
    q.qffn_absmax(st[0:2], dout, N * C, stream=stream)
    d_ln2 = torch.empty(N, C, dtype=torch.int16, device=device)
    dw1 = torch.empty(2 * H, C, dtype=torch.int16, device=device)
    dw2 = torch.empty(C, H, dtype=torch.int16, device=device)
    ws = torch.empty(q.qffn_ffn_backward_workspace_size(N, C, H), dtype=torch.uint8, device=device)
    off = q.qffn_ffn_backward_workspace_offsets(N, C, H)
    sy, sh = d["stats"][1:2], d["stats"][3:4]

    def step():
        q.qffn_ffn_backward(d_ln2, dw1, dw2, st[0:2], st[2:4], dout, d["yq"], sy, d["hq"], sh,
                            d["w1"], d["w1_scale"], d["w2"], d["w2_scale"], N, C, H, False, ws,
                            stream=stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps

    # the same backward accumulating into dW1 and dW2 (gradient accumulation
    # over micro-batches): the weight-gradient epilogues read the previous dW
    def step_acc():
        q.qffn_ffn_backward(d_ln2, dw1, dw2, st[0:2], st[2:4], dout, d["yq"], sy, d["hq"], sh,
                            d["w1"], d["w1_scale"], d["w2"], d["w2_scale"], N, C, H, True, ws,
                            stream=stream)

    step_acc()
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(steps):
        step_acc()
    b.record(stream)
    torch.cuda.synchronize()
    ms_acc = a.elapsed_time(b) / steps
    # staged: the three building blocks of the chain with events between them
    dh = ws[off[0]:].view(torch.int16)
    dgu = ws[off[1]:].view(torch.int16)
    bq = torch.empty(max(q.qffn_backward_qmm_workspace_size(N, H, C),
                         q.qffn_backward_qmm_workspace_size(N, C, 2 * H)), dtype=torch.uint8, device=device)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    ev[0].record(stream)
    q.qffn_backward_qmm(dh, dw2, st[0:2], dout, d["hq"], sh, d["w2"], d["w2_scale"], N, H, C, False, bq,
                        stream=stream)
    ev[1].record(stream)
    q.qffn_gate_up_swiglu_backward(dgu, st[2:4], dh, d["yq"], sy, d["w1"], d["w1_scale"], N, C, H,
                                   stream=stream)
    ev[2].record(stream)
    q.qffn_backward_qmm(d_ln2, dw1, st[2:4], dgu, d["yq"], sy, d["w1"], d["w1_scale"], N, C, 2 * H, False,
                        bq, stream=stream)
    ev[3].record(stream)
    torch.cuda.synchronize()
    q.qffn_check_status(stream)
    stage = [ev[i].elapsed_time(ev[i + 1]) for i in range(3)]
    flop = 16.0 * N * C * H
    return {
        "workload": "llama3-8b FFN backward: N=16384, C=4096, H=14336 (down and up backward_qmm, "
                    "recomputed up projection fused with swiglu_backward)",
        "ms_per_step": ms, "tflops": flop / (ms * 1e-3) / 1e12,
        "tflops_without_recompute": 12.0 * N * C * H / (ms * 1e-3) / 1e12,
        "launches_per_step": 7,
        "ms_per_step_accumulating_dw": ms_acc,
        "stages_ms": {"backward_qmm_down": stage[0], "gate_up_swiglu_backward": stage[1],
                      "backward_qmm_up": stage[2]},
        "gate_up_swiglu_backward_tflops": 2.0 * N * C * 2 * H / (stage[1] * 1e-3) / 1e12,
    }


# Dense FP8 (E4M3, kind::f8f6f4) tensor-core rate per SM per clock: twice the
# dense BF16 rate of 8192 FLOP/clk/SM.  The nominal 4.5 PFLOP/s dense FP8 of a
# 152-SM part corresponds to this rate at about 1.81 GHz.
FP8_FLOP_PER_CLK_PER_SM = 16384


def fp8_peak_computed(torch, device, clocks, peaks):
    """SMs x SM clock x per-SM dense FP8 rate, reported beside the measured
    ceilings: at the SM clock seen under load in the timed region and at the
    part's maximum clock."""
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    out = {"sms": sms, "flop_per_clk_per_sm": FP8_FLOP_PER_CLK_PER_SM,
           "note": "dense FP8 rate per SM per clock (2 x the BF16 rate); the nominal 4.5 PFLOP/s "
                   "corresponds to it at about 1.81 GHz"}
    for key, mhz in (("at_max_clock", clocks.get("sm_max_mhz") or peaks.get("sm_max_mhz")),
                     ("at_clock_under_load", clocks.get("sm_mhz"))):
        if mhz:
            out[key] = {"sm_mhz": mhz, "tflops": sms * mhz * 1e6 * FP8_FLOP_PER_CLK_PER_SM / 1e12}
    return out


def fp8_library_ceiling(torch, device, steps=10):
    """Context only, not on the library's path: the FP8 rate of the vendor GEMM
    (cuBLASLt through torch._scaled_mm, E4M3 x E4M3 -> bf16, per-tensor
    scales) at 8192^3 and at the gate|up shape.  The roofline denominator stays
    the measured bf16 peak x 2."""
    res = {"what": "torch._scaled_mm (cuBLASLt) E4M3 GEMM, bf16 out, per-tensor scales"}
    try:
        g = torch.Generator(device="cpu").manual_seed(7)
        one = torch.ones((), dtype=torch.float32, device=device)
        for name, (m, n, k) in (("8192^3", (8192, 8192, 8192)), ("gate_up 16384x28672x4096", (16384, 28672, 4096))):
            a = (torch.randn(m, k, generator=g) * 0.5).to(device).to(torch.float8_e4m3fn)
            b = (torch.randn(n, k, generator=g) * 0.5).to(device).to(torch.float8_e4m3fn)
            for _ in range(3):
                torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(steps):
                torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / steps
            res[name] = {"ms": ms, "tflops": 2.0 * m * n * k / (ms * 1e-3) / 1e12}
            del a, b
    except Exception as exc:          # reported, never fatal: this is context
        res["unavailable"] = f"{type(exc).__name__}: {exc}"[:200]
    return res


def bench_decode(q, torch, device, iters, dist, peaks):
    cfg = DECODE_CFG
    C, H = cfg.C, cfg.H
    di = decode_inputs(cfg)
    # One decode token through the model's FFN layers: a copy of the weights per
    # layer (32 layers x 176 MB; at least enough copies that no call finds its
    # weights in L2), the records built once on the GPU and cloned.
    copies = max(DECODE_LAYERS, -(-2 * L2_BYTES // cfg.weight_bytes) + 1)
    first = {}
    for k, rows, cols in (("w_gate", H, C), ("w_up", H, C), ("w_down", C, H)):
        wb = to_dev(di[k], torch, device)
        codes = torch.empty(rows, cols, dtype=torch.uint8, device=device)
        sc = torch.empty(rows, dtype=torch.float32, device=device)
        q.qffn_quantize_rows(codes, sc, wb, rows, cols)
        first[k] = (codes, sc)
        del wb
    sets = [first] + [{k: (c.clone(), sc.clone()) for k, (c, sc) in first.items()} for _ in range(copies - 1)]
    x = to_dev(di["x"], torch, device)
    out = torch.empty(C, dtype=torch.int16, device=device)
    ws = torch.zeros(q.qffn_decode_workspace_size(C, H), dtype=torch.uint8, device=device)
    stream = torch.cuda.Stream(device)
    torch.cuda.synchronize()

    def call(s, flags):
        # a decode step on weights built long before: the weight stream may start
        # before the previous step's kernel has finished
        q.qffn_decode_forward_ex(out, x, *s["w_gate"], *s["w_up"], *s["w_down"], C, H, ws, flags,
                                 stream=stream)

    def graph_us(flags, calls=None):
        calls = calls or copies
        for i in range(6):
            call(sets[i % copies], flags)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for s in sets[:calls]:
                call(s, flags)
        reps = max(2, -(-iters // calls))
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        barrier(dist)
        with torch.cuda.stream(stream):
            t0.record(stream)
            for _ in range(reps):
                graph.replay()
            t1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(dist, t0.elapsed_time(t1)) * 1e3 / (reps * calls), reps * calls

    stable = q.QFFN_DECODE_WEIGHTS_STABLE
    us_graph, n_calls = graph_us(stable)
    us_graph_default, _ = graph_us(0)
    us_graph3, _ = graph_us(stable, 3)     # a graph of 3 calls replayed (graph launch every 3 calls)

    def eager_us(flags):
        e_calls = max(1, iters // copies) * copies
        for i in range(copies):
            call(sets[i], flags)
        torch.cuda.synchronize()
        t2 = torch.cuda.Event(enable_timing=True)
        t3 = torch.cuda.Event(enable_timing=True)
        t2.record(stream)
        for i in range(e_calls):
            call(sets[i % copies], flags)
        t3.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(dist, t2.elapsed_time(t3)) * 1e3 / e_calls

    us_eager = eager_us(stable)
    # one call between events (its two launches), each on a weight copy not in L2
    kev = []
    for i in range(60):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        e[0].record(stream)
        call(sets[i % copies], 0)
        e[1].record(stream)
        kev.append(e)
    torch.cuda.synchronize()
    call_us = statistics.mean(e[0].elapsed_time(e[1]) for e in kev[10:]) * 1e3
    # the standalone kernels of the split arm, for context (dual GEMV, silu_mul, down GEMV)
    g = torch.empty(H, dtype=torch.int16, device=device)
    u = torch.empty(H, dtype=torch.int16, device=device)
    o2 = torch.empty(C, dtype=torch.int16, device=device)
    evs = []
    for i in range(60):
        s = sets[i % copies]
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        e[0].record(stream)
        q.qffn_gemv_dual(g, u, x, *s["w_gate"], *s["w_up"], H, C, stream=stream)
        e[1].record(stream)
        q.qffn_silu_mul(g, u, H, stream=stream)
        e[2].record(stream)
        q.qffn_gemv(o2, g, *s["w_down"], C, H, stream=stream)
        e[3].record(stream)
        evs.append(e)
    torch.cuda.synchronize()
    q.qffn_check_status(stream)
    dual_us = statistics.mean(e[0].elapsed_time(e[1]) for e in evs[10:]) * 1e3
    silu_us = statistics.mean(e[1].elapsed_time(e[2]) for e in evs[10:]) * 1e3
    down_us = statistics.mean(e[2].elapsed_time(e[3]) for e in evs[10:]) * 1e3
    split_us = statistics.mean(e[0].elapsed_time(e[3]) for e in evs[10:]) * 1e3
    gbs = cfg.weight_bytes / (us_graph * 1e-6) / 1e9
    dual_bytes = 2 * H * C + 8 * H + 2 * C + 4 * H
    dual_gbs = dual_bytes / (dual_us * 1e-6) / 1e9
    return {
        "metric": DECODE_METRIC, "unit": "GB/s", "value": gbs, "us_per_call": us_graph,
        "bytes_per_call": cfg.weight_bytes, "calls": n_calls, "graph": True,
        "form": f"qffn_decode_forward_ex with QFFN_DECODE_WEIGHTS_STABLE (weights built before the "
                f"timed region): one token through {copies} FFN layers, each with its own weight copy, "
                f"captured as one CUDA graph of {copies} calls and replayed",
        "graph_of_3_us_per_call": us_graph3,
        "default_form_us_per_call": us_graph_default,
        "default_form_gbs": cfg.weight_bytes / (us_graph_default * 1e-6) / 1e9,
        "weight_copies_rotated": copies,
        "eager_back_to_back_us_per_call": us_eager,
        "eager_back_to_back_gbs": cfg.weight_bytes / (us_eager * 1e-6) / 1e9,
        "single_call_us": call_us,
        "roofline": {"bound": "hbm", "kernel": "gemv_kernel<dual> (gate+up GEMV, the decode's first launch)",
                     "achieved": dual_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": dual_gbs / peaks["hbm_gbs"], "traffic": TRAFFIC_DUAL_GEMV_BYTES,
                     "traffic_unit": "bytes per launch", "us_per_launch": dual_us,
                     "peak_note": f"{peaks['source']} HBM copy bandwidth"},
        "split_arm_us": {"gemv_dual": dual_us, "silu_mul": silu_us, "gemv_down": down_us, "total": split_us},
        "frac_of_peak": gbs / peaks["hbm_gbs"],
        "frac_of_8tbs": gbs / 8000.0,
        "gpu_launches": 2 * n_calls,        # dual GEMV (+silu_mul) and down GEMV per call, graph region
    }


# ---------------------------------------------------------------- CPU oracle legs
def _oracle_bytes(cfg, tokens):
    """Algorithmic bytes of the chain on `tokens` tokens: res, x in; r, out out (bf16);
    rstd; gain and both FP8 weight matrices read once."""
    C, H = cfg.C, cfg.H
    return 8 * tokens * C + 4 * tokens + 2 * C + 3 * H * C


def oracle_time(cfg, tokens, threads):
    """The C++ oracle's prefill chain on the first `tokens` tokens of `cfg` with `threads`
    OpenMP threads (0 = every processor); the library's own steady-clock time."""
    import oracle as o
    inp = prefill_inputs(cfg)
    w1q, w1s = o.quantize_tensor(inp["w1"])
    w2q, w2s = o.quantize_tensor(inp["w2"])
    n0 = o.max_threads()
    o.set_threads(threads)
    used = o.max_threads()
    try:
        t = {}
        o.ffn_forward(inp["res"][:tokens], inp["x"][:tokens], inp["gain"], inp["eps"], w1q, w1s, w2q,
                      w2s, cfg.H, timing=t)
    finally:
        o.set_threads(n0)
    secs = t["seconds"]
    flop = cfg.gemm_flop / cfg.N * tokens
    return {"workload": cfg.name, "tokens": tokens, "of_tokens": cfg.N, "threads": used,
            "seconds": secs, "gflops": flop / secs / 1e9,
            "gbs": _oracle_bytes(cfg, tokens) / secs / 1e9}


def cpu_baseline():
    """The oracle on the host cores: every workload, bounded samples (about 20-30 s in all).
    tiny in full and the Llama-3.2-1B sample single-threaded and on every core; the 8B
    sample (the headline figure) on every core."""
    runs = [oracle_time(PREFILL["tiny"], PREFILL["tiny"].N, 1),
            oracle_time(PREFILL["tiny"], PREFILL["tiny"].N, 0),
            oracle_time(PREFILL["llama3.2-1b"], 16, 1),
            oracle_time(PREFILL["llama3.2-1b"], 256, 0),
            oracle_time(PREFILL["qwen2.5-7b"], 64, 0)]
    head = oracle_time(PREFILL_CFG, 128, 0)
    runs.append(head)
    return {"value": head["gflops"] / 1e3, "unit": "TFLOP/s", "cores": head["threads"], "kind": "oracle",
            "sample": f"C++ oracle chain (exact int64 GEMM sums, fp64 norm/SwiGLU) on the first "
                      f"{head['tokens']} of {PREFILL_CFG.N} tokens of the Llama-3-8B FFN workload, weights "
                      f"pre-quantised, {head['threads']} OpenMP threads (os.cpu_count() = {os.cpu_count()}); "
                      f"{head['seconds']:.2f} s by std::chrono::steady_clock",
            "runs": runs}


def run_reference(args, rank, world, dist):
    if rank != 0:
        return
    import oracle as o
    cfg = PREFILL_CFG
    inp = prefill_inputs(cfg)
    w1q, w1s = o.quantize_tensor(inp["w1"])
    w2q, w2s = o.quantize_tensor(inp["w2"])
    o.set_threads(0)
    tokens = 64
    per_tok = cfg.gemm_flop / cfg.N

    def step():
        t = {}
        o.ffn_forward(inp["res"][:tokens], inp["x"][:tokens], inp["gain"], inp["eps"], w1q, w1s,
                      w2q, w2s, cfg.H, timing=t)
        return t["seconds"]

    for _ in range(args.warmup):
        step()
    secs = sum(step() for _ in range(args.steps))
    value = per_tok * tokens * args.steps / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int64 exact GEMM sums, f64 elementwise",
        "data": "synthetic",
        "config": {"workload": f"llama3-8b FFN fwd, {tokens}-token sample per step (of N={cfg.N}), "
                               f"C={cfg.C}, H={cfg.H}", "global_batch": tokens, "seq_len": cfg.T},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": o.max_threads(), "kind": "oracle",
                         "sample": f"C++ oracle, first {tokens} tokens of the 8B workload per step, "
                                   f"{o.max_threads()} OpenMP threads, std::chrono::steady_clock"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def profile_case(q, torch, device):
    """A case sized for ncu captures: the prefill chain at N=2048 tokens of the 8B FFN
    (C=4096, H=14336; weights alone 176 MB, larger than L2; a few GB on the device at most)
    three times, one recompute forward and one FP8 backward on the same tokens, then
    the 8B decode FFN twice.  Launch order per forward: rmsnorm, quantize, gate|up
    GEMM, quantize, down GEMM."""
    global PREFILL_CFG
    from ffn_inputs import PrefillConfig
    PREFILL_CFG = PrefillConfig("llama3-8b-2k", B=1, T=2048, C=4096, H=14336, eps=1e-5)
    d = prefill_setup(q, torch, device)
    torch.cuda.empty_cache()
    stream = torch.cuda.current_stream(device)
    for _ in range(3):
        forward(q, d, stream)
    torch.cuda.synchronize()
    q.qffn_check_status(stream)
    # the recompute form and the FP8 backward on the same tokens (GEMM launches
    # 6-7 and 8-12 of this process: recompute gate|up with the E4M3 epilogue and
    # down; backward down dgrad, down wgrad, fused recompute + swiglu_backward,
    # up dgrad, up wgrad)
    pc = PREFILL_CFG
    st_rec = d["stats"].clone()
    q.qffn_forward_recompute(d["res_out"], d["out"], d["rstd"], st_rec[0:2], st_rec[2:4], d["res"],
                             d["x"], d["gain"], pc.eps, d["w1"], d["w1_scale"], d["w2"], d["w2_scale"],
                             pc.B, pc.T, pc.C, pc.H, d["ws"], stream=stream)
    from ffn_inputs import random_bf16
    dout = to_dev(random_bf16((pc.N, pc.C), seed=401, std=1e-3), torch, device)
    bst = torch.zeros(4, dtype=torch.float32, device=device)
    q.qffn_absmax(bst[0:2], dout, pc.N * pc.C, stream=stream)
    d_ln2 = torch.empty(pc.N, pc.C, dtype=torch.int16, device=device)
    dw1 = torch.empty(2 * pc.H, pc.C, dtype=torch.int16, device=device)
    dw2 = torch.empty(pc.C, pc.H, dtype=torch.int16, device=device)
    bws = torch.empty(q.qffn_ffn_backward_workspace_size(pc.N, pc.C, pc.H), dtype=torch.uint8, device=device)
    q.qffn_ffn_backward(d_ln2, dw1, dw2, bst[0:2], bst[2:4], dout, d["yq"], d["stats"][1:2], d["hq"],
                        d["stats"][3:4], d["w1"], d["w1_scale"], d["w2"], d["w2_scale"], pc.N, pc.C, pc.H,
                        False, bws, stream=stream)
    torch.cuda.synchronize()
    q.qffn_check_status(stream)
    del bws, d_ln2, dw1, dw2
    cfg = DECODE_CFG
    di = decode_inputs(cfg)
    recs = []
    for k, rows, cols in (("w_gate", cfg.H, cfg.C), ("w_up", cfg.H, cfg.C), ("w_down", cfg.C, cfg.H)):
        wb = to_dev(di[k], torch, device)
        codes = torch.empty(rows, cols, dtype=torch.uint8, device=device)
        sc = torch.empty(rows, dtype=torch.float32, device=device)
        q.qffn_quantize_rows(codes, sc, wb, rows, cols)
        recs += [codes, sc]
    del wb
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    x = to_dev(di["x"], torch, device)
    out = torch.empty(cfg.C, dtype=torch.int16, device=device)
    ws = torch.zeros(q.qffn_decode_workspace_size(cfg.C, cfg.H), dtype=torch.uint8, device=device)
    for _ in range(2):
        q.qffn_decode_forward(out, x, *recs, cfg.C, cfg.H, ws, stream=stream)
    torch.cuda.synchronize()
    print("profile case done")


def profile_workload(q, torch, device, cfg):
    """The prefill chain of one of the pages' workloads three times, untimed (for ncu
    captures of the small workloads; launch order per forward: rmsnorm, quantize, gate|up
    GEMM, quantize, down GEMM)."""
    d = prefill_setup(q, torch, device, cfg)
    stream = torch.cuda.current_stream(device)
    for _ in range(3):
        forward(q, d, stream, cfg)
    torch.cuda.synchronize()
    q.qffn_check_status(stream)


def traffic_case(q, torch, device):
    """A case for one ncu capture of DRAM bytes per launch (about 1.2 GB on the device):
    the gate|up GEMM with the SwiGLU epilogue and the down GEMM at the 8B prefill shape
    (N=16384, C=4096, H=14336) twice each on random codes, then two 8B decode calls.
    Launch order: gate|up, down, gate|up, down, then per decode call the dual GEMV and
    the down GEMV."""
    cfg = PREFILL_CFG
    N, C, H = cfg.N, cfg.C, cfg.H
    g = torch.Generator(device=device).manual_seed(0)
    yq = torch.randint(0, 0x70, (N, C), dtype=torch.uint8, device=device, generator=g)
    w1 = torch.randint(0, 0x70, (2 * H, C), dtype=torch.uint8, device=device, generator=g)
    hq = torch.randint(0, 0x70, (N, H), dtype=torch.uint8, device=device, generator=g)
    w2 = torch.randint(0, 0x70, (C, H), dtype=torch.uint8, device=device, generator=g)
    sc = torch.tensor([1e-3, 1e-3], dtype=torch.float32, device=device)
    h = torch.empty(N, H, dtype=torch.int16, device=device)
    out = torch.empty(N, C, dtype=torch.int16, device=device)
    st = torch.zeros(2, dtype=torch.float32, device=device)
    for _ in range(2):
        q.qffn_gate_up_swiglu(h, st, yq, sc[0:1], w1, sc[1:2], N, C, H)
        q.qffn_fp8_gemm_scaled(out, hq, sc[0:1], w2, sc[1:2], N, C, H)
    torch.cuda.synchronize()
    del yq, w1, hq, w2, h, out
    dc = DECODE_CFG
    di = decode_inputs(dc)
    recs = []
    for k, rows, cols in (("w_gate", dc.H, dc.C), ("w_up", dc.H, dc.C), ("w_down", dc.C, dc.H)):
        codes = torch.empty(rows, cols, dtype=torch.uint8, device=device)
        scales = torch.empty(rows, dtype=torch.float32, device=device)
        q.qffn_quantize_rows(codes, scales, to_dev(di[k], torch, device), rows, cols)
        recs += [codes, scales]
    x = to_dev(di["x"], torch, device)
    o = torch.empty(dc.C, dtype=torch.int16, device=device)
    ws = torch.empty(q.qffn_decode_workspace_size(dc.C, dc.H), dtype=torch.uint8, device=device)
    for _ in range(2):
        q.qffn_decode_forward(o, x, *recs, dc.C, dc.H, ws)
    torch.cuda.synchronize()
    print("traffic case done")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="qffn", choices=["qffn", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-iters", type=int, default=300)
    ap.add_argument("--profile-case", action="store_true",
                    help="run a small case once (for ncu captures) and exit without timing")
    ap.add_argument("--profile-workload", choices=sorted(PREFILL),
                    help="run the prefill chain of one workload three times (for ncu captures) and exit")
    ap.add_argument("--traffic-case", action="store_true",
                    help="run the full-size GEMMs and decode twice (for an ncu DRAM-bytes capture) and exit")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, local, world, dist = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, world, dist)
        return

    import torch
    import transformer_ffn_block_gb300 as q
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if args.profile_case:
        profile_case(q, torch, device)
        return
    if args.traffic_case:
        traffic_case(q, torch, device)
        return
    if args.profile_workload:
        profile_workload(q, torch, device, PREFILL[args.profile_workload])
        return
    peaks = load_peaks()
    pre = bench_prefill(q, torch, device, args.steps, args.warmup, dist, peaks)
    dec = bench_decode(q, torch, device, args.decode_iters, dist, peaks)
    att = bench_attention_projections(q, torch, device, args.steps, args.warmup)
    bwd = bench_backward(q, torch, device, max(3, args.steps // 4), args.warmup, peaks)
    ceiling = fp8_library_ceiling(torch, device)
    computed = fp8_peak_computed(torch, device, pre["clocks"], peaks)
    workloads = {name: bench_workload(q, torch, device, PREFILL[name], max(5, args.steps // 2), args.warmup, peaks)
                 for name in ("tiny", "llama3.2-1b", "qwen2.5-7b")}
    cfg = PREFILL_CFG
    value = job_throughput(cfg.gemm_flop, world, pre["ms_per_step"])
    e2e_value = job_throughput(cfg.gemm_flop, world, pre["e2e_ms"])
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": pre["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp8-e4m3 (fp32 accumulate, bf16 out)",
        "data": "synthetic (seeded Gaussian activations, N(0,0.02) weights quantised to E4M3)",
        "config": {"workload": "llama3-8b FFN fwd: B=8, T=2048 (N=16384), C=4096, H=14336",
                   "global_batch": cfg.B * world, "seq_len": cfg.T, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (per-step working set ~3 GB)"},
        "roofline": pre["roofline"],
        "clocks": pre["clocks"],
        "gemm_clock": pre["gemm_clock"],
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": pre["e2e_bytes"][0],
                "d2h_bytes_per_step": pre["e2e_bytes"][1]},
        "gpu_launches": pre["launches_per_step"] * args.steps,
        "stages_ms": pre["stage_ms"],
        "elementwise_gbs": pre["elementwise_gbs"],
        "down_gemm_tflops": pre["down_gemm_tflops"],
        "recompute": pre["recompute"],
        "attention_projections": att,
        "backward": bwd,
        "fp8_library_ceiling": ceiling,
        "fp8_peak_computed": computed,
        "decode": dec,
        "workloads": workloads,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
