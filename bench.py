"""Benchmark of the FP8-Linear hot path (MXFP8 quantise + MXFP8 GEMMs) on GB300.

One step = the whole hot path once over one batch of synthetic input:
  dense FFN layer (8192 tokens, hidden 7168, ffn 18432):
    quantise X [8192x7168] row+col, W [18432x7168] row, dY [8192x18432] row+col;
    fprop  D, AUX = GELU-tanh(X W^T + b)       (M=8192,  N=18432, K=7168)
    wgrad  dW = dY^T X on column-wise operands (M=18432, N=7168,  K=8192)
  MoE expert layer (16384 tokens, top-8 of 128 experts, Zipf(1.1) routing):
    quantise X [131072x4096] row, W [128*1536x4096] row;
    grouped D, AUX = GELU-tanh(X_e W_e^T) over the ragged groups, one launch.
value = the step's GEMM FLOPs / step time (TFLOP/s; quantisation time included).

`--impl reference` times the CPU oracle on a bounded sample of the same step.
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
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MXFP8 GEMM TFLOPS & quantize GB/s at 1 GB300, as % of FP8/HBM roofline"
UNIT = "TFLOP/s"
WORKLOAD = ("ffn fprop+wgrad (tokens 8192, hidden 7168, ffn 18432) + moe grouped "
            "(16384 tokens top-8 of 128 experts, 1536x4096), with all MXFP8 quantisation")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16": p["bf16_tflops"],
                "bf16_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


KERNEL_SOURCES = {"gemm": ["gemm.cu", "ptx.cuh", "tcgen05.cuh"], "quant": ["quantize.cu", "e4m3.cuh", "ptx.cuh", "units.cuh"],
                  "grouped": ["grouped_quantize.cu", "e4m3.cuh", "ptx.cuh", "units.cuh"],
                  "block": ["block_quantize.cu", "e4m3.cuh", "ptx.cuh"],
                  "ln": ["layernorm_quantize.cu", "e4m3.cuh", "ptx.cuh", "units.cuh"]}


def code_only(text: str) -> str:
    """A source's code lines: line comments and blank lines dropped (the
    sources hold no block comments and no "//" inside string literals)."""
    lines = (line.split("//", 1)[0].rstrip() for line in text.splitlines())
    return "\n".join(line for line in lines if line)


def source_sha256(kernel_name: str) -> str:
    """Hash of the code (comments aside) of the sources that build the kernel
    behind a bench kernel name."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel_name.split("_")[0]]:
        with open(os.path.join(ROOT, "mxfp8_block_scaled_quantize_gb300", "csrc", f)) as fh:
            h.update(code_only(fh.read()).encode())
    return h.hexdigest()


def measured_traffic(kernel_name: str):
    """DRAM bytes (read + write) per launch from profiles/traffic.json, recorded
    by ncu for this workload; None unless the kernel's code (comments aside)
    is unchanged since that capture."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            entry = json.load(f).get(kernel_name)
    except (OSError, ValueError):
        return None
    if not entry or entry.get("source_sha256") != source_sha256(kernel_name):
        return None
    return entry["bytes_per_launch"]


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- workload

def build_inputs(dev):
    from mxfp8_block_scaled_quantize_gb300 import workloads
    ffn = workloads.make_ffn()
    moe = workloads.make_moe()
    host = {"ffn_X": ffn["X"], "ffn_W": ffn["W"], "ffn_b": ffn["bias"], "ffn_dY": ffn["dY"],
            "moe_X": moe["X"], "moe_W": moe["W"].view(128 * 1536, 4096), "moe_m": moe["group_m"]}
    return host


class Step:
    """Device buffers and the launch sequence of one step (all on one stream)."""

    def __init__(self, host, dev):
        import mxfp8_block_scaled_quantize_gb300 as temx
        self.temx = temx
        self.d = {k: v.to(dev) for k, v in host.items()}
        d = self.d
        from mxfp8_block_scaled_quantize_gb300 import workloads
        d["ln_g"], d["ln_b"] = (t.to(dev) for t in workloads.layernorm_params(host["ffn_X"].shape[1], 410))
        # the MoE output gradient for the expert wgrad row (made on the device side
        # only: it is not an input of the timed step)
        d["moe_dY"] = workloads.normal_bf16((int(host["moe_m"].sum()), 1536), 1e-3, 503).to(dev)
        e = lambda *s, dt=torch.uint8: torch.empty(*s, dtype=dt, device=dev)
        pitch = temx.te_mx_scale_pitch
        T, H, F = 8192, 7168, 18432
        self.o = o = {}
        o["x_row"] = {"q_row": e(T, H), "s_row": e(T, pitch(H)), "q_col": e(H, T), "s_col": e(H, pitch(T))}
        o["w_row"] = {"q_row": e(F, H), "s_row": e(F, pitch(H))}
        o["dy"] = {"q_row": e(T, F), "s_row": e(T, pitch(F)), "q_col": e(F, T), "s_col": e(F, pitch(T))}
        o["fprop"] = (e(T, F, dt=torch.bfloat16), e(T, F, dt=torch.bfloat16))
        o["wgrad"] = (e(F, H, dt=torch.bfloat16), None)
        MT, G, N, K = 131072, 128, 1536, 4096
        o["mx"] = {"q_row": e(MT, K), "s_row": e(MT, pitch(K))}
        o["mw"] = {"q_row": e(G * N, K), "s_row": e(G * N, pitch(K))}
        o["moe"] = (e(MT, N, dt=torch.bfloat16), e(MT, N, dt=torch.bfloat16))
        counts = host["moe_m"].numpy()
        self.flops = {"gemm_fprop": 2.0 * T * F * H, "gemm_wgrad": 2.0 * F * H * T,
                      "gemm_grouped": 2.0 * float(counts.sum()) * N * K}
        qb = lambda r, c, both: (2.0 + (2 if both else 1) * (1 + 1 / 32)) * r * c
        self.bytes = {"quant_ffn_x": qb(T, H, True), "quant_ffn_w": qb(F, H, False),
                      "quant_ffn_dy": qb(T, F, True), "quant_moe_x": qb(MT, K, False),
                      "quant_moe_w": qb(G * N, K, False)}
        self.kernels = [
            ("quant_ffn_x", lambda: temx.quantize(d["ffn_X"], True, True, out=o["x_row"])),
            ("quant_ffn_w", lambda: temx.quantize(d["ffn_W"], True, False, out=o["w_row"])),
            ("quant_ffn_dy", lambda: temx.quantize(d["ffn_dY"], True, True, out=o["dy"])),
            ("gemm_fprop", lambda: temx.gemm(o["x_row"]["q_row"], o["x_row"]["s_row"], o["w_row"]["q_row"],
                                             o["w_row"]["s_row"], bias=d["ffn_b"], gelu=True, out=o["fprop"])),
            ("gemm_wgrad", lambda: temx.gemm(o["dy"]["q_col"], o["dy"]["s_col"], o["x_row"]["q_col"],
                                             o["x_row"]["s_col"], out=o["wgrad"])),
            ("quant_moe_x", lambda: temx.quantize(d["moe_X"], True, False, out=o["mx"])),
            ("quant_moe_w", lambda: temx.quantize(d["moe_W"], True, False, out=o["mw"])),
            ("gemm_grouped", lambda: temx.grouped_gemm(d["moe_m"], o["mx"]["q_row"], o["mx"]["s_row"],
                                                       o["mw"]["q_row"].view(G, N, K), o["mw"]["s_row"],
                                                       gelu=True, out=o["moe"])),
        ]
        self.outputs = [o["fprop"][0], o["fprop"][1], o["wgrad"][0], o["moe"][0], o["moe"][1]]
        # Backward kernels outside the step (reported under "next_rows"):
        #   dgrad  dX = dY W (M=8192, N=7168, K=18432) on the column-wise weight;
        #   dgelu  the GELU-backward GEMM at fprop shape (8192x18432x7168) reading
        #          the fprop's AUX (operands reused from the step: timing only);
        #   quant_dbias  dY row+col quantisation fused with its bias gradient.
        o["w_col"] = {"q_col": e(H, F), "s_col": e(H, pitch(F))}
        o["dx"] = (e(T, H, dt=torch.bfloat16), None)
        o["dgelu"] = (e(T, F, dt=torch.bfloat16), None)
        o["dy_b"] = {"q_row": e(T, F), "s_row": e(T, pitch(F)), "q_col": e(F, T), "s_col": e(F, pitch(T)),
                     "dbias": e(F, dt=torch.bfloat16)}
        o["ws"] = e(max(1, temx.binding.te_mx_quantize_dbias_workspace_size(T, F)))
        self.next_flops = {"gemm_dgrad": 2.0 * T * H * F, "gemm_dgelu": 2.0 * T * F * H}
        self.next_bytes = {"quant_dbias_ffn_dy": qb(T, F, True) + 2.0 * F,
                           "block_quant_ffn_x": qb(T, H, True), "block_quant_ffn_w": qb(F, H, True),
                           "block_quant_ffn_dy": qb(T, F, True),
                           "ln_quant_ffn_x": qb(T, H, True) + 8.0 * T + 4.0 * H,
                           "grouped_quant_moe_x": qb(MT, K, False), "grouped_quant_moe_dy": qb(MT, N, False)}
        self.next_flops["gemm_moe_wgrad"] = 2.0 * float(counts.sum()) * N * K
        self.next_flops["gemm_wgrad_accum_f32"] = 2.0 * F * H * T
        self.next_flops["gemm_fp32_scales_fprop"] = 2.0 * T * F * H
        self.next_bytes["block_quant_fp32_ffn_x"] = qb(T, H, True)     # fp32 scale per 128 = 1/32 B per element
        self.next_bytes["block_quant_fp32_ffn_w"] = qb(F, H, True)
        p32 = temx.te_mx_block_scale_pitch_fp32
        f32 = lambda r, c: torch.empty(r, c, dtype=torch.float32, device=dev)
        o["x32"] = {"q_row": e(T, H), "s_row": f32(T, p32(H)), "q_col": e(H, T), "s_col": f32(H, p32(T))}
        o["w32"] = {"q_row": e(F, H), "s_row": f32(F, p32(H)), "q_col": e(H, F), "s_col": f32(H, p32(F))}
        o["main_grad"] = torch.zeros(F, H, dtype=torch.float32, device=dev)   # fp32 weight-gradient accumulator
        # MoE expert wgrad: per-expert column-wise copies of X and dY, then dW_e = dY_e^T X_e
        gdev = d["moe_m"].to(torch.int32)
        o["gx"] = temx.quantize_colwise_grouped(d["moe_X"], gdev)
        o["gdy"] = temx.quantize_colwise_grouped(d["moe_dY"], gdev)
        o["dw"] = e(G, N, K, dt=torch.bfloat16)
        # Float8BlockScaling (E8M0-cast scales) quantisation of the same tensors:
        # 1x128 / 128x1 blocks for X and dY, 128x128 blocks for W (both copies).
        # LayerNorm -> MXFP8 of the ffn input (both orientations + mu / rsigma);
        # X stands in for the residual stream that the LayerNorm normalises.
        o["ln"] = {"q_row": o["x_row"]["q_row"], "s_row": o["x_row"]["s_row"], "q_col": o["x_row"]["q_col"],
                   "s_col": o["x_row"]["s_col"], "mu": e(T, dt=torch.float32), "rsigma": e(T, dt=torch.float32)}
        o["w_both"] = {"q_row": o["w_row"]["q_row"], "s_row": o["w_row"]["s_row"],
                       "q_col": o["w_col"]["q_col"], "s_col": o["w_col"]["s_col"]}
        self.next_kernels = [
            ("gemm_dgrad", lambda: temx.gemm(o["dy"]["q_row"], o["dy"]["s_row"], o["w_col"]["q_col"],
                                             o["w_col"]["s_col"], out=o["dx"])),
            ("gemm_dgelu", lambda: temx.gemm(o["x_row"]["q_row"], o["x_row"]["s_row"], o["w_row"]["q_row"],
                                             o["w_row"]["s_row"], out=o["dgelu"], dgelu_aux=o["fprop"][1])),
            ("quant_dbias_ffn_dy", lambda: temx.quantize(d["ffn_dY"], True, True, out=o["dy_b"], dbias=True,
                                                         workspace=o["ws"])),
            ("block_quant_ffn_x", lambda: temx.block_quantize(d["ffn_X"], False, True, True, out=o["x_row"])),
            ("block_quant_ffn_w", lambda: temx.block_quantize(d["ffn_W"], True, True, True, out=o["w_both"])),
            ("block_quant_ffn_dy", lambda: temx.block_quantize(d["ffn_dY"], False, True, True, out=o["dy_b"])),
            ("ln_quant_ffn_x", lambda: temx.layernorm_quantize(d["ffn_X"], d["ln_g"], d["ln_b"], 1e-5, True, True,
                                                               out=o["ln"])),
            ("grouped_quant_moe_x", lambda: temx.quantize_colwise_grouped(d["moe_X"], gdev, out=o["gx"])),
            ("grouped_quant_moe_dy", lambda: temx.quantize_colwise_grouped(d["moe_dY"], gdev, out=o["gdy"])),
            ("gemm_moe_wgrad", lambda: temx.grouped_gemm_wgrad(gdev, MT, o["gdy"], o["gx"], out=o["dw"])),
            ("gemm_wgrad_accum_f32", lambda: temx.gemm(o["dy"]["q_col"], o["dy"]["s_col"], o["x_row"]["q_col"],
                                                       o["x_row"]["s_col"], accumulate=o["main_grad"])),
            # Float8BlockScaling keeping FP32 scales: X (1x128 blocks) and W (128x128),
            # then the ffn fprop computed with those scales (bias + GELU + AUX)
            ("block_quant_fp32_ffn_x", lambda: temx.block_quantize_fp32(d["ffn_X"], False, True, True, out=o["x32"])),
            ("block_quant_fp32_ffn_w", lambda: temx.block_quantize_fp32(d["ffn_W"], True, True, True, out=o["w32"])),
            ("gemm_fp32_scales_fprop", lambda: temx.gemm_fp32_scales(o["x32"]["q_row"], o["x32"]["s_row"],
                                                                     o["w32"]["q_row"], o["w32"]["s_row"], True,
                                                                     bias=d["ffn_b"], gelu=True, out=o["fprop"])),
        ]
        temx.quantize(d["ffn_W"], False, True, out=o["w_col"])

    def run(self, events=None):
        for i, (_, fn) in enumerate(self.kernels):
            if events is not None:
                events[i][0].record()
            fn()
            if events is not None:
                events[i][1].record()


def time_device(step, steps, warmup, sampler):
    for _ in range(warmup):
        step.run()
    step.temx.te_mx_device_status()
    n = len(step.kernels)
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
           for _ in range(steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    start.record()
    for s in range(steps):
        step.run(evs[s])
    stop.record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    barrier()
    step.temx.te_mx_device_status()
    total_ms = start.elapsed_time(stop)
    per_kernel = {}
    for i, (name, _) in enumerate(step.kernels):
        per_kernel[name] = sum(evs[s][i][0].elapsed_time(evs[s][i][1]) for s in range(steps)) / steps
    return total_ms, per_kernel, clocks


def time_next(step, reps, fp8_peak, hbm_gbs, batches=5):
    """CUDA-event time of each backward kernel (after the step ran once): the
    median over `batches` batches of `reps` back-to-back launches (a single
    batch swung by up to 8 % between runs on the longer kernels)."""
    step.run()
    torch.cuda.synchronize()
    res = {}
    for name, fn in step.next_kernels:
        fn()
        torch.cuda.synchronize()
        per = []
        for _ in range(batches):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(reps):
                fn()
            b.record()
            torch.cuda.synchronize()
            per.append(a.elapsed_time(b) / reps)
        ms = sorted(per)[len(per) // 2]
        if name in step.next_flops:
            ach = step.next_flops[name] / (ms * 1e-3) / 1e12
            res[name] = {"us": ms * 1e3, "achieved": ach, "unit": "TFLOP/s", "frac": ach / fp8_peak}
        else:
            ach = step.next_bytes[name] / (ms * 1e-3) / 1e9
            res[name] = {"us": ms * 1e3, "achieved": ach, "unit": "GB/s", "frac": ach / hbm_gbs}
        res[name]["traffic"] = measured_traffic(name)
    step.temx.te_mx_device_status()
    return res


def time_e2e(pair, host, steps, warmup):
    """Same step through the public API with host buffers: every step copies
    its inputs host->device from pinned memory and its outputs back.  The
    steps are pipelined over two independent step instances (their own
    device buffers and pinned result buffers): while one instance computes,
    the other's inputs arrive on a copy stream and the previous results leave
    on another, so the two copy directions and the compute overlap.  Events
    keep every buffer from being reused before its last reader is done."""
    pinned_in = {k: v.pin_memory() for k, v in host.items()}
    pinned_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in st.outputs] for st in pair]
    h2d = sum(t.numel() * t.element_size() for t in pinned_in.values())
    d2h = sum(t.numel() * t.element_size() for t in pinned_out[0])
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = {k: [torch.cuda.Event(), torch.cuda.Event()] for k in ("in", "cmp", "out")}
    used = [False, False]

    def one(i):
        j = i % 2
        st = pair[j]
        with torch.cuda.stream(s_in):
            if used[j]:
                s_in.wait_event(ev["cmp"][j])        # this instance's last step has read its inputs
            for k, v in pinned_in.items():
                st.d[k].copy_(v, non_blocking=True)
            ev["in"][j].record(s_in)
        with torch.cuda.stream(s_cmp):
            s_cmp.wait_event(ev["in"][j])
            if used[j]:
                s_cmp.wait_event(ev["out"][j])       # its last results have left
            st.run()
            ev["cmp"][j].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["cmp"][j])
            for dst, src in zip(pinned_out[j], st.outputs):
                dst.copy_(src, non_blocking=True)
            ev["out"][j].record(s_out)
        used[j] = True

    for i in range(max(2, warmup // 2)):
        one(i)
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        one(i)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    barrier()
    return dt * 1e3 / steps, h2d, d2h


# ----------------------------------------------------------------------------- the smaller workloads

L2_BYTES = 129 << 20


def graph_time_us(launch, nsets, per_graph=24, replays=12):
    """Average device time of one launch, back to back: ``launch(i)`` enqueues
    the kernel on set i (its own inputs and outputs); ``per_graph`` launches
    cycling through the ``nsets`` sets are captured in one CUDA graph (so host
    launch cost does not pace kernels of a few microseconds) and the graph is
    replayed ``replays`` times between two CUDA events on the capture stream."""
    for i in range(nsets):                     # first calls: one-time host set-up outside the capture
        launch(i)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for j in range(per_graph):
            launch(j % nsets)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(replays):
            g.replay()
        b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e3 / (replays * per_graph)


def sets_for(bytes_per_set):
    """Rotating sets so that back-to-back launches touch more than twice the L2."""
    return max(2, int(np.ceil(2 * L2_BYTES / bytes_per_set)))


def qbytes(rows, cols, orientations):
    """Algorithmic bytes of an MXFP8 quantisation: 2 B read, 1 + 1/32 B written per element and orientation."""
    return (2.0 + orientations * (1 + 1 / 32)) * rows * cols


def gemm_bytes(M, N, K, bias, outputs):
    """Algorithmic bytes of a GEMM: each operand's codes and scales once, the bias, the bf16 outputs."""
    return (M + N) * K * (1 + 1 / 32) + (2.0 * N if bias else 0.0) + 2.0 * M * N * outputs


def time_configs(dev, fp8_peak, hbm_gbs):
    """Per-kernel device time of the tiny, QKV and FC1 workloads: every kernel
    launched back to back over rotating input/output sets larger than L2 (the
    tiny workload is smaller than L2 by nature), replayed from a CUDA graph.
    GEMMs report TFLOP/s against the FP8 peak and their algorithmic bytes
    against HBM; quantisers report GB/s against HBM."""
    import mxfp8_block_scaled_quantize_gb300 as temx
    from mxfp8_block_scaled_quantize_gb300 import workloads
    pitch = temx.te_mx_scale_pitch
    u8 = lambda *s: torch.empty(*s, dtype=torch.uint8, device=dev)
    bf = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device=dev)

    def quant_row(x, n):
        r, c = x.shape
        outs = [{"q_row": u8(r, c), "s_row": u8(r, pitch(c))} for _ in range(n)]
        xs = [x] + [x.clone() for _ in range(n - 1)]
        return lambda i: temx.quantize(xs[i], True, False, out=outs[i])

    def quant_both(x, n):
        r, c = x.shape
        outs = [{"q_row": u8(r, c), "s_row": u8(r, pitch(c)), "q_col": u8(c, r), "s_col": u8(c, pitch(r))}
                for _ in range(n)]
        xs = [x] + [x.clone() for _ in range(n - 1)]
        return lambda i: temx.quantize(xs[i], True, True, out=outs[i])

    def gemm_sets(qa, sa, qb, sb, n, bias=None, gelu=False):
        M, N = qa.shape[0], qb.shape[0]
        ops = [(qa, sa, qb, sb)] + [(qa.clone(), sa.clone(), qb.clone(), sb.clone()) for _ in range(n - 1)]
        outs = [(bf(M, N), bf(M, N) if gelu else None) for _ in range(n)]
        return lambda i: temx.gemm(*ops[i], bias=bias, gelu=gelu, out=outs[i])

    def row(us, flops=None, nbytes=None, n_sets=1):
        r = {"us": us, "sets": n_sets}
        if flops is not None:
            r.update({"tflops": flops / us / 1e6, "frac_fp8": flops / us / 1e6 / fp8_peak, "flops": flops})
        if nbytes is not None:
            r.update({"gbs": nbytes / us / 1e3, "frac_hbm": nbytes / us / 1e3 / hbm_gbs, "bytes": nbytes})
        return r

    res = {}
    # tiny: A, B [256x256], bias [256]
    t = workloads.make_tiny()
    a, b, bias = (t[k].to(dev) for k in ("A", "B", "bias"))
    qa = temx.quantize(a, True, True)
    qbm = temx.quantize(b, True, False)
    res["tiny"] = {
        "quant_a_both": row(graph_time_us(quant_both(a, 1), 1), nbytes=qbytes(256, 256, 2)),
        "quant_b_row": row(graph_time_us(quant_row(b, 1), 1), nbytes=qbytes(256, 256, 1)),
        "gemm_bias": row(graph_time_us(gemm_sets(qa["q_row"], qa["s_row"], qbm["q_row"], qbm["s_row"], 1, bias), 1),
                         flops=2.0 * 256 ** 3, nbytes=gemm_bytes(256, 256, 256, True, 1)),
        "note": "L2-resident by size; latency-bound",
    }
    # QKV: X [4096x1024], W [3072x1024], D = X W^T + b
    q = workloads.make_qkv()
    x, w, bias = (q[k].to(dev) for k in ("X", "W", "bias"))
    M, N, K = 4096, 3072, 1024
    qx, qw = temx.quantize(x, True, False), temx.quantize(w, True, False)
    n = sets_for(qbytes(M, K, 1)); res_q = {"quant_x_row": row(graph_time_us(quant_row(x, n), n), nbytes=qbytes(M, K, 1), n_sets=n)}
    n = sets_for(qbytes(N, K, 1)); res_q["quant_w_row"] = row(graph_time_us(quant_row(w, n), n), nbytes=qbytes(N, K, 1), n_sets=n)
    nb = gemm_bytes(M, N, K, True, 1)
    n = sets_for(nb)
    res_q["gemm_bias"] = row(graph_time_us(gemm_sets(qx["q_row"], qx["s_row"], qw["q_row"], qw["s_row"], n, bias), n),
                             flops=2.0 * M * N * K, nbytes=nb, n_sets=n)
    res["qkv"] = res_q
    del qx, qw
    # FC1: X [4096x1024] (outlier columns), W1 [4096x1024], dY [4096x4096]
    f = workloads.make_fc1()
    x, w, bias, dy = (f[k].to(dev) for k in ("X", "W", "bias", "dY"))
    M, N, K, T = 4096, 4096, 1024, 4096
    res_f = {}
    n = sets_for(qbytes(T, K, 2)); res_f["quant_x_both"] = row(graph_time_us(quant_both(x, n), n), nbytes=qbytes(T, K, 2), n_sets=n)
    n = sets_for(qbytes(N, K, 1)); res_f["quant_w_row"] = row(graph_time_us(quant_row(w, n), n), nbytes=qbytes(N, K, 1), n_sets=n)
    n = sets_for(qbytes(T, N, 2)); res_f["quant_dy_both"] = row(graph_time_us(quant_both(dy, n), n), nbytes=qbytes(T, N, 2), n_sets=n)
    qx, qw, qd = temx.quantize(x, True, True), temx.quantize(w, True, False), temx.quantize(dy, False, True)
    nb = gemm_bytes(M, N, K, True, 2)
    n = sets_for(nb)
    res_f["gemm_fprop_bias_gelu_aux"] = row(
        graph_time_us(gemm_sets(qx["q_row"], qx["s_row"], qw["q_row"], qw["s_row"], n, bias, True), n),
        flops=2.0 * M * N * K, nbytes=nb, n_sets=n)
    # wgrad dW [N x K] = dY^T X over T tokens: A = colwise(dY) [N x T], B = colwise(X) [K x T]
    nb = gemm_bytes(N, K, T, False, 1)
    n = sets_for(nb)
    res_f["gemm_wgrad"] = row(graph_time_us(gemm_sets(qd["q_col"], qd["s_col"], qx["q_col"], qx["s_col"], n), n),
                              flops=2.0 * N * K * T, nbytes=nb, n_sets=n)
    res["fc1"] = res_f
    temx.te_mx_device_status()
    return res


# ----------------------------------------------------------------------------- CPU oracle leg
#
# The oracle (numpy, fp64) is timed kernel by kernel on bounded samples of
# every workload, each on its own inputs:
#   quantisers  a slab of 64 rows (two 32-row blocks down each column), full
#               width, in the workload's orientations; GB/s of algorithmic
#               bytes (2 B read + 1 + 1/32 B written per element and
#               orientation) on 1 core (best of three), and on all cores with
#               every core of a spawn process pool quantising the slab for
#               about a second;
#   GEMMs       a 256 x 256 output block (the whole output for the tiny
#               workload), full K, with the workload's epilogue, on operands
#               the oracle quantised beforehand; TFLOP/s of 2 m n K (best of
#               two; numpy matmul on the BLAS threads of all cores).
# A full-size time is the work divided by that rate ("extrapolated").

CPU_SLAB_ROWS = 64
CPU_BLOCK = 256


def _workload_tensors(host=None):
    """Host (CPU) inputs of the five workloads; the ffn and moe ones are
    reused from the bench's own inputs when given."""
    from mxfp8_block_scaled_quantize_gb300 import workloads
    t, q, f = workloads.make_tiny(), workloads.make_qkv(), workloads.make_fc1()
    if host is None:
        ffn, moe = workloads.make_ffn(), workloads.make_moe()
        host = {"ffn_X": ffn["X"], "ffn_W": ffn["W"], "ffn_b": ffn["bias"], "ffn_dY": ffn["dY"],
                "moe_X": moe["X"], "moe_W": moe["W"].reshape(128 * 1536, 4096), "moe_m": moe["group_m"]}
    return {"tiny": {"A": t["A"], "B": t["B"], "bias": t["bias"]},
            "qkv": {"X": q["X"], "W": q["W"], "bias": q["bias"]},
            "fc1": {"X": f["X"], "W": f["W"], "bias": f["bias"], "dY": f["dY"]},
            "ffn": {"X": host["ffn_X"], "W": host["ffn_W"], "bias": host["ffn_b"], "dY": host["ffn_dY"]},
            "moe": {"X": host["moe_X"], "W": host["moe_W"], "m": host["moe_m"]}}


# (workload, kernel, kind, details): quant (tensor, orientations); gemm (M, N, K, how)
ORACLE_KERNELS = [
    ("tiny", "quant_a_both", "quant", ("A", 2)), ("tiny", "quant_b_row", "quant", ("B", 1)),
    ("tiny", "gemm_bias", "gemm", (256, 256, 256, "fprop_bias")),
    ("qkv", "quant_x_row", "quant", ("X", 1)), ("qkv", "quant_w_row", "quant", ("W", 1)),
    ("qkv", "gemm_bias", "gemm", (4096, 3072, 1024, "fprop_bias")),
    ("fc1", "quant_x_both", "quant", ("X", 2)), ("fc1", "quant_w_row", "quant", ("W", 1)),
    ("fc1", "quant_dy_both", "quant", ("dY", 2)),
    ("fc1", "gemm_fprop_bias_gelu_aux", "gemm", (4096, 4096, 1024, "fprop_gelu")),
    ("fc1", "gemm_wgrad", "gemm", (4096, 1024, 4096, "wgrad")),
    ("ffn", "quant_x_both", "quant", ("X", 2)), ("ffn", "quant_w_row", "quant", ("W", 1)),
    ("ffn", "quant_dy_both", "quant", ("dY", 2)),
    ("ffn", "gemm_fprop_bias_gelu_aux", "gemm", (8192, 18432, 7168, "fprop_gelu")),
    ("ffn", "gemm_wgrad", "gemm", (18432, 7168, 8192, "wgrad")),
    ("moe", "quant_x_row", "quant", ("X", 1)), ("moe", "quant_w_row", "quant", ("W", 1)),
    ("moe", "gemm_grouped_gelu_aux", "gemm", (131072, 1536, 4096, "grouped_gelu")),
]
# the kernels of the timed step (ffn + moe), with their names in the GPU line
STEP_ORACLE = {("ffn", "quant_x_both"): "quant_ffn_x", ("ffn", "quant_w_row"): "quant_ffn_w",
               ("ffn", "quant_dy_both"): "quant_ffn_dy", ("ffn", "gemm_fprop_bias_gelu_aux"): "gemm_fprop",
               ("ffn", "gemm_wgrad"): "gemm_wgrad", ("moe", "quant_x_row"): "quant_moe_x",
               ("moe", "quant_w_row"): "quant_moe_w", ("moe", "gemm_grouped_gelu_aux"): "gemm_grouped"}


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _quant_tasks(x, orient, rows):
    """The oracle calls of one quantiser sample: (function, bf16 slab) pairs."""
    from oracle import mx_oracle as O
    slab = _bits(x[:rows])
    return [(O.quantize_rowwise, slab)] + ([(O.quantize_colwise, slab)] if orient == 2 else [])


def _oracle_quantize_repeat(colwise, slab, reps):
    """Worker task of the all-cores quantiser rate: ``reps`` oracle
    quantisations of one slab (results dropped, so that only the slab
    travels to the worker)."""
    from oracle import mx_oracle as O
    for _ in range(reps):
        (O.quantize_colwise if colwise else O.quantize_rowwise)(slab)


def _gemm_sample(w, how, block):
    """Oracle operands of one GEMM sample (quantised outside the timing) and
    the call: returns (fn, flops)."""
    from oracle import mx_oracle as O
    if how == "wgrad":                        # dW = dY^T X: A = colwise(dY), B = colwise(X)
        qa, sa = O.quantize_colwise(_bits(w["dY"][:, :block]))
        qb, sb = O.quantize_colwise(_bits(w["X"][:, :block]))
        bias, gelu = None, False
    else:
        qa, sa = O.quantize_rowwise(_bits(w["X" if "X" in w else "A"][:block]))
        wb = w["W" if "W" in w else "B"][:block]
        qb, sb = O.quantize_rowwise(_bits(wb))
        bias = None if how == "grouped_gelu" else _bits(w["bias"][:block])
        gelu = how != "fprop_bias"
    return (lambda: O.mx_gemm(qa, sa, qb, sb, bias, gelu)), 2.0 * qa.shape[0] * qb.shape[0] * qa.shape[1]


def oracle_rates(tensors, pool=None, slab_rows=CPU_SLAB_ROWS, block=CPU_BLOCK, only=None, all_core_s=1.0):
    """Oracle rate of every kernel in ORACLE_KERNELS (or of those in ``only``):
    {(workload, kernel): {"value", "unit", "cores", "full_s_extrapolated", ...}}."""
    res = {}
    ncores = os.cpu_count() or 1
    for wl, name, kind, det in ORACLE_KERNELS:
        if only is not None and (wl, name) not in only:
            continue
        w = tensors[wl]
        if kind == "quant":
            key, orient = det
            x = w[key]
            rows = min(slab_rows, x.shape[0])
            nbytes = qbytes(rows, x.shape[1], orient)
            tasks = _quant_tasks(x, orient, rows)
            t1 = float("inf")
            for _ in range(3):                   # best of three (the first call pays numpy's warm-up)
                t0 = time.perf_counter()
                for fn, arg in tasks:
                    fn(arg)
                t1 = min(t1, time.perf_counter() - t0)
            r = {"value": nbytes / t1 / 1e9, "unit": "GB/s", "cores": 1,
                 "sample": f"{rows} x {x.shape[1]} rows, {orient} orientation(s)",
                 "full_s_extrapolated": qbytes(*x.shape, orient) / (nbytes / t1)}
            if pool is not None:
                # every core quantises the slab `reps` times (about all_core_s of work each)
                reps = max(1, int(round(all_core_s / t1)))
                slab = tasks[0][1]
                t0 = time.perf_counter()
                futs = [pool.submit(_oracle_quantize_repeat, o == 1, slab, reps)
                        for _ in range(ncores) for o in range(orient)]
                for f in futs:
                    f.result()
                tn = time.perf_counter() - t0
                done = ncores * reps * nbytes
                r["all_cores"] = {"value": done / tn / 1e9, "unit": "GB/s", "cores": ncores,
                                  "full_s_extrapolated": qbytes(*x.shape, orient) / (done / tn)}
        else:
            M, N, K, how = det
            fn, flops = _gemm_sample(w, how, block)
            t1 = float("inf")
            for _ in range(2):                   # best of two
                t0 = time.perf_counter()
                fn()
                t1 = min(t1, time.perf_counter() - t0)
            full = 2.0 * M * N * K
            r = {"value": flops / t1 / 1e12, "unit": "TFLOP/s", "cores": ncores,
                 "sample": ("whole output" if flops >= full else f"{block} x {block} output block, full K"),
                 "full_s_extrapolated": full / (flops / t1)}
        res[(wl, name)] = r
    return res


def _spawn_pool():
    """One worker process per host core (spawn: safe after CUDA initialised),
    started and warmed up before any timing."""
    import multiprocessing
    from concurrent.futures import ProcessPoolExecutor
    pool = ProcessPoolExecutor(max_workers=os.cpu_count() or 1, mp_context=multiprocessing.get_context("spawn"))
    warm = np.zeros((32, 32), np.uint16)
    for f in [pool.submit(_oracle_quantize_repeat, False, warm, 1) for _ in range(os.cpu_count() or 1)]:
        f.result()
    return pool


def step_gemm_flops():
    """GEMM FLOPs of the timed step (the ffn fprop and wgrad and the moe grouped GEMM)."""
    return sum(2.0 * det[0] * det[1] * det[2] for wl, name, kind, det in ORACLE_KERNELS
               if kind == "gemm" and (wl, name) in STEP_ORACLE)


def step_oracle_estimate(rates, all_cores=True):
    """Oracle time of one full step (extrapolated from the kernel rates) and
    the step's GEMM FLOPs / that time."""
    secs = 0.0
    for key in STEP_ORACLE:
        r = rates[key]
        secs += r["all_cores"]["full_s_extrapolated"] if (all_cores and "all_cores" in r) else r["full_s_extrapolated"]
    return secs, step_gemm_flops() / secs / 1e12


def cpu_baseline(host):
    """The oracle on the host cores, per kernel of every workload, and the
    step's rate extrapolated from the step kernels' rates."""
    tensors = _workload_tensors(host)
    pool = _spawn_pool()
    try:
        t0 = time.perf_counter()
        rates = oracle_rates(tensors, pool)
        spent = time.perf_counter() - t0
    finally:
        pool.shutdown()
    secs, v = step_oracle_estimate(rates)
    per = {}
    for (wl, name), r in rates.items():
        per.setdefault(wl, {})[name] = r
    return {"value": v, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": (f"extrapolated: the step's GEMM FLOPs / the sum of its kernels' oracle times, each "
                       f"extrapolated from a sample ({CPU_SLAB_ROWS}-row slabs of the quantisers on all cores, "
                       f"{CPU_BLOCK}x{CPU_BLOCK} output blocks of the GEMMs, full K); oracle step "
                       f"{secs:.1f} s; {spent:.1f} s of sampling"),
            "kernels": per}


# ----------------------------------------------------------------------------- distributed

_dist = False


def barrier():
    if _dist:
        torch.distributed.barrier()


def dist_max(x: float) -> float:
    """Max of x over all ranks (replicas report the slowest rank's time)."""
    if not _dist:
        return x
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank: float, world: int, ms_step_max: float) -> float:
    """Whole-job throughput of `world` replicas: all ranks' FLOPs / the slowest rank's step time."""
    return world * flops_per_rank / (ms_step_max * 1e-3) / 1e12


CASES = {
    "quant_both": "ffn X [8192x7168] row- and column-wise",
    "quant_row": "ffn W [18432x7168] row-wise",
    "block_quant_x": "Float8BlockScaling ffn X [8192x7168], 1x128 and 128x1 blocks, both orientations",
    "block_quant_w": "Float8BlockScaling ffn W [18432x7168], 128x128 blocks, both orientations",
    "ln_quant_x": "LayerNorm -> MXFP8 of ffn X [8192x7168], both orientations + mu/rsigma",
    "gemm_moe_wgrad": "moe expert wgrad dW_e = dY_e^T X_e, 128 experts, 1536 x 4096, per-expert column-wise operands",
    "grouped_quant_x": "per-expert column-wise MXFP8 of moe X [131072x4096] (experts padded to 128 tokens)",
    "gemm_qkv": "qkv fprop 4096x3072x1024, bias",
    "gemm_fc1": "fc1 fprop 4096x4096x1024, bias + GELU + AUX",
    "gemm_fc1_wgrad": "fc1 wgrad 4096x1024x4096 on column-wise operands",
    "gemm_ffn": "ffn fprop 8192x18432x7168, bias + GELU + AUX",
    "gemm_ffn_fp32": "ffn fprop 8192x18432x7168 with FP32 block scales (X 1x128, W 128x128), bias + GELU + AUX",
    "gemm_wgrad": "ffn wgrad 18432x7168x8192 on column-wise operands",
    "gemm_moe": "moe grouped 128 experts x 1536 x 4096, GELU + AUX",
}


def run_case(case: str, reps: int):
    """Run one kernel of the step `reps` times (for profilers); prints per-launch ms."""
    import mxfp8_block_scaled_quantize_gb300 as temx
    from mxfp8_block_scaled_quantize_gb300 import workloads
    dev = torch.device("cuda", 0)
    if case in ("quant_both", "quant_row", "block_quant_x", "block_quant_w", "ln_quant_x", "gemm_ffn", "gemm_wgrad",
                "gemm_ffn_fp32"):
        w = workloads.make_ffn()
    elif case in ("gemm_fc1", "gemm_fc1_wgrad"):
        w = workloads.make_fc1()
    elif case == "gemm_qkv":
        w = workloads.make_qkv()
    elif case in ("gemm_moe_wgrad", "grouped_quant_x"):
        w = None
    else:
        w = workloads.make_moe()
    if case == "quant_both":
        x = w["X"].to(dev)
        fn = lambda: temx.quantize(x, True, True)
    elif case == "quant_row":
        x = w["W"].to(dev)
        fn = lambda: temx.quantize(x, True, False)
    elif case == "block_quant_x":
        x = w["X"].to(dev)
        fn = lambda: temx.block_quantize(x, False, True, True)
    elif case == "block_quant_w":
        x = w["W"].to(dev)
        fn = lambda: temx.block_quantize(x, True, True, True)
    elif case == "ln_quant_x":
        x = w["X"].to(dev)
        g, b = (t.to(dev) for t in workloads.layernorm_params(x.shape[1], 410))
        fn = lambda: temx.layernorm_quantize(x, g, b, 1e-5, True, True)
    elif case in ("gemm_fc1", "gemm_ffn", "gemm_qkv"):
        qx = temx.quantize(w["X"].to(dev), True, False)
        qw = temx.quantize(w["W"].to(dev), True, False)
        b = w["bias"].to(dev)
        gelu = case != "gemm_qkv"
        fn = lambda: temx.gemm(qx["q_row"], qx["s_row"], qw["q_row"], qw["s_row"], bias=b, gelu=gelu)
    elif case == "gemm_ffn_fp32":
        qx = temx.block_quantize_fp32(w["X"].to(dev), False)
        qw = temx.block_quantize_fp32(w["W"].to(dev), True)
        b = w["bias"].to(dev)
        fn = lambda: temx.gemm_fp32_scales(qx["q_row"], qx["s_row"], qw["q_row"], qw["s_row"], True, bias=b,
                                           gelu=True)
    elif case in ("gemm_wgrad", "gemm_fc1_wgrad"):
        qd = temx.quantize(w["dY"].to(dev), False, True)
        qx = temx.quantize(w["X"].to(dev), False, True)
        fn = lambda: temx.gemm(qd["q_col"], qd["s_col"], qx["q_col"], qx["s_col"])
    elif case == "grouped_quant_x":
        g = workloads.make_moe_wgrad()
        gm = g["group_m"].to(torch.int32).to(dev)
        x = g["X"].to(dev)
        out = temx.quantize_colwise_grouped(x, gm)
        fn = lambda: temx.quantize_colwise_grouped(x, gm, out=out)
    elif case == "gemm_moe_wgrad":
        g = workloads.make_moe_wgrad()
        gm = g["group_m"].to(torch.int32).to(dev)
        gx = temx.quantize_colwise_grouped(g["X"].to(dev), gm)
        gdy = temx.quantize_colwise_grouped(g["dY"].to(dev), gm)
        total = int(g["group_m"].sum())
        fn = lambda: temx.grouped_gemm_wgrad(gm, total, gdy, gx)
    else:
        qx = temx.quantize(w["X"].to(dev), True, False)
        qw = temx.quantize(w["W"].view(128 * 1536, 4096).to(dev), True, False)
        gm = w["group_m"].to(dev)
        fn = lambda: temx.grouped_gemm(gm, qx["q_row"], qx["s_row"], qw["q_row"].view(128, 1536, 4096),
                                       qw["s_row"], gelu=True)
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(); fn(); b_.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b_))
    temx.te_mx_device_status()
    print(json.dumps({"case": case, "desc": CASES[case], "ms": times}))


def main():
    global _dist
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="temx", choices=["temx", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", choices=sorted(CASES), help="run one kernel of the step (for profilers)")
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args()
    if args.case:
        run_case(args.case, args.reps)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if world == 1 and args.gpus > 1 and args.impl == "temx":
        # not under torchrun: start one replica process per GPU through it
        sys.exit(run_replicas(args.gpus, sys.argv[1:]))

    if args.impl == "reference":
        if rank != 0:
            return
        reference_arm(args)
        return

    if world > 1:
        torch.distributed.init_process_group("nccl")
        _dist = True
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import mxfp8_block_scaled_quantize_gb300 as temx
    temx.binding.lib()
    peaks = load_peaks()
    host = build_inputs(dev)
    step = Step(host, dev)
    sampler = ClockSampler(local)
    total_ms, per_kernel, clocks = time_device(step, args.steps, args.warmup, sampler)
    ms_step = dist_max(total_ms / args.steps)
    gemm_flops = sum(step.flops.values())
    value = whole_job_tflops(gemm_flops, world, ms_step)

    # FP8 peak = 2 x the measured bf16 GEMM rate (nominal fp8:bf16 = 4.5:2.25); the
    # burst figure, since every timed region here lasts well under a second
    fp8_peak = 2.0 * peaks["bf16"]
    fp8_sustained = 2.0 * peaks["bf16_sustained"]
    kern = {}
    for name, ms in per_kernel.items():
        if name in step.flops:
            ach = step.flops[name] / (ms * 1e-3) / 1e12
            kern[name] = {"us": ms * 1e3, "achieved": ach, "unit": "TFLOP/s", "frac": ach / fp8_peak,
                          "frac_of_sustained": ach / fp8_sustained, "flops": step.flops[name]}
        else:
            ach = step.bytes[name] / (ms * 1e-3) / 1e9
            kern[name] = {"us": ms * 1e3, "achieved": ach, "unit": "GB/s", "frac": ach / peaks["hbm_gbs"],
                          "bytes": step.bytes[name]}
        kern[name]["traffic"] = measured_traffic(name)
    dom = max(per_kernel, key=per_kernel.get)
    dk = kern[dom]
    traffic = measured_traffic(dom)
    roofline = {"kernel": dom, "bound": "tensor" if dk["unit"] == "TFLOP/s" else "hbm",
                "achieved": dk["achieved"], "peak": fp8_peak if dk["unit"] == "TFLOP/s" else peaks["hbm_gbs"],
                "unit": dk["unit"], "frac": dk["frac"], "traffic": traffic,
                "traffic_source": ("ncu dram__bytes_read.sum + dram__bytes_write.sum per launch, recorded in "
                                   "profiles/traffic.json for this kernel's current source (matched by hash)"
                                   if traffic is not None else "no capture of the current source"),
                "peak_source": (f"{peaks['source']}: 2 x bf16 burst {peaks['bf16']} TFLOP/s"
                                if dk["unit"] == "TFLOP/s" else f"{peaks['source']}: HBM copy {peaks['hbm_gbs']} GB/s")}
    if dk["unit"] == "TFLOP/s":
        roofline["frac_of_sustained"] = dk["achieved"] / fp8_sustained
    q_total = sum(step.bytes.values())
    qms = sum(per_kernel[n] for n in step.bytes)
    gms = sum(per_kernel[n] for n in step.flops)

    next_rows = time_next(step, 6, fp8_peak, peaks["hbm_gbs"])
    configs = time_configs(dev, fp8_peak, peaks["hbm_gbs"])
    e2e_ms, h2d, d2h = time_e2e((step, Step(host, dev)), host, max(4, args.steps // 4), args.warmup)
    e2e_ms = dist_max(e2e_ms)
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 x e4m3 -> fp32 accumulate, bf16 in/out",
        "data": "synthetic (seeded generators, shapes and distributions of the workloads)",
        "config": {"workload": WORKLOAD, "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (every operand > 126 MB except bias/group sizes)"},
        "gemm_tflops": gemm_flops / (gms * 1e-3) / 1e12, "gemm_frac": gemm_flops / (gms * 1e-3) / 1e12 / fp8_peak,
        "quantize_gbs": q_total / (qms * 1e-3) / 1e9, "quantize_frac": q_total / (qms * 1e-3) / 1e9 / peaks["hbm_gbs"],
        "kernels": kern, "roofline": roofline, "clocks": clocks, "next_rows": next_rows, "configs": configs,
        "gpu_launches": len(step.kernels) * args.steps,
        "e2e": {"value": whole_job_tflops(gemm_flops, world, e2e_ms), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
    }
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline({k: v.cpu() if v.is_cuda else v for k, v in host.items()})
    if rank == 0:
        print(json.dumps(out))
    if _dist:
        torch.distributed.destroy_process_group()


def replica_command(n: int, script: str, argv, port: int):
    """torchrun command line that starts ``n`` processes of ``script`` on this
    node (one per GPU), rendezvous on 127.0.0.1."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
            "--master-addr=127.0.0.1", f"--master-port={port}", script, *argv]


def run_replicas(n: int, argv) -> int:
    """Start ``n`` replicas of this bench (one per GPU) under torchrun and
    return its exit status; rank 0 prints the JSON line."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    return subprocess.call(replica_command(n, os.path.abspath(__file__), list(argv), port))


def reference_arm(args):
    """The oracle's rate on the timed step's workload: every step samples each
    step kernel (quantiser slabs on all host cores, GEMM blocks on the BLAS
    threads) and extrapolates the full step; value = the step's GEMM FLOPs /
    the mean extrapolated step time."""
    tensors = _workload_tensors()
    pool = _spawn_pool()
    only = set(STEP_ORACLE)
    slab, block = CPU_SLAB_ROWS, CPU_BLOCK
    # keep the whole run within a few minutes: about 150 s over all steps
    budget = 150.0 / max(1, args.steps + args.warmup)
    core_s = min(1.0, max(0.05, budget / 10))
    t0 = time.perf_counter()
    oracle_rates(tensors, pool, slab, block, only, core_s)
    if time.perf_counter() - t0 > budget:
        slab, block = 32, 128
    for _ in range(max(0, args.warmup - 1)):
        oracle_rates(tensors, pool, slab, block, only, core_s)
    secs, wall = [], time.perf_counter()
    for _ in range(args.steps):
        rates = oracle_rates(tensors, pool, slab, block, only, core_s)
        secs.append(step_oracle_estimate(rates)[0])
    wall = time.perf_counter() - wall
    pool.shutdown()
    step_s = statistics.mean(secs)
    v = step_gemm_flops() / step_s / 1e12
    sample = (f"extrapolated: per step, {slab}-row slabs of each quantiser (all {os.cpu_count()} cores, one slab "
              f"per core) and a {block}x{block} output block (full K) of each GEMM (BLAS threads); the step "
              f"time is the sum of the kernels' extrapolated full-size times; {wall:.1f} s of sampling")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded generators)", "config": {"workload": WORKLOAD, "sample": sample},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))


if __name__ == "__main__":
    main()
