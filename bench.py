#!/usr/bin/env python
"""Benchmark of the block-scaled microscaling hot path on GB300.

Default step (workload ``dense_mlp``, the Qwen3-8B-shaped MLP linear): MXFP8 row-wise + column-wise
quantization of X [8192, 4096], W [12288, 4096] and dY [8192, 12288], then the three MXFP8
block-scaled GEMMs FPROP (Y = X W^T), DGRAD (dX = dY W) and WGRAD (dW = dY^T X) with BF16 output.
The metric is the step's GEMM throughput with its quantization included: 2.474 TFLOP per step /
step time.  Other workloads (``--workload moe|moe_mxfp8|dense_fp8_blockwise|dense_nvfp4|wgrad|weight_sync``)
time the NVFP4 paths, the grouped MXFP8 MoE layer, blockwise FP8 (power-of-two scales on the MXFP8 GEMM) and
the NVFP4 pretraining linear layer with the dequantized-backward GEMM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mxnum|reference] [--workload ...]

Under torchrun (N > 1) every rank runs an independent replica of the step (the path has no
exchange step); the reported value is all ranks' work over the slowest rank's time.  ``--impl
reference`` times the CPU oracle on a bounded sample of the same workload on this host's cores.
One JSON line is printed by rank 0.
"""
from __future__ import annotations

import argparse
import csv
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "quantize GB/s vs ~8 TB/s HBM; MXFP8/NVFP4 scaled-GEMM TFLOP/s vs dense peak"
# Tensor peaks of the GEMMs' own types from the measured BF16 peak: NVIDIA's per-GPU dense figures for
# the 8-GPU HGX B300 board (BF16 2.25, FP8 4.5, NVFP4 13.5 PFLOP/s; its datasheet prints 36 / 72 / 144
# PFLOP/s per board with 2:4 sparsity for BF16 and FP8, and 108 dense for FP4) fix the ratios.
FP8_OVER_BF16 = 2.0
FP4_OVER_BF16 = 6.0
# Published dense peaks of one GB300 (the GB300 NVL72 specification: FP4 1,080 PFLOP/s dense, FP8/FP6
# 720 and FP16/BF16 360 PFLOP/s with 2:4 sparsity, per 72 GPUs), the denominators of the >= 60 % bar.
HEAD_START_CYCLES = 2_000_000     # about 1 ms of SM clock: longer than the host needs to queue the first calls
DATASHEET = {"bf16": 2500.0, "fp8": 5000.0, "fp4": 15000.0,
             "source": "GB300 NVL72 specification / 72 GPUs, dense (FP4 1080 PF dense; FP8 720 and BF16 360 PF "
                       "sparse, halved)"}


def recorded_traffic(kernel: str):
    """Per-launch DRAM bytes (read + write) of `kernel` from the committed ncu capture, or None when
    the kernel's source has changed since the counters were taken."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic_dense_mlp.json")) as f:
            rec = json.load(f)["kernels"][kernel]
        with open(os.path.join(ROOT, rec["source"]), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != rec["sha256"]:
                return None
        return int(rec["mean_bytes_per_launch"])
    except Exception:
        return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------------------------------------
# clocks sampling during the timed region
# ------------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"mxnum_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu_index), "-lms", "100"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for r in csv.reader(f):
                if len(r) >= 9:
                    rows.append([c.strip() for c in r])
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        # samples under load: power above the midpoint of the observed range
        if power:
            thr = (max(power) + min(power)) / 2
            loaded = [float(r[1]) for r in rows if r[3].replace(".", "").isdigit() and float(r[3]) >= thr
                      and r[1].replace(".", "").isdigit()]
        else:
            loaded = sm
        return {"sm_mhz": statistics.median(loaded or sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons, "samples": len(rows),
                "power_w_max": max(power) if power else None}


# ------------------------------------------------------------------------------------------------
# workloads on the device
# ------------------------------------------------------------------------------------------------
class Tiny:
    """The tiny check: MXFP8 row + column quantize of X [256, 1024] (N(0, 1) with 0.5 % outliers x50, an
    all-zero block and a subnormal-only block) and W [512, 1024] N(0, 0.02) in one launch, the
    dequantize round trip of X, and the MXFP8 FPROP GEMM 256 x 512 x 1024 with BF16 output.  Every
    kernel here is latency-bound (a few microseconds each)."""
    name = "tiny"
    unit = "TFLOP/s"
    dtype = "e4m3 (f32 accumulate, bf16 out)"
    graph = True          # launch-bound: also timed as one CUDA graph per step
    e2e_pipelined = False  # and its end-to-end copies run serially (staging copies would only add launches)

    def __init__(self, mx, torch, dev, data=None):
        import synthetic
        self.mx, self.torch, self.dev = mx, torch, dev
        d = data or synthetic.tiny()
        bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        self.x, self.w = bf(d["x"]), bf(d["w"])
        self.M, self.K = self.x.shape
        self.N = self.w.shape[0]
        self.qx = mx.alloc_mxfp8(self.M, self.K, dev)
        self.qw = mx.alloc_mxfp8(self.N, self.K, dev)
        self.xdq = torch.empty_like(self.x)
        self.y = torch.empty((self.M, self.N), dtype=torch.bfloat16, device=dev)
        self.launches_per_step = 3

    def ops(self):
        mx, M, N, K = self.mx, self.M, self.N, self.K
        return [
            ("quant", "mxfp8 row+col X+W (one launch)", 1, (M + N) * K * (2 + 2 + 2 / 32),
             lambda: mx.mx_quantize_mxfp8_batched([(self.x, self.qx), (self.w, self.qw)])),
            ("dq", "mxfp8 DQ X", 1, M * K * (1 + 1 / 32 + 2),
             lambda: mx.mx_dequantize_bf16(mx.MX_FMT_MXFP8, self.qx["q_row"], self.qx["s_row"], None, 0, M, K, self.xdq)),
            ("gemm8", "FPROP", 0, 2.0 * M * N * K,
             lambda: mx.mx_scaled_gemm(mx.MX_FMT_MXFP8, self.qx["q_row"], self.qx["s_row"], None, 0, self.qw["q_row"],
                                       self.qw["s_row"], None, 0, M, N, K, self.y)),
        ]

    def e2e_inputs(self):
        return [self.x, self.w]

    def e2e_outputs(self):
        return [self.y, self.xdq]

    def config(self):
        return {"workload": "tiny: MXFP8 row+col quantize X 256x1024 + W 512x1024, DQ round trip, FPROP 256x512x1024",
                "note": "latency-bound at this size (parity case)"}


class DenseMLP:
    """MXFP8 quantize X, W, dY (row + column) + FPROP, DGRAD, WGRAD (Qwen3-8B MLP shapes)."""
    name = "dense_mlp"

    def __init__(self, mx, torch, dev, tokens=8192, hidden=4096, ffn=12288, host_inputs=None):
        import synthetic
        self.mx, self.torch, self.dev = mx, torch, dev
        self.T, self.H, self.F = tokens, hidden, ffn
        data = host_inputs or synthetic.dense_mlp(tokens, hidden, ffn)
        self.host = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16) for k, v in data.items()}
        self.x = self.host["x"].to(dev)
        self.w = self.host["w"].to(dev)
        self.dy = self.host["dy"].to(dev)
        self.qx = mx.alloc_mxfp8(tokens, hidden, dev)
        self.qw = mx.alloc_mxfp8(ffn, hidden, dev)
        self.qdy = mx.alloc_mxfp8(tokens, ffn, dev)
        self.y = torch.empty((tokens, ffn), dtype=torch.bfloat16, device=dev)
        self.dx = torch.empty((tokens, hidden), dtype=torch.bfloat16, device=dev)
        self.dw = torch.empty((ffn, hidden), dtype=torch.bfloat16, device=dev)
        T, H, F = tokens, hidden, ffn
        self.gemm_flops = [2.0 * T * F * H, 2.0 * T * H * F, 2.0 * F * H * T]
        self.quant_elems = [T * H + F * H + T * F]      # X, W, dY in one batched launch
        self.launches_per_step = 4

    def ops(self):
        """The step as a list of (kind, label, callable); kinds: quant / gemm."""
        mx = self.mx
        F8 = mx.MX_FMT_MXFP8
        T, H, F = self.T, self.H, self.F
        return [
            ("quant", "mxfp8_quantize X+W+dY (one launch)",
             lambda: mx.mx_quantize_mxfp8_batched([(self.x, self.qx), (self.w, self.qw), (self.dy, self.qdy)])),
            ("gemm", "FPROP", lambda: mx.mx_scaled_gemm(F8, self.qx["q_row"], self.qx["s_row"], None, 0,
                                                         self.qw["q_row"], self.qw["s_row"], None, 0, T, F, H, self.y)),
            ("gemm", "DGRAD", lambda: mx.mx_scaled_gemm(F8, self.qdy["q_row"], self.qdy["s_row"], None, 0,
                                                         self.qw["q_col"], self.qw["s_col"], None, 0, T, H, F, self.dx)),
            ("gemm", "WGRAD", lambda: mx.mx_scaled_gemm(F8, self.qdy["q_col"], self.qdy["s_col"], None, 0,
                                                         self.qx["q_col"], self.qx["s_col"], None, 0, F, H, T, self.dw)),
        ]

    def units_per_step(self):
        return sum(self.gemm_flops) / 1e12      # TFLOP

    def quant_bytes(self):
        # row + column copies: 2 B read + 2 x 1 B codes + 2 x 1/32 B scales per element
        return [e * (2 + 2 + 2 / 32) for e in self.quant_elems]

    # end-to-end: every step's inputs come from pinned host memory and its results go back to pinned
    # host memory; two device buffer sets and separate copy streams let the copies of one step overlap
    # the kernels of its neighbours (the inputs of step i + 1 arrive while step i computes, the results of
    # step i - 1 leave meanwhile)
    def e2e_setup(self):
        t = self.torch
        self.hx = self.host["x"].pin_memory()
        self.hw = self.host["w"].pin_memory()
        self.hdy = self.host["dy"].pin_memory()
        self.slots = []
        for _ in range(2):
            self.slots.append({
                "x": t.empty_like(self.x), "w": t.empty_like(self.w), "dy": t.empty_like(self.dy),
                "y": t.empty_like(self.y), "dx": t.empty_like(self.dx), "dw": t.empty_like(self.dw),
                "hy": t.empty(self.y.shape, dtype=t.bfloat16).pin_memory(),
                "hdx": t.empty(self.dx.shape, dtype=t.bfloat16).pin_memory(),
                "hdw": t.empty(self.dw.shape, dtype=t.bfloat16).pin_memory()})
        self.s_in, self.s_out = t.cuda.Stream(), t.cuda.Stream()
        ev = lambda: [t.cuda.Event(), t.cuda.Event()]
        self.ev_in, self.ev_done, self.ev_out = ev(), ev(), ev()
        self.h2d = sum(a.numel() * 2 for a in (self.hx, self.hw, self.hdy))
        self.d2h = sum(self.slots[0][k].numel() * 2 for k in ("hy", "hdx", "hdw"))

    def e2e_run(self, steps):
        """Run `steps` pipelined end-to-end steps; returns ms per step (CUDA events around all of it)."""
        t = self.torch
        cur = t.cuda.current_stream()
        start, end = t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True)
        start.record(self.s_in)
        for i in range(steps):
            k = i % 2
            sl = self.slots[k]
            with t.cuda.stream(self.s_in):
                if i >= 2:
                    self.s_in.wait_event(self.ev_done[k])          # step i - 2 has read these inputs
                sl["x"].copy_(self.hx, non_blocking=True)
                sl["w"].copy_(self.hw, non_blocking=True)
                sl["dy"].copy_(self.hdy, non_blocking=True)
                self.ev_in[k].record(self.s_in)
            cur.wait_event(self.ev_in[k])
            if i >= 2:
                cur.wait_event(self.ev_out[k])                     # step i - 2's results have left
            self.x, self.w, self.dy = sl["x"], sl["w"], sl["dy"]
            self.y, self.dx, self.dw = sl["y"], sl["dx"], sl["dw"]
            for _, _, f in self.ops():
                f()
            self.ev_done[k].record(cur)
            with t.cuda.stream(self.s_out):
                self.s_out.wait_event(self.ev_done[k])
                sl["hy"].copy_(sl["y"], non_blocking=True)
                sl["hdx"].copy_(sl["dx"], non_blocking=True)
                sl["hdw"].copy_(sl["dw"], non_blocking=True)
                self.ev_out[k].record(self.s_out)
        end.record(self.s_out)
        t.cuda.synchronize()
        return start.elapsed_time(end) / steps


class MoE:
    """Qwen3-30B-A3B expert layer, NVFP4 forward with dequantized-BF16 backward operands:
    per-token quantize of the 65536 expert-sorted rows, 16x16 2D quantize of 128 experts' gate|up
    (1536x2048) and down (2048x768) weights, the two grouped NVFP4 GEMMs, per-token quantize of the
    down-projection input, and DQ(Q(w)) of both weight stacks."""
    name = "moe"

    unit = "TFLOP/s"

    def __init__(self, mx, torch, dev, experts=128, data=None):
        import synthetic
        self.mx, self.torch, self.dev = mx, torch, dev
        d = data or synthetic.moe(experts=experts)
        bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        x = bf(d["x"])
        self.rows = int(d["group_offsets"][-1])
        # the expert-sorted activation rows are the GEMM's input (the routing gather is setup)
        self.a = x.index_select(0, torch.from_numpy(d["row_token"]).to(dev)).contiguous()
        del x
        self.down_in = bf(d["down_in"])
        self.wgu = bf(d["w_gate_up"])
        self.wd = bf(d["w_down"])
        self.offs = torch.from_numpy(d["group_offsets"]).to(dev)
        G, O1, H = self.wgu.shape
        _, O2, F = self.wd.shape
        self.G, self.H, self.F, self.O1, self.O2 = G, H, F, O1, O2
        self.qa = mx.alloc_nvfp4_rows_grouped(self.rows, G, H, dev)
        self.qdn = mx.alloc_nvfp4_rows_grouped(self.rows, G, F, dev)
        self.qgu = mx.alloc_nvfp4_weight_2d(G, O1, H, dev)
        self.qwd = mx.alloc_nvfp4_weight_2d(G, O2, F, dev)
        self.y1 = torch.empty((self.rows, O1), dtype=torch.bfloat16, device=dev)
        self.y2 = torch.empty((self.rows, O2), dtype=torch.bfloat16, device=dev)
        self.dq_gu = torch.empty((G * O1, H), dtype=torch.bfloat16, device=dev)
        self.dq_d = torch.empty((G * O2, F), dtype=torch.bfloat16, device=dev)
        self.launches_per_step = 10

    def gemm_min_bytes(self, N, K):
        """HBM bytes a grouped NVFP4 GEMM cannot avoid: A and B codes and block scales read once, the
        FP32 row and group scales, the BF16 output written once."""
        R, G = self.rows, self.G
        return R * K * (0.5 + 1 / 16) + G * N * K * (0.5 + 1 / 16) + 4 * R + 4 * G + 2 * R * N

    def ops(self):
        mx, F4 = self.mx, self.mx.MX_FMT_NVFP4
        G, H, F, O1, O2, R = self.G, self.H, self.F, self.O1, self.O2, self.rows
        q = self.qgu
        w = self.qwd
        return [
            ("quant", "nvfp4_per_token A", 1, R * H * (2 + 0.5 + 1 / 16) + 4 * R,
             lambda: mx.mx_nvfp4_quantize_per_token_grouped(self.a, self.offs, self.qa["q"], self.qa["s"], self.qa["s2"])),
            ("quant", "nvfp4_weight_2d gate_up", 1, G * O1 * H * (2 + 1 + 2 / 16),
             lambda: mx.mx_nvfp4_quantize_weight_2d(self.wgu, q["q_row"], q["s_row"], q["q_col"], q["s_col"], q["s_w"], q["ws"])),
            ("quant", "nvfp4_weight_2d down", 1, G * O2 * F * (2 + 1 + 2 / 16),
             lambda: mx.mx_nvfp4_quantize_weight_2d(self.wd, w["q_row"], w["s_row"], w["q_col"], w["s_col"], w["s_w"], w["ws"])),
            ("gemm4", "grouped gate_up", 0, 2.0 * R * O1 * H,
             lambda: mx.mx_grouped_scaled_gemm(F4, self.offs, self.qa["q"], self.qa["s"], self.qa["s2"], q["q_row"],
                                               q["s_row"], q["s_w"], O1, H, self.y1),
             self.gemm_min_bytes(O1, H)),
            ("quant", "nvfp4_per_token down input", 1, R * F * (2 + 0.5 + 1 / 16) + 4 * R,
             lambda: mx.mx_nvfp4_quantize_per_token_grouped(self.down_in, self.offs, self.qdn["q"], self.qdn["s"],
                                                            self.qdn["s2"])),
            ("gemm4", "grouped down", 0, 2.0 * R * O2 * F,
             lambda: mx.mx_grouped_scaled_gemm(F4, self.offs, self.qdn["q"], self.qdn["s"], self.qdn["s2"], w["q_row"],
                                               w["s_row"], w["s_w"], O2, F, self.y2),
             self.gemm_min_bytes(O2, F)),
            ("dq", "dequantize gate_up DQ(Q(w))", 1, G * O1 * H * (0.5 + 1 / 16 + 2),
             lambda: mx.mx_dequantize_bf16(F4, q["q_row"], q["s_row"], q["s_w"], mx.MX_SCOPE_GROUP, G * O1, H, self.dq_gu,
                                           group_rows=O1)),
            ("dq", "dequantize down DQ(Q(w))", 1, G * O2 * F * (0.5 + 1 / 16 + 2),
             lambda: mx.mx_dequantize_bf16(F4, w["q_row"], w["s_row"], w["s_w"], mx.MX_SCOPE_GROUP, G * O2, F, self.dq_d,
                                           group_rows=O2)),
        ]

    def config(self):
        return {"workload": "moe: Qwen3-30B-A3B expert layer, NVFP4 per-token + 2D weights + grouped GEMMs + DQ(Q(w))",
                "tokens": 8192, "routed_rows": self.rows, "experts": self.G, "hidden": self.H, "ffn": self.F}

    def e2e_inputs(self):
        return [self.a, self.down_in, self.wgu, self.wd]

    def e2e_outputs(self):
        return [self.y1, self.y2, self.dq_gu, self.dq_d]


    def aux_ops(self):
        """Four-over-Six variants of the two NVFP4 quantizers on the same tensors (reported beside the
        step, not part of it)."""
        mx, G, H, O1, R = self.mx, self.G, self.H, self.O1, self.rows
        if not hasattr(self, "q46"):
            self.q46 = mx.alloc_nvfp4_rows(R, H, self.dev)
            self.w46 = mx.alloc_nvfp4_weight_2d(G, O1, H, self.dev)
        q, w = self.q46, self.w46
        return [
            ("quant", "nvfp4_per_token 4/6 A", 1, R * H * (2 + 0.5 + 1 / 16) + 4 * R,
             lambda: mx.mx_nvfp4_quantize_per_token_46(self.a, q["q"], q["s"], q["s2"])),
            ("quant", "nvfp4_weight_2d 4/6 gate_up", 1, G * O1 * H * (2 + 1 + 2 / 16),
             lambda: mx.mx_nvfp4_quantize_weight_2d_46(self.wgu, w["q_row"], w["s_row"], w["q_col"], w["s_col"],
                                                       w["s_w"], w["ws"])),
        ]


class MoE8(MoE):
    """The same Qwen3-30B-A3B expert layer with MXFP8 instead of NVFP4: row-wise MXFP8 of the 65536
    expert-sorted rows (grouped scale layout) and of the 128 experts' stacked gate|up and down weights,
    the two grouped MXFP8 GEMMs, row-wise MXFP8 of the down-projection input."""
    name = "moe_mxfp8"
    unit = "TFLOP/s"
    dtype = "e4m3 (f32 accumulate, bf16 out)"

    def __init__(self, mx, torch, dev, experts=128):
        import synthetic
        self.mx, self.torch, self.dev = mx, torch, dev
        d = synthetic.moe(experts=experts)
        bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        x = bf(d["x"])
        self.rows = int(d["group_offsets"][-1])
        self.a = x.index_select(0, torch.from_numpy(d["row_token"]).to(dev)).contiguous()
        self.down_in = bf(d["down_in"])
        G, O1, H = d["w_gate_up"].shape
        _, O2, F = d["w_down"].shape
        self.wgu = bf(d["w_gate_up"]).reshape(G * O1, H)
        self.wd = bf(d["w_down"]).reshape(G * O2, F)
        self.offs = torch.from_numpy(d["group_offsets"]).to(dev)
        self.G, self.H, self.F, self.O1, self.O2 = G, H, F, O1, O2
        u8 = lambda n: torch.zeros(n, dtype=torch.uint8, device=dev)
        R = self.rows
        self.qa, self.sa = torch.empty((R, H), dtype=torch.uint8, device=dev), u8(mx.grouped_scale_bytes(R, G, H, 32))
        self.qdn, self.sdn = torch.empty((R, F), dtype=torch.uint8, device=dev), u8(mx.grouped_scale_bytes(R, G, F, 32))
        self.qgu = mx.alloc_mxfp8(G * O1, H, dev, rowwise=True, colwise=False)
        self.qwd = mx.alloc_mxfp8(G * O2, F, dev, rowwise=True, colwise=False)
        self.y1 = torch.empty((R, O1), dtype=torch.bfloat16, device=dev)
        self.y2 = torch.empty((R, O2), dtype=torch.bfloat16, device=dev)
        self.launches_per_step = 6

    def gemm_min_bytes(self, N, K):
        """HBM bytes a grouped MXFP8 GEMM cannot avoid: A and B codes and scales read once, the BF16
        output written once."""
        R, G = self.rows, self.G
        return R * K * (1 + 1 / 32) + G * N * K * (1 + 1 / 32) + 2 * R * N

    def ops(self):
        mx, F8 = self.mx, self.mx.MX_FMT_MXFP8
        G, H, F, O1, O2, R = self.G, self.H, self.F, self.O1, self.O2, self.rows
        per = 2 + 1 + 1 / 32
        return [
            ("quant", "mxfp8 routed rows A", 1, R * H * per,
             lambda: mx.mx_quantize_mxfp8_grouped(self.a, self.offs, self.qa, self.sa)),
            ("quant", "mxfp8 weights gate_up", 1, G * O1 * H * per,
             lambda: mx.mx_quantize_mxfp8(self.wgu, self.qgu["q_row"], self.qgu["s_row"])),
            ("quant", "mxfp8 weights down", 1, G * O2 * F * per,
             lambda: mx.mx_quantize_mxfp8(self.wd, self.qwd["q_row"], self.qwd["s_row"])),
            ("gemm8", "grouped gate_up", 0, 2.0 * R * O1 * H,
             lambda: mx.mx_grouped_scaled_gemm(F8, self.offs, self.qa, self.sa, None, self.qgu["q_row"],
                                               self.qgu["s_row"], None, O1, H, self.y1),
             self.gemm_min_bytes(O1, H)),
            ("quant", "mxfp8 down input", 1, R * F * per,
             lambda: mx.mx_quantize_mxfp8_grouped(self.down_in, self.offs, self.qdn, self.sdn)),
            ("gemm8", "grouped down", 0, 2.0 * R * O2 * F,
             lambda: mx.mx_grouped_scaled_gemm(F8, self.offs, self.qdn, self.sdn, None, self.qwd["q_row"],
                                               self.qwd["s_row"], None, O2, F, self.y2),
             self.gemm_min_bytes(O2, F)),
        ]

    def aux_ops(self):
        return []

    def config(self):
        c = super().config()
        c["workload"] = "moe_mxfp8: Qwen3-30B-A3B expert layer, MXFP8 routed rows + weights + grouped MXFP8 GEMMs"
        return c


class WGrad:
    """Llama-3-8B MLP WGRAD in NVFP4: RHT16 along tokens + 1x16 column-wise quantize with a
    per-tensor scale (SR on dY, RNE on X), then dW = dY^T X over K = 32768 tokens."""
    name = "wgrad"
    unit = "TFLOP/s"

    def __init__(self, mx, torch, dev, data=None, tokens=32768):
        import synthetic
        self.mx, self.torch, self.dev = mx, torch, dev
        d = data or synthetic.wgrad(tokens=tokens)
        bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        self.x, self.dy = bf(d["x"]), bf(d["dy"])
        self.rht_seed, self.sr_seed = d["rht_seed"], d["sr_seed"]
        T, H = self.x.shape
        F = self.dy.shape[1]
        self.T, self.H, self.F = T, H, F
        u8 = lambda n: torch.empty(n, dtype=torch.uint8, device=dev)
        self.qdy, self.sdy = torch.empty((F, T // 2), dtype=torch.uint8, device=dev), u8(mx.scale_bytes(F, T, 16))
        self.qx, self.sx = torch.empty((H, T // 2), dtype=torch.uint8, device=dev), u8(mx.scale_bytes(H, T, 16))
        self.Sdy = torch.empty(1, dtype=torch.float32, device=dev)
        self.Sx = torch.empty(1, dtype=torch.float32, device=dev)
        self.ws1, self.ws2 = u8(16), u8(16)
        self.dw = torch.empty((F, H), dtype=torch.bfloat16, device=dev)
        self.rht_out = torch.empty((T, F), dtype=torch.bfloat16, device=dev)
        self.launches_per_step = 5

    def ops(self):
        mx, F4 = self.mx, self.mx.MX_FMT_NVFP4
        T, H, F = self.T, self.H, self.F
        per = 2 * 2 + 0.5 + 1 / 16          # two reads (amax pass, quantize pass) + codes + scales
        return [
            ("quant", "rht16+nvfp4_1x16 colwise SR dY", 1, T * F * per,
             lambda: mx.mx_nvfp4_quantize_1x16(self.dy, True, True, self.rht_seed, True, self.sr_seed, self.qdy, self.sdy,
                                               self.Sdy, self.ws1)),
            ("quant", "rht16+nvfp4_1x16 colwise RNE X", 1, T * H * per,
             lambda: mx.mx_nvfp4_quantize_1x16(self.x, True, True, self.rht_seed, False, 0, self.qx, self.sx, self.Sx,
                                               self.ws2)),
            ("gemm4", "WGRAD", 0, 2.0 * F * H * T,
             lambda: mx.mx_scaled_gemm(F4, self.qdy, self.sdy, self.Sdy, mx.MX_SCOPE_TENSOR, self.qx, self.sx, self.Sx,
                                       mx.MX_SCOPE_TENSOR, F, H, T, self.dw)),
        ]

    def aux_ops(self):
        """Standalone RHT16 (the unfused transform), timed apart from the step."""
        return [("rht", "rht16 dY standalone", 1, self.T * self.F * 4.0,
                 lambda: self.mx.mx_rht16(self.dy, self.rht_seed, self.rht_out))]

    def config(self):
        return {"workload": "wgrad: Llama-3-8B MLP WGRAD, RHT16 + NVFP4 1x16 colwise (SR dY, RNE X) + NVFP4 GEMM",
                "tokens": self.T, "hidden": self.H, "ffn": self.F}

    def e2e_inputs(self):
        return [self.x, self.dy]

    def e2e_outputs(self):
        return [self.dw]


class DenseBlockwise:
    """The Qwen3-8B MLP linear of the default step with DeepSeek-V3-style blockwise FP8 and power-of-two
    scales (the learner's form on Blackwell): [1, 128] row + column tiles of X and dY from one read each,
    [128, 128] blocks of W in both orientations, E8M0 scale bytes written straight into the MXFP8 GEMM
    layout, then FPROP, DGRAD and WGRAD on the MXFP8 tensor-core GEMM.  Aux: the FP32-scale quantizers
    (the sampler's form) of X, dY and W and the FP32-scale FPROP and WGRAD (per-K-block scaling around the
    tensor cores)."""
    name = "dense_fp8_blockwise"
    unit = "TFLOP/s"
    dtype = "e4m3 (f32 accumulate, bf16 out)"

    def __init__(self, mx, torch, dev, tokens=8192, hidden=4096, ffn=12288):
        import synthetic
        self.mx, self.torch, self.dev = mx, torch, dev
        data = synthetic.dense_mlp(tokens, hidden, ffn)
        bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        self.x, self.w, self.dy = bf(data["x"]), bf(data["w"]), bf(data["dy"])
        T, H, F = tokens, hidden, ffn
        self.T, self.H, self.F = T, H, F
        u8 = lambda *shape: torch.zeros(shape, dtype=torch.uint8, device=dev)
        f32 = lambda *shape: torch.zeros(shape, dtype=torch.float32, device=dev)

        def act(R, C):
            return {"q_row": u8(R, C), "s_row": f32(R, C // 128), "sf_row": u8(mx.scale_bytes(R, C, 32)),
                    "q_col": u8(C, R), "s_col": f32(C, R // 128), "sf_col": u8(mx.scale_bytes(C, R, 32))}
        self.qx, self.qdy = act(T, H), act(T, F)
        self.qw = {"q_row": u8(1, F, H), "q_col": u8(1, H, F), "s": f32(1, F // 128, H // 128),
                   "sf_row": u8(mx.scale_bytes(F, H, 32)), "sf_col": u8(mx.scale_bytes(H, F, 32))}
        self.fx = {"q_row": u8(T, H), "s_row": f32(T, H // 128), "q_col": u8(H, T), "s_col": f32(H, T // 128)}
        self.fdy = {"q_col": u8(F, T), "s_col": f32(F, T // 128)}
        self.fw = {"q_row": u8(1, F, H), "q_col": u8(1, H, F), "s": f32(1, F // 128, H // 128)}
        self.y = torch.empty((T, F), dtype=torch.bfloat16, device=dev)
        self.dx = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        self.dw = torch.empty((F, H), dtype=torch.bfloat16, device=dev)
        self.launches_per_step = 6

    def ops(self):
        mx, F8 = self.mx, self.mx.MX_FMT_MXFP8
        T, H, F = self.T, self.H, self.F
        act_per = 2 + 2 + 2 * (4 + 4) / 128      # BF16 read, two code copies, FP32 + E8M0 scales per copy
        w_per = 2 + 2
        qx, qdy, qw = self.qx, self.qdy, self.qw
        return [
            ("quant", "blockwise 1x128 row+col X", 1, T * H * act_per,
             lambda: mx.mx_fp8_blockwise_quantize_1x128(self.x, True, **qx)),
            ("quant", "blockwise 128x128 W", 1, F * H * w_per,
             lambda: mx.mx_fp8_blockwise_quantize_128x128(self.w[None], True, qw["q_row"], qw["q_col"], qw["s"],
                                                          sf_row=qw["sf_row"], sf_col=qw["sf_col"])),
            ("quant", "blockwise 1x128 row+col dY", 1, T * F * act_per,
             lambda: mx.mx_fp8_blockwise_quantize_1x128(self.dy, True, **qdy)),
            ("gemm8", "FPROP", 0, 2.0 * T * F * H,
             lambda: mx.mx_scaled_gemm(F8, qx["q_row"], qx["sf_row"], None, 0, qw["q_row"][0], qw["sf_row"], None, 0,
                                       T, F, H, self.y)),
            ("gemm8", "DGRAD", 0, 2.0 * T * H * F,
             lambda: mx.mx_scaled_gemm(F8, qdy["q_row"], qdy["sf_row"], None, 0, qw["q_col"][0], qw["sf_col"], None, 0,
                                       T, H, F, self.dx)),
            ("gemm8", "WGRAD", 0, 2.0 * F * H * T,
             lambda: mx.mx_scaled_gemm(F8, qdy["q_col"], qdy["sf_col"], None, 0, qx["q_col"], qx["sf_col"], None, 0,
                                       F, H, T, self.dw)),
        ]

    def aux_ops(self):
        """FP32-scale blockwise quantizers (the sampler's form): X row- and column-wise, dY column-wise, W both
        orientations; the FP32-scale FPROP and WGRAD GEMMs on them."""
        mx, T, H, F = self.mx, self.T, self.H, self.F
        return [
            ("quant", "blockwise 1x128 row+col FP32-scale X", 1, T * H * (2 + 2 + 2 * 4 / 128),
             lambda: mx.mx_fp8_blockwise_quantize_1x128(self.x, False, q_row=self.fx["q_row"], s_row=self.fx["s_row"],
                                                        q_col=self.fx["q_col"], s_col=self.fx["s_col"])),
            ("quant", "blockwise 1x128 col FP32-scale dY", 1, T * F * (2 + 1 + 4 / 128),
             lambda: mx.mx_fp8_blockwise_quantize_1x128(self.dy, False, q_col=self.fdy["q_col"], s_col=self.fdy["s_col"])),
            ("quant", "blockwise 128x128 FP32-scale W", 1, F * H * 4,
             lambda: mx.mx_fp8_blockwise_quantize_128x128(self.w[None], False, self.fw["q_row"], self.fw["q_col"],
                                                          self.fw["s"])),
            ("gemm8", "FPROP FP32-scale blockwise (scaling around the tensor cores)", 0, 2.0 * T * F * H,
             lambda: mx.mx_fp8_blockwise_gemm(self.fx["q_row"], self.fx["s_row"], self.fw["q_row"][0], self.fw["s"][0],
                                              T, F, H, self.y)),
            ("gemm8", "WGRAD FP32-scale blockwise (per-row scales of both operands around the tensor cores)", 0,
             2.0 * F * H * T,
             lambda: mx.mx_fp8_blockwise_gemm_wgrad(self.fdy["q_col"], self.fdy["s_col"], self.fx["q_col"],
                                                    self.fx["s_col"], F, H, T, self.dw)),
        ]

    def config(self):
        return {"workload": "dense_fp8_blockwise: Qwen3-8B MLP linear, blockwise FP8 (power-of-two scales) "
                            "X/dY 1x128 row+col, W 128x128 + FPROP/DGRAD/WGRAD on the MXFP8 GEMM",
                "tokens": self.T, "hidden": self.H, "ffn": self.F}


class DenseNVFP4:
    """The NVFP4 pretraining linear layer (MaxText recipe) at Llama-3-8B MLP shapes: W in 16x16 2D blocks
    (both orientations), X and dY 1x16 row-wise under per-tensor scales (RNE for X, SR for dY), FPROP and
    DGRAD as NVFP4 GEMMs with the 2D weight, RHT16 + column-wise 1x16 of dY (SR) and X (RNE) and the NVFP4
    WGRAD.  Aux: the dequantized-backward DGRAD (BF16 dY times DQ(W) expanded inside the GEMM, no BF16
    weight copy) and WGRAD (BF16 dY^T times DQ(X) of the forward's X codes) and, for comparison, the
    materialized DQ(W) the DGRAD avoids."""
    name = "dense_nvfp4"
    unit = "TFLOP/s"

    def __init__(self, mx, torch, dev, tokens=32768):
        import synthetic
        self.mx, self.torch, self.dev = mx, torch, dev
        d = synthetic.dense_nvfp4(tokens=tokens)
        bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        self.x, self.dy, self.w = bf(d["x"]), bf(d["dy"]), bf(d["w"])
        self.rht_seed, self.sr_seed = d["rht_seed"], d["sr_seed"]
        T, H = self.x.shape
        F = self.dy.shape[1]
        self.T, self.H, self.F = T, H, F
        u8 = lambda *shape: torch.empty(shape, dtype=torch.uint8, device=dev)
        z8 = lambda n: torch.zeros(n, dtype=torch.uint8, device=dev)
        f32 = lambda n: torch.empty(n, dtype=torch.float32, device=dev)
        self.qw = mx.alloc_nvfp4_weight_2d(1, F, H, dev)
        self.qx, self.sx, self.Sx = u8(T, H // 2), z8(mx.scale_bytes(T, H, 16)), f32(1)
        self.qdy, self.sdy, self.Sdy = u8(T, F // 2), z8(mx.scale_bytes(T, F, 16)), f32(1)
        self.qdy_c, self.sdy_c, self.Sdy_c = u8(F, T // 2), z8(mx.scale_bytes(F, T, 16)), f32(1)
        self.qx_c, self.sx_c, self.Sx_c = u8(H, T // 2), z8(mx.scale_bytes(H, T, 16)), f32(1)
        self.ws = [z8(16) for _ in range(4)]
        self.y = torch.empty((T, F), dtype=torch.bfloat16, device=dev)
        self.dx = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        self.dw = torch.empty((F, H), dtype=torch.bfloat16, device=dev)
        self.dx_dq = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        self.dw_dq = torch.empty((F, H), dtype=torch.bfloat16, device=dev)
        self.wdq = torch.empty((H, F), dtype=torch.bfloat16, device=dev)
        self.launches_per_step = 13

    def ops(self):
        mx, F4 = self.mx, self.mx.MX_FMT_NVFP4
        T, H, F = self.T, self.H, self.F
        TS = mx.MX_SCOPE_TENSOR
        qw = self.qw
        per_tensor_1x16 = 2 * 2 + 0.5 + 1 / 16           # amax pass + quantize pass reads, codes, scales
        return [
            ("quant", "nvfp4 2D W", 1, F * H * (2 + 1 + 2 / 16),
             lambda: mx.mx_nvfp4_quantize_weight_2d(self.w[None], qw["q_row"], qw["s_row"], qw["q_col"], qw["s_col"],
                                                    qw["s_w"], qw["ws"])),
            ("quant", "nvfp4 1x16 X", 1, T * H * per_tensor_1x16,
             lambda: mx.mx_nvfp4_quantize_1x16(self.x, False, False, 0, False, 0, self.qx, self.sx, self.Sx, self.ws[0])),
            ("gemm4", "FPROP", 0, 2.0 * T * F * H,
             lambda: mx.mx_scaled_gemm(F4, self.qx, self.sx, self.Sx, TS, qw["q_row"][0], qw["s_row"], qw["s_w"], TS,
                                       T, F, H, self.y)),
            ("quant", "nvfp4 1x16 SR dY", 1, T * F * per_tensor_1x16,
             lambda: mx.mx_nvfp4_quantize_1x16(self.dy, False, False, 0, True, self.sr_seed, self.qdy, self.sdy, self.Sdy,
                                               self.ws[1])),
            ("gemm4", "DGRAD", 0, 2.0 * T * H * F,
             lambda: mx.mx_scaled_gemm(F4, self.qdy, self.sdy, self.Sdy, TS, qw["q_col"][0], qw["s_col"], qw["s_w"], TS,
                                       T, H, F, self.dx)),
            ("quant", "rht16+nvfp4 colwise SR dY", 1, T * F * per_tensor_1x16,
             lambda: mx.mx_nvfp4_quantize_1x16(self.dy, True, True, self.rht_seed, True, self.sr_seed, self.qdy_c,
                                               self.sdy_c, self.Sdy_c, self.ws[2])),
            ("quant", "rht16+nvfp4 colwise X", 1, T * H * per_tensor_1x16,
             lambda: mx.mx_nvfp4_quantize_1x16(self.x, True, True, self.rht_seed, False, 0, self.qx_c, self.sx_c,
                                               self.Sx_c, self.ws[3])),
            ("gemm4", "WGRAD", 0, 2.0 * F * H * T,
             lambda: mx.mx_scaled_gemm(F4, self.qdy_c, self.sdy_c, self.Sdy_c, TS, self.qx_c, self.sx_c, self.Sx_c, TS,
                                       F, H, T, self.dw)),
        ]

    def aux_ops(self):
        mx, T, H, F = self.mx, self.T, self.H, self.F
        qw = self.qw
        return [
            ("gemm16", "DGRAD dequantized backward (BF16 dY x DQ(W) in the mainloop)", 0, 2.0 * T * H * F,
             lambda: mx.mx_gemm_bf16_dq_nvfp4(self.dy, qw["q_col"][0], qw["s_col"], qw["s_w"], mx.MX_SCOPE_TENSOR,
                                              T, H, F, self.dx_dq)),
            ("gemm16", "WGRAD dequantized backward (BF16 dY^T x DQ(X) in the mainloop)", 0, 2.0 * F * H * T,
             lambda: mx.mx_wgrad_bf16_dq_nvfp4(self.dy, self.qx, self.sx, self.Sx, mx.MX_SCOPE_TENSOR, self.dw_dq)),
            ("quant", "DQ(W) materialized (the BF16 copy the fused GEMM avoids)", 1, F * H * (0.5 + 1 / 16 + 2),
             lambda: mx.mx_dequantize_bf16(mx.MX_FMT_NVFP4, qw["q_col"][0], qw["s_col"], qw["s_w"], mx.MX_SCOPE_TENSOR,
                                           H, F, self.wdq)),
        ]

    def config(self):
        return {"workload": "dense_nvfp4: Llama-3-8B MLP linear in NVFP4 (MaxText recipe: 2D weights, 1x16 per-tensor "
                            "X/dY, RHT16 + SR on WGRAD inputs) FPROP/DGRAD/WGRAD",
                "tokens": self.T, "hidden": self.H, "ffn": self.F}


class WeightSync:
    """Weight-sync sweep: 48 layers of 128 experts x {2048x768, 768x2048, 768x2048}; per matrix
    stack MXFP8 row+col quantize, dequantize, re-quantize and byte compare; NVFP4 2D quantize,
    dequantize, re-quantize and byte compare.  The per-matrix maxima that the NVFP4 2D quantizer needs
    come from the calls that already read the values (the MXFP8 quantize of the weights, the NVFP4
    dequantize for the re-quantize), so the 2D quantizer reads its input once.  One layer's weights are
    drawn on the device per step (torch generator seeded 1000 + layer) outside the timed kernels."""
    name = "weight_sync"
    unit = "GB/s"

    def __init__(self, mx, torch, dev, layers=48, experts=128):
        self.mx, self.torch, self.dev = mx, torch, dev
        self.layers = layers
        self.shapes = [(experts, 2048, 768), (experts, 768, 2048), (experts, 768, 2048)]
        self.layer = 0
        self.bufs = []
        for (G, O, H) in self.shapes:
            b = {"w": torch.empty((G, O, H), dtype=torch.bfloat16, device=dev),
                 "m8": mx.alloc_mxfp8(G * O, H, dev), "m8b": mx.alloc_mxfp8(G * O, H, dev, colwise=False),
                 "n4": mx.alloc_nvfp4_weight_2d(G, O, H, dev), "n4b": mx.alloc_nvfp4_weight_2d(G, O, H, dev),
                 "y": torch.empty((G * O, H), dtype=torch.bfloat16, device=dev),
                 "amax_w": torch.empty(G, dtype=torch.int32, device=dev), "amax_y": torch.empty(G, dtype=torch.int32, device=dev)}
            self.bufs.append(b)
        self.count = torch.zeros(1, dtype=torch.int64, device=dev)
        # per shape: Q, DQ, re-Q, 2 compares (MXFP8); Q, DQ, re-Q, 3 compares (NVFP4 2D)
        self.launches_per_step = 3 * (1 + 1 + 1 + 2 + 1 + 1 + 1 + 3)

    def draw(self, layer):
        gen = self.torch.Generator(device=self.dev)
        gen.manual_seed(1000 + layer)
        for b in self.bufs:
            b["w"].normal_(0.0, 0.02, generator=gen)

    def ops(self):
        mx = self.mx
        out = []
        for (G, O, H), b in zip(self.shapes, self.bufs):
            n = G * O * H
            R = G * O
            m8, m8b, n4, n4b = b["m8"], b["m8b"], b["n4"], b["n4b"]
            w2 = b["w"].view(R, H)
            out += [
                ("quant", f"mxfp8 Q {O}x{H} (+ matrix maxima)", 1, n * (2 + 2 + 2 / 32),
                 lambda w2=w2, m8=m8, b=b, O=O: mx.mx_quantize_mxfp8_amax(w2, O, b["amax_w"], **m8)),
                ("dq", f"mxfp8 DQ {O}x{H}", 1, n * (1 + 1 / 32 + 2),
                 lambda m8=m8, b=b, R=R, H=H: mx.mx_dequantize_bf16(mx.MX_FMT_MXFP8, m8["q_row"], m8["s_row"], None, 0, R, H, b["y"])),
                ("quant", f"mxfp8 re-Q {O}x{H}", 1, n * (2 + 1 + 1 / 32), lambda b=b, m8b=m8b: mx.mx_quantize_mxfp8(b["y"], **m8b)),
                ("cmp", f"mxfp8 compare {O}x{H}", 1, 2 * n * (1 + 1 / 32),
                 lambda m8=m8, m8b=m8b: (mx.mx_count_mismatch(m8["q_row"], m8b["q_row"], self.count),
                                         mx.mx_count_mismatch(m8["s_row"], m8b["s_row"], self.count))),
                ("quant", f"nvfp4 2D Q {O}x{H}", 1, n * (2 + 1 + 2 / 16),
                 lambda b=b, n4=n4: mx.mx_nvfp4_quantize_weight_2d_given_amax(b["w"], n4["q_row"], n4["s_row"], n4["q_col"],
                                                                               n4["s_col"], n4["s_w"], b["amax_w"])),
                ("dq", f"nvfp4 DQ {O}x{H} (+ matrix maxima)", 1, n * (0.5 + 1 / 16 + 2),
                 lambda n4=n4, b=b, R=R, H=H, O=O: mx.mx_dequantize_nvfp4_amax(n4["q_row"], n4["s_row"], n4["s_w"], O, R, H,
                                                                             b["y"], b["amax_y"])),
                ("quant", f"nvfp4 2D re-Q {O}x{H}", 1, n * (2 + 1 + 2 / 16),
                 lambda b=b, n4b=n4b, G=G, O=O, H=H: mx.mx_nvfp4_quantize_weight_2d_given_amax(
                     b["y"].view(G, O, H), n4b["q_row"], n4b["s_row"], n4b["q_col"], n4b["s_col"], n4b["s_w"], b["amax_y"])),
                ("cmp", f"nvfp4 compare {O}x{H}", 1, 2 * n * (0.5 + 0.5 + 2 / 16),
                 lambda n4=n4, n4b=n4b: (mx.mx_count_mismatch(n4["q_row"], n4b["q_row"], self.count),
                                         mx.mx_count_mismatch(n4["q_col"], n4b["q_col"], self.count),
                                         mx.mx_count_mismatch(n4["s_row"], n4b["s_row"], self.count))),
            ]
        return out

    def config(self):
        return {"workload": "weight_sync: 48 layers x 128 experts x {2048x768, 768x2048, 768x2048}, MXFP8 + NVFP4-2D "
                            "quantize, dequantize, re-quantize, byte compare (matrix maxima carried into the 2D quantizer)",
                "layers": self.layers}

    def e2e_inputs(self):
        return [b["w"] for b in self.bufs]

    def e2e_outputs(self):
        return [self.count]


def max_over_ranks(x: float, dist=None, device=None) -> float:
    """The largest value of x over all ranks (x itself on a single process)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank_step: float, world: int, ms_per_step: float) -> float:
    """Work per second of the whole job: every rank processes units_per_rank_step per step, and a step
    takes the slowest rank's time."""
    return world * units_per_rank_step / (ms_per_step / 1e3)


def time_device(work, torch, steps, warmup, dist=None):
    """Warm up, then time `steps` steps with CUDA events on the current stream; per-op events too."""
    ops = work.ops()
    for _ in range(warmup):
        for _, _, f in ops:
            f()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    n = len(ops)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n + 1)] for _ in range(steps)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    head_start(torch)
    start.record()
    for s in range(steps):
        e = evs[s]
        e[0].record()
        for i, (_, _, f) in enumerate(ops):
            f()
            e[i + 1].record()
    end.record()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    total_ms = start.elapsed_time(end)
    per_op = [statistics.mean(evs[s][i].elapsed_time(evs[s][i + 1]) for s in range(steps)) for i in range(n)]
    return total_ms, per_op


def head_start(torch):
    """Just before a timed region (after its synchronize): a short device-side spin on the current stream,
    so that the host queues the timed calls behind it and the first call's time does not include the host's
    submission of that call to an idle GPU.  The spin ends before the start event is recorded."""
    torch.cuda._sleep(HEAD_START_CYCLES)


def time_ops(ops, torch, steps, warmup):
    """Per-op CUDA-event times (ms, averaged over `steps`) for a list of 5-tuples."""
    for _ in range(warmup):
        for op in ops:
            op[4]()
    torch.cuda.synchronize()
    n = len(ops)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n + 1)] for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    head_start(torch)
    start.record()
    for st in range(steps):
        evs[st][0].record()
        for i, op in enumerate(ops):
            op[4]()
            evs[st][i + 1].record()
    end.record()
    torch.cuda.synchronize()
    per_op = [statistics.mean(evs[st][i].elapsed_time(evs[st][i + 1]) for st in range(steps)) for i in range(n)]
    return start.elapsed_time(end), per_op


def tensor_peaks(kind, peaks):
    """(measured-derived peak, published dense peak, report key) in TFLOP/s for a GEMM op kind:
    gemm8 = FP8, gemm16 = BF16, otherwise NVFP4."""
    if kind == "gemm8":
        return peaks["bf16_tflops"] * FP8_OVER_BF16, DATASHEET["fp8"], "frac_fp8_peak"
    if kind == "gemm16":
        return peaks["bf16_tflops"], DATASHEET["bf16"], "frac_bf16_peak"
    return peaks["bf16_tflops"] * FP4_OVER_BF16, DATASHEET["fp4"], "frac_fp4_peak"


def op_report(ops, per_op, peaks):
    """Achieved rate and roofline fraction per op: byte-moving ops against the HBM copy bandwidth;
    FP4 GEMMs against the FP4 peak and, when the op carries its minimum HBM traffic (a sixth tuple
    element: operand codes and scales read once, output written once), against the memory roofline
    too -- the bound is whichever of the two takes longer at peak."""
    rep, by_kind = {}, {}
    for op, ms in zip(ops, per_op):
        kind, label, is_bytes, units = op[:4]
        mem = op[5] if len(op) > 5 else None
        if is_bytes:
            ach = units / (ms / 1e3) / 1e9
            rep[label] = {"ms": round(ms, 4), "GBps": round(ach, 1), "frac_hbm": round(ach / peaks["hbm_gbs"], 4)}
        else:
            peak, ds, tag = tensor_peaks(kind, peaks)
            ach = units / (ms / 1e3) / 1e12
            rep[label] = {"ms": round(ms, 4), "TFLOPs": round(ach, 1), tag: round(ach / peak, 4),
                          "frac_datasheet": round(ach / ds, 4)}
            if mem:
                t_flop = units / (peak * 1e12) * 1e3
                t_mem = mem / (peaks["hbm_gbs"] * 1e9) * 1e3
                rep[label].update({"min_hbm_bytes": int(mem), "GBps": round(mem / (ms / 1e3) / 1e9, 1),
                                   "frac_hbm": round(mem / (ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
                                   "bound": "hbm" if t_mem > t_flop else "tensor",
                                   "frac_roofline": round(max(t_flop, t_mem) / ms, 4)})
        k = by_kind.setdefault(kind, [0.0, 0.0, is_bytes])
        k[0] += ms
        k[1] += units
    return rep, by_kind


def kind_roofline(kind, kms, kunits, is_bytes, kmem, peaks):
    """Roofline of the ops of one kind taken together: HBM for byte-moving ops; for GEMMs the tensor
    peak of their type, or HBM on their minimum traffic when that takes longer at peak."""
    if is_bytes:
        ach = kunits / (kms / 1e3) / 1e9
        return {"kernel": kind, "bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(ach / peaks["hbm_gbs"], 4), "traffic": None,
                "peak_source": f"{peaks['source']} copy bandwidth"}
    tpeak, ds, _ = tensor_peaks(kind, peaks)
    ach = kunits / (kms / 1e3) / 1e12
    ratio = tpeak / peaks["bf16_tflops"]
    roof = {"kernel": kind, "bound": "tensor", "achieved": round(ach, 1), "peak": round(tpeak, 1), "unit": "TFLOP/s",
            "frac": round(ach / tpeak, 4), "traffic": None,
            "peak_source": f"{peaks['source']} bf16 burst x {ratio:g} (nominal dense ratio)",
            "datasheet_peak": ds, "frac_datasheet": round(ach / ds, 4), "datasheet_source": DATASHEET["source"]}
    if kmem and kmem / (peaks["hbm_gbs"] * 1e9) > kunits / (tpeak * 1e12):
        gbs = kmem / (kms / 1e3) / 1e9
        roof.update({"bound": "hbm", "min_hbm_bytes": int(kmem), "achieved_GBps": round(gbs, 1),
                     "frac": round(gbs / peaks["hbm_gbs"], 4),
                     "note": "the minimum HBM traffic takes longer at peak than the flops: frac is against HBM"})
    return roof


def step_units(work, ops):
    """Work per step in the config's unit base: its GEMM flops (reported in TFLOP/s) or its algorithmic
    bytes (reported in GB/s)."""
    if work.unit == "GB/s":
        return sum(op[3] for op in ops if op[2])
    return sum(op[3] for op in ops if not op[2])


def unit_scale(unit):
    return 1e9 if unit == "GB/s" else 1e12


def step_value(work, ops, ms):
    return step_units(work, ops) / (ms / 1e3) / unit_scale(work.unit)


def dominant_roofline(ops, per_op, peaks):
    kinds = {}
    for op, ms in zip(ops, per_op):
        k = kinds.setdefault(op[0], [0.0, 0.0, op[2], 0.0])
        k[0] += ms
        k[1] += op[3]
        k[3] += op[5] if len(op) > 5 and op[5] else 0.0
    kind, (kms, kunits, is_bytes, kmem) = max(kinds.items(), key=lambda kv: kv[1][0])
    return kind_roofline(kind, kms, kunits, is_bytes, kmem, peaks)


def e2e_generic(work, torch, steps, ops=None, units_per_step=None, warmup=2, pipelined=True):
    """End to end through the same calls: every step copies the step's inputs in from pinned host
    memory, runs the ops and copies the results out to pinned host memory; CUDA events around all steps.
    Reported two ways.  `value`: pipelined -- the host-to-device copies land in one of two device
    staging sets on their own stream while the previous step computes, the step moves them into place
    device-to-device, and its results leave through a second pair of staging sets on a third stream while
    the next step computes.  `serial_value`: the same copies and calls one after the other on one stream
    (the reported value as well when `pipelined` is false: a latency-bound step, where the staging copies
    would only add launches)."""
    ins, outs = work.e2e_inputs(), work.e2e_outputs()
    ops = ops if ops is not None else work.ops()
    h_in = [t.cpu().pin_memory() for t in ins]
    h_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs]
    units = units_per_step if units_per_step is not None else step_units(work, ops)
    to_value = lambda ms: round(units / (ms / 1e3) / unit_scale(work.unit), 2)

    def serial_step():
        for d, h in zip(ins, h_in):
            d.copy_(h, non_blocking=True)
        for op in ops:
            op[4]()
        for d, h in zip(outs, h_out):
            h.copy_(d, non_blocking=True)

    def timed(run, first_stream, last_stream):
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(first_stream)
        run()
        end.record(last_stream)
        torch.cuda.synchronize()
        return start.elapsed_time(end) / steps

    cur = torch.cuda.current_stream()
    for _ in range(warmup):
        serial_step()
    serial_ms = timed(lambda: [serial_step() for _ in range(steps)], cur, cur)
    common = {"unit": work.unit, "steps": steps,
              "h2d_bytes_per_step": int(sum(h.numel() * h.element_size() for h in h_in)),
              "d2h_bytes_per_step": int(sum(h.numel() * h.element_size() for h in h_out))}
    if not pipelined:
        return {"value": to_value(serial_ms), "ms_per_step": round(serial_ms, 4), **common,
                "serial_value": to_value(serial_ms), "serial_ms_per_step": round(serial_ms, 4),
                "note": "inputs copied in from pinned host memory, kernels, results copied out, every step, serially "
                        "(a latency-bound step: no staging pipeline)"}

    st_in = [[torch.empty_like(t) for t in ins] for _ in range(2)]
    st_out = [[torch.empty_like(t) for t in outs] for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: [torch.cuda.Event(), torch.cuda.Event()]
    ev_in, ev_used, ev_done, ev_out = ev(), ev(), ev(), ev()

    def piped(n):
        for i in range(n):
            k = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_used[k])            # step i - 2 has moved staging set k into place
                for st, h in zip(st_in[k], h_in):
                    st.copy_(h, non_blocking=True)
                ev_in[k].record(s_in)
            cur.wait_event(ev_in[k])
            for d, st in zip(ins, st_in[k]):
                d.copy_(st)
            ev_used[k].record(cur)
            for op in ops:
                op[4]()
            if i >= 2:
                cur.wait_event(ev_out[k])                   # step i - 2's results have left staging set k
            for st, d in zip(st_out[k], outs):
                st.copy_(d)
            ev_done[k].record(cur)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[k])
                for h, st in zip(h_out, st_out[k]):
                    h.copy_(st, non_blocking=True)
                ev_out[k].record(s_out)

    piped(warmup)
    s_in.wait_stream(s_out)                                 # the timed steps start after the warm-up's copies
    ms = timed(lambda: piped(steps), s_in, s_out)
    out = {"value": to_value(ms), "ms_per_step": round(ms, 4), **common,
           "serial_value": to_value(serial_ms), "serial_ms_per_step": round(serial_ms, 4),
           "note": "inputs copied in from pinned host memory and results copied out to pinned host memory every "
                   "step; value: the copies of neighbouring steps overlap the kernels through two device staging "
                   "sets (moved into place device-to-device inside the step); serial_value: copies and kernels "
                   "one after the other on one stream"}
    del h_in, h_out, st_in, st_out
    return out


def graph_step(work, torch, ops, steps, warmup):
    """Capture one step's calls into a CUDA graph and time `steps` replays with CUDA events; returns the
    replay value and ms per step (the eager ones kept under eager_*)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for op in ops:
            op[4]()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for op in ops:
            op[4]()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    head_start(torch)
    start.record()
    for _ in range(steps):
        g.replay()
    end.record()
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / steps
    return {"graph_ms_per_step": round(ms, 4), "graph_value": round(step_value(work, ops, ms), 2),
            "graph_note": "the step's calls captured once into a CUDA graph and replayed (the value and ms_per_step "
                          "above are the eager calls through the Python binding)"}


def measure(work, torch, mx, peaks, steps, warmup, e2e=True, gpu_index=0):
    """Device-timed steps of a workload (CUDA events per op), its roofline, clocks and end-to-end run."""
    ops = work.ops()
    sampler = ClockSampler(gpu_index)
    sampler.start()
    total_ms, per_op = time_ops(ops, torch, steps, warmup)
    clocks = sampler.stop()
    status = mx.mx_check_device_status()
    ms = total_ms / steps
    rep, _ = op_report(ops, per_op, peaks)
    out = {"value": round(step_value(work, ops, ms), 2), "unit": work.unit, "ms_per_step": round(ms, 4),
           "steps": steps, "warmup": warmup, "dtype": getattr(work, "dtype", "e2m1 (f32 accumulate, bf16 out)"),
           "config": work.config(), "per_op": rep, "roofline": dominant_roofline(ops, per_op, peaks),
           "clocks": clocks, "gpu_launches": work.launches_per_step * steps,
           "watchdog": "ok" if status == 0 else f"status {status}"}
    if getattr(work, "graph", False):
        # a launch-bound step: the same calls captured once into a CUDA graph and replayed, so the host's
        # per-call work (argument checks, tensor-map encoding, launch) leaves the step time
        out.update(graph_step(work, torch, ops, steps, warmup))
    if hasattr(work, "aux_ops"):
        aops = work.aux_ops()
        if aops:
            _, aper = time_ops(aops, torch, steps, warmup)
            out["aux"], _ = op_report(aops, aper, peaks)
    if e2e and hasattr(work, "e2e_inputs"):
        out["e2e"] = e2e_generic(work, torch, steps, ops, pipelined=getattr(work, "e2e_pipelined", True))
    return out


def measure_weight_sync(work, torch, mx, peaks, warmup, e2e=True, gpu_index=0):
    """The weight-sync sweep: one layer per step (its weights drawn on the device before its ops, outside
    the timed kernels), every layer once; the value is all layers' algorithmic bytes over their time."""
    ops = work.ops()
    acc = [0.0] * len(ops)
    sampler = ClockSampler(gpu_index)
    work.count.zero_()
    sampler.start()
    for layer in range(work.layers):
        work.draw(layer)
        _, per = time_ops(ops, torch, 1, warmup if layer == 0 else 0)
        acc = [a + b for a, b in zip(acc, per)]
    clocks = sampler.stop()
    status = mx.mx_check_device_status()
    mismatched = int(work.count.item())
    total_ms = sum(acc)
    bytes_layer = sum(op[3] for op in ops)
    value = bytes_layer * work.layers / (total_ms / 1e3) / 1e9
    per_op = [a / work.layers for a in acc]
    rep, _ = op_report(ops, per_op, peaks)
    out = {"value": round(value, 1), "unit": "GB/s", "ms_per_step": round(total_ms / work.layers, 4),
           "steps": work.layers, "warmup": warmup, "dtype": "bf16 -> e4m3/e2m1 codes",
           "config": work.config(), "per_op": rep, "roofline": dominant_roofline(ops, per_op, peaks),
           "frac_hbm": round(value / peaks["hbm_gbs"], 4), "mismatched_bytes": mismatched, "clocks": clocks,
           "gpu_launches": work.launches_per_step * work.layers,
           "watchdog": "ok" if status == 0 else f"status {status}",
           "data": "per-layer N(0, 0.02) draws on the device, seed 1000 + layer"}
    if e2e:
        work.draw(0)
        out["e2e"] = e2e_generic(work, torch, work.layers, ops, units_per_step=bytes_layer)
        out["e2e"]["note"] += "; one layer per step (layer 0's bytes from the host each time)"
    return out


def make_workload(name, mx, torch, dev, args, data=None):
    if name == "tiny":
        return Tiny(mx, torch, dev, data=data)
    if name == "moe":
        return MoE(mx, torch, dev, experts=args.experts, data=data)
    if name == "moe_mxfp8":
        return MoE8(mx, torch, dev, experts=args.experts)
    if name == "dense_fp8_blockwise":
        return DenseBlockwise(mx, torch, dev)
    if name == "dense_nvfp4":
        return DenseNVFP4(mx, torch, dev, tokens=args.tokens)
    if name == "wgrad":
        return WGrad(mx, torch, dev, data=data, tokens=args.tokens)
    if name == "weight_sync":
        return WeightSync(mx, torch, dev, layers=args.layers, experts=args.experts)
    raise ValueError(name)


def run_workload(args):
    import torch
    import microscaled_precision_numerics_gb300 as mx
    torch.cuda.set_device(0)
    dev = torch.device("cuda:0")
    mx.lib()
    peaks = load_peaks()
    work = make_workload(args.workload, mx, torch, dev, args)
    if args.workload == "weight_sync":
        res = measure_weight_sync(work, torch, mx, peaks, args.warmup, e2e=not args.no_e2e)
    else:
        res = measure(work, torch, mx, peaks, args.steps, args.warmup, e2e=not args.no_e2e)
    line = {"metric": METRIC, "value": res.pop("value"), "unit": res.pop("unit"), "n_gpus": 1,
            "steps": res.pop("steps"), "warmup": res.pop("warmup"), "ms_per_step": res.pop("ms_per_step"),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": res.pop("dtype"),
            "data": res.pop("data", "synthetic (seeded draws)")}
    line.update(res)
    print(json.dumps(line), flush=True)


def run_device(args):
    import torch
    import microscaled_precision_numerics_gb300 as mx

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as td
        td.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
        dist = td
    torch.cuda.set_device(local)
    dev = torch.device(f"cuda:{local}")
    mx.lib()

    # the CPU baselines run before any GPU work (oracle threads, no forked pool after CUDA init)
    cpu = None
    run_configs = world == 1 and not args.no_configs
    cfg_data, cfg_cpu = {}, {}
    if run_configs:
        cfg_data = config_inputs()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.workload)
        if run_configs:
            cfg_cpu = cpu_baseline_configs(cfg_data)

    work = DenseMLP(mx, torch, dev)
    peaks = load_peaks()
    sampler = ClockSampler(local)
    sampler.start()
    total_ms, per_op = time_device(work, torch, args.steps, args.warmup, dist)
    clocks = sampler.stop()
    mx.check_device_status()

    total_ms = max_over_ranks(total_ms, dist, dev)
    ms_per_step = total_ms / args.steps
    value = whole_job_rate(work.units_per_step(), world, ms_per_step)

    ops = work.ops()
    gemm_ms = sum(per_op[i] for i, (k, _, _) in enumerate(ops) if k == "gemm")
    quant_ms = sum(per_op[i] for i, (k, _, _) in enumerate(ops) if k == "quant")
    gemm_tflops = sum(work.gemm_flops) / (gemm_ms / 1e3) / 1e12
    quant_gbs = sum(work.quant_bytes()) / (quant_ms / 1e3) / 1e9
    fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    dominant = "gemm" if gemm_ms >= quant_ms else "quant"
    if dominant == "gemm":
        roofline = {"kernel": "bs_gemm_pair_kernel<MXFP8> (FPROP+DGRAD+WGRAD)", "bound": "tensor",
                    "achieved": round(gemm_tflops, 1), "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                    "frac": round(gemm_tflops / fp8_peak, 4), "traffic": recorded_traffic("bs_gemm_pair_kernel<MXFP8>"),
                    "traffic_unit": "DRAM bytes per launch (mean of FPROP, DGRAD, WGRAD; ncu)",
                    "peak_source": f"{peaks['source']} bf16 burst x {FP8_OVER_BF16:g} (nominal FP8/BF16)"}
    else:
        roofline = {"kernel": "mxfp8_quantize_kernel", "bound": "hbm", "achieved": round(quant_gbs, 1),
                    "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(quant_gbs / peaks["hbm_gbs"], 4),
                    "traffic": recorded_traffic("mxfp8_quantize_kernel<row,col> batched"),
                    "peak_source": f"{peaks['source']} copy bandwidth"}

    launches = work.launches_per_step * args.steps
    T, H, F, gemm_flops = work.T, work.H, work.F, list(work.gemm_flops)
    labels = [(k, lbl) for (k, lbl, _) in ops]
    del ops
    roofline.update({"datasheet_peak": DATASHEET["fp8"], "frac_datasheet": round(gemm_tflops / DATASHEET["fp8"], 4),
                     "datasheet_source": DATASHEET["source"]} if dominant == "gemm" else {})
    e2e = None
    if not args.no_e2e:
        work.e2e_setup()
        e2e_steps = max(4, min(args.steps, 20))
        work.e2e_run(2)                                            # warm-up
        if dist is not None:
            dist.barrier()
        e_ms = work.e2e_run(e2e_steps)
        e_ms = max_over_ranks(e_ms, dist, dev)
        e2e = {"value": round(whole_job_rate(work.units_per_step(), world, e_ms), 2), "unit": "TFLOP/s",
               "ms_per_step": round(e_ms, 3), "steps": e2e_steps,
               "h2d_bytes_per_step": work.h2d, "d2h_bytes_per_step": work.d2h,
               "note": "pinned host inputs in, BF16 results out, every step; copies of neighbouring steps overlap the kernels"}

    # the other four configurations, one after the other on this GPU (single-GPU runs only)
    configs = {}
    if run_configs:
        del work
        torch.cuda.empty_cache()
        for key, name in (("C1_tiny", "tiny"), ("C3_moe", "moe"), ("C4_wgrad", "wgrad"),
                          ("C5_weight_sync", "weight_sync")):
            w = make_workload(name, mx, torch, dev, args, data=cfg_data.pop(name, None))
            if name == "weight_sync":
                res = measure_weight_sync(w, torch, mx, peaks, args.warmup, e2e=not args.no_e2e, gpu_index=local)
            else:
                res = measure(w, torch, mx, peaks, args.steps, args.warmup, e2e=not args.no_e2e, gpu_index=local)
            res["cpu_baseline"] = cfg_cpu.get(name)
            configs[key] = res
            del w
            torch.cuda.empty_cache()

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 (f32 accumulate, bf16 out)",
            "data": "synthetic (seeded numpy draws; no dataset or trained weights needed)",
            "config": {"workload": "dense_mlp: Qwen3-8B MLP linear, MXFP8 quantize X/W/dY row+col + FPROP/DGRAD/WGRAD",
                       "tokens": T, "hidden": H, "ffn": F, "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2 (369 MB BF16 read per step, 129 MB L2)"},
            "components": {
                "quantize_ms": round(quant_ms, 4), "quantize_GBps": round(quant_gbs, 1),
                "quantize_frac_hbm": round(quant_gbs / peaks["hbm_gbs"], 4),
                "gemm_ms": round(gemm_ms, 4), "gemm_TFLOPs": round(gemm_tflops, 1),
                "per_op_ms": {lbl: round(per_op[i], 4) for i, (_, lbl) in enumerate(labels)},
                "per_gemm_TFLOPs": {lbl: round(gemm_flops[j] / (per_op[i] / 1e3) / 1e12, 1)
                                    for j, (i, (_, lbl)) in enumerate([(i, o) for i, o in enumerate(labels) if o[0] == "gemm"])},
            },
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clocks,
        }
        if configs:
            line["configs"] = configs
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


# ------------------------------------------------------------------------------------------------
# CPU oracle (reported baseline / reference arm)
# ------------------------------------------------------------------------------------------------
SLICE = 8     # the oracle sample is 1/8 of the tokens and 1/8 of the output features


def oracle_sample_step(orc, data):
    """A proportional slice of the dense_mlp step: S = T/8 tokens and Fs = F/8 output features.
    MXFP8 row+col quantization of X[:S], W[:Fs] and dY[:S, :Fs]; FP64 reference FPROP
    (Y[:S, :Fs]), DGRAD (dX[:S] over K = Fs) and WGRAD (dW[:Fs] over K = S)."""
    T, F = data["x"].shape[0], data["w"].shape[0]
    S, Fs = T // SLICE, F // SLICE
    x = np.ascontiguousarray(data["x"][:S])
    w = np.ascontiguousarray(data["w"][:Fs])
    dy = np.ascontiguousarray(data["dy"][:S, :Fs])
    qx, sx = orc.mxfp8_quantize_rowwise(x)
    qxc, sxc = orc.mxfp8_quantize_colwise(x)
    qw, sw = orc.mxfp8_quantize_rowwise(w)
    qwc, swc = orc.mxfp8_quantize_colwise(w)
    qd, sd = orc.mxfp8_quantize_rowwise(dy)
    qdc, sdc = orc.mxfp8_quantize_colwise(dy)
    orc.gemm_ref_mxfp8(qx, sx, qw, sw)          # FPROP
    orc.gemm_ref_mxfp8(qd, sd, qwc, swc)        # DGRAD
    orc.gemm_ref_mxfp8(qdc, sdc, qxc, sxc)      # WGRAD
    return 3 * 2.0 * S * Fs * x.shape[1]


def sample_text(data):
    T, H = data["x"].shape
    F = data["w"].shape[0]
    S, Fs = T // SLICE, F // SLICE
    return (f"1/{SLICE} slice of the dense_mlp step: tokens [0, {S}) and output features [0, {Fs}); MXFP8 row+col "
            f"quantize of X[:{S}], W[:{Fs}], dY[:{S}, :{Fs}] (C oracle, OpenMP) and FP64 FPROP/DGRAD/WGRAD "
            f"references (numpy), {3 * 2.0 * S * Fs * H / 1e9:.1f} GFLOP")


def cpu_baseline(workload: str, data=None):
    import oracle as orc
    import synthetic
    orc.build()
    cores = os.cpu_count() or 1
    orc.set_threads(cores)
    if data is None:
        data = synthetic.dense_mlp()
    # the sample is repeated until about 10 s of host work has been timed (at most 32 repetitions)
    t0 = time.perf_counter()
    flops, reps = 0.0, 0
    while reps < 32 and (reps == 0 or time.perf_counter() - t0 < 10.0):
        flops += oracle_sample_step(orc, data)
        reps += 1
    dt = time.perf_counter() - t0
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "seconds": round(dt, 2), "repetitions": reps, "sample": sample_text(data)}


# Algorithmic bytes per element of one weight-sync pass, the sum of the per-op counts WeightSync.ops()
# uses: MXFP8 quantize row+col, dequantize, re-quantize row-wise, compare codes and scales; NVFP4 2D
# quantize, dequantize, re-quantize, compare both code copies and the row scales.
WS_BYTES_PER_ELEM = ((2 + 2 + 2 / 32) + (1 + 1 / 32 + 2) + (2 + 1 + 1 / 32) + 2 * (1 + 1 / 32)
                     + (2 + 1 + 2 / 16) + (0.5 + 1 / 16 + 2) + (2 + 1 + 2 / 16) + 2 * (0.5 + 0.5 + 2 / 16))


def oracle_tiny(orc, d):
    """The whole tiny check on the oracle: MXFP8 row + column quantize of X and W, the dequantize of X,
    the FP64 FPROP reference.  Returns the step's GEMM flops."""
    x, w = d["x"], d["w"]
    qx, sx = orc.mxfp8_quantize_rowwise(x)
    orc.mxfp8_quantize_colwise(x)
    qw, sw = orc.mxfp8_quantize_rowwise(w)
    orc.mxfp8_quantize_colwise(w)
    orc.dequant_mxfp8(qx, sx)
    orc.gemm_ref_mxfp8(qx, sx, qw, sw)
    return 2.0 * x.shape[0] * w.shape[0] * x.shape[1]


def oracle_moe(orc, d):
    """Expert 0's slice of the MoE layer: its routed rows (per-token NVFP4 of the activations and of the
    down-projection input), its gate|up and down weights (16x16 NVFP4, DQ(Q(w))), and the FP64 references
    of its two grouped GEMMs.  Returns their flops."""
    o0, o1 = int(d["group_offsets"][0]), int(d["group_offsets"][1])
    a = np.ascontiguousarray(d["x"][d["row_token"][o0:o1]])
    dn = np.ascontiguousarray(d["down_in"][o0:o1])
    qa, sa, ta = orc.nvfp4_quantize_per_token(a)
    qd, sd, td = orc.nvfp4_quantize_per_token(dn)
    wgu, wd = np.ascontiguousarray(d["w_gate_up"][0]), np.ascontiguousarray(d["w_down"][0])
    q1, _, t1, s1 = orc.nvfp4_quantize_weight_2d(wgu)
    q2, _, t2, s2 = orc.nvfp4_quantize_weight_2d(wd)
    r1, r2 = orc.weight_2d_operand_scales(t1, "row"), orc.weight_2d_operand_scales(t2, "row")
    orc.dequant_nvfp4(q1, r1, s1, per_row=False)
    orc.dequant_nvfp4(q2, r2, s2, per_row=False)
    orc.gemm_ref_nvfp4(qa, sa, ta, q1, r1, s1)
    orc.gemm_ref_nvfp4(qd, sd, td, q2, r2, s2)
    m = o1 - o0
    return 2.0 * m * wgu.shape[0] * wgu.shape[1] + 2.0 * m * wd.shape[0] * wd.shape[1]


WGRAD_SLICE = 32


def oracle_wgrad(orc, d):
    """1/32 of the columns of the WGRAD path over all 32768 tokens: RHT16 + column-wise NVFP4 (both passes)
    of X[:, :128] (RNE) and dY[:, :448] (SR), each slab taken as its own tensor, and the FP64 reference of
    dW[:448, :128].  Returns its flops."""
    H, F = d["x"].shape[1] // WGRAD_SLICE, d["dy"].shape[1] // WGRAD_SLICE
    x = np.ascontiguousarray(d["x"][:, :H])
    dy = np.ascontiguousarray(d["dy"][:, :F])
    qx, sx, Sx = orc.nvfp4_quantize_1x16(x, True, True, d["rht_seed"], False, 0)
    qd, sd, Sd = orc.nvfp4_quantize_1x16(dy, True, True, d["rht_seed"], True, d["sr_seed"])
    orc.gemm_ref_nvfp4(qd, sd, Sd, qx, sx, Sx)
    return 2.0 * F * H * x.shape[0]


def weight_sync_sample(matrices=("down", "gate", "up")):
    """Expert 0 of the chosen matrices of layer 0 (host draws of the same shape and distribution)."""
    import synthetic
    shapes = {"down": (2048, 768), "gate": (768, 2048), "up": (768, 2048)}
    return [synthetic.normal(np.random.default_rng([1000, i, 0]), shapes[m], 0.02) for i, m in enumerate(matrices)]


def oracle_weight_sync(orc, mats):
    """One weight-sync pass over each matrix: MXFP8 quantize (row + column), dequantize, re-quantize and
    byte compare; NVFP4 16x16 quantize, dequantize, re-quantize and byte compare.  Returns the algorithmic
    bytes (the same per-element count as the GPU pass)."""
    total = 0.0
    for w in mats:
        qr, sr = orc.mxfp8_quantize_rowwise(w)
        orc.mxfp8_quantize_colwise(w)
        q2, s2 = orc.mxfp8_quantize_rowwise(orc.dequant_mxfp8(qr, sr))
        assert np.array_equal(q2, qr) and np.array_equal(s2, sr)
        n1, n1c, t1, sw = orc.nvfp4_quantize_weight_2d(w)
        y = orc.dequant_nvfp4(n1, orc.weight_2d_operand_scales(t1, "row"), sw, per_row=False)
        m1, m1c, u1, sw2 = orc.nvfp4_quantize_weight_2d(y)
        assert np.array_equal(m1, n1) and np.array_equal(m1c, n1c) and np.array_equal(u1, t1) and sw2 == sw
        total += w.size * WS_BYTES_PER_ELEM
    return total


def timed_oracle(orc, fn, arg, threads, unit, sample):
    orc.set_threads(threads)
    t0 = time.perf_counter()
    units = fn(orc, arg)
    dt = time.perf_counter() - t0
    return {"value": round(units / dt / unit_scale(unit), 6), "unit": unit, "cores": threads, "kind": "oracle",
            "seconds": round(dt, 2), "sample": sample}


def config_inputs():
    """Host inputs of the tiny, MoE and WGRAD configs (the weight-sync sweep draws on the device)."""
    import synthetic
    return {"tiny": synthetic.tiny(), "moe": synthetic.moe(), "wgrad": synthetic.wgrad()}


def cpu_baseline_configs(data):
    """The oracle, as it stands, on a bounded sample of each further config, at all cores; the tiny check
    and a one-matrix slice of a weight-sync layer also on one thread."""
    import oracle as orc
    orc.build()
    cores = os.cpu_count() or 1
    out = {}
    out["tiny"] = timed_oracle(orc, oracle_tiny, data["tiny"], cores, "TFLOP/s", "the whole tiny check")
    out["tiny"]["one_thread"] = timed_oracle(orc, oracle_tiny, data["tiny"], 1, "TFLOP/s", "the whole tiny check")
    out["moe"] = timed_oracle(orc, oracle_moe, data["moe"], cores, "TFLOP/s",
                              "expert 0: its routed rows' per-token NVFP4 (activations and down input), its gate|up "
                              "and down 2D NVFP4 + DQ, FP64 references of its two grouped GEMMs")
    out["wgrad"] = timed_oracle(orc, oracle_wgrad, data["wgrad"], cores, "TFLOP/s",
                                f"1/{WGRAD_SLICE} of the columns of X and dY over all tokens: RHT16 + column-wise NVFP4 "
                                "(RNE X, SR dY, both passes) and the FP64 WGRAD reference of that block")
    mats = weight_sync_sample()
    out["weight_sync"] = timed_oracle(orc, oracle_weight_sync, mats, cores, "GB/s",
                                      "expert 0 of down, gate and up of one layer: MXFP8 + NVFP4-2D Q, DQ, re-Q, compare")
    out["weight_sync"]["one_thread"] = timed_oracle(orc, oracle_weight_sync, mats[:1], 1, "GB/s",
                                                    "expert 0 of the down matrix of one layer")
    orc.set_threads(cores)
    return out


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle as orc
    import synthetic
    orc.build()
    cores = os.cpu_count() or 1
    orc.set_threads(cores)
    data = synthetic.dense_mlp()
    for _ in range(args.warmup):
        oracle_sample_step(orc, data)
    times, flops = [], 0.0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        flops = oracle_sample_step(orc, data)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = flops / (ms / 1e3) / 1e12
    T, H = data["x"].shape
    F = data["w"].shape[0]
    line = {"metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 2), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64 (oracle)", "data": "synthetic",
            "config": {"workload": "dense_mlp: Qwen3-8B MLP linear, MXFP8 quantize X/W/dY row+col + FPROP/DGRAD/WGRAD",
                       "tokens": T, "hidden": H, "ffn": F, "parallelism": "cpu"},
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample_text(data)},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["mxnum", "reference"], default="mxnum")
    ap.add_argument("--workload", choices=["dense_mlp", "tiny", "moe", "moe_mxfp8", "dense_fp8_blockwise", "dense_nvfp4", "wgrad",
                                           "weight_sync"], default="dense_mlp")
    ap.add_argument("--layers", type=int, default=48, help="weight_sync: layers swept")
    ap.add_argument("--experts", type=int, default=128, help="moe / weight_sync: experts (fewer only for profiling)")
    ap.add_argument("--tokens", type=int, default=32768, help="wgrad / dense_nvfp4: tokens (fewer only for profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="dense_mlp only, without the other four configurations")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
        return
    if args.workload != "dense_mlp":
        run_workload(args)
        return
    run_device(args)


if __name__ == "__main__":
    main()
