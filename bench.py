"""Benchmark of the adaptive-LayerNorm activation producers on GB300.

One step = one call of every producer on its workload (the shapes of the
producers' benchmark tables), all inputs resident in HBM, in this order:

  fp8 broadcast 4096x3072 | fp8 layer norm 4096x3072 | fp8 per-token 2520x3072 |
  fp8 table 4096x3072 (6 chunks) | nvfp4 broadcast 5070x3072 | nvfp4 layer norm
  5070x3072 | modulation6 1x5070x6x3072

Every producer reads its own buffers and one step streams ~0.9 GB, so no
input is still in the 129 MB L2 when its producer runs again.

metric: µs/call and achieved HBM GB/s per producer; the headline `value` is
the step's algorithmic bytes (what the producers must read and write) divided
by the step's device time, in GB/s, summed over ranks.  `e2e` is the same
metric through the Python API with host buffers: every step copies its inputs
from pinned host memory and its outputs back.  `roofline` is for the kernel
with the largest share of the step; `per_op` lists every producer.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--sweep] [--out FILE]

`--impl reference` times the CPU oracle (the only reference implementation of
this path) on a bounded sample of the same workload on the host cores.
Under torchrun each rank runs the whole step on its own GPU (weak scaling, no
collective on the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import platform
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "µs/call and achieved HBM GB/s (fraction of GB300 peak) per producer op/shape"
WORKLOAD = ("adaLN producer step: fp8 broadcast 4096x3072, fp8 layer-norm 4096x3072, fp8 per-token 2520x3072 "
            "(1% rows x8), fp8 table 4096x3072 (temb 6 chunks, fp32 table), nvfp4 broadcast 5070x3072, "
            "nvfp4 layer-norm 5070x3072, modulation6 1x5070x6x3072")


# ---------------------------------------------------------------------------
# workload
# ---------------------------------------------------------------------------

def step_workloads():
    return [
        ("fp8_broadcast", synth.fp8_broadcast(4096, 3072, 2001)),
        ("fp8_layer_norm", synth.fp8_ln(4096, 3072, 2002)),
        ("fp8_per_token", synth.fp8_ptok(2520, 3072, 1002)),
        ("fp8_table", synth.fp8_table(4096, 3072, 1003)),
        ("nvfp4_broadcast", synth.nvfp4_broadcast(5070, 3072, 1004)),
        ("nvfp4_layer_norm", synth.nvfp4_ln(5070, 3072, 2004)),
        ("modulation6", synth.modulation6(1, 5070, 3072, 1005)),
    ]


# The FP8 producers at the shapes of the pages' RTX 5090 table (benchmarks/
# RESULTS.md, "AdaLN->FP8 / LN->FP8"; 4096x3072 is in the step) and at 32768
# rows: (rows, dim, the page's AdaLN->FP8 us, the page's LN->FP8 us) -- the
# page's figures are another GPU's, context only.
PAGE_FP8_SHAPES = ((16, 2048, 4.117, 3.962), (64, 3072, 4.133, 4.117), (256, 3072, 4.140, 4.108),
                   (2520, 3072, 12.330, 10.267), (4096, 3072, 18.465, 16.412))
SWEEP_EXTRA = ((32768, 3072),)
# below this many rows a producer is bound by launch latency and ramp, not by
# HBM: its per_op line carries no bandwidth fraction
LAUNCH_BOUND_ROWS = 2500


def op_kind(name: str) -> str:
    """The producer of a per_op line: names with a trailing _<rows>x<dim> are
    the same producer at another shape."""
    m = re.match(r"^(.*)_(\d+)x(\d+)$", name)
    return m.group(1) if m else name


def page_context(name: str, rows: int, dim: int):
    """The pages' own figure for this producer and shape, if they print one
    (another GPU's: context only)."""
    kind = op_kind(name)
    for R, D, ada, ln in PAGE_FP8_SHAPES:
        if (R, D) == (rows, dim) and kind in ("fp8_broadcast", "fp8_layer_norm"):
            us = ada if kind == "fp8_broadcast" else ln
            return {"us": us, "hw": "RTX 5090, --iters 100 on identical buffers (benchmarks/RESULTS.md)"}
    if kind == "modulation6" and (rows, dim) == (5070, 3072):
        return {"us": 347.251, "hw": "RTX 5090 (benchmarks/RESULTS.md, adaln_modulation6 B1 S5070 D3072)"}
    return None


def page_shape_workloads():
    """The FP8 broadcast and layer-norm producers at the pages' shapes (but the
    step's 4096x3072) and at SWEEP_EXTRA."""
    shapes = []
    for R, D, _, _ in PAGE_FP8_SHAPES:
        if (R, D) == (4096, 3072):
            continue
        seed = 1001 if (R, D) == (16, 2048) else 1006
        shapes.append((f"fp8_broadcast_{R}x{D}", synth.fp8_broadcast(R, D, seed)))
        shapes.append((f"fp8_layer_norm_{R}x{D}", synth.fp8_ln(R, D, seed)))
    for R, D in SWEEP_EXTRA:
        shapes.append((f"fp8_broadcast_{R}x{D}", synth.fp8_broadcast(R, D, 1006)))
        shapes.append((f"fp8_layer_norm_{R}x{D}", synth.fp8_ln(R, D, 1006)))
    return shapes


def extra_workloads():
    """Producers measured beside the step (same shapes as their broadcast
    counterparts, the pages' FP8 shapes, a large row count), reported in
    `per_op` with "in_step": false."""
    return page_shape_workloads() + [
        ("fp8_modfp8", synth.fp8_modfp8(4096, 3072, 2006)),
        ("fp8_awq", synth.fp8_awq(4096, 3072, 2007)),
        ("nvfp4_modfp8", synth.nvfp4_modfp8(5070, 3072, 2008)),
        ("fp8_seg_h3", synth.segmented(37810, 5376, 2010)),
        ("nvfp4_2level_seg_h3", synth.segmented(37810, 5376, 2011)),
        ("nvfp4_2level_layer_norm", synth.nvfp4_ln(5070, 3072, 2012)),
        ("swiglu_values_h3", synth.swiglu(37810, 14336, 2013)),
        ("nvfp4_2level_swiglu_h3", synth.swiglu(37810, 14336, 2014)),
    ]


def alg_bytes(name: str, w) -> int:
    """Bytes the producer must move: every input element it uses read once,
    every output byte written once (per-op formulas of the design notes)."""
    R, D = w.rows, w.dim
    name = op_kind(name)
    if name == "fp8_broadcast":
        return 2 * R * D + 4 * D + R * D + 4
    if name == "fp8_modfp8":
        return 2 * R * D + 2 * D + 8 + R * D + 4          # e4m3 vectors, two deq scalars
    if name == "fp8_awq":
        return 2 * R * D + 6 * D + R * D + 4              # scale, shift, inv_s
    if name == "fp8_seg_h3":
        nseg = w.inputs["seg_scale"].shape[0]
        return 2 * R * D + 4 * R + 4 * nseg * D + R * D + 4   # x, segment index, tables, codes
    if name == "swiglu_values_h3":
        return 4 * R * D + 2 * R * D                       # gate and up, bf16 values
    if name == "nvfp4_2level_swiglu_h3":
        # two passes over gate and up (the tensor scale needs every value first)
        sf = ((R + 127) // 128 * 128) * ((D // 16 + 3) // 4 * 4)
        return 2 * 4 * R * D + R * D // 2 + sf + 4
    if name in ("nvfp4_2level_seg_h3", "nvfp4_2level_layer_norm"):
        # the input once per pass (no block can be encoded before the whole
        # tensor's maximum is known: two passes, or one where the library
        # stages the whole tensor in shared memory), then codes, scales and
        # the tensor scale
        sf = ((R + 127) // 128 * 128) * ((D // 16 + 3) // 4 * 4)
        src = 0
        if name == "nvfp4_2level_seg_h3":
            src = 4 * R + 4 * w.inputs["seg_scale"].shape[0] * D
        return two_level_passes(name, w) * (2 * R * D + src) + R * D // 2 + sf + 4
    if name == "fp8_layer_norm":
        return 2 * R * D + R * D + 4
    if name == "fp8_per_token":
        return 6 * R * D + R * D + 4
    if name == "fp8_table":
        return 2 * R * D + 4 * R * D + 8 * D + R * D + 4   # 2 of the temb chunks, 2 table rows
    if name in ("nvfp4_broadcast", "nvfp4_layer_norm", "nvfp4_modfp8"):
        mod = {"nvfp4_broadcast": 4 * D, "nvfp4_layer_norm": 0, "nvfp4_modfp8": 2 * D + 8}[name]
        sf = ((R + 127) // 128 * 128) * ((D // 16 + 3) // 4 * 4)
        return 2 * R * D + mod + R * D // 2 + sf
    if name == "modulation6":
        return 24 * R * D + 24 * D + 12 * R * D
    raise KeyError(name)


def two_level_passes(name: str, w) -> int:
    """Passes over the input of a two-level LayerNorm producer on the current
    device: 1 where the library reads the tensor once (its rows fit in the SMs'
    shared memory), else 2 (also without a CUDA device)."""
    if not torch.cuda.is_available():
        return 2
    mod = "segmented" if op_kind(name) == "nvfp4_2level_seg_h3" else "none"
    try:
        import nvfp4_activation_producer_gb300 as ap
        return 1 if ap.two_level_single_read(w.rows, w.dim, mod) else 2
    except (OSError, RuntimeError):
        return 2


def launches_per_call(name: str, w=None) -> int:
    """Kernels one call of the producer launches: the two-level producers (the
    LayerNorm forms and SwiGLU) clear their words, then run the maximum and the
    quantising pass, or one cooperative kernel where a LayerNorm form reads the
    tensor once."""
    kind = op_kind(name)
    if kind in ("nvfp4_2level_seg_h3", "nvfp4_2level_layer_norm") and w is not None:
        return 1 + two_level_passes(name, w)
    return 3 if kind.startswith("nvfp4_2level") else 1


class DeviceOp:
    """Inputs resident on the device, outputs preallocated, one call = one launch."""

    def __init__(self, ap, name, w, dev):
        self.ap, self.name, self.w = ap, name, w
        self.d = {k: v.to(dev) for k, v in w.inputs.items()}
        R, D = w.rows, w.dim
        if name.startswith("fp8"):
            self.out = (torch.empty((R, D), dtype=torch.float8_e4m3fn, device=dev),)
        elif name.startswith("swiglu"):
            self.out = (torch.empty((R, D), dtype=torch.bfloat16, device=dev),)
        elif name.startswith("nvfp4_2level"):
            self.out = (torch.empty((R, D // 2), dtype=torch.uint8, device=dev),
                        torch.empty((ap.swizzled_sf_size(R, D),), dtype=torch.uint8, device=dev),
                        torch.empty((1,), dtype=torch.float32, device=dev),
                        torch.zeros((ap.workspace_2level_bytes(R),), dtype=torch.uint8, device=dev))
        elif name.startswith("nvfp4"):
            self.out = (torch.empty((R, D // 2), dtype=torch.uint8, device=dev),
                        torch.empty((ap.swizzled_sf_size(R, D),), dtype=torch.uint8, device=dev))
        else:
            self.out = (torch.empty((6, 1, R, D), dtype=torch.bfloat16, device=dev),)
        self.bytes = alg_bytes(name, w)

    def api_call(self):
        """The producer through the Python API (tensor checks, then the C ABI)."""
        ap, d, o, p = self.ap, self.d, self.out, self.w.params
        n = op_kind(self.name)
        if n == "fp8_broadcast":
            ap.ada_layer_norm_quant_fp8_bf16(d["x"], d["scale"], d["shift"], d["act_scale"], p["eps"], out=o[0])
        elif n == "fp8_layer_norm":
            ap.layer_norm_no_affine_quant_fp8_static_bf16(d["x"], d["act_scale"], p["eps"], out=o[0])
        elif n == "fp8_per_token":
            ap.ada_layer_norm_quant_fp8_ptok_bf16(d["x"], d["scale"], d["shift"], d["act_scale"], p["eps"], out=o[0])
        elif n == "fp8_table":
            ap.ada_layer_norm_quant_fp8_ptok_table_bf16(d["x"], d["temb"], d["table"], d["act_scale"],
                                                        p["shift_idx"], p["scale_idx"], p["eps"], out=o[0])
        elif n == "nvfp4_broadcast":
            ap.ada_layer_norm_quant_nvfp4_swizzled_bf16(d["x"], d["scale"], d["shift"], p["eps"],
                                                        packed=o[0], sf_swizzled=o[1])
        elif n == "nvfp4_layer_norm":
            ap.layer_norm_no_affine_quant_nvfp4_swizzled_bf16(d["x"], p["eps"], packed=o[0], sf_swizzled=o[1])
        elif n == "fp8_modfp8":
            ap.ada_layer_norm_quant_fp8_modfp8_bf16(d["x"], d["scale_fp8"], d["shift_fp8"], d["scale_deq"],
                                                    d["shift_deq"], d["act_scale"], p["eps"], out=o[0])
        elif n == "fp8_awq":
            ap.awq_ada_layer_norm_quant_fp8_bf16(d["x"], d["scale"], d["shift"], d["inv_s"], d["act_scale"],
                                                 p["eps"], out=o[0])
        elif n == "nvfp4_modfp8":
            ap.ada_layer_norm_quant_nvfp4_swizzled_modfp8_bf16(d["x"], d["scale_fp8"], d["shift_fp8"],
                                                               d["scale_deq"], d["shift_deq"], p["eps"],
                                                               packed=o[0], sf_swizzled=o[1])
        elif n == "fp8_seg_h3":
            ap.ada_layer_norm_quant_fp8_seg_bf16(d["x"], d["seg_idx"], d["seg_scale"], d["seg_shift"],
                                                 d["act_scale"], p["eps"], out=o[0])
        elif n == "nvfp4_2level_seg_h3":
            ap.ada_layer_norm_quant_nvfp4_2level_seg_bf16(d["x"], d["seg_idx"], d["seg_scale"], d["seg_shift"],
                                                          p["eps"], packed=o[0], sf_swizzled=o[1], tensor_scale=o[2],
                                                          workspace=o[3])
        elif n == "nvfp4_2level_layer_norm":
            ap.layer_norm_no_affine_quant_nvfp4_2level_bf16(d["x"], p["eps"], packed=o[0], sf_swizzled=o[1],
                                                            tensor_scale=o[2], workspace=o[3])
        elif n == "swiglu_values_h3":
            ap.swiglu_bf16(d["fc1"][:, :self.w.dim], d["fc1"][:, self.w.dim:], out=o[0])
        elif n == "nvfp4_2level_swiglu_h3":
            ap.swiglu_quant_nvfp4_2level_bf16(d["fc1"][:, :self.w.dim], d["fc1"][:, self.w.dim:], packed=o[0],
                                              sf_swizzled=o[1], tensor_scale=o[2], workspace=o[3])
        elif n == "modulation6":
            ap.adaln_modulation6_bf16(d["params"], d["modulation"], out=o[0])

    def bind_raw(self, stream: int):
        """Pre-marshalled C-ABI call (pointers fixed), so the timed loop adds
        only the ctypes call and the launch to each producer."""
        import ctypes
        L = self.ap._load()
        d, o, p, R, D = self.d, self.out, self.w.params, self.w.rows, self.w.dim
        P = lambda t: t.data_ptr()
        n = op_kind(self.name)
        if n == "fp8_broadcast":
            fn, a = L.ada_layer_norm_quant_fp8_bf16, (P(d["x"]), P(d["scale"]), P(d["shift"]), P(d["act_scale"]),
                                                      p["eps"], P(o[0]), R, D, stream)
        elif n == "fp8_layer_norm":
            fn, a = L.layer_norm_no_affine_quant_fp8_static_bf16, (P(d["x"]), P(d["act_scale"]), p["eps"], P(o[0]),
                                                                   R, D, stream)
        elif n == "fp8_per_token":
            fn, a = L.ada_layer_norm_quant_fp8_ptok_bf16, (P(d["x"]), P(d["scale"]), P(d["shift"]),
                                                           P(d["act_scale"]), p["eps"], P(o[0]), R, D, stream)
        elif n == "fp8_table":
            fn, a = L.ada_layer_norm_quant_fp8_ptok_table_bf16, (P(d["x"]), P(d["temb"]), P(d["table"]),
                                                                 d["temb"].shape[1], p["shift_idx"], p["scale_idx"],
                                                                 P(d["act_scale"]), p["eps"], P(o[0]), R, D, stream)
        elif n == "nvfp4_broadcast":
            fn, a = L.ada_layer_norm_quant_nvfp4_swizzled_bf16, (P(d["x"]), P(d["scale"]), P(d["shift"]), p["eps"],
                                                                 P(o[0]), P(o[1]), R, D, stream)
        elif n == "nvfp4_layer_norm":
            fn, a = L.layer_norm_no_affine_quant_nvfp4_swizzled_bf16, (P(d["x"]), p["eps"], P(o[0]), P(o[1]), R, D,
                                                                       stream)
        elif n == "fp8_modfp8":
            fn, a = L.ada_layer_norm_quant_fp8_modfp8_bf16, (P(d["x"]), P(d["scale_fp8"]), P(d["shift_fp8"]),
                                                             P(d["scale_deq"]), P(d["shift_deq"]), P(d["act_scale"]),
                                                             p["eps"], P(o[0]), R, D, stream)
        elif n == "fp8_awq":
            fn, a = L.awq_ada_layer_norm_quant_fp8_bf16, (P(d["x"]), P(d["scale"]), P(d["shift"]), P(d["inv_s"]),
                                                          P(d["act_scale"]), p["eps"], P(o[0]), R, D, stream)
        elif n == "nvfp4_modfp8":
            fn, a = L.ada_layer_norm_quant_nvfp4_swizzled_modfp8_bf16, (P(d["x"]), P(d["scale_fp8"]),
                                                                        P(d["shift_fp8"]), P(d["scale_deq"]),
                                                                        P(d["shift_deq"]), p["eps"], P(o[0]), P(o[1]),
                                                                        R, D, stream)
        elif n == "fp8_seg_h3":
            fn, a = L.ada_layer_norm_quant_fp8_seg_bf16, (P(d["x"]), P(d["seg_idx"]), P(d["seg_scale"]),
                                                          P(d["seg_shift"]), d["seg_scale"].shape[0], P(d["act_scale"]),
                                                          p["eps"], P(o[0]), R, D, stream)
        elif n == "nvfp4_2level_seg_h3":
            fn, a = L.ada_layer_norm_quant_nvfp4_2level_seg_bf16, (P(d["x"]), P(d["seg_idx"]), P(d["seg_scale"]),
                                                                   P(d["seg_shift"]), d["seg_scale"].shape[0],
                                                                   p["eps"], P(o[0]), P(o[1]), P(o[2]), P(o[3]),
                                                                   R, D, stream)
        elif n == "nvfp4_2level_layer_norm":
            fn, a = L.layer_norm_no_affine_quant_nvfp4_2level_bf16, (P(d["x"]), p["eps"], P(o[0]), P(o[1]), P(o[2]),
                                                                     P(o[3]), R, D, stream)
        elif n == "swiglu_values_h3":
            g = P(d["fc1"])
            fn, a = L.swiglu_bf16, (g, g + 2 * D, 2 * D, P(o[0]), R, D, stream)
        elif n == "nvfp4_2level_swiglu_h3":
            g = P(d["fc1"])
            fn, a = L.swiglu_quant_nvfp4_2level_bf16, (g, g + 2 * D, 2 * D, P(o[0]), P(o[1]), P(o[2]), P(o[3]),
                                                       R, D, stream)
        else:
            self._outs6 = (ctypes.c_void_p * 6)(*[o[0][i].data_ptr() for i in range(6)])
            fn, a = L.adaln_modulation6_bf16, (P(d["params"]), P(d["modulation"]), self._outs6, 1, R, D, stream)
        name = self.name

        def call():
            rc = fn(*a)
            if rc:
                raise RuntimeError(f"{name}: status {rc}")
        self.raw = call
        return call


# ---------------------------------------------------------------------------
# measurement helpers
# ---------------------------------------------------------------------------

def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return None


def sources_digest(files) -> str:
    """Digest of the named kernel source files (csrc/), to tell whether a
    committed counter capture was taken on the current sources."""
    csrc = os.path.join(ROOT, "nvfp4_activation_producer_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(files):
        h.update(f.encode())
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def committed_traffic(op: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current sources of that producer's kernel (else None)."""
    try:
        t = json.load(open(os.path.join(ROOT, "profiles", "dram_traffic.json")))
        rec = t.get("per_launch", {}).get(op)
        if not rec or rec.get("sources_digest") != sources_digest(rec["sources"]):
            return None
    except (OSError, ValueError, KeyError):
        return None
    return rec.get("dram_bytes")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, every 50 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = [s for t, s in self.samples if self.t0 and self.t1 and self.t0 - 0.06 <= t <= self.t1 + 0.06]
        if not rows:
            rows = [s for _, s in self.samples]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------

def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time: every rank runs the same step on its own rows
    (replicas, no data-path collective), so the job takes as long as the
    slowest.  `device` is where the reduction tensor lives (the rank's GPU
    under NCCL, the CPU under gloo)."""
    if world <= 1:
        return float(ms)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_gbs(step_bytes: int, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: the algorithmic bytes all ranks moved per step
    over the (slowest rank's) step time."""
    return step_bytes * world / (ms_per_step * 1e-3) / 1e9


def run_ours(args, rank, world, local_rank):
    import nvfp4_activation_producer_gb300 as ap
    from nvfp4_activation_producer_gb300 import build as b
    b.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    works = step_workloads()
    extras = [] if args.no_extra else extra_workloads()
    if args.only:
        keep = set(args.only.split(","))
        works = [(n, w) for n, w in works if n in keep]
        extras = [(n, w) for n, w in extras if n in keep]
    if not works:  # only producers outside the step were asked for: time them as the step
        works, extras = extras, []
    ops = [DeviceOp(ap, n, w, dev) for n, w in works]
    extra_ops = [DeviceOp(ap, n, w, dev) for n, w in extras]
    stream = torch.cuda.Stream(dev)
    step_bytes = sum(o.bytes for o in ops)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    calls = [o.bind_raw(stream.cuda_stream) for o in ops]
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            for o in ops + extra_ops:
                o.api_call()       # the public API once per op and warm-up step
            for c in calls:
                c()
    barrier()

    # Timed region, two phases, both CUDA graphs replayed on `stream` and timed
    # with CUDA events on it (the host never starves the GPU between launches):
    #  1. the step: M steps (7 launches each) per graph, replayed R times;
    #     `value` and `ms_per_step` come from here;
    #  2. each producer alone: a graph of `per_op_launches` back-to-back calls
    #     over rotating copies of its buffers (together > 3x L2, so every call
    #     reads HBM), replayed 3 times; `per_op` and `roofline` come from here.
    M = max(1, min(args.graph_steps, args.steps))
    R = max(1, -(-args.steps // M))
    steps = M * R
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for _ in range(M):
            for c in calls:
                c()
    with torch.cuda.stream(stream):
        graph.replay()
    barrier()

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size if hasattr(
        torch.cuda.get_device_properties(dev), "L2_cache_size") else 129 * 2 ** 20
    per_op_graphs = []
    for o in ops + extra_ops:
        # rotating buffer sets > 3x L2 (at most one per call of the graph: the
        # launch-bound shapes then run from L2, which bounds them no more than
        # their launches do)
        nsets = min(args.per_op_launches, max(2, -(-3 * l2 // o.bytes)))
        copies = [o] + [DeviceOp(ap, o.name, o.w, dev) for _ in range(nsets - 1)]
        ccalls = [c.bind_raw(stream.cuda_stream) for c in copies]
        with torch.cuda.stream(stream):
            for c in ccalls:
                c()
        g = torch.cuda.CUDAGraph()
        n = args.per_op_launches
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                ccalls[i % nsets]()
        with torch.cuda.stream(stream):
            g.replay()
        per_op_graphs.append((o, g, n, copies, nsets))
    barrier()

    # Copy reference per producer: a graph of the same number of back-to-back
    # SM copy kernels (torch's vectorised elementwise int32 "+ 0") that move the
    # producer's algorithmic bytes (read half, write half) over rotating buffers
    # (> 3x L2), timed the same way: the bandwidth a plain streaming kernel of
    # that size reaches on this GPU, launch ramp and drain included.
    copy_graphs = []
    for o in ops + extra_ops:
        words = max(4, (o.bytes // 8) // 4 * 4)
        nsets = min(args.per_op_launches, max(2, -(-3 * l2 // (8 * words))))
        bufs = [(torch.zeros(words, dtype=torch.int32, device=dev), torch.empty(words, dtype=torch.int32, device=dev))
                for _ in range(nsets)]
        g = torch.cuda.CUDAGraph()
        n = args.per_op_launches
        with torch.cuda.stream(stream):
            for src, dst in bufs:
                torch.add(src, 0, out=dst)
            with torch.cuda.graph(g, stream=stream):
                for i in range(n):
                    torch.add(bufs[i % nsets][0], 0, out=bufs[i % nsets][1])
            g.replay()
        copy_graphs.append((g, n, bufs))
    barrier()

    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    smi_index = vis.split(",")[local_rank] if vis else str(local_rank)
    clocks = ClockSampler(smi_index)
    clocks.start()
    time.sleep(0.3)
    barrier()
    clocks.mark("t0")
    op_events = []
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for _ in range(R):
            graph.replay()
        t_end.record(stream)
        for o, g, n, _, _ in per_op_graphs:
            evs = []
            for _ in range(args.op_replays):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                g.replay()
                e1.record(stream)
                evs.append((e0, e1))
            op_events.append(evs)
        copy_events = []
        for g, n, _ in copy_graphs:
            evs = []
            for _ in range(3):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                g.replay()
                e1.record(stream)
                evs.append((e0, e1))
            copy_events.append(evs)
    barrier()
    # the same step graph replayed enough times for ~400 steps, after the timed
    # K steps: a longer look at the step time (context beside `value`)
    rep_n = max(1, -(-400 // M))
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        r0.record(stream)
        for _ in range(rep_n):
            graph.replay()
        r1.record(stream)
    barrier()
    clocks.mark("t1")
    clocks.stop()
    rep_ms = max_over_ranks(r0.elapsed_time(r1), world, dev)
    step_repeat = {"steps": rep_n * M, "ms_per_step": round(rep_ms / (rep_n * M), 5),
                   "value": round(job_gbs(step_bytes, world, rep_ms / (rep_n * M)), 1), "unit": "GB/s"}
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    ms_per_step = elapsed_ms / steps
    value = job_gbs(step_bytes, world, ms_per_step)
    args.steps = steps
    launches = sum(launches_per_call(o.name, o.w) for o in ops) * steps + \
        sum(launches_per_call(o.name, o.w) * n * args.op_replays for o, _, n, _, _ in per_op_graphs)
    del per_op_graphs, copy_graphs

    peaks = measured_peaks()
    hbm = peaks.get("hbm_gbs") if peaks else None
    peak_src = "measured" if hbm else "fallback"
    hbm = hbm or 6800.0
    per_op = []
    for i, o in enumerate(ops + extra_ops):
        n = args.per_op_launches
        calls = [e0.elapsed_time(e1) * 1e3 / n for e0, e1 in op_events[i]]
        us = statistics.median(calls)
        gbs = o.bytes / (us * 1e-6) / 1e9
        copy_us = statistics.median(e0.elapsed_time(e1) for e0, e1 in copy_events[i]) * 1e3 / n
        launch_bound = o.w.rows < LAUNCH_BOUND_ROWS
        rec = {"op": o.name, "rows": o.w.rows, "dim": o.w.dim, "us_per_call": round(us, 3),
               "us_p10": round(float(np.percentile(calls, 10)), 3),
               "us_p90": round(float(np.percentile(calls, 90)), 3),
               "alg_bytes": o.bytes, "gbs": round(gbs, 1),
               "frac_of_hbm_peak": None if launch_bound else round(gbs / hbm, 4),
               "copy_us": round(copy_us, 3), "frac_of_copy": None if launch_bound else round(copy_us / us, 4),
               "in_step": i < len(ops)}
        if launch_bound:
            rec["launch_bound"] = True
        kind = op_kind(o.name)
        if kind.startswith("nvfp4_2level"):
            # passes over the input counted in alg_bytes (SwiGLU: always two)
            rec["input_passes"] = two_level_passes(o.name, o.w) if kind != "nvfp4_2level_swiglu_h3" else 2
        page = page_context(o.name, o.w.rows, o.w.dim)
        if page:
            rec["page"] = page
        per_op.append(rec)
    dom = max(range(len(ops)), key=lambda i: per_op[i]["us_per_call"])  # largest share of the step
    d = per_op[dom]
    roofline = {"bound": "hbm", "kernel": d["op"], "achieved": d["gbs"], "peak": hbm, "peak_source": peak_src,
                "unit": "GB/s", "frac": round(d["gbs"] / hbm, 4), "alg_bytes_per_launch": d["alg_bytes"],
                "traffic": committed_traffic(d["op"])}

    # end to end through the Python API with host buffers (pinned), fewer steps
    e2e = None if args.no_e2e else run_e2e(ap, works, dev, stream, args, world, step_bytes, barrier)
    # the NVFP4 producer feeding a block-scaled GEMM (context, outside the step)
    chain = None if (args.no_chain or args.only) else run_chain(ap, dev, stream)

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "step_alg_bytes": step_bytes,
                   "l2": "no flush: each step streams ~0.9 GB of distinct buffers (> 129 MB L2) between repeats "
                         "of any producer", "parallelism": f"replicas x{world} (rows shard, no collective)"},
        "roofline": roofline, "per_op": per_op, "e2e": e2e, "chain": chain,
        "step_repeat": step_repeat,
        "gpu_launches": launches + rep_n * M * sum(launches_per_call(o.name, o.w) for o in ops),
        "clocks": clocks.summary(),
        "timing": ("step: exactly %d steps timed, %d replay(s) of a CUDA graph of %d steps (%.2f ms of GPU time); "
                   "step_repeat: the same graph replayed %d times (%d steps) right after, a longer look at the same "
                   "step; per_op: graph of %d back-to-back calls per producer over rotating buffers > 3x L2 (at most "
                   "one set per call: shapes below %d rows are launch-bound, run from L2 and carry no bandwidth "
                   "fraction), median (us_per_call), p10 and p90 of the per-call time over %d replays; copy_us: the "
                   "same for a streaming copy kernel (torch int32 add of 0) moving the producer's algorithmic bytes, "
                   "median of 3 replays, frac_of_copy = copy_us / us_per_call"
                   % (steps, R, M, elapsed_ms, rep_n, rep_n * M, args.per_op_launches, LAUNCH_BOUND_ROWS,
                      args.op_replays)),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(works, budget_s=args.cpu_seconds)
    return result


def run_chain(ap, dev, stream, reps: int = 16):
    """NVFP4 broadcast producer (5070x3072) followed by cuBLASLt's NVFP4
    block-scaled GEMM against a (3072, 3072) NVFP4 weight made by the plain
    producer: the chain and the GEMM alone, each a CUDA graph of `reps`
    iterations timed with CUDA events.  The GEMM is library code; it is here
    to show the producer's output consumed in place and what the producer adds
    in front of its consumer."""
    if not hasattr(torch, "float4_e2m1fn_x2"):
        return {"unavailable": "this torch build has no float4_e2m1fn_x2 (no NVFP4 scaled GEMM)"}
    M, N, K = 5070, 3072, 3072
    wa, wb = synth.nvfp4_broadcast(M, K, 1004), synth.nvfp4_ln(N, K, 2009)
    x, sc, sh = (wa.inputs[k].to(dev) for k in ("x", "scale", "shift"))
    a_pk = torch.empty((M, K // 2), dtype=torch.uint8, device=dev)
    a_sf = torch.empty((ap.swizzled_sf_size(M, K),), dtype=torch.uint8, device=dev)
    fp4, e4 = torch.float4_e2m1fn_x2, torch.float8_e4m3fn
    with torch.cuda.stream(stream):
        b_pk, b_sf = ap.layer_norm_no_affine_quant_nvfp4_swizzled_bf16(wb.inputs["x"].to(dev))

        def produce():
            ap.ada_layer_norm_quant_nvfp4_swizzled_bf16(x, sc, sh, packed=a_pk, sf_swizzled=a_sf)

        def gemm():
            return torch._scaled_mm(a_pk.view(fp4), b_pk.view(fp4).t(), a_sf.view(e4), b_sf.view(e4),
                                    out_dtype=torch.bfloat16)
        produce()
        gemm()
        graphs = {}
        for name, body in (("gemm", gemm), ("chain", lambda: (produce(), gemm()))):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(reps):
                    body()
            g.replay()
            graphs[name] = g
        stream.synchronize()
        us = {}
        for name in ("gemm", "chain", "gemm", "chain"):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graphs[name].replay()
            e1.record(stream)
            e1.synchronize()
            t = e0.elapsed_time(e1) * 1e3 / reps
            us[name] = min(us.get(name, t), t)
    return {"producer": f"ada_layer_norm_quant_nvfp4_swizzled_bf16 {M}x{K}",
            "consumer": f"cuBLASLt NVFP4 block-scaled GEMM (torch._scaled_mm) {M}x{N}x{K}, bf16 out",
            "us_gemm": round(us["gemm"], 3), "us_chain": round(us["chain"], 3),
            "us_producer_in_chain": round(us["chain"] - us["gemm"], 3),
            "gemm_tflops": round(2.0 * M * N * K / (us["gemm"] * 1e-6) / 1e12, 1),
            "timing": f"CUDA graphs of {reps} iterations, best of 2 replays"}


def run_e2e(ap, works, dev, stream, args, world, step_bytes, barrier):
    """The step through the Python API with host buffers, pipelined: every step
    copies all of its inputs from pinned host memory (stream h2d), runs the
    seven producers (stream comp) and copies all of their outputs back to
    pinned host memory (stream d2h).  Two device buffer sets alternate, so
    step k+1's inputs travel while step k computes and step k-1's outputs
    travel back; host->device and device->host copies use separate copy
    engines."""
    host_in, host_out = [], []
    h2d = d2h = 0
    for name, w in works:
        host_in.append({k: v.pin_memory() for k, v in w.inputs.items()})
        h2d += sum(v.numel() * v.element_size() for v in w.inputs.values())
    sets = []
    for _ in range(2):
        ops = []
        for (name, w), hin in zip(works, host_in):
            op = DeviceOp.__new__(DeviceOp)
            op.ap, op.name, op.w = ap, name, w
            op.d = {k: torch.empty_like(v, device=dev) for k, v in hin.items()}
            R, D = w.rows, w.dim
            if name.startswith("fp8"):
                op.out = (torch.empty((R, D), dtype=torch.float8_e4m3fn, device=dev),)
            elif name.startswith("nvfp4"):
                op.out = (torch.empty((R, D // 2), dtype=torch.uint8, device=dev),
                          torch.empty((ap.swizzled_sf_size(R, D),), dtype=torch.uint8, device=dev))
            else:
                op.out = (torch.empty((6, 1, R, D), dtype=torch.bfloat16, device=dev),)
            ops.append(op)
        sets.append(ops)
    for op in sets[0]:
        host_out.append(tuple(torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in op.out))
        d2h += sum(o.numel() * o.element_size() for o in op.out)

    s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    free = [torch.cuda.Event(), torch.cuda.Event()]   # set's outputs copied out
    ready = [torch.cuda.Event(), torch.cuda.Event()]  # set's inputs copied in
    done = [torch.cuda.Event(), torch.cuda.Event()]   # set's producers finished

    def one_step(k):
        b = k % 2
        ops = sets[b]
        with torch.cuda.stream(s_in):
            if k >= 2:
                s_in.wait_event(free[b])
            for op, hin in zip(ops, host_in):
                for key, v in hin.items():
                    op.d[key].copy_(v, non_blocking=True)
            ready[b].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(ready[b])
            for op in ops:
                op.api_call()
            done[b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(done[b])
            for op, hout in zip(ops, host_out):
                for h, o in zip(hout, op.out):
                    h.copy_(o, non_blocking=True)
            free[b].record(s_out)

    steps = max(3, min(args.e2e_steps, args.steps))
    for k in range(2):
        one_step(k)
    barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    for k in range(steps):
        one_step(k)
    with torch.cuda.stream(s_out):
        t1.record(s_out)
    barrier()
    ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    ms_step = ms / steps
    return {"value": round(job_gbs(step_bytes, world, ms_step), 1), "unit": "GB/s",
            "ms_per_step": round(ms_step, 4), "steps": steps, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "pipeline": "h2d / producers / d2h on three streams, two device buffer sets",
            "binding": ap.marshalling()}


# ---------------------------------------------------------------------------
# CPU oracle (reported baseline and the reference arm)
# ---------------------------------------------------------------------------

def oracle_sample_step(works, frac_rows: int, nthreads: int):
    """Run the oracle on the first rows/frac_rows rows of every producer; returns the
    algorithmic bytes of the sample."""
    import oracle
    total = 0
    for name, w in works:
        n = max(1, w.rows // frac_rows)
        x = synth.u16(w.inputs["x"][:n]) if "x" in w.inputs else None
        eps = w.params.get("eps", 1e-5)
        if name == "fp8_broadcast":
            oracle.ln_quant_fp8(x, 0.025, oracle.MOD_BCAST, eps, nthreads, scale=synth.u16(w.inputs["scale"]),
                                shift=synth.u16(w.inputs["shift"]))
        elif name == "fp8_layer_norm":
            oracle.ln_quant_fp8(x, 0.025, oracle.MOD_NONE, eps, nthreads)
        elif name == "fp8_per_token":
            oracle.ln_quant_fp8(x, 0.025, oracle.MOD_PTOK, eps, nthreads, scale=synth.u16(w.inputs["scale"][:n]),
                                shift=synth.u16(w.inputs["shift"][:n]))
        elif name == "fp8_table":
            oracle.ln_quant_fp8(x, 0.025, oracle.MOD_TABLE, eps, nthreads, temb=synth.u16(w.inputs["temb"][:n]),
                                table=w.inputs["table"].numpy(), shift_idx=w.params["shift_idx"],
                                scale_idx=w.params["scale_idx"])
        elif name == "nvfp4_broadcast":
            oracle.ln_quant_nvfp4(x, oracle.MOD_BCAST, eps, nthreads, scale=synth.u16(w.inputs["scale"]),
                                  shift=synth.u16(w.inputs["shift"]))
        elif name == "nvfp4_layer_norm":
            oracle.ln_quant_nvfp4(x, oracle.MOD_NONE, eps, nthreads)
        elif name in ("fp8_modfp8", "nvfp4_modfp8"):
            src = dict(scale_fp8=w.inputs["scale_fp8"].view(torch.uint8).numpy(),
                       shift_fp8=w.inputs["shift_fp8"].view(torch.uint8).numpy(),
                       scale_deq=float(w.inputs["scale_deq"][0]), shift_deq=float(w.inputs["shift_deq"][0]))
            if name == "fp8_modfp8":
                oracle.ln_quant_fp8(x, 0.025, oracle.MOD_MODFP8, eps, nthreads, **src)
            else:
                oracle.ln_quant_nvfp4(x, oracle.MOD_MODFP8, eps, nthreads, **src)
        elif name == "fp8_awq":
            oracle.ln_quant_fp8(x, 0.025, oracle.MOD_AWQ, eps, nthreads, scale=synth.u16(w.inputs["scale"]),
                                shift=synth.u16(w.inputs["shift"]), inv_s=synth.u16(w.inputs["inv_s"]))
        elif name in ("fp8_seg_h3", "nvfp4_2level_seg_h3"):
            src = dict(seg_idx=w.inputs["seg_idx"][:n].numpy(), seg_scale=synth.u16(w.inputs["seg_scale"]),
                       seg_shift=synth.u16(w.inputs["seg_shift"]))
            if name == "fp8_seg_h3":
                oracle.ln_quant_fp8(x, 0.025, oracle.MOD_SEG, eps, nthreads, **src)
            else:
                oracle.ln_quant_nvfp4_2level(x, oracle.MOD_SEG, eps, nthreads, **src)
        elif name == "nvfp4_2level_layer_norm":
            oracle.ln_quant_nvfp4_2level(x, oracle.MOD_NONE, eps, nthreads)
        elif name == "modulation6":
            oracle.adaln_modulation6(w.inputs["params"][:, :n].numpy(), w.inputs["modulation"].numpy(), nthreads)
        sub = synth.Workload(w.op, n, w.dim)
        total += alg_bytes(name, sub)
    return total


def host_cpu() -> str:
    """The host CPU's model as the OS reports it (lscpu's model name, else
    /proc/cpuinfo), for the oracle timings."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def cpu_baseline(works, budget_s: float = 15.0, frac_rows: int = 8, single_s: float = 3.0):
    """The oracle timed on the host cores: row-parallel over every core for
    ~budget_s, then single-threaded for ~single_s (smaller samples)."""
    import oracle
    oracle.build()
    nthreads = oracle.default_threads()
    oracle_sample_step(works, 64, nthreads)  # warm the page cache / code
    t0 = time.perf_counter()
    reps, total = 0, 0
    while True:
        total += oracle_sample_step(works, frac_rows, nthreads)
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    t1 = time.perf_counter()
    reps1, total1 = 0, 0
    while True:
        total1 += oracle_sample_step(works, frac_rows * 16, 1)
        reps1 += 1
        if time.perf_counter() - t1 >= single_s:
            break
    dt1 = time.perf_counter() - t1
    return {"value": round(total / dt / 1e9, 3), "unit": "GB/s", "cores": nthreads, "kind": "oracle",
            "sample": f"first 1/{frac_rows} of the rows of every producer of the step, repeated {reps}x "
                      f"({dt:.1f} s, {total / 1e9:.2f} GB algorithmic)",
            "single_thread": {"value": round(total1 / dt1 / 1e9, 4), "unit": "GB/s",
                              "sample": f"first 1/{frac_rows * 16} of the rows, repeated {reps1}x ({dt1:.1f} s)"},
            "host_cpu": host_cpu(), "nproc": os.cpu_count()}


def run_reference(args):
    works = step_workloads()
    step_bytes = sum(alg_bytes(n, w) for n, w in works)
    import oracle
    oracle.build()
    nthreads = oracle.default_threads()
    frac = 16
    for _ in range(max(0, min(args.warmup, 1))):
        oracle_sample_step(works, frac, nthreads)
    times, sample_bytes = [], 0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        sample_bytes = oracle_sample_step(works, frac, nthreads)
        times.append(time.perf_counter() - t0)
    dt = sum(times)
    value = sample_bytes * len(times) / dt / 1e9
    ms_full = step_bytes / (value * 1e9) * 1e3
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_full, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "sampled": True,
            "sample_wall_s": round(dt, 3), "ms_per_step_sampled": round(dt / len(times) * 1e3, 3),
            "config": {"workload": WORKLOAD, "step_alg_bytes": step_bytes,
                       "sample": f"sampled: each step runs the CPU oracle on the first 1/{frac} of the rows of every "
                                 f"producer ({sample_bytes} algorithmic bytes, {dt / len(times) * 1e3:.1f} ms per "
                                 f"step, {dt:.2f} s for all steps); value is those bytes over that time, and "
                                 f"ms_per_step ({ms_full:.1f} ms) the full step's bytes at that rate -- an "
                                 f"extrapolation, not a timed full step"},
            "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": nthreads, "kind": "oracle",
                             "sample": f"first 1/{frac} of the rows of every producer, {args.steps} steps"},
            "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------------------
# row sweep of the FP8 broadcast producer (optional)
# ---------------------------------------------------------------------------

# the pages' RTX 5090 shapes of the FP8 broadcast and layer-norm producers
PAGE_SHAPES = ((16, 2048), (64, 3072), (256, 3072), (2520, 3072), (4096, 3072))


def eager_context(op, xs, sc, sh, act, nsets, st):
    """Context only: the PyTorch eager chain the pages time beside their
    producers (F.layer_norm, then *(1+scale)+shift for the broadcast form,
    / act_scale, clamp to +-448, .to(float8_e4m3fn)), on this GPU, timed the
    same two ways as the producer: device time per call from a CUDA graph of
    32 calls over the rotating buffers, and one direct call.  It is not the
    product path and no output of it is used."""
    import torch.nn.functional as F
    D = xs[0].shape[1]

    def chain(i):
        y = F.layer_norm(xs[i], (D,), eps=1e-5)
        if op == "fp8_broadcast":
            y = y * (1 + sc) + sh
        return (y / act).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)

    with torch.cuda.stream(st):
        for i in range(nsets):
            chain(i)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            for i in range(32):
                chain(i % nsets)
        g.replay()
        ts = []
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            g.replay()
            e1.record(st)
            st.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3 / 32)
        single = []
        for k in range(20):
            st.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            chain(k % nsets)
            e1.record(st)
            st.synchronize()
            single.append(e0.elapsed_time(e1) * 1e3)
    del g
    return {"eager_us_per_call": round(statistics.median(ts), 3),
            "eager_us_single_launch": round(statistics.median(single), 3)}


def run_sweep(args, dev):
    """FP8 broadcast row sweep (dims 1536 and 3072, rows 51...32768) plus the pages'
    RTX 5090 shapes for the broadcast and layer-norm producers.  Per shape: device
    time per call (a graph of 32 back-to-back calls over rotating buffers > 3x L2,
    median of 3 replays) and single-launch time (CUDA events around one direct
    call after a synchronize, median of 20: host launch latency included); at
    the pages' shapes also the PyTorch eager chain, as context (eager_context)."""
    import nvfp4_activation_producer_gb300 as ap
    l2 = 129 * 2 ** 20
    shapes = [("fp8_broadcast", R, D) for D in synth.SWEEP_DIMS for R in synth.SWEEP_ROWS]
    shapes += [(op, R, D) for op in ("fp8_broadcast", "fp8_layer_norm") for R, D in PAGE_SHAPES]
    res = []
    eager_done = set()
    st = torch.cuda.Stream(dev)
    for op, R, D in shapes:
        w = synth.fp8_broadcast(R, D, synth.SWEEP_SEED)
        one = alg_bytes(op, w)
        nsets = min(max(2, int(np.ceil(3 * l2 / one))), 512)
        xs = [w.inputs["x"].to(dev) for _ in range(nsets)]
        outs = [torch.empty((R, D), dtype=torch.float8_e4m3fn, device=dev) for _ in range(nsets)]
        sc, sh, act = (w.inputs[k].to(dev) for k in ("scale", "shift", "act_scale"))

        def call(i):
            if op == "fp8_broadcast":
                ap.ada_layer_norm_quant_fp8_bf16(xs[i], sc, sh, act, out=outs[i])
            else:
                ap.layer_norm_no_affine_quant_fp8_static_bf16(xs[i], act, out=outs[i])
        with torch.cuda.stream(st):
            for i in range(nsets):
                call(i)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                for i in range(32):
                    call(i % nsets)
            g.replay()
            ts = []
            for _ in range(3):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(st)
                g.replay()
                e1.record(st)
                st.synchronize()
                ts.append(e0.elapsed_time(e1) * 1e3 / 32)
            single = []
            for k in range(20):
                st.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(st)
                call(k % nsets)
                e1.record(st)
                st.synchronize()
                single.append(e0.elapsed_time(e1) * 1e3)
        us = statistics.median(ts)
        rec = {"op": op, "rows": R, "dim": D, "us_per_call": round(us, 3),
               "us_single_launch": round(statistics.median(single), 3), "gbs": round(one / us / 1e3, 1),
               "rows_per_s": round(R / us * 1e6), "buffer_sets": nsets}
        if (R, D) in PAGE_SHAPES and (op, R, D) not in eager_done:
            rec.update(eager_context(op, xs, sc, sh, act, nsets, st))
            eager_done.add((op, R, D))
        res.append(rec)
        del xs, outs, g
    return res


def main():
    ap_ = argparse.ArgumentParser()
    ap_.add_argument("--gpus", type=int, default=1)
    ap_.add_argument("--steps", type=int, default=2000)
    ap_.add_argument("--warmup", type=int, default=20)
    ap_.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap_.add_argument("--e2e-steps", type=int, default=20)
    ap_.add_argument("--graph-steps", type=int, default=25, help="steps captured per CUDA graph")
    ap_.add_argument("--per-op-launches", type=int, default=32, help="back-to-back calls per producer graph")
    ap_.add_argument("--op-replays", type=int, default=11,
                     help="replays of each producer graph (median, p10 and p90 of the per-call time)")
    ap_.add_argument("--only", default=None, help="comma list of producers to run (for profiling one kernel)")
    ap_.add_argument("--cpu-seconds", type=float, default=15.0)
    ap_.add_argument("--no-cpu-baseline", action="store_true")
    ap_.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap_.add_argument("--no-chain", action="store_true", help="skip the producer -> NVFP4 GEMM chain leg")
    ap_.add_argument("--no-extra", action="store_true",
                     help="skip the producers measured beside the step (modfp8, AWQ)")
    ap_.add_argument("--sweep", action="store_true", help="also time the FP8 broadcast row sweep")
    ap_.add_argument("--out", default=None, help="also write the JSON line (and the sweep) to this file")
    args = ap_.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            line = run_reference(args)
            print(json.dumps(line), flush=True)
        return

    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    result = run_ours(args, rank, world, local_rank)
    if args.sweep and rank == 0:
        result["sweep"] = run_sweep(args, torch.device("cuda", local_rank))
    if rank == 0:
        line = json.dumps(result)
        print(line, flush=True)
        if args.out:
            with open(args.out, "w") as f:
                f.write(line + "\n")
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
