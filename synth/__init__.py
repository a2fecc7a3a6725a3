"""Seeded synthetic inputs for the producers.

This module only draws random numbers and lays them out in the shapes and
dtypes of the producers' tensor contract (adaptive-layernorm-producers README,
"Tensor Contract").  It holds none of the producers' arithmetic, so both the
CPU oracle's tests and the CUDA path can take their inputs from it.

Every tensor is drawn from numpy's PCG64 generator seeded with
``seed * 1000 + k`` (k = position of the tensor in the workload), as float32
normals times the stated standard deviation, then converted with torch's
float32 -> bfloat16 conversion where the contract says bf16.  Outlier rows are
multiplied by 8, which is exact in bf16.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


def normal(seed: int, k: int, shape, std: float) -> np.ndarray:
    rng = np.random.default_rng(seed * 1000 + k)
    a = rng.standard_normal(size=int(np.prod(shape)), dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a.reshape(shape)


def bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def u16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (CPU) -> its uint16 bit patterns as a numpy array."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def outlier_rows(seed: int, rows: int, frac: float = 0.01) -> np.ndarray:
    rng = np.random.default_rng(seed * 1000 + 999)
    n = int(round(frac * rows))
    return np.sort(rng.permutation(rows)[:n])


@dataclass
class Workload:
    """One producer call: op name, sizes and the CPU tensors of its inputs."""
    op: str
    rows: int
    dim: int
    inputs: dict = field(default_factory=dict)
    params: dict = field(default_factory=dict)

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in self.inputs.values())


def fp8_broadcast(rows: int, dim: int, seed: int, act_scale: float = 0.025,
                  eps: float = 1e-5, outliers: float = 0.0) -> Workload:
    x = normal(seed, 0, (rows, dim), 1.0)
    if outliers:
        x[outlier_rows(seed, rows, outliers)] *= 8.0
    return Workload("ada_layer_norm_quant_fp8_bf16", rows, dim,
                    {"x": bf16(x), "scale": bf16(normal(seed, 1, (dim,), 0.1)),
                     "shift": bf16(normal(seed, 2, (dim,), 0.1)),
                     "act_scale": torch.tensor([act_scale], dtype=torch.float32)},
                    {"eps": eps})


def fp8_ln(rows: int, dim: int, seed: int, act_scale: float = 0.025,
           eps: float = 1e-5) -> Workload:
    x = normal(seed, 0, (rows, dim), 1.0)
    return Workload("layer_norm_no_affine_quant_fp8_static_bf16", rows, dim,
                    {"x": bf16(x), "act_scale": torch.tensor([act_scale], dtype=torch.float32)},
                    {"eps": eps})


def fp8_ptok(rows: int, dim: int, seed: int, act_scale: float = 0.025,
             eps: float = 1e-5, outliers: float = 0.01) -> Workload:
    x = normal(seed, 0, (rows, dim), 1.0)
    if outliers:
        x[outlier_rows(seed, rows, outliers)] *= 8.0
    return Workload("ada_layer_norm_quant_fp8_ptok_bf16", rows, dim,
                    {"x": bf16(x), "scale": bf16(normal(seed, 1, (rows, dim), 0.1)),
                     "shift": bf16(normal(seed, 2, (rows, dim), 0.1)),
                     "act_scale": torch.tensor([act_scale], dtype=torch.float32)},
                    {"eps": eps})


def fp8_table(rows: int, dim: int, seed: int, chunks: int = 6, shift_idx: int = 0,
              scale_idx: int = 1, act_scale: float = 0.025, eps: float = 1e-5) -> Workload:
    x = normal(seed, 0, (rows, dim), 1.0)
    return Workload("ada_layer_norm_quant_fp8_ptok_table_bf16", rows, dim,
                    {"x": bf16(x), "temb": bf16(normal(seed, 1, (rows, chunks, dim), 0.1)),
                     "table": torch.from_numpy(normal(seed, 2, (chunks, dim), 0.05)),
                     "act_scale": torch.tensor([act_scale], dtype=torch.float32)},
                    {"eps": eps, "shift_idx": shift_idx, "scale_idx": scale_idx})


def nvfp4_broadcast(rows: int, dim: int, seed: int, eps: float = 1e-5) -> Workload:
    x = normal(seed, 0, (rows, dim), 1.0)
    return Workload("ada_layer_norm_quant_nvfp4_swizzled_bf16", rows, dim,
                    {"x": bf16(x), "scale": bf16(normal(seed, 1, (dim,), 0.1)),
                     "shift": bf16(normal(seed, 2, (dim,), 0.1))},
                    {"eps": eps})


def nvfp4_ln(rows: int, dim: int, seed: int, eps: float = 1e-5) -> Workload:
    x = normal(seed, 0, (rows, dim), 1.0)
    return Workload("layer_norm_no_affine_quant_nvfp4_swizzled_bf16", rows, dim,
                    {"x": bf16(x)}, {"eps": eps})


def e4m3(a: np.ndarray) -> torch.Tensor:
    """float32 -> torch.float8_e4m3fn (torch's conversion; |a| kept below 448)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)


def fp8_modfp8(rows: int, dim: int, seed: int, act_scale: float = 0.025, eps: float = 1e-5,
               scale_deq: float = 0.05, shift_deq: float = 0.05) -> Workload:
    """modfp8 broadcast form: scale_fp8/shift_fp8 are e4m3 draws of N(0, 2), so that
    code * 0.05 has the spread N(0, 0.1) of the bf16 broadcast vectors."""
    x = normal(seed, 0, (rows, dim), 1.0)
    return Workload("ada_layer_norm_quant_fp8_modfp8_bf16", rows, dim,
                    {"x": bf16(x), "scale_fp8": e4m3(normal(seed, 1, (dim,), 2.0)),
                     "shift_fp8": e4m3(normal(seed, 2, (dim,), 2.0)),
                     "scale_deq": torch.tensor([scale_deq], dtype=torch.float32),
                     "shift_deq": torch.tensor([shift_deq], dtype=torch.float32),
                     "act_scale": torch.tensor([act_scale], dtype=torch.float32)},
                    {"eps": eps})


def nvfp4_modfp8(rows: int, dim: int, seed: int, eps: float = 1e-5,
                 scale_deq: float = 0.05, shift_deq: float = 0.05) -> Workload:
    x = normal(seed, 0, (rows, dim), 1.0)
    return Workload("ada_layer_norm_quant_nvfp4_swizzled_modfp8_bf16", rows, dim,
                    {"x": bf16(x), "scale_fp8": e4m3(normal(seed, 1, (dim,), 2.0)),
                     "shift_fp8": e4m3(normal(seed, 2, (dim,), 2.0)),
                     "scale_deq": torch.tensor([scale_deq], dtype=torch.float32),
                     "shift_deq": torch.tensor([shift_deq], dtype=torch.float32)},
                    {"eps": eps})


def fp8_awq(rows: int, dim: int, seed: int, act_scale: float = 0.025, eps: float = 1e-5) -> Workload:
    """AWQ broadcast form: inv_s = exp(N(0, 0.5)) per channel (positive smoothing
    factors around 1, spread over about a factor of 3 each way)."""
    x = normal(seed, 0, (rows, dim), 1.0)
    return Workload("awq_ada_layer_norm_quant_fp8_bf16", rows, dim,
                    {"x": bf16(x), "scale": bf16(normal(seed, 1, (dim,), 0.1)),
                     "shift": bf16(normal(seed, 2, (dim,), 0.1)),
                     "inv_s": bf16(np.exp(normal(seed, 3, (dim,), 0.5))),
                     "act_scale": torch.tensor([act_scale], dtype=torch.float32)},
                    {"eps": eps})


# The segment layout of the h3-blackwell-runtime compare page's attention-output
# record (37,810 packed tokens): rows [0, 100) use table row 1, [100, 514) row 2,
# the rest row 0.
H3_SEGMENTS = ((0, 100, 1), (100, 514, 2), (514, 37810, 0))


def segment_index(rows: int, segments=H3_SEGMENTS) -> np.ndarray:
    """(rows,) int32 table row per row; the ranges are scaled to `rows` when
    rows differs from the layout's 37,810 (at least one row per range)."""
    total = segments[-1][1]
    idx = np.empty(rows, dtype=np.int32)
    start = 0
    for n, (lo, hi, g) in enumerate(segments):
        end = rows if n == len(segments) - 1 else max(start + 1, min(rows, round(hi * rows / total)))
        idx[start:end] = g
        start = end
    return idx


def segmented(rows: int, dim: int, seed: int, nseg: int = 3, act_scale: float = 0.025,
              eps: float = 1e-5) -> Workload:
    """Segmented modulation: x N(0, 1); (nseg, dim) bf16 scale/shift tables
    N(0, 0.1); the page's segment layout scaled to `rows`."""
    x = normal(seed, 0, (rows, dim), 1.0)
    return Workload("ada_layer_norm_quant_*_seg_bf16", rows, dim,
                    {"x": bf16(x), "seg_idx": torch.from_numpy(segment_index(rows)),
                     "seg_scale": bf16(normal(seed, 1, (nseg, dim), 0.1)),
                     "seg_shift": bf16(normal(seed, 2, (nseg, dim), 0.1)),
                     "act_scale": torch.tensor([act_scale], dtype=torch.float32)},
                    {"eps": eps})


def swiglu(rows: int, dim: int, seed: int) -> Workload:
    """SwiGLU input in the FC1-output layout: one (rows, 2*dim) bf16 tensor
    N(0, 1) whose halves [:, :dim] and [:, dim:] are gate and up."""
    return Workload("swiglu_*_bf16", rows, dim, {"fc1": bf16(normal(seed, 0, (rows, 2 * dim), 1.0))}, {})


def modulation6(batch: int, seq: int, dim: int, seed: int) -> Workload:
    return Workload("adaln_modulation6_bf16", batch * seq, dim,
                    {"params": torch.from_numpy(normal(seed, 0, (batch, seq, 6, dim), 1.0)),
                     "modulation": torch.from_numpy(normal(seed, 1, (6, dim), 0.02))},
                    {"batch": batch, "seq": seq})


# The five workloads of the producers' benchmark table, with their seeds.
CONFIGS = {
    "fp8_broadcast_16x2048": lambda: fp8_broadcast(16, 2048, 1001),
    "fp8_ptok_2520x3072": lambda: fp8_ptok(2520, 3072, 1002),
    "fp8_table_4096x3072": lambda: fp8_table(4096, 3072, 1003),
    "nvfp4_broadcast_5070x3072": lambda: nvfp4_broadcast(5070, 3072, 1004),
    "nvfp4_ln_5070x3072": lambda: nvfp4_ln(5070, 3072, 1004),
    "modulation6_1x5070x3072": lambda: modulation6(1, 5070, 3072, 1005),
}

# Row sweep of the FP8 broadcast producer (dims 1536 and 3072).
SWEEP_ROWS = (51, 105, 256, 1024, 2520, 4096, 5070, 8192, 16384, 32768)
SWEEP_DIMS = (1536, 3072)
SWEEP_SEED = 1006
