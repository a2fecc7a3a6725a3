"""CPU oracle for the adaptive-LayerNorm activation producers (Python side).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
CUDA library and its Python binding never do.

The arithmetic lives in ``orc.c`` (plain scalar C, fp64 statistics); this file
compiles it with gcc and marshals numpy arrays through ctypes.  bf16 arrays are
passed as ``uint16`` bit patterns, e4m3 and packed e2m1 as ``uint8``.

Sources: the adaptive-layernorm-producers README ("Available Functions",
"Tensor Contract", "Minimal Usage", "Validation") and the NVFP4 facts of the
h3-blackwell-runtime compare page (see ``orc.c`` for the readings R1-R8, R15, R16).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "orc.c")
_HDR = os.path.join(_HERE, "orc.h")
_SO = os.path.join(_HERE, "liborc.so")

MOD_NONE, MOD_BCAST, MOD_PTOK, MOD_TABLE, MOD_MODFP8, MOD_AWQ, MOD_SEG = 0, 1, 2, 3, 4, 5, 6


def build(force: bool = False) -> str:
    """Compile ``orc.c`` into ``liborc.so`` (no fast-math, no FP contraction)."""
    stale = (not os.path.exists(_SO)) or any(
        os.path.getmtime(p) > os.path.getmtime(_SO) for p in (_SRC, _HDR))
    if force or stale:
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


class _Mod(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int),
                ("scale", ctypes.c_void_p), ("shift", ctypes.c_void_p),
                ("temb", ctypes.c_void_p), ("table", ctypes.c_void_p),
                ("chunks", ctypes.c_int64), ("shift_idx", ctypes.c_int64),
                ("scale_idx", ctypes.c_int64),
                ("scale_fp8", ctypes.c_void_p), ("shift_fp8", ctypes.c_void_p),
                ("scale_deq", ctypes.c_float), ("shift_deq", ctypes.c_float),
                ("inv_s", ctypes.c_void_p),
                ("seg_idx", ctypes.c_void_p), ("seg_scale", ctypes.c_void_p), ("seg_shift", ctypes.c_void_p),
                ("nseg", ctypes.c_int64)]


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        i64, p, f32, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int
        L.orc_bf16_to_f64.restype = ctypes.c_double
        L.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.orc_bf16_from_f32.restype = ctypes.c_uint16
        L.orc_bf16_from_f32.argtypes = [f32]
        L.orc_e4m3_decode.restype = ctypes.c_double
        L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_e4m3_encode.argtypes = [ctypes.c_double]
        L.orc_e2m1_decode.restype = ctypes.c_double
        L.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
        L.orc_e2m1_encode.restype = ctypes.c_uint8
        L.orc_e2m1_encode.argtypes = [ctypes.c_double, ctypes.c_double]
        L.orc_swizzled_sf_size.restype = i64
        L.orc_swizzled_sf_size.argtypes = [i64, i64]
        L.orc_sf_offset.restype = i64
        L.orc_sf_offset.argtypes = [i64, i64, i64]
        L.orc_swizzle_scales.restype = None
        L.orc_swizzle_scales.argtypes = [p, i64, i64, p]
        L.orc_row_stats.restype = None
        L.orc_row_stats.argtypes = [p, i64, f32, ctypes.POINTER(ctypes.c_double),
                                    ctypes.POINTER(ctypes.c_double)]
        L.orc_modulated_rows.restype = i32
        L.orc_modulated_rows.argtypes = [p, ctypes.POINTER(_Mod), f32, p, i64, i64, i32]
        L.orc_ln_quant_fp8.restype = i32
        L.orc_ln_quant_fp8.argtypes = [p, ctypes.POINTER(_Mod), f32, f32, p, i64, i64, i32]
        L.orc_ln_quant_nvfp4.restype = i32
        L.orc_ln_quant_nvfp4.argtypes = [p, ctypes.POINTER(_Mod), f32, p, p, i64, i64, i32]
        L.orc_ln_quant_nvfp4_swizzled.restype = i32
        L.orc_ln_quant_nvfp4_swizzled.argtypes = [p, ctypes.POINTER(_Mod), f32, p, p, i64, i64, i32]
        L.orc_ln_staged_bf16.restype = i32
        L.orc_ln_staged_bf16.argtypes = [p, ctypes.POINTER(_Mod), f32, p, i64, i64, i32]
        L.orc_nvfp4_2level.restype = i32
        L.orc_nvfp4_2level.argtypes = [p, i64, i64, p, p, ctypes.POINTER(ctypes.c_float), i32]
        L.orc_ln_quant_nvfp4_2level.restype = i32
        L.orc_ln_quant_nvfp4_2level.argtypes = [p, ctypes.POINTER(_Mod), f32, p, p,
                                                ctypes.POINTER(ctypes.c_float), i64, i64, i32]
        L.orc_swiglu_values.restype = i32
        L.orc_swiglu_values.argtypes = [p, p, i64, p, i64, i64, i32]
        L.orc_swiglu_quant_nvfp4_2level.restype = i32
        L.orc_swiglu_quant_nvfp4_2level.argtypes = [p, p, i64, p, p, ctypes.POINTER(ctypes.c_float), i64, i64, i32]
        L.orc_adaln_modulation6.restype = i32
        L.orc_adaln_modulation6.argtypes = [p, p, p, i64, i64, i32]
        _lib = L
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# --------------------------------------------------------------------------
# scalar codecs
# --------------------------------------------------------------------------

def bf16_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_from_f32(v: float) -> int:
    return int(lib().orc_bf16_from_f32(float(v)))


def e4m3_decode(code: int) -> float:
    return float(lib().orc_e4m3_decode(int(code)))


def e4m3_encode(v: float) -> int:
    return int(lib().orc_e4m3_encode(float(v)))


def e2m1_decode(code: int) -> float:
    return float(lib().orc_e2m1_decode(int(code)))


def e2m1_encode(v: float, s_dec: float) -> int:
    return int(lib().orc_e2m1_encode(float(v), float(s_dec)))


def swizzled_sf_size(rows: int, dim: int) -> int:
    return int(lib().orc_swizzled_sf_size(int(rows), int(dim)))


def sf_offset(r: int, c: int, dim: int) -> int:
    return int(lib().orc_sf_offset(int(r), int(c), int(dim)))


def sf_offsets(rows: np.ndarray, cols: np.ndarray, dim: int) -> np.ndarray:
    """Vector of orc_sf_offset(r, c, dim), one ctypes call per pair."""
    L = lib()
    return np.array([L.orc_sf_offset(int(r), int(c), int(dim)) for r, c in zip(rows, cols)],
                    dtype=np.int64)


def swizzle_scales(sf_logical: np.ndarray, rows: int, dim: int) -> np.ndarray:
    sf_logical = np.ascontiguousarray(sf_logical, dtype=np.uint8)
    out = np.empty(swizzled_sf_size(rows, dim), dtype=np.uint8)
    lib().orc_swizzle_scales(sf_logical.ctypes.data, rows, dim, out.ctypes.data)
    return out


def row_stats(x_row: np.ndarray, eps: float):
    x_row = np.ascontiguousarray(x_row, dtype=np.uint16)
    mean, rstd = ctypes.c_double(), ctypes.c_double()
    lib().orc_row_stats(x_row.ctypes.data, x_row.size, eps, ctypes.byref(mean), ctypes.byref(rstd))
    return mean.value, rstd.value


# --------------------------------------------------------------------------
# producers
# --------------------------------------------------------------------------

class _Keep:
    """Holds the contiguous arrays a _Mod points into."""

    def __init__(self):
        self.arrays = []

    def ptr(self, a, dtype):
        if a is None:
            return None
        a = np.ascontiguousarray(a, dtype=dtype)
        self.arrays.append(a)
        return a.ctypes.data


def _mod(keep: _Keep, kind: int, scale=None, shift=None, temb=None, table=None,
         shift_idx: int = 0, scale_idx: int = 0, scale_fp8=None, shift_fp8=None,
         scale_deq: float = 1.0, shift_deq: float = 1.0, inv_s=None, seg_idx=None, seg_scale=None,
         seg_shift=None) -> _Mod:
    m = _Mod()
    m.kind = kind
    m.scale = keep.ptr(scale, np.uint16)
    m.shift = keep.ptr(shift, np.uint16)
    m.temb = keep.ptr(temb, np.uint16)
    m.table = keep.ptr(table, np.float32)
    m.chunks = int(temb.shape[1]) if temb is not None else 0
    m.shift_idx = int(shift_idx)
    m.scale_idx = int(scale_idx)
    m.scale_fp8 = keep.ptr(scale_fp8, np.uint8)
    m.shift_fp8 = keep.ptr(shift_fp8, np.uint8)
    m.scale_deq = float(scale_deq)
    m.shift_deq = float(shift_deq)
    m.inv_s = keep.ptr(inv_s, np.uint16)
    m.seg_idx = keep.ptr(seg_idx, np.int32)
    m.seg_scale = keep.ptr(seg_scale, np.uint16)
    m.seg_shift = keep.ptr(seg_shift, np.uint16)
    m.nseg = int(np.asarray(seg_scale).shape[0]) if seg_scale is not None else 0
    return m


def _check(rc: int):
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")


def modulated(x, kind=MOD_NONE, eps=1e-5, nthreads=None, **mod) -> np.ndarray:
    """Unquantised y = LN(x)*(1+scale)+shift in double, shape (rows, dim)."""
    keep = _Keep()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    rows, dim = x.shape
    m = _mod(keep, kind, **mod)
    y = np.empty((rows, dim), dtype=np.float64)
    _check(lib().orc_modulated_rows(x.ctypes.data, ctypes.byref(m), eps, y.ctypes.data,
                                    rows, dim, nthreads or default_threads()))
    return y


def ln_quant_fp8(x, act_scale: float, kind=MOD_NONE, eps=1e-5, nthreads=None, **mod) -> np.ndarray:
    """e4m3 bytes (rows, dim) of the FP8 producers (K1-K4 by modulation kind)."""
    keep = _Keep()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    rows, dim = x.shape
    m = _mod(keep, kind, **mod)
    out = np.empty((rows, dim), dtype=np.uint8)
    _check(lib().orc_ln_quant_fp8(x.ctypes.data, ctypes.byref(m), act_scale, eps,
                                  out.ctypes.data, rows, dim, nthreads or default_threads()))
    return out


def ln_quant_nvfp4(x, kind=MOD_NONE, eps=1e-5, nthreads=None, swizzled=True, **mod):
    """(packed (rows, dim/2) uint8, scales) of the NVFP4 producers.

    ``swizzled=True`` returns the swizzled scale buffer of
    swizzled_sf_size(rows, dim) bytes, else the logical (rows, dim/16) matrix.
    """
    keep = _Keep()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    rows, dim = x.shape
    m = _mod(keep, kind, **mod)
    packed = np.empty((rows, dim // 2), dtype=np.uint8)
    nt = nthreads or default_threads()
    if swizzled:
        sf = np.empty(max(swizzled_sf_size(rows, dim), 0), dtype=np.uint8)
        _check(lib().orc_ln_quant_nvfp4_swizzled(x.ctypes.data, ctypes.byref(m), eps,
                                                 packed.ctypes.data, sf.ctypes.data, rows, dim, nt))
    else:
        sf = np.empty((rows, dim // 16), dtype=np.uint8)
        _check(lib().orc_ln_quant_nvfp4(x.ctypes.data, ctypes.byref(m), eps,
                                        packed.ctypes.data, sf.ctypes.data, rows, dim, nt))
    return packed, sf


def staged(x, kind=MOD_NONE, eps=1e-5, nthreads=None, **mod) -> np.ndarray:
    """bf16 bits (rows, dim) of v = bf16(fp32(y)), the NVFP4 producers' staged values."""
    keep = _Keep()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    rows, dim = x.shape
    m = _mod(keep, kind, **mod)
    v = np.empty((rows, dim), dtype=np.uint16)
    _check(lib().orc_ln_staged_bf16(x.ctypes.data, ctypes.byref(m), eps, v.ctypes.data, rows, dim,
                                    nthreads or default_threads()))
    return v


def nvfp4_2level(v, nthreads=None):
    """Two-level NVFP4 of bf16 bits v (rows, dim): (packed, swizzled scales, tensor scale)."""
    v = np.ascontiguousarray(v, dtype=np.uint16)
    rows, dim = v.shape
    packed = np.empty((rows, dim // 2), dtype=np.uint8)
    sf = np.empty(max(swizzled_sf_size(rows, dim), 0), dtype=np.uint8)
    ts = ctypes.c_float()
    _check(lib().orc_nvfp4_2level(v.ctypes.data, rows, dim, packed.ctypes.data, sf.ctypes.data, ctypes.byref(ts),
                                  nthreads or default_threads()))
    return packed, sf, ts.value


def ln_quant_nvfp4_2level(x, kind=MOD_NONE, eps=1e-5, nthreads=None, **mod):
    """LayerNorm producer with two-level NVFP4 output: (packed, swizzled scales, tensor scale)."""
    keep = _Keep()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    rows, dim = x.shape
    m = _mod(keep, kind, **mod)
    packed = np.empty((rows, dim // 2), dtype=np.uint8)
    sf = np.empty(max(swizzled_sf_size(rows, dim), 0), dtype=np.uint8)
    ts = ctypes.c_float()
    _check(lib().orc_ln_quant_nvfp4_2level(x.ctypes.data, ctypes.byref(m), eps, packed.ctypes.data, sf.ctypes.data,
                                           ctypes.byref(ts), rows, dim, nthreads or default_threads()))
    return packed, sf, ts.value


def swiglu_values(gate, up, nthreads=None) -> np.ndarray:
    """bf16 bits (rows, dim) of v = bf16(bf16(silu(gate)) * up); gate, up bf16 bits (rows, dim)."""
    gate = np.ascontiguousarray(gate, dtype=np.uint16)
    up = np.ascontiguousarray(up, dtype=np.uint16)
    rows, dim = gate.shape
    assert up.shape == gate.shape
    v = np.empty((rows, dim), dtype=np.uint16)
    _check(lib().orc_swiglu_values(gate.ctypes.data, up.ctypes.data, dim, v.ctypes.data, rows, dim,
                                   nthreads or default_threads()))
    return v


def swiglu_quant_nvfp4_2level(gate, up, nthreads=None):
    """SwiGLU producer, two-level NVFP4: (packed, swizzled scales, tensor scale)."""
    gate = np.ascontiguousarray(gate, dtype=np.uint16)
    up = np.ascontiguousarray(up, dtype=np.uint16)
    rows, dim = gate.shape
    packed = np.empty((rows, dim // 2), dtype=np.uint8)
    sf = np.empty(max(swizzled_sf_size(rows, dim), 0), dtype=np.uint8)
    ts = ctypes.c_float()
    _check(lib().orc_swiglu_quant_nvfp4_2level(gate.ctypes.data, up.ctypes.data, dim, packed.ctypes.data,
                                               sf.ctypes.data, ctypes.byref(ts), rows, dim,
                                               nthreads or default_threads()))
    return packed, sf, ts.value


def adaln_modulation6(params, modulation, nthreads=None) -> np.ndarray:
    """Six bf16 outputs as uint16 (6, batch, seq, dim) from fp32 (batch, seq, 6, dim)."""
    params = np.ascontiguousarray(params, dtype=np.float32)
    modulation = np.ascontiguousarray(modulation, dtype=np.float32)
    b, s, six, dim = params.shape
    assert six == 6 and modulation.shape == (6, dim)
    out = np.empty((6, b, s, dim), dtype=np.uint16)
    _check(lib().orc_adaln_modulation6(params.ctypes.data, modulation.ctypes.data, out.ctypes.data,
                                       b * s, dim, nthreads or default_threads()))
    return out


# --------------------------------------------------------------------------
# helpers used by the comparisons (decoding only)
# --------------------------------------------------------------------------

def e4m3_table() -> np.ndarray:
    """Decoded value of every e4m3 byte, float64[256] (NaN at 0x7F, 0xFF)."""
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


def e2m1_table() -> np.ndarray:
    """Decoded value of every e2m1 nibble, float64[16]."""
    return np.array([e2m1_decode(c) for c in range(16)], dtype=np.float64)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    """(rows, dim/2) bytes -> (rows, dim) nibble codes, low nibble first."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out
