"""GB300 (sm_103a) adaptive-LayerNorm activation producers: Python binding.

Thin ctypes binding of ``libnvfp4ap.so`` (C ABI in ``include/nvfp4ap.h``).
The functions follow the adaptive-layernorm-producers README ("Available
Functions", "Tensor Contract"): torch CUDA tensors in, outputs allocated when
``out``/``packed``/``sf_swizzled`` are None, every launch on the current CUDA
stream of the input's device.  This module only checks dtypes/shapes and
passes pointers; all arithmetic runs in the library's CUDA kernels.  If the
library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

__all__ = [
    "ada_layer_norm_quant_fp8_bf16",
    "ada_layer_norm_quant_fp8_ptok_bf16",
    "ada_layer_norm_quant_fp8_ptok_table_bf16",
    "ada_layer_norm_quant_fp8_modfp8_bf16",
    "awq_ada_layer_norm_quant_fp8_bf16",
    "layer_norm_no_affine_quant_fp8_static_bf16",
    "ada_layer_norm_quant_nvfp4_swizzled_bf16",
    "ada_layer_norm_quant_nvfp4_swizzled_modfp8_bf16",
    "ada_layer_norm_quant_fp8_seg_bf16",
    "ada_layer_norm_quant_nvfp4_swizzled_seg_bf16",
    "layer_norm_no_affine_quant_nvfp4_2level_bf16",
    "ada_layer_norm_quant_nvfp4_2level_bf16",
    "ada_layer_norm_quant_nvfp4_2level_seg_bf16",
    "swiglu_quant_nvfp4_2level_bf16",
    "swiglu_bf16",
    "workspace_2level_bytes",
    "SWIGLU_WORKSPACE_BYTES",
    "layer_norm_no_affine_quant_nvfp4_swizzled_bf16",
    "adaln_modulation6_bf16",
    "swizzled_sf_size",
    "library_path",
    "marshalling",
    "take_device_fault",
    "set_wait_limit",
    "wait_limit",
    "noalloc_progress",
    "NvFp4ApError",
    "NvFp4ApArgumentError",
]

LIB_PATH = _build.LIB

(OK, ERR_NULL, ERR_SHAPE, ERR_DIM, ERR_INDEX, ERR_ALIGN, ERR_LAUNCH, ERR_TIMEOUT, ERR_VALUE, ERR_SCRATCH,
 ERR_FAULT) = range(11)
# statuses that report a bad argument (the binding raises them as ValueError too)
_ARG_ERRORS = (ERR_NULL, ERR_SHAPE, ERR_DIM, ERR_INDEX, ERR_ALIGN, ERR_VALUE, ERR_SCRATCH)
MAX_DIM = 32768
SWIGLU_WORKSPACE_BYTES = 4  # the SwiGLU two-level producer keeps only the maximum word


def workspace_2level_bytes(rows: int) -> int:
    """Bytes of the workspace of the two-level LayerNorm producers for `rows`
    rows: the maximum word (padded to 16 bytes) and a 16-byte statistics slot
    per row (the C ABI's NVFP4AP_2LEVEL_WORKSPACE_BYTES(rows))."""
    if rows < 0:
        raise ValueError("rows must be >= 0")
    return 16 + 16 * rows


class NvFp4ApError(RuntimeError):
    """A non-zero status from the C ABI (launch, timeout and device-fault
    statuses are raised as this class)."""

    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: status {status}: {msg}")
        self.status = status


class NvFp4ApArgumentError(NvFp4ApError, ValueError):
    """A status that reports a bad argument (null pointer, shape, dim, index,
    alignment, eps, scratch size): both a NvFp4ApError and a ValueError."""


_lib = None

# the producer entry points the Python API calls: through the C marshalling
# module (_pycall, built beside the library when Python's headers are present)
# when it is there, else through ctypes; NVFP4AP_PYCALL=0 forces ctypes
_PRODUCERS = (
    "ada_layer_norm_quant_fp8_bf16", "ada_layer_norm_quant_fp8_ptok_bf16",
    "ada_layer_norm_quant_fp8_ptok_table_bf16", "ada_layer_norm_quant_fp8_modfp8_bf16",
    "awq_ada_layer_norm_quant_fp8_bf16", "ada_layer_norm_quant_fp8_seg_bf16",
    "layer_norm_no_affine_quant_fp8_static_bf16", "ada_layer_norm_quant_nvfp4_swizzled_bf16",
    "ada_layer_norm_quant_nvfp4_swizzled_modfp8_bf16", "layer_norm_no_affine_quant_nvfp4_swizzled_bf16",
    "ada_layer_norm_quant_nvfp4_swizzled_seg_bf16", "layer_norm_no_affine_quant_nvfp4_2level_bf16",
    "ada_layer_norm_quant_nvfp4_2level_bf16", "ada_layer_norm_quant_nvfp4_2level_seg_bf16",
    "swiglu_quant_nvfp4_2level_bf16", "swiglu_bf16", "adaln_modulation6_bf16",
)


class _Api:
    """The library's entry points.  Attribute lookup falls through to the
    ctypes library; the producers are replaced by the C marshalling module's
    functions of the same name when it is available (``marshalling`` says
    which: "c" or "ctypes").  adaln_modulation6_bf16 takes its six output
    pointers as any sequence of six ints on both paths."""

    def __init__(self, cdll: ctypes.CDLL, fast):
        self._cdll = cdll
        self.marshalling = "ctypes" if fast is None else "c"
        if fast is not None:
            for name in _PRODUCERS:
                setattr(self, name, getattr(fast, name))
        else:
            mod6 = cdll.adaln_modulation6_bf16

            def adaln_modulation6_bf16(params, modulation, outs, *rest):
                if not isinstance(outs, ctypes.Array):
                    outs = (ctypes.c_void_p * 6)(*outs)
                return mod6(params, modulation, outs, *rest)
            self.adaln_modulation6_bf16 = adaln_modulation6_bf16

    def __getattr__(self, name):
        return getattr(self._cdll, name)


def _fast_marshalling():
    """The bound C marshalling module, or None when it is not built (or
    NVFP4AP_PYCALL=0)."""
    if os.environ.get("NVFP4AP_PYCALL", "1") == "0":
        return None
    try:
        from . import _pycall
    except ImportError:
        return None
    _pycall.bind(LIB_PATH)
    return _pycall


def _load() -> "_Api":
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libnvfp4ap.so is not built ({LIB_PATH}); run "
                           "nvfp4_activation_producer_gb300.build.build() or __graft_entry__.build()")
    L = ctypes.CDLL(LIB_PATH)
    _declare(L)
    _lib = _Api(L, _fast_marshalling())
    return _lib


def marshalling() -> str:
    """How the producers' arguments reach the library: "c" (the C marshalling
    module) or "ctypes"."""
    return _load().marshalling


def _declare(L: ctypes.CDLL) -> None:
    """ctypes argument and result types of every C ABI entry point."""
    p, i64, f32, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int
    L.nvfp4ap_status_string.restype = ctypes.c_char_p
    L.nvfp4ap_status_string.argtypes = [i32]
    L.nvfp4ap_version.restype = i32
    L.nvfp4ap_version.argtypes = []
    L.nvfp4ap_take_device_fault.restype = i32
    L.nvfp4ap_take_device_fault.argtypes = []
    L.nvfp4ap_set_wait_limit.restype = i32
    L.nvfp4ap_set_wait_limit.argtypes = [i64]
    L.nvfp4ap_wait_limit.restype = i64
    L.nvfp4ap_wait_limit.argtypes = []
    L.nvfp4ap_noalloc_progress.restype = i32
    L.nvfp4ap_noalloc_progress.argtypes = [p, i64, ctypes.POINTER(ctypes.c_int64)]
    L.nvfp4ap_2level_single_read.restype = i32
    L.nvfp4ap_2level_single_read.argtypes = [i64, i64, i32, ctypes.POINTER(ctypes.c_int)]
    for name in ("ada_layer_norm_quant_fp8_bf16", "ada_layer_norm_quant_fp8_ptok_bf16"):
        fn = getattr(L, name)
        fn.restype = i32
        fn.argtypes = [p, p, p, p, f32, p, i64, i64, p]
    L.ada_layer_norm_quant_fp8_bf16_noalloc.restype = i32
    L.ada_layer_norm_quant_fp8_bf16_noalloc.argtypes = [p, p, p, p, f32, p, i64, i64, p]
    L.ada_layer_norm_quant_fp8_ptok_table_bf16.restype = i32
    L.ada_layer_norm_quant_fp8_ptok_table_bf16.argtypes = [p, p, p, i64, i64, i64, p, f32, p, i64, i64, p]
    L.ada_layer_norm_quant_fp8_modfp8_bf16.restype = i32
    L.ada_layer_norm_quant_fp8_modfp8_bf16.argtypes = [p, p, p, p, p, p, f32, p, i64, i64, p]
    L.awq_ada_layer_norm_quant_fp8_bf16.restype = i32
    L.awq_ada_layer_norm_quant_fp8_bf16.argtypes = [p, p, p, p, p, f32, p, i64, i64, p]
    L.ada_layer_norm_quant_nvfp4_swizzled_modfp8_bf16.restype = i32
    L.ada_layer_norm_quant_nvfp4_swizzled_modfp8_bf16.argtypes = [p, p, p, p, p, f32, p, p, i64, i64, p]
    L.ada_layer_norm_quant_fp8_seg_bf16.restype = i32
    L.ada_layer_norm_quant_fp8_seg_bf16.argtypes = [p, p, p, p, i64, p, f32, p, i64, i64, p]
    L.ada_layer_norm_quant_nvfp4_swizzled_seg_bf16.restype = i32
    L.ada_layer_norm_quant_nvfp4_swizzled_seg_bf16.argtypes = [p, p, p, p, i64, f32, p, p, i64, i64, p]
    L.layer_norm_no_affine_quant_nvfp4_2level_bf16.restype = i32
    L.layer_norm_no_affine_quant_nvfp4_2level_bf16.argtypes = [p, f32, p, p, p, p, i64, i64, p]
    L.ada_layer_norm_quant_nvfp4_2level_bf16.restype = i32
    L.ada_layer_norm_quant_nvfp4_2level_bf16.argtypes = [p, p, p, f32, p, p, p, p, i64, i64, p]
    L.ada_layer_norm_quant_nvfp4_2level_seg_bf16.restype = i32
    L.ada_layer_norm_quant_nvfp4_2level_seg_bf16.argtypes = [p, p, p, p, i64, f32, p, p, p, p, i64, i64, p]
    L.swiglu_bf16.restype = i32
    L.swiglu_bf16.argtypes = [p, p, i64, p, i64, i64, p]
    L.swiglu_quant_nvfp4_2level_bf16.restype = i32
    L.swiglu_quant_nvfp4_2level_bf16.argtypes = [p, p, i64, p, p, p, p, i64, i64, p]
    L.layer_norm_no_affine_quant_fp8_static_bf16.restype = i32
    L.layer_norm_no_affine_quant_fp8_static_bf16.argtypes = [p, p, f32, p, i64, i64, p]
    L.ada_layer_norm_quant_nvfp4_swizzled_bf16.restype = i32
    L.ada_layer_norm_quant_nvfp4_swizzled_bf16.argtypes = [p, p, p, f32, p, p, i64, i64, p]
    L.layer_norm_no_affine_quant_nvfp4_swizzled_bf16.restype = i32
    L.layer_norm_no_affine_quant_nvfp4_swizzled_bf16.argtypes = [p, f32, p, p, i64, i64, p]
    L.swizzled_sf_size.restype = i64
    L.swizzled_sf_size.argtypes = [i64, i64]
    L.nvfp4ap_2level_workspace_bytes.restype = i64
    L.nvfp4ap_2level_workspace_bytes.argtypes = [i64]
    L.adaln_modulation6_bf16.restype = i32
    L.adaln_modulation6_bf16.argtypes = [p, p, ctypes.POINTER(ctypes.c_void_p), i64, i64, i64, p]


def take_device_fault() -> None:
    """Raise NvFp4ApError if a producer kernel on the current device ran out of
    its bounded wait (status ERR_TIMEOUT) or met an out-of-range segment index
    (ERR_FAULT) since the last check (synchronises with the device)."""
    _raise("nvfp4ap_take_device_fault", _load().nvfp4ap_take_device_fault())


def set_wait_limit(cycles: int) -> None:
    """Bound of the TMA kernels' waits in SM clock cycles (<= 0: the default,
    about one second); for tests of the failure path."""
    _raise("nvfp4ap_set_wait_limit", _load().nvfp4ap_set_wait_limit(int(cycles)))


def wait_limit() -> int:
    """The bound of the TMA kernels' waits in effect, in SM clock cycles."""
    return int(_load().nvfp4ap_wait_limit())


def noalloc_progress():
    """Per-CTA progress words of the last allocation-free launch on the current
    device, as a list of ints (rows finished in bits 0-30, bit 31 if a wait
    ran out); a blocking read."""
    L = _load()
    used = ctypes.c_int64(0)
    _raise("nvfp4ap_noalloc_progress", L.nvfp4ap_noalloc_progress(None, 0, ctypes.byref(used)))
    n = used.value
    words = (ctypes.c_uint32 * max(n, 1))()
    _raise("nvfp4ap_noalloc_progress", L.nvfp4ap_noalloc_progress(words, n, ctypes.byref(used)))
    return [int(w) for w in words[:n]]


_MODULATION = {"none": 0, "broadcast": 1, "segmented": 2}


def two_level_single_read(rows: int, dim: int, modulation: str = "none") -> bool:
    """Whether the two-level LayerNorm producers read a (rows, dim) tensor from
    HBM once on the current device (one cooperative launch) rather than twice,
    with the default kernel choice; modulation: "none", "broadcast" or
    "segmented"."""
    if modulation not in _MODULATION:
        raise ValueError(f"modulation must be one of {sorted(_MODULATION)}")
    flag = ctypes.c_int(0)
    _raise("nvfp4ap_2level_single_read",
           _load().nvfp4ap_2level_single_read(int(rows), int(dim), _MODULATION[modulation], ctypes.byref(flag)))
    return bool(flag.value)


def library_path() -> str:
    _load()
    return LIB_PATH


def _raise(fn: str, rc: int):
    if rc != OK:
        msg = _load().nvfp4ap_status_string(rc).decode()
        raise (NvFp4ApArgumentError if rc in _ARG_ERRORS else NvFp4ApError)(fn, rc, msg)


# ---------------------------------------------------------------------------
# tensor-contract checks (README "Tensor Contract")
# ---------------------------------------------------------------------------

def _need(t: torch.Tensor, name: str, dtype, shape, device=None):
    # the common case in one expression; anything else takes the checks below,
    # which name what is wrong
    if (type(t) is torch.Tensor and t.dtype is dtype and (t.is_cuda if device is None else t.device == device) and
            t.shape == shape and t.is_contiguous()):
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _scalar(t: torch.Tensor, name: str, device):
    if type(t) is torch.Tensor and t.dtype is torch.float32 and t.device == device and t.numel() == 1:
        return
    if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or not t.is_cuda or t.numel() != 1:
        raise TypeError(f"{name} must be a CUDA float32 tensor with one element")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _x(x: torch.Tensor):
    if type(x) is torch.Tensor and x.dtype is torch.bfloat16 and x.is_cuda and x.dim() == 2 and x.is_contiguous():
        rows, dim = x.shape
        return rows, dim, x.device
    if not isinstance(x, torch.Tensor) or x.dim() != 2:
        raise ValueError("x must be a 2-D (rows, dim) tensor")
    _need(x, "x", torch.bfloat16, x.shape)
    return x.shape[0], x.shape[1], x.device


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(device) -> int:
    """The current CUDA stream of `device` as an integer handle (torch's raw
    accessor when present: ~0.1 us against ~2 us for the Stream object)."""
    if _raw_stream is not None and device.index is not None:
        return _raw_stream(device.index)
    return torch.cuda.current_stream(device).cuda_stream


def _ptr(t):
    return t.data_ptr() if t is not None else None


def _fp8_out(out, rows, dim, device):
    if out is None:
        return torch.empty((rows, dim), dtype=torch.float8_e4m3fn, device=device)
    _need(out, "out", torch.float8_e4m3fn, (rows, dim), device)
    return out


# ---------------------------------------------------------------------------
# FP8 producers
# ---------------------------------------------------------------------------

def ada_layer_norm_quant_fp8_bf16(x, scale, shift, act_scale, eps: float = 1e-5, out=None):
    """LayerNorm(x)*(1+scale)+shift -> e4m3fn(. / act_scale); scale/shift (dim,) bf16."""
    rows, dim, dev = _x(x)
    _need(scale, "scale", torch.bfloat16, (dim,), dev)
    _need(shift, "shift", torch.bfloat16, (dim,), dev)
    _scalar(act_scale, "act_scale", dev)
    out = _fp8_out(out, rows, dim, dev)
    rc = _load().ada_layer_norm_quant_fp8_bf16(_ptr(x), _ptr(scale), _ptr(shift), _ptr(act_scale), eps,
                                               _ptr(out), rows, dim, _stream(dev))
    _raise("ada_layer_norm_quant_fp8_bf16", rc)
    return out


def ada_layer_norm_quant_fp8_ptok_bf16(x, scale, shift, act_scale, eps: float = 1e-5, out=None):
    """Per-token form: scale/shift (rows, dim) bf16."""
    rows, dim, dev = _x(x)
    _need(scale, "scale", torch.bfloat16, (rows, dim), dev)
    _need(shift, "shift", torch.bfloat16, (rows, dim), dev)
    _scalar(act_scale, "act_scale", dev)
    out = _fp8_out(out, rows, dim, dev)
    rc = _load().ada_layer_norm_quant_fp8_ptok_bf16(_ptr(x), _ptr(scale), _ptr(shift), _ptr(act_scale), eps,
                                                    _ptr(out), rows, dim, _stream(dev))
    _raise("ada_layer_norm_quant_fp8_ptok_bf16", rc)
    return out


def ada_layer_norm_quant_fp8_ptok_table_bf16(x, temb, table, act_scale, shift_idx: int, scale_idx: int,
                                             eps: float = 1e-5, out=None):
    """Table form: scale/shift = temb[:, idx, :] + table[idx, :]; temb (rows, chunks, dim) bf16,
    table (chunks, dim) fp32."""
    rows, dim, dev = _x(x)
    if not isinstance(temb, torch.Tensor) or temb.dim() != 3:
        raise ValueError("temb must be a 3-D (rows, chunks, dim) tensor")
    chunks = temb.shape[1]
    _need(temb, "temb", torch.bfloat16, (rows, chunks, dim), dev)
    _need(table, "table", torch.float32, (chunks, dim), dev)
    _scalar(act_scale, "act_scale", dev)
    out = _fp8_out(out, rows, dim, dev)
    rc = _load().ada_layer_norm_quant_fp8_ptok_table_bf16(_ptr(x), _ptr(temb), _ptr(table), chunks,
                                                          int(shift_idx), int(scale_idx), _ptr(act_scale),
                                                          eps, _ptr(out), rows, dim, _stream(dev))
    _raise("ada_layer_norm_quant_fp8_ptok_table_bf16", rc)
    return out


def ada_layer_norm_quant_fp8_modfp8_bf16(x, scale_fp8, shift_fp8, scale_deq, shift_deq, act_scale,
                                         eps: float = 1e-5, out=None):
    """Broadcast form with e4m3 (dim,) scale/shift, each times its fp32 scalar:
    scale = scale_fp8 * scale_deq, shift = shift_fp8 * shift_deq."""
    rows, dim, dev = _x(x)
    _need(scale_fp8, "scale_fp8", torch.float8_e4m3fn, (dim,), dev)
    _need(shift_fp8, "shift_fp8", torch.float8_e4m3fn, (dim,), dev)
    _scalar(scale_deq, "scale_deq", dev)
    _scalar(shift_deq, "shift_deq", dev)
    _scalar(act_scale, "act_scale", dev)
    out = _fp8_out(out, rows, dim, dev)
    rc = _load().ada_layer_norm_quant_fp8_modfp8_bf16(_ptr(x), _ptr(scale_fp8), _ptr(shift_fp8), _ptr(scale_deq),
                                                      _ptr(shift_deq), _ptr(act_scale), eps, _ptr(out), rows, dim,
                                                      _stream(dev))
    _raise("ada_layer_norm_quant_fp8_modfp8_bf16", rc)
    return out


def awq_ada_layer_norm_quant_fp8_bf16(x, scale, shift, inv_s, act_scale, eps: float = 1e-5, out=None):
    """Broadcast form with a bf16 (dim,) AWQ smoothing vector:
    e4m3fn((LayerNorm(x)*(1+scale)+shift) * inv_s / act_scale)."""
    rows, dim, dev = _x(x)
    _need(scale, "scale", torch.bfloat16, (dim,), dev)
    _need(shift, "shift", torch.bfloat16, (dim,), dev)
    _need(inv_s, "inv_s", torch.bfloat16, (dim,), dev)
    _scalar(act_scale, "act_scale", dev)
    out = _fp8_out(out, rows, dim, dev)
    rc = _load().awq_ada_layer_norm_quant_fp8_bf16(_ptr(x), _ptr(scale), _ptr(shift), _ptr(inv_s),
                                                   _ptr(act_scale), eps, _ptr(out), rows, dim, _stream(dev))
    _raise("awq_ada_layer_norm_quant_fp8_bf16", rc)
    return out


def layer_norm_no_affine_quant_fp8_static_bf16(x, act_scale, eps: float = 1e-5, out=None):
    """LayerNorm(x) (no affine) -> e4m3fn(. / act_scale)."""
    rows, dim, dev = _x(x)
    _scalar(act_scale, "act_scale", dev)
    out = _fp8_out(out, rows, dim, dev)
    rc = _load().layer_norm_no_affine_quant_fp8_static_bf16(_ptr(x), _ptr(act_scale), eps, _ptr(out), rows,
                                                            dim, _stream(dev))
    _raise("layer_norm_no_affine_quant_fp8_static_bf16", rc)
    return out


# ---------------------------------------------------------------------------
# NVFP4 producers
# ---------------------------------------------------------------------------

def swizzled_sf_size(rows: int, dim: int) -> int:
    """Bytes of the 128x4-swizzled e4m3 scale buffer for a (rows, dim) activation."""
    n = int(_load().swizzled_sf_size(int(rows), int(dim)))
    if n < 0:
        raise ValueError(f"swizzled_sf_size: invalid rows={rows}, dim={dim} (dim must be a positive multiple of 16)")
    return n


def _nvfp4_outs(packed, sf, rows, dim, dev):
    if dim % 16 != 0:
        raise ValueError("dim must be divisible by 16 for NVFP4 outputs")
    if packed is None:
        packed = torch.empty((rows, dim // 2), dtype=torch.uint8, device=dev)
    else:
        _need(packed, "packed", torch.uint8, (rows, dim // 2), dev)
    n = swizzled_sf_size(rows, dim)
    if sf is None:
        sf = torch.empty((n,), dtype=torch.uint8, device=dev)
    else:
        if not isinstance(sf, torch.Tensor) or sf.dtype != torch.uint8 or not sf.is_cuda:
            raise TypeError("sf_swizzled must be a CUDA uint8 tensor")
        if sf.device != dev or not sf.is_contiguous() or sf.numel() != n:
            raise ValueError(f"sf_swizzled must be a contiguous uint8 tensor of swizzled_sf_size = {n} elements")
    return packed, sf


def ada_layer_norm_quant_nvfp4_swizzled_bf16(x, scale, shift, eps: float = 1e-5, packed=None, sf_swizzled=None):
    """LayerNorm(x)*(1+scale)+shift -> NVFP4 (packed e2m1, 128x4-swizzled e4m3 block scales)."""
    rows, dim, dev = _x(x)
    _need(scale, "scale", torch.bfloat16, (dim,), dev)
    _need(shift, "shift", torch.bfloat16, (dim,), dev)
    packed, sf_swizzled = _nvfp4_outs(packed, sf_swizzled, rows, dim, dev)
    rc = _load().ada_layer_norm_quant_nvfp4_swizzled_bf16(_ptr(x), _ptr(scale), _ptr(shift), eps, _ptr(packed),
                                                          _ptr(sf_swizzled), rows, dim, _stream(dev))
    _raise("ada_layer_norm_quant_nvfp4_swizzled_bf16", rc)
    return packed, sf_swizzled


def ada_layer_norm_quant_nvfp4_swizzled_modfp8_bf16(x, scale_fp8, shift_fp8, scale_deq, shift_deq,
                                                    eps: float = 1e-5, packed=None, sf_swizzled=None):
    """NVFP4 broadcast form with e4m3 (dim,) scale/shift times fp32 scalars."""
    rows, dim, dev = _x(x)
    _need(scale_fp8, "scale_fp8", torch.float8_e4m3fn, (dim,), dev)
    _need(shift_fp8, "shift_fp8", torch.float8_e4m3fn, (dim,), dev)
    _scalar(scale_deq, "scale_deq", dev)
    _scalar(shift_deq, "shift_deq", dev)
    packed, sf_swizzled = _nvfp4_outs(packed, sf_swizzled, rows, dim, dev)
    rc = _load().ada_layer_norm_quant_nvfp4_swizzled_modfp8_bf16(_ptr(x), _ptr(scale_fp8), _ptr(shift_fp8),
                                                                 _ptr(scale_deq), _ptr(shift_deq), eps,
                                                                 _ptr(packed), _ptr(sf_swizzled), rows, dim,
                                                                 _stream(dev))
    _raise("ada_layer_norm_quant_nvfp4_swizzled_modfp8_bf16", rc)
    return packed, sf_swizzled


def layer_norm_no_affine_quant_nvfp4_swizzled_bf16(x, eps: float = 1e-5, packed=None, sf_swizzled=None):
    """LayerNorm(x) (no affine) -> NVFP4."""
    rows, dim, dev = _x(x)
    packed, sf_swizzled = _nvfp4_outs(packed, sf_swizzled, rows, dim, dev)
    rc = _load().layer_norm_no_affine_quant_nvfp4_swizzled_bf16(_ptr(x), eps, _ptr(packed), _ptr(sf_swizzled),
                                                                rows, dim, _stream(dev))
    _raise("layer_norm_no_affine_quant_nvfp4_swizzled_bf16", rc)
    return packed, sf_swizzled


# ---------------------------------------------------------------------------
# segmented modulation and two-level NVFP4
# ---------------------------------------------------------------------------

def _seg(seg_idx, seg_scale, seg_shift, rows, dim, dev):
    if not isinstance(seg_scale, torch.Tensor) or seg_scale.dim() != 2:
        raise ValueError("seg_scale must be a 2-D (nseg, dim) tensor")
    nseg = seg_scale.shape[0]
    _need(seg_idx, "seg_idx", torch.int32, (rows,), dev)
    _need(seg_scale, "seg_scale", torch.bfloat16, (nseg, dim), dev)
    _need(seg_shift, "seg_shift", torch.bfloat16, (nseg, dim), dev)
    return nseg


def ada_layer_norm_quant_fp8_seg_bf16(x, seg_idx, seg_scale, seg_shift, act_scale, eps: float = 1e-5, out=None):
    """Segmented modulation: row r uses row seg_idx[r] of the (nseg, dim) bf16 scale/shift tables."""
    rows, dim, dev = _x(x)
    nseg = _seg(seg_idx, seg_scale, seg_shift, rows, dim, dev)
    _scalar(act_scale, "act_scale", dev)
    out = _fp8_out(out, rows, dim, dev)
    rc = _load().ada_layer_norm_quant_fp8_seg_bf16(_ptr(x), _ptr(seg_idx), _ptr(seg_scale), _ptr(seg_shift), nseg,
                                                   _ptr(act_scale), eps, _ptr(out), rows, dim, _stream(dev))
    _raise("ada_layer_norm_quant_fp8_seg_bf16", rc)
    return out


def ada_layer_norm_quant_nvfp4_swizzled_seg_bf16(x, seg_idx, seg_scale, seg_shift, eps: float = 1e-5, packed=None,
                                                 sf_swizzled=None):
    """Single-level NVFP4 with segmented modulation."""
    rows, dim, dev = _x(x)
    nseg = _seg(seg_idx, seg_scale, seg_shift, rows, dim, dev)
    packed, sf_swizzled = _nvfp4_outs(packed, sf_swizzled, rows, dim, dev)
    rc = _load().ada_layer_norm_quant_nvfp4_swizzled_seg_bf16(_ptr(x), _ptr(seg_idx), _ptr(seg_scale),
                                                              _ptr(seg_shift), nseg, eps, _ptr(packed),
                                                              _ptr(sf_swizzled), rows, dim, _stream(dev))
    _raise("ada_layer_norm_quant_nvfp4_swizzled_seg_bf16", rc)
    return packed, sf_swizzled


def _twolevel_extra(tensor_scale, workspace, dev, need: int):
    """tensor_scale (1,) fp32 and a workspace of at least `need` bytes,
    16-byte aligned; allocated when None."""
    if tensor_scale is None:
        tensor_scale = torch.empty((1,), dtype=torch.float32, device=dev)
    else:
        _scalar(tensor_scale, "tensor_scale", dev)
    if workspace is None:
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    elif (not isinstance(workspace, torch.Tensor) or not workspace.is_cuda or workspace.device != dev or
          not workspace.is_contiguous() or workspace.numel() * workspace.element_size() < need):
        raise ValueError(f"workspace must be a contiguous CUDA tensor of at least {need} bytes on {dev}")
    return tensor_scale, workspace


def layer_norm_no_affine_quant_nvfp4_2level_bf16(x, eps: float = 1e-5, packed=None, sf_swizzled=None,
                                                 tensor_scale=None, workspace=None):
    """LayerNorm (no affine) -> two-level NVFP4: (packed, sf_swizzled, tensor_scale)."""
    rows, dim, dev = _x(x)
    packed, sf_swizzled = _nvfp4_outs(packed, sf_swizzled, rows, dim, dev)
    tensor_scale, workspace = _twolevel_extra(tensor_scale, workspace, dev, workspace_2level_bytes(rows))
    rc = _load().layer_norm_no_affine_quant_nvfp4_2level_bf16(_ptr(x), eps, _ptr(packed), _ptr(sf_swizzled),
                                                              _ptr(tensor_scale), _ptr(workspace), rows, dim,
                                                              _stream(dev))
    _raise("layer_norm_no_affine_quant_nvfp4_2level_bf16", rc)
    return packed, sf_swizzled, tensor_scale


def ada_layer_norm_quant_nvfp4_2level_bf16(x, scale, shift, eps: float = 1e-5, packed=None, sf_swizzled=None,
                                           tensor_scale=None, workspace=None):
    """Broadcast modulation -> two-level NVFP4: (packed, sf_swizzled, tensor_scale)."""
    rows, dim, dev = _x(x)
    _need(scale, "scale", torch.bfloat16, (dim,), dev)
    _need(shift, "shift", torch.bfloat16, (dim,), dev)
    packed, sf_swizzled = _nvfp4_outs(packed, sf_swizzled, rows, dim, dev)
    tensor_scale, workspace = _twolevel_extra(tensor_scale, workspace, dev, workspace_2level_bytes(rows))
    rc = _load().ada_layer_norm_quant_nvfp4_2level_bf16(_ptr(x), _ptr(scale), _ptr(shift), eps, _ptr(packed),
                                                        _ptr(sf_swizzled), _ptr(tensor_scale), _ptr(workspace),
                                                        rows, dim, _stream(dev))
    _raise("ada_layer_norm_quant_nvfp4_2level_bf16", rc)
    return packed, sf_swizzled, tensor_scale


def ada_layer_norm_quant_nvfp4_2level_seg_bf16(x, seg_idx, seg_scale, seg_shift, eps: float = 1e-5, packed=None,
                                               sf_swizzled=None, tensor_scale=None, workspace=None):
    """Segmented modulation -> two-level NVFP4: (packed, sf_swizzled, tensor_scale)."""
    rows, dim, dev = _x(x)
    nseg = _seg(seg_idx, seg_scale, seg_shift, rows, dim, dev)
    packed, sf_swizzled = _nvfp4_outs(packed, sf_swizzled, rows, dim, dev)
    tensor_scale, workspace = _twolevel_extra(tensor_scale, workspace, dev, workspace_2level_bytes(rows))
    rc = _load().ada_layer_norm_quant_nvfp4_2level_seg_bf16(_ptr(x), _ptr(seg_idx), _ptr(seg_scale),
                                                            _ptr(seg_shift), nseg, eps, _ptr(packed),
                                                            _ptr(sf_swizzled), _ptr(tensor_scale), _ptr(workspace),
                                                            rows, dim, _stream(dev))
    _raise("ada_layer_norm_quant_nvfp4_2level_seg_bf16", rc)
    return packed, sf_swizzled, tensor_scale


def _gate_up(gate, up):
    for name, t in (("gate", gate), ("up", up)):
        if not isinstance(t, torch.Tensor) or t.dim() != 2 or t.dtype != torch.bfloat16 or not t.is_cuda:
            raise TypeError(f"{name} must be a 2-D CUDA bfloat16 tensor")
    if gate.shape != up.shape or gate.device != up.device:
        raise ValueError("gate and up must have the same shape and device")
    rows, dim = gate.shape
    if gate.stride(1) != 1 or up.stride(1) != 1 or gate.stride(0) != up.stride(0):
        raise ValueError("gate and up must have unit column stride and the same row stride")
    return rows, dim, (gate.stride(0) if rows > 1 else dim), gate.device


def swiglu_bf16(gate, up, out=None):
    """bf16(bf16(silu(gate)) * up), (rows, dim) bf16 (the materialised SwiGLU values)."""
    rows, dim, ld, dev = _gate_up(gate, up)
    if out is None:
        out = torch.empty((rows, dim), dtype=torch.bfloat16, device=dev)
    else:
        _need(out, "out", torch.bfloat16, (rows, dim), dev)
    rc = _load().swiglu_bf16(_ptr(gate), _ptr(up), ld, _ptr(out), rows, dim, _stream(dev))
    _raise("swiglu_bf16", rc)
    return out


def swiglu_quant_nvfp4_2level_bf16(gate, up, packed=None, sf_swizzled=None, tensor_scale=None, workspace=None):
    """bf16(bf16(silu(gate)) * up) -> two-level NVFP4: (packed, sf_swizzled, tensor_scale).

    gate and up are (rows, dim) bf16 views with the same row stride: two
    contiguous tensors, or the two halves x[:, :dim], x[:, dim:] of one
    contiguous (rows, 2*dim) tensor."""
    rows, dim, ld, dev = _gate_up(gate, up)
    packed, sf_swizzled = _nvfp4_outs(packed, sf_swizzled, rows, dim, dev)
    tensor_scale, workspace = _twolevel_extra(tensor_scale, workspace, dev, SWIGLU_WORKSPACE_BYTES)
    rc = _load().swiglu_quant_nvfp4_2level_bf16(_ptr(gate), _ptr(up), ld, _ptr(packed), _ptr(sf_swizzled),
                                                _ptr(tensor_scale), _ptr(workspace), rows, dim, _stream(dev))
    _raise("swiglu_quant_nvfp4_2level_bf16", rc)
    return packed, sf_swizzled, tensor_scale


# ---------------------------------------------------------------------------
# six-way modulation
# ---------------------------------------------------------------------------

def adaln_modulation6_bf16(adaln_params, layer_modulation, out=None):
    """Six bf16 (batch, seq, dim) tensors from fp32 (batch, seq, 6, dim) params + (6, dim) modulation.

    ``out`` may be a (6, batch, seq, dim) bf16 tensor or a sequence of six
    (batch, seq, dim) bf16 tensors; the result is a tuple of six tensors.
    """
    p = adaln_params
    if not isinstance(p, torch.Tensor) or p.dim() != 4 or p.shape[2] != 6:
        raise ValueError("adaln_params must be a (batch, seq, 6, dim) tensor")
    b, s, _, dim = p.shape
    dev = p.device
    _need(p, "adaln_params", torch.float32, (b, s, 6, dim), dev)
    _need(layer_modulation, "layer_modulation", torch.float32, (6, dim), dev)
    if out is None:
        buf = torch.empty((6, b, s, dim), dtype=torch.bfloat16, device=dev)
        outs = tuple(buf[i] for i in range(6))
    elif isinstance(out, torch.Tensor):
        _need(out, "out", torch.bfloat16, (6, b, s, dim), dev)
        outs = tuple(out[i] for i in range(6))
    else:
        outs = tuple(out)
        if len(outs) != 6:
            raise ValueError("out must hold six tensors")
        for i, o in enumerate(outs):
            _need(o, f"out[{i}]", torch.bfloat16, (b, s, dim), dev)
    ptrs = tuple(o.data_ptr() for o in outs)
    rc = _load().adaln_modulation6_bf16(_ptr(p), _ptr(layer_modulation), ptrs, b, s, dim, _stream(dev))
    _raise("adaln_modulation6_bf16", rc)
    return outs
