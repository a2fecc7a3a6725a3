"""Comparison of the CUDA path's outputs with the oracle's (used by the gpu tests).

Acceptance, per producer output (the tolerance is stated here and used by every
parity test):
  - FP8 / NVFP4 codes: at least CODE_MATCH_MIN of the elements equal, and every
    mismatch exactly one step in the ordered code index (magnitude +-1 with the
    same sign, or +0 <-> -0 / +-0 <-> the smallest magnitude).
  - per row: at most ROW_MISMATCH_FRAC of the row's codes (and never fewer
    than ROW_MISMATCH_MIN) differ, so one row whose every code is one step off
    fails even where it is a small part of a large tensor.
  - dequantised output: ||deq_gpu - deq_orc||_2 / ||deq_orc||_2 over the whole
    output tensor below DEQ_REL_MAX ("max relative error" is read as the largest
    of these over every compared output; a row-wise ratio cannot be the bound
    everywhere, since on short rows one permitted one-step mismatch alone
    exceeds 1e-2).  Row-wise the same bound is asserted where it is
    meaningful: FP8 rows of at least ROW_REL_MIN_DIM elements with at most one
    mismatch (one e4m3 step of a value within four standard deviations of the
    row is below 1e-2 of such a row's norm).  The largest row-wise ratio is
    reported for every output.
  - NVFP4 block-scale bytes: equal, except for blocks whose oracle amax lies
    within one bf16 ulp of an e4m3 rounding boundary of amax/6 (there the fp32
    and fp64 routes to the staged bf16 value may differ by one ulp); the
    padding of the swizzled buffer is all zero.
  - six-way modulation: bit-exact.
"""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle

CODE_MATCH_MIN = 0.999
MAX_STEP = 1
DEQ_REL_MAX = 1e-2
ROW_MISMATCH_FRAC = 0.01
ROW_MISMATCH_MIN = 2
ROW_REL_MIN_DIM = 2048

_E4M3 = None
_E2M1 = None


def e4m3_table():
    global _E4M3
    if _E4M3 is None:
        _E4M3 = oracle.e4m3_table()
    return _E4M3


def e2m1_table():
    global _E2M1
    if _E2M1 is None:
        _E2M1 = oracle.e2m1_table()
    return _E2M1


def _ordinal(codes: np.ndarray, sign_bit: int) -> np.ndarray:
    c = codes.astype(np.int64)
    mag = c & (sign_bit - 1)
    return np.where(c & sign_bit, -mag, mag)


def _row_rel(deq_g: np.ndarray, deq_o: np.ndarray) -> float:
    num = np.sqrt(((deq_g - deq_o) ** 2).sum(axis=1))
    den = np.sqrt((deq_o ** 2).sum(axis=1))
    zero = den == 0
    assert np.all(num[zero] == 0), "rows with an all-zero oracle output differ"
    if (~zero).any():
        return float((num[~zero] / den[~zero]).max())
    return 0.0


def _tensor_rel(deq_g: np.ndarray, deq_o: np.ndarray) -> float:
    num = float(np.sqrt(((deq_g - deq_o) ** 2).sum()))
    den = float(np.sqrt((deq_o ** 2).sum()))
    if den == 0.0:
        assert num == 0.0, "an all-zero oracle output differs"
        return 0.0
    return num / den


def check_codes(gpu: np.ndarray, orc: np.ndarray, sign_bit: int, what: str) -> dict:
    assert gpu.shape == orc.shape, (gpu.shape, orc.shape)
    eq = gpu == orc
    frac = float(eq.mean()) if eq.size else 1.0
    step = np.abs(_ordinal(gpu, sign_bit) - _ordinal(orc, sign_bit))
    bad = (~eq) & (step > MAX_STEP)
    assert not bad.any(), f"{what}: {int(bad.sum())} codes more than {MAX_STEP} step off, first at {np.argwhere(bad)[:5].tolist()}"
    assert frac >= CODE_MATCH_MIN, f"{what}: only {frac:.6f} of codes equal"
    if gpu.ndim == 2 and gpu.size:
        per_row = (~eq).sum(axis=1)
        cap = max(ROW_MISMATCH_MIN, int(np.ceil(ROW_MISMATCH_FRAC * gpu.shape[1])))
        worst = int(per_row.max())
        assert worst <= cap, f"{what}: row {int(per_row.argmax())} has {worst} mismatched codes (cap {cap})"
    return {"equal_frac": frac, "mismatches": int((~eq).sum())}


def _row_rel_all(deq_g: np.ndarray, deq_o: np.ndarray) -> np.ndarray:
    num = np.sqrt(((deq_g - deq_o) ** 2).sum(axis=1))
    den = np.sqrt((deq_o ** 2).sum(axis=1))
    return np.where(den > 0, num / np.where(den > 0, den, 1.0), 0.0)


def check_fp8(gpu_codes: np.ndarray, orc_codes: np.ndarray, act_scale: float, what: str = "fp8") -> dict:
    st = check_codes(gpu_codes, orc_codes, 0x80, what)
    t = e4m3_table()
    dg, do = t[gpu_codes].astype(np.float64) * act_scale, t[orc_codes].astype(np.float64) * act_scale
    rel = _tensor_rel(dg, do)
    assert rel < DEQ_REL_MAX, f"{what}: relative error {rel}"
    st["rel_err"] = rel
    st["row_rel_err_max"] = _row_rel(dg, do)
    if gpu_codes.ndim == 2 and gpu_codes.shape[1] >= ROW_REL_MIN_DIM:
        rows_ok = (gpu_codes != orc_codes).sum(axis=1) <= 1
        rr = _row_rel_all(dg, do)[rows_ok]
        assert rr.size == 0 or rr.max() < DEQ_REL_MAX, f"{what}: row-wise relative error {rr.max()}"
    return st


def unswizzle(sf: np.ndarray, rows: int, dim: int) -> np.ndarray:
    """Logical (rows, dim/16) scales read from a swizzled buffer via the oracle's offsets."""
    return sf[_offsets(rows, dim)].reshape(rows, dim // 16)


@functools.lru_cache(maxsize=64)
def _offsets(rows: int, dim: int) -> np.ndarray:
    # the oracle's layout, expanded once per (rows, dim) through its swizzler:
    # swizzle an index matrix and invert the permutation
    nblk = dim // 16
    n = rows * nblk
    size = oracle.swizzled_sf_size(rows, dim)
    if n == 0:
        return np.zeros(0, dtype=np.int64)
    # encode each logical index (plus one) in four byte planes
    idx = np.arange(n, dtype=np.int64) + 1
    off = np.zeros(size, dtype=np.int64)
    for plane in range(4):
        b = ((idx >> (8 * plane)) & 0xFF).astype(np.uint8).reshape(rows, nblk)
        off |= oracle.swizzle_scales(b, rows, dim).astype(np.int64) << (8 * plane)
    pos = np.full(n, -1, dtype=np.int64)
    nz = np.nonzero(off)[0]
    pos[off[nz] - 1] = nz
    assert (pos >= 0).all()
    return pos


def padding_mask(rows: int, dim: int) -> np.ndarray:
    size = oracle.swizzled_sf_size(rows, dim)
    m = np.ones(size, dtype=bool)
    m[_offsets(rows, dim)] = False
    return m


def _bf16_neighbours(a: np.ndarray):
    b = torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().astype(np.int64)
    lo = (b - 1).astype(np.int16)
    hi = (b + 1).astype(np.int16)
    f = lambda x: torch.from_numpy(x).view(torch.bfloat16).double().numpy()
    return np.abs(f(lo)), np.abs(f(hi))


def check_nvfp4(gpu_packed: np.ndarray, gpu_sf: np.ndarray, orc_packed: np.ndarray, orc_sf: np.ndarray,
                rows: int, dim: int, v_orc: np.ndarray | None = None, what: str = "nvfp4",
                ts: float | None = None) -> dict:
    """Compare packed codes and the swizzled scale buffer.  v_orc: the oracle's
    staged bf16 values (rows, dim) as float64, used to explain scale mismatches.
    ts: the tensor scale of the two-level contract (block scale
    e4m3(min(fp32(fp32(amax / 6) / ts), 448))), None for single level."""
    nblk = dim // 16
    gcodes, ocodes = oracle.unpack_e2m1(gpu_packed), oracle.unpack_e2m1(orc_packed)
    st = check_codes(gcodes, ocodes, 0x8, what + " codes")
    # padding
    pad = padding_mask(rows, dim)
    assert not gpu_sf[pad].any(), f"{what}: non-zero padding bytes in the swizzled scales"
    gs, os_ = unswizzle(gpu_sf, rows, dim), unswizzle(orc_sf, rows, dim)
    diff = gs != os_
    st["scale_mismatches"] = int(diff.sum())
    if diff.any():
        assert v_orc is not None, f"{what}: {int(diff.sum())} scale bytes differ"
        amax = np.abs(v_orc).reshape(rows, nblk, 16).max(axis=2)
        lo, hi = _bf16_neighbours(amax)
        if ts is None:
            enc = lambda a: torch.from_numpy((a / 6).astype(np.float32)).clamp(max=448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        else:
            def enc(a):
                q = ((a.astype(np.float32) / np.float32(6.0)).astype(np.float32) / np.float32(ts)).astype(np.float32)
                q = np.where(np.isnan(q), np.float32(448.0), np.minimum(q, np.float32(448.0)))
                return torch.from_numpy(q.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        ok = (gs == enc(lo)) | (gs == enc(hi))
        bad = diff & ~ok
        assert not bad.any(), f"{what}: scale bytes differ without an amax explanation at {np.argwhere(bad)[:5].tolist()}"
    e2, e4 = e2m1_table(), e4m3_table()
    deq_g = e2[gcodes].reshape(rows, nblk, 16) * e4[gs][..., None]
    deq_o = e2[ocodes].reshape(rows, nblk, 16) * e4[os_][..., None]
    rel = _tensor_rel(deq_g, deq_o)
    assert rel < DEQ_REL_MAX, f"{what}: relative error {rel}"
    st["rel_err"] = rel
    st["row_rel_err_max"] = _row_rel(deq_g.reshape(rows, dim), deq_o.reshape(rows, dim))
    return st
