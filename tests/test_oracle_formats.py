"""Pins of the oracle's number formats (CPU only).

Each check compares the oracle with something other than itself: torch's own
bfloat16 and float8_e4m3fn conversions, the OCP e2m1 value table, exact
rational arithmetic (fractions.Fraction), and the byte dump of the
h3-blackwell-runtime compare page (benchmarks/gb10-cute-nvfp4-conversion-
contract.json, tile-producer clamp byte).
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch


# ---------------------------------------------------------------- bf16 ----

def test_bf16_decode_all_patterns(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    L = orc.lib()
    got = np.array([L.orc_bf16_to_f64(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def test_bf16_encode_matches_torch_rne(orc):
    rng = np.random.default_rng(7)
    u = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    # ties (low half exactly 0x8000) and exact values, both parities of the kept half
    u[:2000] = (u[:2000] & 0xFFFF0000) | 0x8000
    u[2000:3000] &= 0xFFFF0000
    # the overflow band: every pattern from the largest finite bf16 up to the
    # largest binary32 (round-to-nearest overflows to infinity from the midpoint on)
    band = np.arange(0x7F7F0000, 0x7F800000, 7, dtype=np.uint64).astype(np.uint32)
    band = np.concatenate([band, np.array([0x7F7F7FFF, 0x7F7F8000, 0x7F7F8001, 0x7F7FFFFF], dtype=np.uint32)])
    u = np.concatenate([u, band, band | np.uint32(0x80000000)])
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    L = orc.lib()
    got = np.array([L.orc_bf16_from_f32(float(v)) for v in f], dtype=np.uint16)
    assert np.array_equal(got, ref)
    # the band's midpoint 0x7F7F8000 ties to the even pattern: infinity (0x7F80)
    assert L.orc_bf16_from_f32(float(np.uint32(0x7F7F8000).view(np.float32))) == 0x7F80
    assert L.orc_bf16_from_f32(float(np.uint32(0x7F7F7FFF).view(np.float32))) == 0x7F7F


# ---------------------------------------------------------------- e4m3 ----

def test_e4m3_decode_all_codes(orc):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    got = orc.e4m3_table()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert nan.sum() == 2  # 0x7F and 0xFF only
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_encode_roundtrip_every_finite_code(orc):
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert orc.e4m3_encode(orc.e4m3_decode(c)) == c


def _torch_e4m3(vals):
    t = torch.tensor(vals, dtype=torch.float64).float()
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_encode_ties_and_random_match_torch(orc):
    table = orc.e4m3_table()
    pos = table[:0x7F]                       # 0 .. 448, increasing
    mids = list((pos[:-1] + pos[1:]) / 2)    # every midpoint: ties to even
    nudged = [m * (1 + 2**-20) for m in mids] + [m * (1 - 2**-20) for m in mids]
    rng = np.random.default_rng(11)
    rand = list(rng.uniform(-464, 464, 4000)) + list(rng.standard_normal(4000) * 1e-2)
    vals = mids + [-m for m in mids] + nudged + rand + [0.0, -0.0, 464.0, -464.0, 2**-10, 2**-11]
    # torch converts through float32: feed values that are exact in float32
    vals = [float(np.float32(v)) for v in vals]
    ref = _torch_e4m3(vals)
    got = np.array([orc.e4m3_encode(v) for v in vals], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_saturates_at_clamp_byte(orc, golden_dir):
    g = json.load(open(os.path.join(golden_dir, "e4m3_block_scale_clamp.json")))
    assert orc.e4m3_decode(g["clamp_byte"]) == g["clamp_value"]
    for v in (448.0, 465.0, 500.0, 1e4, 1e30):
        assert orc.e4m3_encode(v) == g["clamp_byte"]
        assert orc.e4m3_encode(-v) == 0x80 | g["clamp_byte"]


def test_e4m3_signed_zero_and_subnormals(orc):
    assert orc.e4m3_encode(0.0) == 0x00
    assert orc.e4m3_encode(-0.0) == 0x80
    assert orc.e4m3_encode(-1e-30) == 0x80
    assert orc.e4m3_encode(2.0**-9) == 0x01           # smallest subnormal
    assert orc.e4m3_encode(2.0**-10) == 0x00          # tie with 0 -> even
    assert orc.e4m3_encode(3 * 2.0**-10) == 0x02      # tie 1|2 -> even 2
    assert orc.e4m3_encode(15 * 2.0**-10) == 0x08     # tie 7|8 -> 8 = 2^-6


# ---------------------------------------------------------------- e2m1 ----

# OCP Microscaling spec, FP4 E2M1: magnitudes of codes 0..7
E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_decode_table(orc):
    got = orc.e2m1_table()
    assert list(got[:8]) == E2M1_VALUES
    assert list(got[8:]) == [-v for v in E2M1_VALUES]
    assert np.signbit(got[8])  # code 0x8 is -0


def test_e2m1_ties_go_to_even_code(orc):
    # midpoint -> expected code (the even one of its two neighbours)
    ties = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}
    for s in (1.0, 0.5, 1.125, 448.0, 2.0**-9, 0.0703125):
        for m, code in ties.items():
            v = m * s
            assert orc.e2m1_encode(v, s) == code, (m, s)
            assert orc.e2m1_encode(-v, s) == 8 | code, (m, s)


def test_e2m1_nearest_by_exact_rationals(orc):
    rng = np.random.default_rng(3)
    scales = [orc.e4m3_decode(c) for c in range(1, 0x7F)]
    for _ in range(3000):
        s = scales[rng.integers(len(scales))]
        # bf16-representable v within a few multiples of 6*s
        v = float(torch.tensor(rng.uniform(-7.5, 7.5) * s).to(torch.bfloat16).double())
        code = orc.e2m1_encode(v, s)
        q = Fraction(v) / Fraction(s)
        dists = [abs(abs(q) - Fraction(g)) for g in E2M1_VALUES]
        best = min(dists)
        cands = [k for k, d in enumerate(dists) if d == best]
        expect = cands[0] if len(cands) == 1 else [k for k in cands if k % 2 == 0][0]
        assert code & 7 == expect, (v, s)
        assert (code >> 3) == (1 if np.signbit(v) else 0)


def test_e2m1_signed_zero_and_zero_scale(orc):
    assert orc.e2m1_encode(-0.0, 1.0) == 0x8
    assert orc.e2m1_encode(0.0, 1.0) == 0x0
    assert orc.e2m1_encode(-0.1, 1.0) == 0x8   # rounds to -0
    assert orc.e2m1_encode(-3.0, 0.0) == 0x8   # zero scale: signed zero
    assert orc.e2m1_encode(3.0, 0.0) == 0x0
    assert orc.e2m1_encode(100.0, 1.0) == 0x7  # saturates at 6
    assert orc.e2m1_encode(-100.0, 1.0) == 0xF


def test_e2m1_page_byte_dump_is_low_nibble_first(orc, golden_dir):
    g = json.load(open(os.path.join(golden_dir, "e2m1_conversion_contract.json")))
    storage = np.array(g["fp4_bytes"], dtype=np.uint8)
    b = np.array(g["expected_low_first_bytes"], dtype=np.uint8)
    assert np.array_equal(storage[: b.size], b) and not storage[b.size:].any()
    codes = orc.unpack_e2m1(b[None, :])[0]
    assert codes.size == g["padded_value_count"]
    vals = orc.e2m1_table()[codes[: g["value_count"]]]
    # a monotone sweep read low nibble first is non-decreasing, with -0 before +0
    assert np.all(np.diff(vals) >= 0)
    assert 0x8 in codes[: g["value_count"]] and 0x0 in codes[: g["value_count"]]
    first_neg0 = list(codes).index(0x8)
    first_pos0 = list(codes).index(0x0)
    assert first_neg0 < first_pos0
    # read high nibble first, the same bytes are not monotone
    swapped = np.empty_like(codes)
    swapped[0::2], swapped[1::2] = codes[1::2], codes[0::2]
    assert not np.all(np.diff(orc.e2m1_table()[swapped[: g["value_count"]]]) >= 0)
    # the padding codes are +0
    assert np.all(codes[g["value_count"]:] == 0)
    # every value of the sweep re-encodes (unit scale) to its own code
    for c in codes[: g["value_count"]]:
        assert orc.e2m1_encode(orc.e2m1_decode(int(c)), 1.0) == c
