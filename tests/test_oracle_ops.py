"""Pins of the oracle's producers (CPU only).

Library routines: torch.nn.functional.layer_norm in float64 (LayerNorm
without affine), numpy float32 addition and torch's bf16 conversion (six-way).
Closed forms: a constant row normalises to 0; an alternating +-a row to
+-a/sqrt(a^2+eps); with eps = 0 LayerNorm is invariant to power-of-two
scaling.  Special cases from the README ("Minimal Usage"): zero scale/shift is
plain LayerNorm; the table form equals the per-token form on temb + table.
Properties: every FP8 code is the nearest e4m3 value of y/act_scale; every
NVFP4 block scale bounds its block and every code is nearest.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import synth


def _u16(a):
    return synth.u16(synth.bf16(a))


def _f64(bits):
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double()


# ------------------------------------------------------------ statistics --

def test_layer_norm_matches_torch_float64(orc):
    rng = np.random.default_rng(0)
    for rows, dim, eps in [(7, 48, 1e-5), (33, 3072, 1e-5), (5, 2050, 1e-6)]:
        a = rng.standard_normal((rows, dim)).astype(np.float32) * 3 + 0.5
        x = _u16(a)
        y = orc.modulated(x, orc.MOD_NONE, eps=eps)
        ref = F.layer_norm(_f64(x), (dim,), eps=float(np.float32(eps))).numpy()
        np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_constant_row_normalises_to_zero(orc):
    x = _u16(np.full((3, 64), 1.75, dtype=np.float32))
    y = orc.modulated(x, orc.MOD_NONE)
    assert np.all(y == 0.0)
    mean, rstd = orc.row_stats(x[0], 1e-5)
    assert mean == 1.75 and rstd == 1.0 / np.sqrt(np.float64(np.float32(1e-5)))


def test_alternating_row_closed_form(orc):
    for a in (0.5, 3.0, 1e-3):
        row = np.array([a, -a] * 32, dtype=np.float32)
        x = _u16(row[None, :])
        eps = np.float32(1e-5)
        av = float(_f64(x)[0, 0])
        y = orc.modulated(x, orc.MOD_NONE, eps=float(eps))[0]
        expect = av / np.sqrt(av * av + np.float64(eps))
        np.testing.assert_allclose(y[0::2], expect, rtol=1e-14)
        np.testing.assert_allclose(y[1::2], -expect, rtol=1e-14)


def test_power_of_two_invariance_eps0(orc):
    rng = np.random.default_rng(1)
    a = rng.standard_normal((4, 512)).astype(np.float32)
    x = _u16(a)
    y = orc.modulated(x, orc.MOD_NONE, eps=0.0)
    for k in (3, -5, 8):
        xk = _u16(_f64(x).numpy().astype(np.float32) * np.float32(2.0**k))
        yk = orc.modulated(xk, orc.MOD_NONE, eps=0.0)
        assert np.array_equal(y, yk)


# ------------------------------------------------------------ modulation --

def test_modulation_forms_match_torch(orc):
    w = synth.fp8_table(9, 96, seed=5)
    x = synth.u16(w.inputs["x"])
    temb = synth.u16(w.inputs["temb"])
    table = w.inputs["table"].numpy()
    si, ci = w.params["shift_idx"], w.params["scale_idx"]
    ln = F.layer_norm(_f64(x), (96,), eps=float(np.float32(1e-5))).numpy()
    # broadcast
    sc, sh = _u16(np.linspace(-0.3, 0.3, 96, dtype=np.float32)), _u16(np.linspace(0.2, -0.1, 96, dtype=np.float32))
    y = orc.modulated(x, orc.MOD_BCAST, scale=sc, shift=sh)
    np.testing.assert_allclose(y, ln * (1 + _f64(sc).numpy()) + _f64(sh).numpy(), rtol=1e-12, atol=1e-12)
    # per token
    sc2, sh2 = temb[:, 3], temb[:, 4]
    y = orc.modulated(x, orc.MOD_PTOK, scale=sc2, shift=sh2)
    np.testing.assert_allclose(y, ln * (1 + _f64(sc2).numpy()) + _f64(sh2).numpy(), rtol=1e-12, atol=1e-12)
    # table
    y = orc.modulated(x, orc.MOD_TABLE, temb=temb, table=table, shift_idx=si, scale_idx=ci)
    scale = _f64(temb[:, ci]).numpy() + table[ci].astype(np.float64)
    shift = _f64(temb[:, si]).numpy() + table[si].astype(np.float64)
    np.testing.assert_allclose(y, ln * (1 + scale) + shift, rtol=1e-12, atol=1e-12)


def test_zero_modulation_is_plain_layer_norm(orc):
    w = synth.fp8_broadcast(17, 256, seed=9)
    x = synth.u16(w.inputs["x"])
    z = np.zeros(256, dtype=np.uint16)
    a = orc.ln_quant_fp8(x, 0.025, orc.MOD_BCAST, scale=z, shift=z)
    b = orc.ln_quant_fp8(x, 0.025, orc.MOD_NONE)
    assert np.array_equal(a, b)
    zp = np.zeros((17, 256), dtype=np.uint16)
    c = orc.ln_quant_fp8(x, 0.025, orc.MOD_PTOK, scale=zp, shift=zp)
    assert np.array_equal(a, c)
    pa, sa = orc.ln_quant_nvfp4(x, orc.MOD_BCAST, scale=z, shift=z)
    pb, sb = orc.ln_quant_nvfp4(x, orc.MOD_NONE)
    assert np.array_equal(pa, pb) and np.array_equal(sa, sb)


def test_broadcast_equals_per_token_with_repeated_rows(orc):
    w = synth.fp8_broadcast(11, 160, seed=4)
    x, sc, sh = (synth.u16(w.inputs[k]) for k in ("x", "scale", "shift"))
    a = orc.ln_quant_fp8(x, 0.025, orc.MOD_BCAST, scale=sc, shift=sh)
    b = orc.ln_quant_fp8(x, 0.025, orc.MOD_PTOK, scale=np.tile(sc, (11, 1)), shift=np.tile(sh, (11, 1)))
    assert np.array_equal(a, b)


def test_table_form_equals_per_token_on_sum(orc):
    rows, chunks, dim = 13, 6, 128
    rng = np.random.default_rng(2)
    x = _u16(rng.standard_normal((rows, dim)).astype(np.float32))
    # multiples of 2^-6 in [-1, 1]: temb + table is exact in bf16
    temb_f = (rng.integers(-64, 65, (rows, chunks, dim)) / 64.0).astype(np.float32)
    table = (rng.integers(-64, 65, (chunks, dim)) / 64.0).astype(np.float32)
    temb = _u16(temb_f)
    si, ci = 2, 5
    a = orc.ln_quant_fp8(x, 0.025, orc.MOD_TABLE, temb=temb, table=table, shift_idx=si, scale_idx=ci)
    s_sum = _u16(temb_f[:, ci] + table[ci])
    h_sum = _u16(temb_f[:, si] + table[si])
    assert np.array_equal(synth.u16(synth.bf16(temb_f[:, ci] + table[ci])), s_sum)
    b = orc.ln_quant_fp8(x, 0.025, orc.MOD_PTOK, scale=s_sum, shift=h_sum)
    assert np.array_equal(a, b)
    # table = 0 reduces to the per-token form on the temb chunks
    c = orc.ln_quant_fp8(x, 0.025, orc.MOD_TABLE, temb=temb, table=np.zeros_like(table),
                         shift_idx=si, scale_idx=ci)
    d = orc.ln_quant_fp8(x, 0.025, orc.MOD_PTOK, scale=temb[:, ci], shift=temb[:, si])
    assert np.array_equal(c, d)
    # shift_idx == scale_idx is allowed
    e = orc.ln_quant_fp8(x, 0.025, orc.MOD_TABLE, temb=temb, table=table, shift_idx=3, scale_idx=3)
    f = orc.ln_quant_fp8(x, 0.025, orc.MOD_PTOK, scale=_u16(temb_f[:, 3] + table[3]),
                         shift=_u16(temb_f[:, 3] + table[3]))
    assert np.array_equal(e, f)


# ------------------------------------------------------------ FP8 codes ---

def test_fp8_codes_are_nearest(orc):
    w = synth.fp8_ptok(64, 512, seed=3, outliers=0.05)
    x, sc, sh = (synth.u16(w.inputs[k]) for k in ("x", "scale", "shift"))
    act = 0.025
    q = orc.ln_quant_fp8(x, act, orc.MOD_PTOK, scale=sc, shift=sh)
    y = orc.modulated(x, orc.MOD_PTOK, scale=sc, shift=sh)
    t = (y / np.float64(np.float32(act))).astype(np.float32).astype(np.float64)
    table = orc.e4m3_table()
    dec = table[q]
    mag = (q & 0x7F).astype(np.int64)
    sgn = np.where(q & 0x80, -1.0, 1.0)
    lower = sgn * table[np.maximum(mag - 1, 0)]
    upper = sgn * table[np.minimum(mag + 1, 0x7E)]
    err = np.abs(t - dec)
    sat = np.abs(t) >= 448
    assert np.all((err <= np.abs(t - lower)) | sat)
    assert np.all((err <= np.abs(t - upper)) | sat)
    assert np.all(np.sign(dec) * np.sign(t) >= 0)
    # saturated values sit at +-448
    assert np.all(np.abs(dec[sat]) == 448)


def test_fp8_constant_row_gives_shift_codes(orc):
    x = _u16(np.full((2, 32), -3.0, dtype=np.float32))
    sh = _u16(np.linspace(-12, 12, 32, dtype=np.float32))
    z = np.zeros(32, dtype=np.uint16)
    q = orc.ln_quant_fp8(x, 0.025, orc.MOD_BCAST, scale=z, shift=sh)
    ref = torch.from_numpy((_f64(sh).numpy() / np.float32(0.025)).astype(np.float32))
    ref = ref.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q[0], ref) and np.array_equal(q[1], ref)


# ------------------------------------------------------------ NVFP4 -------

def test_nvfp4_blocks_bound_and_nearest(orc):
    w = synth.nvfp4_broadcast(40, 1024, seed=8)
    x, sc, sh = (synth.u16(w.inputs[k]) for k in ("x", "scale", "shift"))
    packed, sf = orc.ln_quant_nvfp4(x, orc.MOD_BCAST, swizzled=False, scale=sc, shift=sh)
    y = orc.modulated(x, orc.MOD_BCAST, scale=sc, shift=sh)
    v = torch.from_numpy(y.astype(np.float32)).to(torch.bfloat16).double().numpy()
    codes = orc.unpack_e2m1(packed)
    e4 = orc.e4m3_table()
    e2 = orc.e2m1_table()
    s_dec = e4[sf]
    amax = np.abs(v).reshape(40, 64, 16).max(axis=2)
    # scale byte: the e4m3 value nearest amax/6 (torch's RNE conversion)
    ref_sf = torch.from_numpy((amax / 6).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(sf, ref_sf)
    # the decoded scale covers the block unless amax/6 rounded down
    rounded_down = s_dec < amax / 6
    assert np.all((s_dec * 6 >= amax) | rounded_down)
    # every code is the nearest grid value of v/s (checked against both neighbours)
    q = v / np.repeat(s_dec, 16, axis=1)
    dec = e2[codes]
    mag = (codes & 7).astype(np.int64)
    sgn = np.where(codes & 8, -1.0, 1.0)
    lo = sgn * e2[np.maximum(mag - 1, 0)]
    hi = sgn * e2[np.minimum(mag + 1, 7)]
    assert np.all(np.abs(q - dec) <= np.abs(q - lo))
    assert np.all(np.abs(q - dec) <= np.abs(q - hi))
    assert np.array_equal((codes >> 3).astype(bool), np.signbit(v))


def test_nvfp4_packing_low_nibble_first(orc):
    # constant x -> x_hat = 0 -> y = shift exactly: the shift row sets v directly
    dim = 32
    sh = np.array([6.0, 0.5, -1.0, 3.0] + [0.0] * 12 + [-6.0, -1e-30, 1.5, -4.0] + [2.0] * 12,
                  dtype=np.float32)
    x = _u16(np.ones((1, dim), dtype=np.float32))
    z = np.zeros(dim, dtype=np.uint16)
    packed, sf = orc.ln_quant_nvfp4(x, orc.MOD_BCAST, swizzled=False, scale=z, shift=_u16(sh))
    assert list(sf[0]) == [0x38, 0x38]            # amax 6 -> scale 1.0
    assert packed[0, 0] == (0x7 | (0x1 << 4))      # 6 low, 0.5 high
    assert packed[0, 1] == (0xA | (0x5 << 4))      # -1 low, 3 high
    assert packed[0, 8] == (0xF | (0x8 << 4))      # -6 low, -1e-30 -> -0 high
    assert packed[0, 9] == (0x3 | (0xE << 4))      # 1.5 low, -4 high


def test_nvfp4_zero_block_scale_and_signed_zero(orc):
    dim = 16
    sh = np.array([-1e-30, 1e-30] + [0.0] * 14, dtype=np.float32)  # amax/6 underflows e4m3
    x = _u16(np.ones((1, dim), dtype=np.float32))
    z = np.zeros(dim, dtype=np.uint16)
    packed, sf = orc.ln_quant_nvfp4(x, orc.MOD_BCAST, swizzled=False, scale=z, shift=_u16(sh))
    assert sf[0, 0] == 0
    assert packed[0, 0] == 0x08 and np.all(packed[0, 1:] == 0)


def test_nvfp4_swizzled_matches_logical(orc):
    w = synth.nvfp4_ln(131, 80, seed=12)
    x = synth.u16(w.inputs["x"])
    p1, logical = orc.ln_quant_nvfp4(x, orc.MOD_NONE, swizzled=False)
    p2, swz = orc.ln_quant_nvfp4(x, orc.MOD_NONE, swizzled=True)
    assert np.array_equal(p1, p2)
    assert np.array_equal(swz, orc.swizzle_scales(logical, 131, 80))


# ------------------------------------------------------------ six-way -----

def test_modulation6_matches_numpy_add_and_torch_bf16(orc):
    w = synth.modulation6(2, 37, 200, seed=6)
    p, m = w.inputs["params"].numpy(), w.inputs["modulation"].numpy()
    out = orc.adaln_modulation6(p, m)
    for i in range(6):
        s = p[:, :, i, :] + m[i]   # numpy float32 addition
        ref = synth.u16(torch.from_numpy(np.ascontiguousarray(s)).to(torch.bfloat16))
        assert np.array_equal(out[i], ref)


def test_threads_do_not_change_results(orc):
    w = synth.fp8_table(50, 192, seed=21)
    x, temb = synth.u16(w.inputs["x"]), synth.u16(w.inputs["temb"])
    t = w.inputs["table"].numpy()
    a = orc.ln_quant_fp8(x, 0.025, orc.MOD_TABLE, nthreads=1, temb=temb, table=t, shift_idx=0, scale_idx=1)
    b = orc.ln_quant_fp8(x, 0.025, orc.MOD_TABLE, nthreads=7, temb=temb, table=t, shift_idx=0, scale_idx=1)
    assert np.array_equal(a, b)
