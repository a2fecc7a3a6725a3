"""Pins of the oracle's modfp8 and AWQ modulation sources (CPU only).

modfp8 (README "Available Functions": ada_layer_norm_quant_fp8_modfp8_bf16 and
ada_layer_norm_quant_nvfp4_swizzled_modfp8_bf16; "Tensor Contract": e4m3 (dim,)
scale_fp8/shift_fp8 and fp32 scalar scale_deq/shift_deq).  Reading: scale =
decode(scale_fp8) * scale_deq, shift = decode(shift_fp8) * shift_deq.

AWQ (README "Available Functions": awq_ada_layer_norm_quant_fp8_bf16; "Tensor
Contract": bf16 (dim,) inv_s).  Reading: the FP8 code is e4m3(y * inv_s /
act_scale) with y the modulated activation.

Pins: hand-worked rows whose every intermediate value is exact (alternating
+-1 rows with eps = 0 normalise to exactly +-1), torch's own float8_e4m3fn
decoder and float64 layer_norm, and equalities with the broadcast producer
(itself pinned against torch) where the new source reduces to it exactly.
"""
import numpy as np
import torch
import torch.nn.functional as F

import synth


def _u16(a):
    return synth.u16(synth.bf16(a))


def _f64(bits):
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double()


def _torch_e4m3(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).double()


def _alternating(rows=1, dim=16):
    """x = [+1, -1, +1, ...]: mean 0, variance 1, so with eps = 0 x_hat = +-1 exactly."""
    return _u16(np.tile(np.array([1.0, -1.0], dtype=np.float32), (rows, dim // 2)))


# ---------------------------------------------------------------- modfp8 --

def test_modfp8_fp8_hand_worked_row(orc):
    # columns 0-7: scale 0.5 (0x30) * deq 2 = 1, shift 0.25 (0x28) * deq 4 = 1
    #   -> y = +1*(1+1)+1 = 3 (even cols), -1*2+1 = -1 (odd cols)
    # columns 8-15: shift -0.25 (0xA8) * 4 = -1 -> y = 1 (even), -3 (odd)
    # act_scale 0.5: y/act = 6, -2 | 2, -6 -> e4m3 0x4C, 0xC0 | 0x40, 0xCC
    x = _alternating()
    scale_fp8 = np.full(16, 0x30, dtype=np.uint8)
    shift_fp8 = np.array([0x28] * 8 + [0xA8] * 8, dtype=np.uint8)
    out = orc.ln_quant_fp8(x, 0.5, orc.MOD_MODFP8, eps=0.0, scale_fp8=scale_fp8,
                           shift_fp8=shift_fp8, scale_deq=2.0, shift_deq=4.0)
    expect = np.array([0x4C, 0xC0] * 4 + [0x40, 0xCC] * 4, dtype=np.uint8)
    assert np.array_equal(out[0], expect)


def test_modfp8_nvfp4_hand_worked_row(orc):
    # same modulation: block 0 holds y = 3, -1 (amax 3), block 1 y = 1, -3
    # (amax 3); s = e4m3(3/6 = 0.5) = 0x30 for both; v/s = 6, -2 | 2, -6
    # -> e2m1 magnitudes 6 (code 7), 2 (code 4); negative adds 8
    x = _alternating(dim=32)
    scale_fp8 = np.full(32, 0x30, dtype=np.uint8)
    shift_fp8 = np.array([0x28] * 16 + [0xA8] * 16, dtype=np.uint8)
    packed, sf = orc.ln_quant_nvfp4(x, orc.MOD_MODFP8, eps=0.0, swizzled=False, scale_fp8=scale_fp8,
                                    shift_fp8=shift_fp8, scale_deq=2.0, shift_deq=4.0)
    assert list(sf[0]) == [0x30, 0x30]
    codes = orc.unpack_e2m1(packed)[0]
    assert list(codes[:16]) == [0x7, 0xC] * 8
    assert list(codes[16:]) == [0x4, 0xF] * 8


def test_modfp8_modulation_matches_torch_decoder(orc):
    rng = np.random.default_rng(11)
    rows, dim = 6, 80
    x = _u16(rng.standard_normal((rows, dim)).astype(np.float32))
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    scale_fp8 = rng.choice(finite, dim).astype(np.uint8)
    shift_fp8 = rng.choice(finite, dim).astype(np.uint8)
    sdeq, hdeq = np.float32(0.0123), np.float32(-3.7)
    y = orc.modulated(x, orc.MOD_MODFP8, eps=1e-5, scale_fp8=scale_fp8, shift_fp8=shift_fp8,
                      scale_deq=float(sdeq), shift_deq=float(hdeq))
    ln = F.layer_norm(_f64(x), (dim,), eps=float(np.float32(1e-5)))
    ref = ln * (1.0 + _torch_e4m3(scale_fp8) * float(sdeq)) + _torch_e4m3(shift_fp8) * float(hdeq)
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)


def _representable_codes(rng, n):
    # |value| <= 1 (codes 0x00-0x38 and their negatives): decode * deq below
    # has at most 6 significant bits, so it is exact in bf16
    mags = rng.integers(0, 0x39, n)
    sign = rng.integers(0, 2, n) << 7
    return (mags | sign).astype(np.uint8)


def test_modfp8_equals_broadcast_on_bf16_exact_values(orc):
    rng = np.random.default_rng(12)
    rows, dim = 9, 192
    x = _u16(rng.standard_normal((rows, dim)).astype(np.float32))
    scale_fp8, shift_fp8 = _representable_codes(rng, dim), _representable_codes(rng, dim)
    sdeq, hdeq = 0.375, 3.0  # two significant bits each
    dec = orc.e4m3_table()
    scale_bf = _u16((dec[scale_fp8] * sdeq).astype(np.float32))
    shift_bf = _u16((dec[shift_fp8] * hdeq).astype(np.float32))
    assert np.array_equal(_f64(scale_bf).numpy(), dec[scale_fp8] * sdeq)
    assert np.array_equal(_f64(shift_bf).numpy(), dec[shift_fp8] * hdeq)
    src = dict(scale_fp8=scale_fp8, shift_fp8=shift_fp8, scale_deq=sdeq, shift_deq=hdeq)
    a = orc.ln_quant_fp8(x, 0.025, orc.MOD_MODFP8, **src)
    b = orc.ln_quant_fp8(x, 0.025, orc.MOD_BCAST, scale=scale_bf, shift=shift_bf)
    assert np.array_equal(a, b)
    pa, sa = orc.ln_quant_nvfp4(x, orc.MOD_MODFP8, **src)
    pb, sb = orc.ln_quant_nvfp4(x, orc.MOD_BCAST, scale=scale_bf, shift=shift_bf)
    assert np.array_equal(pa, pb) and np.array_equal(sa, sb)
    # swapping the two scalars changes the result (the pins above tell them apart)
    c = orc.ln_quant_fp8(x, 0.025, orc.MOD_MODFP8, scale_fp8=scale_fp8, shift_fp8=shift_fp8,
                         scale_deq=hdeq, shift_deq=sdeq)
    assert not np.array_equal(a, c)


def test_modfp8_zero_codes_are_plain_layer_norm(orc):
    rng = np.random.default_rng(13)
    x = _u16(rng.standard_normal((5, 64)).astype(np.float32))
    z = np.zeros(64, dtype=np.uint8)
    a = orc.ln_quant_fp8(x, 0.025, orc.MOD_MODFP8, scale_fp8=z, shift_fp8=z, scale_deq=7.0, shift_deq=-2.0)
    b = orc.ln_quant_fp8(x, 0.025, orc.MOD_NONE)
    assert np.array_equal(a, b)


# ------------------------------------------------------------------- AWQ --

def test_awq_hand_worked_row(orc):
    # scale 1 (1+scale = 2), shift 1: y = 3 (even cols), -1 (odd cols)
    # inv_s 0.5 on columns 0-7, 2 on columns 8-15: y*inv_s = 1.5, -0.5 | 6, -2
    # act_scale 0.5: 3, -1 | 12, -4 -> e4m3 0x44, 0xB8 | 0x54, 0xC8
    # (inv_s applied to x_hat before the modulation would give 4, ... instead)
    x = _alternating()
    one = _u16(np.ones(16, dtype=np.float32))
    inv_s = _u16(np.array([0.5] * 8 + [2.0] * 8, dtype=np.float32))
    out = orc.ln_quant_fp8(x, 0.5, orc.MOD_AWQ, eps=0.0, scale=one, shift=one, inv_s=inv_s)
    expect = np.array([0x44, 0xB8] * 4 + [0x54, 0xC8] * 4, dtype=np.uint8)
    assert np.array_equal(out[0], expect)


def test_awq_unit_smoothing_is_broadcast(orc):
    w = synth.fp8_broadcast(7, 320, seed=14)
    x, sc, sh = (synth.u16(w.inputs[k]) for k in ("x", "scale", "shift"))
    one = _u16(np.ones(320, dtype=np.float32))
    a = orc.ln_quant_fp8(x, 0.025, orc.MOD_AWQ, scale=sc, shift=sh, inv_s=one)
    b = orc.ln_quant_fp8(x, 0.025, orc.MOD_BCAST, scale=sc, shift=sh)
    assert np.array_equal(a, b)


def test_awq_power_of_two_smoothing_moves_act_scale(orc):
    # y * 2^k / act == y / (act * 2^-k) exactly, so the codes are identical
    w = synth.fp8_broadcast(7, 320, seed=15)
    x, sc, sh = (synth.u16(w.inputs[k]) for k in ("x", "scale", "shift"))
    for k in (-3, 1, 4):
        inv_s = _u16(np.full(320, 2.0**k, dtype=np.float32))
        a = orc.ln_quant_fp8(x, 0.025, orc.MOD_AWQ, scale=sc, shift=sh, inv_s=inv_s)
        b = orc.ln_quant_fp8(x, float(np.float32(0.025) * np.float32(2.0**-k)), orc.MOD_BCAST, scale=sc, shift=sh)
        assert np.array_equal(a, b), k


def test_awq_modulation_matches_torch(orc):
    rng = np.random.default_rng(16)
    rows, dim = 5, 96
    x = _u16(rng.standard_normal((rows, dim)).astype(np.float32))
    sc = _u16(rng.normal(0, 0.1, dim).astype(np.float32))
    sh = _u16(rng.normal(0, 0.1, dim).astype(np.float32))
    inv_s = _u16(rng.uniform(0.25, 4.0, dim).astype(np.float32))
    y = orc.modulated(x, orc.MOD_AWQ, scale=sc, shift=sh, inv_s=inv_s)
    ln = F.layer_norm(_f64(x), (dim,), eps=float(np.float32(1e-5)))
    ref = (ln * (1.0 + _f64(sc)) + _f64(sh)) * _f64(inv_s)
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)
