"""Pins of the oracle's two-level NVFP4 quantiser and segmented modulation (CPU).

Two-level NVFP4 (h3-blackwell-runtime compare page: NVFP4_STREAMING_DESIGN.md
"Numerical Constraint"; the P1 checkpoint's "numerical_contract").  Readings:
tensor scale ts = bf16(fp32(amax / 2688)); block scale e4m3(fminf((amax_b / 6)
/ ts, 448)); codes e2m1(v / (decode(s) * ts)).  Pins: the page's all-zero case
(tensor scale 0, scale byte 126); a tensor whose global amax is 2688 has ts = 1
and must equal the single-level producer byte for byte; power-of-two scaling of
the whole tensor scales ts and nothing else; hand-worked blocks.

Segmented modulation: row r takes row seg_idx[r] of the tables -- equal to the
per-token form on the gathered rows.
"""
import json
import os

import numpy as np
import torch

import synth


def _u16(a):
    return synth.u16(synth.bf16(a))


def _f64(bits):
    return torch.from_numpy(np.asarray(bits).view(np.int16).copy()).view(torch.bfloat16).double().numpy()


def test_zero_tensor_matches_page(orc, golden_dir):
    g = json.load(open(os.path.join(golden_dir, "h3_two_level_zero_tensor.json")))
    rows, dim = 130, 80
    v = np.zeros((rows, dim), dtype=np.uint16)
    packed, sf, ts = orc.nvfp4_2level(v)
    assert ts == g["tensor_scale"]
    logical = orc.swizzled_sf_size(rows, dim)
    data = sf[orc.sf_offsets(np.repeat(np.arange(rows), dim // 16), np.tile(np.arange(dim // 16), rows), dim)]
    assert set(data.tolist()) == set(g["block_scale_bytes"])
    assert np.all(packed == 0)
    assert logical == sf.size


def test_global_amax_2688_equals_single_level(orc):
    # broadcast modulation with scale 0 and shift 2688 in column 5: every v there is
    # bf16(x_hat + 2688) = 2688 (|x_hat| < 7 < half the bf16 spacing 16 at 2688),
    # so the global amax is 2688 and ts = bf16(2688 / 2688) = 1
    rng = np.random.default_rng(3)
    rows, dim = 70, 48
    x = _u16(rng.standard_normal((rows, dim)).astype(np.float32))
    scale = _u16(rng.normal(0, 0.3, dim).astype(np.float32))
    shift_f = rng.normal(0, 2.0, dim).astype(np.float32)
    shift_f[5] = 2688.0
    scale_f = _f64(scale).astype(np.float32)
    scale_f[5] = 0.0
    scale, shift = _u16(scale_f), _u16(shift_f)
    v = orc.staged(x, orc.MOD_BCAST, scale=scale, shift=shift)
    assert np.abs(_f64(v)).max() == 2688.0 and np.all(_f64(v)[:, 5] == 2688.0)
    p2, s2, ts = orc.ln_quant_nvfp4_2level(x, orc.MOD_BCAST, scale=scale, shift=shift)
    p1, s1 = orc.ln_quant_nvfp4(x, orc.MOD_BCAST, scale=scale, shift=shift)
    assert ts == 1.0
    assert np.array_equal(p1, p2) and np.array_equal(s1, s2)


def test_power_of_two_scaling_moves_only_the_tensor_scale(orc):
    rng = np.random.default_rng(4)
    v = _u16(rng.standard_normal((33, 96)).astype(np.float32) * 3)
    p0, s0, t0 = orc.nvfp4_2level(v)
    for k in (-20, -3, 5, 40):
        vk = _u16(_f64(v).astype(np.float32) * np.float32(2.0 ** k))
        assert np.array_equal(_f64(vk), _f64(v) * 2.0 ** k)           # exact in bf16
        pk, sk, tk = orc.nvfp4_2level(vk)
        assert np.array_equal(pk, p0) and np.array_equal(sk, s0)
        assert tk == t0 * 2.0 ** k


def test_constant_tensor_hand_worked(orc):
    # v = +-2.625: ts = bf16(2.625 / 2688) = 2^-10 exactly; (2.625 / 6) / 2^-10 = 448
    # -> scale byte 0x7E; v / (448 * 2^-10) = +-6 -> codes 0x7 / 0xF
    v = _u16(np.tile(np.array([2.625, -2.625], dtype=np.float32), (4, 16)))
    packed, sf, ts = orc.nvfp4_2level(v)
    assert ts == 2.0 ** -10
    data = sf[orc.sf_offsets(np.repeat(np.arange(4), 2), np.tile(np.arange(2), 4), 32)]
    assert np.all(data == 0x7E)
    assert np.all(packed == 0xF7)


def test_clamp_when_the_tensor_scale_rounds_down(orc):
    # a single 3072 (1.5 * 2^11): 3072 / 2688 = 1.142857... rounds down to the bf16
    # 1.140625, so (3072 / 6) / ts = 448.88 is clamped to 448 (byte 0x7E) and
    # 3072 / (448 * 1.140625) = 6.01 saturates to code 7; the other blocks hold
    # 1.0 with ts 1.140625: (1/6)/1.140625 = 0.14612 -> e4m3 0.140625 (byte 0x22)
    v = np.full((1, 48), 0x3F80, dtype=np.uint16)               # 1.0
    v[0, 0] = _u16(np.array([3072.0], dtype=np.float32))[0]
    packed, sf, ts = orc.nvfp4_2level(v)
    assert ts == 1.140625
    data = sf[orc.sf_offsets(np.zeros(3, dtype=np.int64), np.arange(3), 48)]
    assert data[0] == 0x7E
    assert orc.e4m3_decode(int(data[1])) == 0.140625 and data[1] == data[2]
    codes = orc.unpack_e2m1(packed)[0]
    assert codes[0] == 7
    # 1.0 / (0.140625 * 1.140625) = 6.23 -> 6 (code 7); in block 0: 1 / (448 * 1.140625) -> 0
    assert np.all(codes[16:] == 7) and np.all(codes[1:16] == 0)


def test_segmented_equals_per_token_on_gathered_rows(orc):
    rng = np.random.default_rng(5)
    rows, dim, nseg = 61, 80, 3
    x = _u16(rng.standard_normal((rows, dim)).astype(np.float32))
    tab_s = _u16(rng.normal(0, 0.1, (nseg, dim)).astype(np.float32))
    tab_h = _u16(rng.normal(0, 0.1, (nseg, dim)).astype(np.float32))
    seg = np.array([1] * 10 + [2] * 30 + [0] * 21, dtype=np.int32)   # the page's range form
    src = dict(seg_idx=seg, seg_scale=tab_s, seg_shift=tab_h)
    a = orc.ln_quant_fp8(x, 0.025, orc.MOD_SEG, **src)
    b = orc.ln_quant_fp8(x, 0.025, orc.MOD_PTOK, scale=tab_s[seg], shift=tab_h[seg])
    assert np.array_equal(a, b)
    pa, sa = orc.ln_quant_nvfp4(x, orc.MOD_SEG, **src)
    pb, sb = orc.ln_quant_nvfp4(x, orc.MOD_PTOK, scale=tab_s[seg], shift=tab_h[seg])
    assert np.array_equal(pa, pb) and np.array_equal(sa, sb)
    q1 = orc.ln_quant_nvfp4_2level(x, orc.MOD_SEG, **src)
    q2 = orc.ln_quant_nvfp4_2level(x, orc.MOD_PTOK, scale=tab_s[seg], shift=tab_h[seg])
    assert all(np.array_equal(u, w) for u, w in zip(q1[:2], q2[:2])) and q1[2] == q2[2]


def test_segmented_modulation_matches_torch(orc):
    import torch.nn.functional as F
    rng = np.random.default_rng(6)
    rows, dim = 9, 64
    x = _u16(rng.standard_normal((rows, dim)).astype(np.float32))
    tab_s = _u16(rng.normal(0, 0.2, (2, dim)).astype(np.float32))
    tab_h = _u16(rng.normal(0, 0.2, (2, dim)).astype(np.float32))
    seg = rng.integers(0, 2, rows).astype(np.int32)
    y = orc.modulated(x, orc.MOD_SEG, seg_idx=seg, seg_scale=tab_s, seg_shift=tab_h)
    ln = F.layer_norm(torch.from_numpy(_f64(x)), (dim,), eps=float(np.float32(1e-5))).numpy()
    ref = ln * (1.0 + _f64(tab_s)[seg]) + _f64(tab_h)[seg]
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_block_scale_division_order_does_not_change_bytes():
    # the page prints (amax / 6) / ts; with bf16 amax values and a bf16 tensor
    # scale the reverse order (amax / ts) / 6 gives the same e4m3 byte for every
    # pair: global amax over all 128 bf16 mantissas in [1, 2), block amax over
    # 18 binades below it (power-of-two scaling of the whole tensor is exact)
    g = ((np.arange(0x3F80, 0x4000, dtype=np.uint32)) << 16).view(np.float32)
    a = ((np.arange(0x3780, 0x4000, dtype=np.uint32)) << 16).view(np.float32)
    ts = torch.from_numpy(g / np.float32(2688.0)).to(torch.bfloat16).float().numpy()
    A, T = np.meshgrid(a, ts, indexing="ij")
    G = np.meshgrid(a, g, indexing="ij")[1]
    keep = A <= G
    e4 = lambda q: torch.from_numpy(np.minimum(q, np.float32(448.0))).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    printed = e4(((A / np.float32(6.0)).astype(np.float32) / T).astype(np.float32))
    reverse = e4(((A / T).astype(np.float32) / np.float32(6.0)).astype(np.float32))
    assert np.array_equal(printed[keep], reverse[keep])


# ------------------------------------------------------------------ SwiGLU --

def _silu_bf16_torch(g_bits):
    # torch's float64 silu, rounded to binary32 and then to bf16
    g = torch.from_numpy(_f64(g_bits))
    return torch.nn.functional.silu(g).float().to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_swiglu_silu_boundary_matches_torch(orc):
    # with up = 1 the product is exact, so v is the bf16 silu value itself
    rng = np.random.default_rng(12)
    g = _u16((rng.standard_normal((40, 64)) * 4).astype(np.float32))
    one = _u16(np.ones((40, 64), dtype=np.float32))
    assert np.array_equal(orc.swiglu_values(g, one), _silu_bf16_torch(g))


def test_swiglu_product_boundary_matches_torch(orc):
    rng = np.random.default_rng(13)
    g = _u16((rng.standard_normal((30, 48)) * 3).astype(np.float32))
    u = _u16((rng.standard_normal((30, 48)) * 2).astype(np.float32))
    s = torch.from_numpy(_silu_bf16_torch(g).view(np.int16)).view(torch.bfloat16).double()
    ref = (s * torch.from_numpy(_f64(u))).float().to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.swiglu_values(g, u), ref)
    # power-of-two up scales the bf16 silu exactly
    two = _u16(np.full((30, 48), 0.25, dtype=np.float32))
    assert np.array_equal(_f64(orc.swiglu_values(g, two)), _f64(_silu_bf16_torch(g)) * 0.25)


def test_swiglu_closed_forms(orc):
    # silu(0) = 0 (sign kept: 0 / 1), silu(-inf-like) -> -0-side tiny values, silu(large) = large
    g = _u16(np.array([[0.0, -0.0, 64.0, 1.0]], dtype=np.float32))
    u = _u16(np.ones((1, 4), dtype=np.float32))
    v = _f64(orc.swiglu_values(g, u))[0]
    assert v[0] == 0.0 and v[2] == 64.0
    assert np.float32(v[3]) == torch.tensor(1.0 / (1.0 + np.exp(-1.0))).float().to(torch.bfloat16).float().item()


def test_swiglu_two_level_is_the_quantiser_of_its_values(orc):
    rng = np.random.default_rng(14)
    g = _u16((rng.standard_normal((70, 96)) * 2).astype(np.float32))
    u = _u16(rng.standard_normal((70, 96)).astype(np.float32))
    p1, s1, t1 = orc.swiglu_quant_nvfp4_2level(g, u)
    p2, s2, t2 = orc.nvfp4_2level(orc.swiglu_values(g, u))
    assert np.array_equal(p1, p2) and np.array_equal(s1, s2) and t1 == t2
