"""GPU parity of the modfp8 and AWQ producers against the oracle (C ABI).

ada_layer_norm_quant_fp8_modfp8_bf16, ada_layer_norm_quant_nvfp4_swizzled_
modfp8_bf16 and awq_ada_layer_norm_quant_fp8_bf16 (README "Available
Functions"; readings: scale = decode(scale_fp8) * scale_deq, and the AWQ
code e4m3(y * inv_s / act_scale)).  Tolerance: tests/parity.py.  Cases: the
shapes of the broadcast producers' tests under every kernel family, the
bf16-pair path (dims not a multiple of 8, e4m3 vectors off 8-byte alignment),
deq scalars that are not powers of two, and exact reductions on the GPU
itself: with codes and deq whose products are bf16 values, the modfp8 output
equals the broadcast producer's output bit for bit; with inv_s = 1 the AWQ
output equals it too.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import check_fp8, check_nvfp4

pytestmark = pytest.mark.gpu

FP8_SHAPES = [(1, 32), (3, 48), (8, 2), (40, 16), (127, 1536), (129, 3072), (300, 2048), (64, 2050),
              (17, 1152), (51, 1536), (5, 32768), (33, 6144), (9, 10240)]
NV_SHAPES = [(1, 16), (3, 48), (127, 64), (129, 80), (300, 3072), (64, 5376), (128, 7168), (33, 14336),
             (5, 32768), (257, 1536)]


def _codes(t):
    return t.view(torch.uint8).cpu().numpy()


def _u8(t):
    return t.view(torch.uint8).numpy()


def _d(w, dev):
    return {k: v.to(dev) for k, v in w.inputs.items()}


def _fval(t):
    return float(t[0])


def _modfp8_src(w):
    return dict(scale_fp8=_u8(w.inputs["scale_fp8"]), shift_fp8=_u8(w.inputs["shift_fp8"]),
                scale_deq=_fval(w.inputs["scale_deq"]), shift_deq=_fval(w.inputs["shift_deq"]))


@pytest.mark.parametrize("rows,dim", FP8_SHAPES)
def test_modfp8_fp8(ap, dev, path, rows, dim):
    w = synth.fp8_modfp8(rows, dim, seed=rows * 19 + dim)
    d = _d(w, dev)
    out = ap.ada_layer_norm_quant_fp8_modfp8_bf16(d["x"], d["scale_fp8"], d["shift_fp8"], d["scale_deq"],
                                                  d["shift_deq"], d["act_scale"])
    act = _fval(w.inputs["act_scale"])
    ref = oracle.ln_quant_fp8(synth.u16(w.inputs["x"]), act, oracle.MOD_MODFP8, **_modfp8_src(w))
    check_fp8(_codes(out), ref, act, "modfp8")


@pytest.mark.parametrize("rows,dim", FP8_SHAPES)
def test_awq_fp8(ap, dev, path, rows, dim):
    w = synth.fp8_awq(rows, dim, seed=rows * 23 + dim)
    d = _d(w, dev)
    out = ap.awq_ada_layer_norm_quant_fp8_bf16(d["x"], d["scale"], d["shift"], d["inv_s"], d["act_scale"])
    act = _fval(w.inputs["act_scale"])
    u = {k: synth.u16(w.inputs[k]) for k in ("x", "scale", "shift", "inv_s")}
    ref = oracle.ln_quant_fp8(u["x"], act, oracle.MOD_AWQ, scale=u["scale"], shift=u["shift"], inv_s=u["inv_s"])
    check_fp8(_codes(out), ref, act, "awq")


@pytest.mark.parametrize("rows,dim", NV_SHAPES)
def test_modfp8_nvfp4(ap, dev, path, rows, dim):
    w = synth.nvfp4_modfp8(rows, dim, seed=rows * 29 + dim)
    d = _d(w, dev)
    n = ap.swizzled_sf_size(rows, dim)
    guard = 512
    sfbuf = torch.full((n + 2 * guard,), 0xFF, dtype=torch.uint8, device=dev)
    sf = sfbuf[guard:guard + n]
    packed, _ = ap.ada_layer_norm_quant_nvfp4_swizzled_modfp8_bf16(d["x"], d["scale_fp8"], d["shift_fp8"],
                                                                   d["scale_deq"], d["shift_deq"], sf_swizzled=sf)
    sb = sfbuf.cpu().numpy()
    assert np.all(sb[:guard] == 0xFF) and np.all(sb[-guard:] == 0xFF)
    x = synth.u16(w.inputs["x"])
    src = _modfp8_src(w)
    opk, osf = oracle.ln_quant_nvfp4(x, oracle.MOD_MODFP8, **src)
    y = oracle.modulated(x, oracle.MOD_MODFP8, **src)
    v = torch.from_numpy(y.astype(np.float32)).to(torch.bfloat16).double().numpy()
    check_nvfp4(packed.cpu().numpy(), sb[guard:guard + n], opk, osf, rows, dim, v, "modfp8 nvfp4")


def _exact_codes(rng, n):
    # |value| <= 1: decode * deq (deq with two significant bits) is a bf16 value
    mags = rng.integers(0, 0x39, n)
    return torch.from_numpy(((mags | (rng.integers(0, 2, n) << 7)).astype(np.uint8))).view(torch.float8_e4m3fn)


# Bit-for-bit reductions compare two calls that must run the same kernel: the
# default choice, the register row kernels (NVFP4AP_KERNEL=3) and the
# block-per-lane kernels (NVFP4AP_KERNEL=5).  The TMA family has no modfp8 /
# AWQ variant, so there the two calls run different kernels whose fp32
# rounding order differs (each is compared with the oracle above).
@pytest.fixture(params=["auto", "rows", "blk"])
def same_kernel(request, monkeypatch):
    if request.param == "auto":
        monkeypatch.delenv("NVFP4AP_KERNEL", raising=False)
    else:
        monkeypatch.setenv("NVFP4AP_KERNEL", "3" if request.param == "rows" else "5")
    return request.param


@pytest.mark.parametrize("rows,dim", [(129, 3072), (300, 2048), (64, 2050), (5, 32768)])
def test_modfp8_equals_broadcast_bit_for_bit(ap, dev, same_kernel, rows, dim):
    rng = np.random.default_rng(rows + dim)
    x = synth.bf16(synth.normal(rows + dim, 0, (rows, dim), 1.0)).to(dev)
    s8, h8 = _exact_codes(rng, dim), _exact_codes(rng, dim)
    sdeq, hdeq = 0.375, 3.0
    scale_bf = (s8.float() * sdeq).to(torch.bfloat16)
    shift_bf = (h8.float() * hdeq).to(torch.bfloat16)
    assert torch.equal(scale_bf.float(), s8.float() * sdeq) and torch.equal(shift_bf.float(), h8.float() * hdeq)
    act = torch.tensor([0.025], device=dev)
    sd, hd = torch.tensor([sdeq], device=dev), torch.tensor([hdeq], device=dev)
    s8, h8, scale_bf, shift_bf = s8.to(dev), h8.to(dev), scale_bf.to(dev), shift_bf.to(dev)
    a = ap.ada_layer_norm_quant_fp8_modfp8_bf16(x, s8, h8, sd, hd, act)
    b = ap.ada_layer_norm_quant_fp8_bf16(x, scale_bf, shift_bf, act)
    assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    if dim % 16 == 0:
        pa, sa = ap.ada_layer_norm_quant_nvfp4_swizzled_modfp8_bf16(x, s8, h8, sd, hd)
        pb, sb = ap.ada_layer_norm_quant_nvfp4_swizzled_bf16(x, scale_bf, shift_bf)
        assert torch.equal(pa, pb) and torch.equal(sa, sb)


@pytest.mark.parametrize("rows,dim", [(129, 3072), (64, 2050), (5, 32768)])
def test_awq_unit_smoothing_equals_broadcast_bit_for_bit(ap, dev, same_kernel, rows, dim):
    w = synth.fp8_broadcast(rows, dim, seed=rows + 3 * dim)
    d = _d(w, dev)
    one = torch.ones(dim, dtype=torch.bfloat16, device=dev)
    a = ap.awq_ada_layer_norm_quant_fp8_bf16(d["x"], d["scale"], d["shift"], one, d["act_scale"])
    b = ap.ada_layer_norm_quant_fp8_bf16(d["x"], d["scale"], d["shift"], d["act_scale"])
    assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def _offset_view(t, elems):
    buf = torch.empty(t.numel() + elems + 16, dtype=t.dtype, device=t.device)
    v = buf[elems:elems + t.numel()].view(t.shape)
    v.copy_(t)
    return v


def test_modfp8_pair_path_when_vectors_off_8_byte_alignment(ap, dev):
    w = synth.fp8_modfp8(65, 1536, seed=77)
    d = _d(w, dev)
    s8, h8 = _offset_view(d["scale_fp8"], 2), _offset_view(d["shift_fp8"], 6)  # 2-byte aligned only
    assert s8.data_ptr() % 8 != 0 and h8.data_ptr() % 8 != 0
    out = ap.ada_layer_norm_quant_fp8_modfp8_bf16(d["x"], s8, h8, d["scale_deq"], d["shift_deq"], d["act_scale"])
    act = _fval(w.inputs["act_scale"])
    ref = oracle.ln_quant_fp8(synth.u16(w.inputs["x"]), act, oracle.MOD_MODFP8, **_modfp8_src(w))
    check_fp8(_codes(out), ref, act, "modfp8 pair path")


def test_awq_pair_path_when_off_16_byte_alignment(ap, dev):
    w = synth.fp8_awq(33, 1024, seed=78)
    d = _d(w, dev)
    inv_s = _offset_view(d["inv_s"], 2)  # 4-byte aligned only
    out = ap.awq_ada_layer_norm_quant_fp8_bf16(d["x"], d["scale"], d["shift"], inv_s, d["act_scale"])
    act = _fval(w.inputs["act_scale"])
    u = {k: synth.u16(w.inputs[k]) for k in ("x", "scale", "shift", "inv_s")}
    ref = oracle.ln_quant_fp8(u["x"], act, oracle.MOD_AWQ, scale=u["scale"], shift=u["shift"], inv_s=u["inv_s"])
    check_fp8(_codes(out), ref, act, "awq pair path")


def test_modfp8_nvfp4_misaligned_vectors_take_the_element_wise_kernel(ap, dev):
    w = synth.nvfp4_modfp8(16, 64, seed=79)
    d = _d(w, dev)
    s8 = _offset_view(d["scale_fp8"], 4)
    pk, sf = ap.ada_layer_norm_quant_nvfp4_swizzled_modfp8_bf16(d["x"], s8, d["shift_fp8"], d["scale_deq"],
                                                                d["shift_deq"])
    src = _modfp8_src(w)
    xu = synth.u16(w.inputs["x"])
    op, os_ = oracle.ln_quant_nvfp4(xu, oracle.MOD_MODFP8, **src)
    check_nvfp4(pk.cpu().numpy(), sf.cpu().numpy(), op, os_, 16, 64, what="modfp8 vectors off 8-byte alignment")


def test_modfp8_extreme_codes_and_saturation(ap, dev):
    # every finite e4m3 code appears in the scale and shift vectors (dim 256 = 2 x 128
    # codes per sign); deq 1/64 keeps scale within [-7, 7] and the outputs saturate
    # in places (|y / act| > 448)
    rows, dim = 40, 256
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F] + [0, 0x80], dtype=np.uint8)
    rng = np.random.default_rng(5)
    s8 = torch.from_numpy(rng.permutation(codes)).view(torch.float8_e4m3fn)
    h8 = torch.from_numpy(rng.permutation(codes)).view(torch.float8_e4m3fn)
    x = synth.bf16(synth.normal(80, 0, (rows, dim), 1.0))
    act, sd, hd = 0.0125, 1.0 / 64, 1.0 / 64
    out = ap.ada_layer_norm_quant_fp8_modfp8_bf16(x.to(dev), s8.to(dev), h8.to(dev), torch.tensor([sd], device=dev),
                                                  torch.tensor([hd], device=dev), torch.tensor([act], device=dev))
    ref = oracle.ln_quant_fp8(synth.u16(x), act, oracle.MOD_MODFP8, scale_fp8=_u8(s8), shift_fp8=_u8(h8),
                              scale_deq=sd, shift_deq=hd)
    assert np.any((ref & 0x7F) == 0x7E)  # saturated codes present
    check_fp8(_codes(out), ref, act, "modfp8 extreme codes")
