"""GPU parity of the block-per-lane persistent kernel where it is the default.

The FP8 broadcast sources (bf16, modfp8, AWQ) take it from 4096 rows when its
shape leaves no lane idle and holds three or more rows per 512-thread CTA
(dims 1024, 1536, 2048, 3072, 4096, 5120, 6144); the single-level NVFP4 forms
take it from 2048 rows where the row does not fit the one-row-per-CTA kernel
(dims 1024, 1536, 5120).  Cases: parity with the oracle on both sides of
each row threshold; the default's bytes equal the forced block-per-lane
kernel's (NVFP4AP_KERNEL=5), so the default really runs it; and the exact
reductions of the adaptive-layernorm-producers README's modulation sources
("Available Functions": modfp8 = e4m3 vectors times fp32 scalars, AWQ with a
smoothing vector) hold bit for bit on this kernel too, since the three sources
share one dispatch rule.  Tolerance: tests/parity.py.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import check_fp8, check_nvfp4

pytestmark = pytest.mark.gpu


def _codes(t):
    return t.view(torch.uint8).cpu().numpy()


def _d(w, dev):
    return {k: v.to(dev) for k, v in w.inputs.items()}


def _act(w):
    return float(w.inputs["act_scale"][0])


@pytest.fixture
def auto(monkeypatch):
    monkeypatch.delenv("NVFP4AP_KERNEL", raising=False)
    return monkeypatch


def _fp8_call(ap, op, d):
    if op == "bcast":
        return ap.ada_layer_norm_quant_fp8_bf16(d["x"], d["scale"], d["shift"], d["act_scale"])
    if op == "modfp8":
        return ap.ada_layer_norm_quant_fp8_modfp8_bf16(d["x"], d["scale_fp8"], d["shift_fp8"], d["scale_deq"],
                                                       d["shift_deq"], d["act_scale"])
    return ap.awq_ada_layer_norm_quant_fp8_bf16(d["x"], d["scale"], d["shift"], d["inv_s"], d["act_scale"])


def _fp8_case(op, rows, dim, seed):
    if op == "bcast":
        w = synth.fp8_broadcast(rows, dim, seed)
        u = {k: synth.u16(w.inputs[k]) for k in ("x", "scale", "shift")}
        ref = oracle.ln_quant_fp8(u["x"], _act(w), oracle.MOD_BCAST, scale=u["scale"], shift=u["shift"])
    elif op == "modfp8":
        w = synth.fp8_modfp8(rows, dim, seed)
        src = dict(scale_fp8=w.inputs["scale_fp8"].view(torch.uint8).numpy(),
                   shift_fp8=w.inputs["shift_fp8"].view(torch.uint8).numpy(),
                   scale_deq=float(w.inputs["scale_deq"][0]), shift_deq=float(w.inputs["shift_deq"][0]))
        ref = oracle.ln_quant_fp8(synth.u16(w.inputs["x"]), _act(w), oracle.MOD_MODFP8, **src)
    else:
        w = synth.fp8_awq(rows, dim, seed)
        u = {k: synth.u16(w.inputs[k]) for k in ("x", "scale", "shift", "inv_s")}
        ref = oracle.ln_quant_fp8(u["x"], _act(w), oracle.MOD_AWQ, scale=u["scale"], shift=u["shift"],
                                  inv_s=u["inv_s"])
    return w, ref


@pytest.mark.parametrize("op", ["bcast", "modfp8", "awq"])
@pytest.mark.parametrize("rows,dim", [(4095, 1536), (4096, 1536), (4097, 3072), (4096, 1024), (4103, 2048),
                                      (4096, 4096), (4099, 5120), (4096, 6144)])
def test_fp8_broadcast_sources_default(ap, dev, auto, op, rows, dim):
    w, ref = _fp8_case(op, rows, dim, seed=rows + dim)
    d = _d(w, dev)
    out = _fp8_call(ap, op, d)
    check_fp8(_codes(out), ref, _act(w), f"{op} {rows}x{dim}")
    if rows >= 4096:
        auto.setenv("NVFP4AP_KERNEL", "5")
        forced = _fp8_call(ap, op, d)
        assert torch.equal(out.view(torch.uint8), forced.view(torch.uint8)), "default is not the block-per-lane kernel"


@pytest.mark.parametrize("rows,dim", [(4095, 3072), (4224, 8192), (4096, 2560)])
def test_fp8_broadcast_default_keeps_persistent_kernel(ap, dev, auto, rows, dim):
    # below 4096 rows, at two rows per CTA (8192) and with idle lanes (2560)
    # the broadcast form stays on the persistent kernel: its bytes equal the
    # forced register kernels' (NVFP4AP_KERNEL=3)
    w, ref = _fp8_case("bcast", rows, dim, seed=rows)
    d = _d(w, dev)
    out = _fp8_call(ap, "bcast", d)
    check_fp8(_codes(out), ref, _act(w))
    auto.setenv("NVFP4AP_KERNEL", "3")
    forced = _fp8_call(ap, "bcast", d)
    assert torch.equal(out.view(torch.uint8), forced.view(torch.uint8))


def _exact_codes(rng, n):
    # |value| <= 1: decode * deq (deq with two significant bits) is a bf16 value
    mags = rng.integers(0, 0x39, n)
    return torch.from_numpy(((mags | (rng.integers(0, 2, n) << 7)).astype(np.uint8))).view(torch.float8_e4m3fn)


@pytest.mark.parametrize("rows,dim", [(4096, 1536), (4100, 3072), (2048, 1536), (2050, 5120)])
def test_sources_reduce_bit_for_bit(ap, dev, auto, rows, dim):
    rng = np.random.default_rng(rows * 7 + dim)
    x = synth.bf16(synth.normal(rows + dim, 0, (rows, dim), 1.0)).to(dev)
    s8, h8 = _exact_codes(rng, dim), _exact_codes(rng, dim)
    sdeq, hdeq = 0.375, 3.0
    scale_bf = (s8.float() * sdeq).to(torch.bfloat16)
    shift_bf = (h8.float() * hdeq).to(torch.bfloat16)
    assert torch.equal(scale_bf.float(), s8.float() * sdeq) and torch.equal(shift_bf.float(), h8.float() * hdeq)
    act = torch.tensor([0.025], device=dev)
    sd, hd = torch.tensor([sdeq], device=dev), torch.tensor([hdeq], device=dev)
    s8, h8, scale_bf, shift_bf = s8.to(dev), h8.to(dev), scale_bf.to(dev), shift_bf.to(dev)
    b = ap.ada_layer_norm_quant_fp8_bf16(x, scale_bf, shift_bf, act)
    a = ap.ada_layer_norm_quant_fp8_modfp8_bf16(x, s8, h8, sd, hd, act)
    one = torch.ones(dim, dtype=torch.bfloat16, device=dev)
    c = ap.awq_ada_layer_norm_quant_fp8_bf16(x, scale_bf, shift_bf, one, act)
    assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    assert torch.equal(c.view(torch.uint8), b.view(torch.uint8))
    pa, sa = ap.ada_layer_norm_quant_nvfp4_swizzled_modfp8_bf16(x, s8, h8, sd, hd)
    pb, sb = ap.ada_layer_norm_quant_nvfp4_swizzled_bf16(x, scale_bf, shift_bf)
    assert torch.equal(pa, pb) and torch.equal(sa, sb)


def _nv_call(ap, op, d, sf):
    if op == "ln":
        return ap.layer_norm_no_affine_quant_nvfp4_swizzled_bf16(d["x"], sf_swizzled=sf)
    if op == "bcast":
        return ap.ada_layer_norm_quant_nvfp4_swizzled_bf16(d["x"], d["scale"], d["shift"], sf_swizzled=sf)
    return ap.ada_layer_norm_quant_nvfp4_swizzled_modfp8_bf16(d["x"], d["scale_fp8"], d["shift_fp8"],
                                                              d["scale_deq"], d["shift_deq"], sf_swizzled=sf)


@pytest.mark.parametrize("op", ["ln", "bcast", "modfp8"])
@pytest.mark.parametrize("rows,dim", [(2047, 1536), (2048, 1536), (2177, 1024), (2051, 5120), (2100, 2560)])
def test_nvfp4_default(ap, dev, auto, op, rows, dim):
    seed = rows * 3 + dim
    if op == "ln":
        w = synth.nvfp4_ln(rows, dim, seed)
        x = synth.u16(w.inputs["x"])
        src, mod = {}, oracle.MOD_NONE
    elif op == "bcast":
        w = synth.nvfp4_broadcast(rows, dim, seed)
        x = synth.u16(w.inputs["x"])
        src, mod = dict(scale=synth.u16(w.inputs["scale"]), shift=synth.u16(w.inputs["shift"])), oracle.MOD_BCAST
    else:
        w = synth.nvfp4_modfp8(rows, dim, seed)
        x = synth.u16(w.inputs["x"])
        src = dict(scale_fp8=w.inputs["scale_fp8"].view(torch.uint8).numpy(),
                   shift_fp8=w.inputs["shift_fp8"].view(torch.uint8).numpy(),
                   scale_deq=float(w.inputs["scale_deq"][0]), shift_deq=float(w.inputs["shift_deq"][0]))
        mod = oracle.MOD_MODFP8
    d = _d(w, dev)
    n = ap.swizzled_sf_size(rows, dim)
    guard = 512
    sfbuf = torch.full((n + 2 * guard,), 0xFF, dtype=torch.uint8, device=dev)
    packed, _ = _nv_call(ap, op, d, sfbuf[guard:guard + n])
    sb = sfbuf.cpu().numpy()
    assert np.all(sb[:guard] == 0xFF) and np.all(sb[-guard:] == 0xFF)
    opk, osf = oracle.ln_quant_nvfp4(x, mod, **src)
    y = oracle.modulated(x, mod, **src)
    v = torch.from_numpy(y.astype(np.float32)).to(torch.bfloat16).double().numpy()
    check_nvfp4(packed.cpu().numpy(), sb[guard:guard + n], opk, osf, rows, dim, v, f"{op} {rows}x{dim}")
    if rows >= 2048 and dim != 2560:
        # the default is the block-per-lane kernel: same bytes as when forced
        auto.setenv("NVFP4AP_KERNEL", "5")
        fp, fs = _nv_call(ap, op, d, None)
        assert torch.equal(packed, fp) and torch.equal(sfbuf[guard:guard + n], fs)
