"""GPU parity of the LayerNorm producers on views that are only element-aligned.

The tensor contract (adaptive-layernorm-producers README, "Tensor Contract")
asks for contiguous tensors of the stated dtypes, not for any pointer
alignment, so a slice at an odd element offset is a valid argument.  The
library takes such pointers on its element-wise kernel (one load per element,
byte stores); these tests give every LayerNorm form inputs at odd element
offsets and outputs at odd byte offsets, over ragged shapes, and compare with
the oracle (tolerance: tests/parity.py).  Guard bytes around each output must
stay untouched.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import check_fp8, check_nvfp4

pytestmark = pytest.mark.gpu

GUARD = 64


def _off(t: torch.Tensor, dev, elems: int = 1) -> torch.Tensor:
    """The same values, contiguous, starting `elems` elements past an aligned base."""
    buf = torch.empty(t.numel() + elems + 16, dtype=t.dtype, device=dev)
    v = buf[elems:elems + t.numel()].view(t.shape)
    v.copy_(t.to(dev))
    return v


def _out(nbytes: int, dev, off: int = 3):
    """A uint8 output at an odd byte offset with guard bands filled with 0xA5."""
    buf = torch.full((nbytes + 2 * GUARD + off,), 0xA5, dtype=torch.uint8, device=dev)
    return buf, buf[GUARD + off:GUARD + off + nbytes]


def _guards_ok(buf, nbytes, off=3):
    b = buf.cpu().numpy()
    return bool((b[:GUARD + off] == 0xA5).all() and (b[GUARD + off + nbytes:] == 0xA5).all())


def _act(w):
    return float(w.inputs["act_scale"][0])


FP8_CASES = [(37, 1536), (130, 3072), (5, 2050), (3, 64), (129, 1000)]


@pytest.mark.parametrize("form", ["ln", "bcast", "ptok", "table", "modfp8", "awq", "seg"])
@pytest.mark.parametrize("rows,dim", FP8_CASES)
def test_fp8_element_aligned(ap, dev, form, rows, dim):
    seed = rows * 7 + dim
    if form == "table":
        w = synth.fp8_table(rows, dim, seed, chunks=4, shift_idx=3, scale_idx=1)
    elif form == "modfp8":
        w = synth.fp8_modfp8(rows, dim, seed)
    elif form == "awq":
        w = synth.fp8_awq(rows, dim, seed)
    elif form == "seg":
        w = synth.segmented(rows, dim, seed, nseg=3)
    elif form == "ptok":
        w = synth.fp8_ptok(rows, dim, seed)
    else:
        w = synth.fp8_broadcast(rows, dim, seed, outliers=0.05)
    I = w.inputs
    act = I["act_scale"].to(dev)
    x = _off(I["x"], dev)
    buf, o = _out(rows * dim, dev)
    out = o.view(torch.float8_e4m3fn).view(rows, dim)
    u = lambda k: synth.u16(I[k])
    if form == "ln":
        ap.layer_norm_no_affine_quant_fp8_static_bf16(x, act, out=out)
        ref = oracle.ln_quant_fp8(u("x"), _act(w), oracle.MOD_NONE)
    elif form == "bcast":
        ap.ada_layer_norm_quant_fp8_bf16(x, _off(I["scale"], dev), _off(I["shift"], dev), act, out=out)
        ref = oracle.ln_quant_fp8(u("x"), _act(w), oracle.MOD_BCAST, scale=u("scale"), shift=u("shift"))
    elif form == "ptok":
        ap.ada_layer_norm_quant_fp8_ptok_bf16(x, _off(I["scale"], dev), _off(I["shift"], dev), act, out=out)
        ref = oracle.ln_quant_fp8(u("x"), _act(w), oracle.MOD_PTOK, scale=u("scale"), shift=u("shift"))
    elif form == "table":
        ap.ada_layer_norm_quant_fp8_ptok_table_bf16(x, _off(I["temb"], dev), _off(I["table"], dev), act, 3, 1,
                                                    out=out)
        ref = oracle.ln_quant_fp8(u("x"), _act(w), oracle.MOD_TABLE, temb=u("temb"), table=I["table"].numpy(),
                                  shift_idx=3, scale_idx=1)
    elif form == "modfp8":
        ap.ada_layer_norm_quant_fp8_modfp8_bf16(x, _off(I["scale_fp8"], dev, 3), _off(I["shift_fp8"], dev, 5),
                                                I["scale_deq"].to(dev), I["shift_deq"].to(dev), act, out=out)
        ref = oracle.ln_quant_fp8(u("x"), _act(w), oracle.MOD_MODFP8,
                                  scale_fp8=I["scale_fp8"].view(torch.uint8).numpy(),
                                  shift_fp8=I["shift_fp8"].view(torch.uint8).numpy(),
                                  scale_deq=float(I["scale_deq"][0]), shift_deq=float(I["shift_deq"][0]))
    elif form == "awq":
        ap.awq_ada_layer_norm_quant_fp8_bf16(x, _off(I["scale"], dev), _off(I["shift"], dev), _off(I["inv_s"], dev),
                                             act, out=out)
        ref = oracle.ln_quant_fp8(u("x"), _act(w), oracle.MOD_AWQ, scale=u("scale"), shift=u("shift"),
                                  inv_s=u("inv_s"))
    else:
        idx = I["seg_idx"].to(dev)
        ap.ada_layer_norm_quant_fp8_seg_bf16(x, idx, _off(I["seg_scale"], dev), _off(I["seg_shift"], dev), act,
                                             out=out)
        ref = oracle.ln_quant_fp8(u("x"), _act(w), oracle.MOD_SEG, seg_idx=I["seg_idx"].numpy(),
                                  seg_scale=u("seg_scale"), seg_shift=u("seg_shift"))
    torch.cuda.synchronize()
    check_fp8(o.cpu().numpy().reshape(rows, dim), ref, _act(w), f"fp8 {form} {rows}x{dim} element-aligned")
    assert _guards_ok(buf, rows * dim), "guard bytes written"


NV_CASES = [(37, 1536), (130, 3072), (3, 64), (129, 272)]


@pytest.mark.parametrize("form", ["ln", "bcast", "modfp8", "seg"])
@pytest.mark.parametrize("rows,dim", NV_CASES)
def test_nvfp4_element_aligned(ap, dev, form, rows, dim):
    seed = rows * 11 + dim
    if form == "modfp8":
        w = synth.nvfp4_modfp8(rows, dim, seed)
    elif form == "seg":
        w = synth.segmented(rows, dim, seed, nseg=3)
    else:
        w = synth.nvfp4_broadcast(rows, dim, seed)
    I = w.inputs
    u = lambda k: synth.u16(I[k])
    x = _off(I["x"], dev)
    nsf = ap.swizzled_sf_size(rows, dim)
    pbuf, pk = _out(rows * dim // 2, dev, 5)
    sbuf, sf = _out(nsf, dev, 1)
    pk2 = pk.view(rows, dim // 2)
    if form == "ln":
        ap.layer_norm_no_affine_quant_nvfp4_swizzled_bf16(x, packed=pk2, sf_swizzled=sf)
        mk, mod = oracle.MOD_NONE, {}
    elif form == "bcast":
        ap.ada_layer_norm_quant_nvfp4_swizzled_bf16(x, _off(I["scale"], dev), _off(I["shift"], dev), packed=pk2,
                                                    sf_swizzled=sf)
        mk, mod = oracle.MOD_BCAST, dict(scale=u("scale"), shift=u("shift"))
    elif form == "modfp8":
        ap.ada_layer_norm_quant_nvfp4_swizzled_modfp8_bf16(x, _off(I["scale_fp8"], dev, 1), _off(I["shift_fp8"], dev, 7),
                                                           I["scale_deq"].to(dev), I["shift_deq"].to(dev), packed=pk2,
                                                           sf_swizzled=sf)
        mk = oracle.MOD_MODFP8
        mod = dict(scale_fp8=I["scale_fp8"].view(torch.uint8).numpy(), shift_fp8=I["shift_fp8"].view(torch.uint8).numpy(),
                   scale_deq=float(I["scale_deq"][0]), shift_deq=float(I["shift_deq"][0]))
    else:
        ap.ada_layer_norm_quant_nvfp4_swizzled_seg_bf16(x, I["seg_idx"].to(dev), _off(I["seg_scale"], dev),
                                                        _off(I["seg_shift"], dev), packed=pk2, sf_swizzled=sf)
        mk = oracle.MOD_SEG
        mod = dict(seg_idx=I["seg_idx"].numpy(), seg_scale=u("seg_scale"), seg_shift=u("seg_shift"))
    torch.cuda.synchronize()
    op, os_ = oracle.ln_quant_nvfp4(u("x"), mk, **mod)
    y = oracle.modulated(u("x"), mk, **mod)
    v = torch.from_numpy(y.astype(np.float32)).to(torch.bfloat16).double().numpy()
    check_nvfp4(pk2.cpu().numpy(), sf.cpu().numpy(), op, os_, rows, dim, v_orc=v,
                what=f"nvfp4 {form} {rows}x{dim} element-aligned")
    assert _guards_ok(pbuf, rows * dim // 2, 5) and _guards_ok(sbuf, nsf, 1), "guard bytes written"


def test_out_of_range_segment_index_on_the_element_wise_kernel(ap, dev):
    rows, dim = 40, 1000  # dim % 8 != 0: the element-wise kernel
    w = synth.segmented(rows, dim, 5, nseg=3)
    I = w.inputs
    idx = I["seg_idx"].clone()
    idx[7] = 3  # outside [0, nseg)
    ap.take_device_fault()
    out = ap.ada_layer_norm_quant_fp8_seg_bf16(I["x"].to(dev), idx.to(dev), I["seg_scale"].to(dev),
                                               I["seg_shift"].to(dev), I["act_scale"].to(dev))
    torch.cuda.synchronize()
    with pytest.raises(ap.NvFp4ApError) as e:
        ap.take_device_fault()
    assert e.value.status == ap.ERR_FAULT
    # the bad row is produced with zero modulation: the plain layer norm's codes
    plain = oracle.ln_quant_fp8(synth.u16(I["x"][7:8]), _act(w), oracle.MOD_NONE)
    check_fp8(out.view(torch.uint8).cpu().numpy()[7:8], plain, _act(w), "bad segment row")
