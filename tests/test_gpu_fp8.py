"""GPU parity of the FP8 producers against the oracle (through the C ABI).

Tolerance: tests/parity.py (>= 99.9% equal codes, every mismatch one code
step, row-wise relative error of the dequantised output below 1e-2).  Cases
span one to many thread groups per row, ragged rows, the bf16-pair path
(dim not a multiple of 8, or pointers off 16-byte alignment), the largest
dim, constant rows whose outputs are exact ties, saturation, rows = 0,
guard bands around the output, batch invariance, a side stream and a CUDA
graph capture.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import check_fp8

pytestmark = pytest.mark.gpu

SHAPES = [(1, 32), (3, 48), (8, 2), (40, 16), (127, 1536), (129, 3072), (300, 2048), (64, 2050),
          (17, 1152), (51, 1536), (5, 32768), (33, 6144), (9, 10240)]


def _codes(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.uint8).cpu().numpy()


def _d(w, dev):
    return {k: v.to(dev) for k, v in w.inputs.items()}


def _act(w):
    return float(w.inputs["act_scale"][0])


@pytest.mark.parametrize("rows,dim", SHAPES)
def test_layer_norm_fp8(ap, dev, path, rows, dim):
    w = synth.fp8_ln(rows, dim, seed=rows * 31 + dim)
    d = _d(w, dev)
    out = ap.layer_norm_no_affine_quant_fp8_static_bf16(d["x"], d["act_scale"], eps=1e-5)
    ref = oracle.ln_quant_fp8(synth.u16(w.inputs["x"]), _act(w), oracle.MOD_NONE, eps=1e-5)
    check_fp8(_codes(out), ref, _act(w))


@pytest.mark.parametrize("rows,dim", SHAPES)
def test_broadcast_fp8(ap, dev, path, rows, dim):
    w = synth.fp8_broadcast(rows, dim, seed=rows * 17 + dim, outliers=0.05)
    d = _d(w, dev)
    out = ap.ada_layer_norm_quant_fp8_bf16(d["x"], d["scale"], d["shift"], d["act_scale"])
    u = {k: synth.u16(w.inputs[k]) for k in ("x", "scale", "shift")}
    ref = oracle.ln_quant_fp8(u["x"], _act(w), oracle.MOD_BCAST, scale=u["scale"], shift=u["shift"])
    check_fp8(_codes(out), ref, _act(w))


@pytest.mark.parametrize("rows,dim", SHAPES)
def test_per_token_fp8(ap, dev, path, rows, dim):
    w = synth.fp8_ptok(rows, dim, seed=rows * 13 + dim)
    d = _d(w, dev)
    out = ap.ada_layer_norm_quant_fp8_ptok_bf16(d["x"], d["scale"], d["shift"], d["act_scale"])
    u = {k: synth.u16(w.inputs[k]) for k in ("x", "scale", "shift")}
    ref = oracle.ln_quant_fp8(u["x"], _act(w), oracle.MOD_PTOK, scale=u["scale"], shift=u["shift"])
    check_fp8(_codes(out), ref, _act(w))


@pytest.mark.parametrize("rows,dim,chunks,si,ci", [(1, 32, 6, 0, 1), (129, 3072, 6, 0, 1), (77, 1536, 6, 4, 2),
                                                   (64, 2050, 3, 2, 2), (300, 2048, 2, 1, 0), (5, 32768, 6, 5, 3)])
def test_table_fp8(ap, dev, path, rows, dim, chunks, si, ci):
    w = synth.fp8_table(rows, dim, seed=rows * 7 + dim, chunks=chunks, shift_idx=si, scale_idx=ci)
    d = _d(w, dev)
    out = ap.ada_layer_norm_quant_fp8_ptok_table_bf16(d["x"], d["temb"], d["table"], d["act_scale"], si, ci)
    ref = oracle.ln_quant_fp8(synth.u16(w.inputs["x"]), _act(w), oracle.MOD_TABLE,
                              temb=synth.u16(w.inputs["temb"]), table=w.inputs["table"].numpy(),
                              shift_idx=si, scale_idx=ci)
    check_fp8(_codes(out), ref, _act(w))


def _offset_view(t: torch.Tensor, elems: int) -> torch.Tensor:
    """Same values, contiguous, data pointer moved by `elems` elements."""
    buf = torch.empty(t.numel() + elems + 8, dtype=t.dtype, device=t.device)
    v = buf[elems:elems + t.numel()].view(t.shape)
    v.copy_(t)
    return v


def test_pair_path_when_off_16_byte_alignment(ap, dev):
    w = synth.fp8_ptok(65, 1536, seed=99)
    d = _d(w, dev)
    x, sc, sh = (_offset_view(d[k], 2) for k in ("x", "scale", "shift"))  # 4-byte aligned only
    assert x.data_ptr() % 16 != 0
    out = torch.empty(65 * 1536 + 2, dtype=torch.uint8, device=dev)[2:].view(torch.float8_e4m3fn).view(65, 1536)
    ap.ada_layer_norm_quant_fp8_ptok_bf16(x, sc, sh, d["act_scale"], out=out)
    u = {k: synth.u16(w.inputs[k]) for k in ("x", "scale", "shift")}
    ref = oracle.ln_quant_fp8(u["x"], _act(w), oracle.MOD_PTOK, scale=u["scale"], shift=u["shift"])
    check_fp8(_codes(out), ref, _act(w))
    # an odd element offset (2-byte aligned) takes the element-wise kernel
    out = ap.ada_layer_norm_quant_fp8_ptok_bf16(_offset_view(d["x"], 1), sc, sh, d["act_scale"])
    check_fp8(_codes(out), ref, _act(w), "odd element offset")


def _constant_rows_with_shift(shift_vals: np.ndarray, rows: int):
    dim = shift_vals.size
    x = synth.bf16(np.full((rows, dim), 0.75, dtype=np.float32))
    sh = synth.bf16(shift_vals.astype(np.float32))
    sc = synth.bf16(np.zeros(dim, dtype=np.float32))
    return x, sc, sh


def test_fp8_exact_ties_on_constant_rows(ap, dev, path):
    # constant rows normalise to exactly 0, so y = shift; act_scale = 0.5 is a
    # power of two, so y / act_scale is exact and every midpoint between two
    # e4m3 values is a tie that must round to the even code
    t = oracle.e4m3_table()[:0x7F]
    mids = (t[:-1] + t[1:]) / 2 * 0.5
    vals = np.concatenate([mids, -mids, t * 0.5, [300.0, -300.0, 2.0 ** -100, -(2.0 ** -100), 0.0]])
    dim = int(np.ceil(vals.size / 64) * 64)
    vals = np.concatenate([vals, np.zeros(dim - vals.size)])
    x, sc, sh = _constant_rows_with_shift(vals, 3)
    act = torch.tensor([0.5], dtype=torch.float32)
    out = ap.ada_layer_norm_quant_fp8_bf16(x.to(dev), sc.to(dev), sh.to(dev), act.to(dev))
    ref = oracle.ln_quant_fp8(synth.u16(x), 0.5, oracle.MOD_BCAST, scale=synth.u16(sc), shift=synth.u16(sh))
    assert np.array_equal(_codes(out), ref)
    # saturation to +-448 and signed zero are part of it
    assert (ref == 0x7E).any() and (ref == 0xFE).any() and (ref == 0x80).any()


def test_rows_zero_is_a_no_op(ap, dev):
    x = torch.empty((0, 64), dtype=torch.bfloat16, device=dev)
    act = torch.tensor([0.025], device=dev)
    out = ap.layer_norm_no_affine_quant_fp8_static_bf16(x, act)
    assert out.shape == (0, 64)
    torch.cuda.synchronize()


def test_guard_bands_untouched(ap, dev):
    rows, dim = 129, 3072
    w = synth.fp8_broadcast(rows, dim, seed=5)
    d = _d(w, dev)
    pad = 4096
    buf = torch.full((rows * dim + 2 * pad,), 0xA5, dtype=torch.uint8, device=dev)
    out = buf[pad:pad + rows * dim].view(torch.float8_e4m3fn).view(rows, dim)
    ap.ada_layer_norm_quant_fp8_bf16(d["x"], d["scale"], d["shift"], d["act_scale"], out=out)
    b = buf.cpu().numpy()
    assert np.all(b[:pad] == 0xA5) and np.all(b[-pad:] == 0xA5)


def test_batch_invariance(ap, dev, path):
    w = synth.fp8_broadcast(1024, 3072, seed=77)
    d = _d(w, dev)
    full = _codes(ap.ada_layer_norm_quant_fp8_bf16(d["x"], d["scale"], d["shift"], d["act_scale"]))
    for n in (1, 7, 128, 333, 1000):
        for start in (0, 24):
            part = _codes(ap.ada_layer_norm_quant_fp8_bf16(d["x"][start:start + n].contiguous(), d["scale"],
                                                          d["shift"], d["act_scale"]))
            assert np.array_equal(part, full[start:start + n])


def test_side_stream_and_graph_capture(ap, dev, path):
    w = synth.fp8_table(256, 3072, seed=8)
    d = _d(w, dev)
    ref = _codes(ap.ada_layer_norm_quant_fp8_ptok_table_bf16(d["x"], d["temb"], d["table"], d["act_scale"], 0, 1))
    s = torch.cuda.Stream(device=dev)
    out = torch.empty((256, 3072), dtype=torch.float8_e4m3fn, device=dev)
    with torch.cuda.stream(s):
        ap.ada_layer_norm_quant_fp8_ptok_table_bf16(d["x"], d["temb"], d["table"], d["act_scale"], 0, 1, out=out)
    s.synchronize()
    assert np.array_equal(_codes(out), ref)
    g = torch.cuda.CUDAGraph()
    out2 = torch.zeros_like(out)
    with torch.cuda.graph(g):
        ap.ada_layer_norm_quant_fp8_ptok_table_bf16(d["x"], d["temb"], d["table"], d["act_scale"], 0, 1, out=out2)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(_codes(out2), ref)


@pytest.mark.parametrize("rows,dim", [(40000, 256), (6000, 3072)])
def test_noalloc_ring_wraps_many_rows_per_warp(ap, dev, rows, dim):
    # the allocation-free producer's warp-per-row ring kernel: with more rows
    # than warps in its persistent grid every warp walks several rows, so each
    # stage's mbarrier goes through many phases and refills
    import ctypes
    w = synth.fp8_broadcast(rows, dim, seed=rows % 97)
    d = _d(w, dev)
    out = torch.empty((rows, dim), dtype=torch.uint8, device=dev)
    rc = ap._load().ada_layer_norm_quant_fp8_bf16_noalloc(
        d["x"].data_ptr(), d["scale"].data_ptr(), d["shift"].data_ptr(), d["act_scale"].data_ptr(),
        ctypes.c_float(1e-5), out.data_ptr(), rows, dim, torch.cuda.current_stream(dev).cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    u = {k: synth.u16(w.inputs[k]) for k in ("x", "scale", "shift")}
    ref = oracle.ln_quant_fp8(u["x"], _act(w), oracle.MOD_BCAST, scale=u["scale"], shift=u["shift"])
    check_fp8(out.cpu().numpy(), ref, _act(w))
    words = ap.noalloc_progress()
    assert sum(words) == rows and len(words) * 8 < rows  # every warp had several rows
    ap.take_device_fault()  # no bounded wait ran out


@pytest.mark.parametrize("rows,dim", [(131, 2048), (3001, 4096), (257, 6144), (129, 8192), (77, 4608), (1, 3072)])
def test_rowblk_layer_norm_shapes(ap, dev, rows, dim, monkeypatch):
    # the FP8 layer norm on the one-row-per-CTA block-per-lane kernel (its
    # default where a row is exactly 64-128 threads x 2-4 blocks): 3 blocks per
    # lane at dims 3072, 4608, 6144, 2 at 2048 and 4096, 4 at 8192
    monkeypatch.delenv("NVFP4AP_KERNEL", raising=False)
    w = synth.fp8_ln(rows, dim, seed=rows + dim)
    d = _d(w, dev)
    out = ap.layer_norm_no_affine_quant_fp8_static_bf16(d["x"], d["act_scale"])
    ref = oracle.ln_quant_fp8(synth.u16(w.inputs["x"]), _act(w), oracle.MOD_NONE)
    check_fp8(_codes(out), ref, _act(w))


@pytest.mark.parametrize("op", ["bcast", "modfp8", "awq"])
def test_rowblk_broadcast_sources_when_forced(ap, dev, op, monkeypatch):
    # the FP8 broadcast sources on the same kernel (NVFP4AP_KERNEL=8)
    monkeypatch.setenv("NVFP4AP_KERNEL", "8")
    rows, dim = 517, 3072
    if op == "bcast":
        w = synth.fp8_broadcast(rows, dim, seed=5)
        d = _d(w, dev)
        out = ap.ada_layer_norm_quant_fp8_bf16(d["x"], d["scale"], d["shift"], d["act_scale"])
        u = {k: synth.u16(w.inputs[k]) for k in ("x", "scale", "shift")}
        ref = oracle.ln_quant_fp8(u["x"], _act(w), oracle.MOD_BCAST, scale=u["scale"], shift=u["shift"])
    elif op == "modfp8":
        w = synth.fp8_modfp8(rows, dim, seed=6)
        d = _d(w, dev)
        out = ap.ada_layer_norm_quant_fp8_modfp8_bf16(d["x"], d["scale_fp8"], d["shift_fp8"], d["scale_deq"],
                                                      d["shift_deq"], d["act_scale"])
        src = dict(scale_fp8=w.inputs["scale_fp8"].view(torch.uint8).numpy(),
                   shift_fp8=w.inputs["shift_fp8"].view(torch.uint8).numpy(),
                   scale_deq=float(w.inputs["scale_deq"][0]), shift_deq=float(w.inputs["shift_deq"][0]))
        ref = oracle.ln_quant_fp8(synth.u16(w.inputs["x"]), _act(w), oracle.MOD_MODFP8, **src)
    else:
        w = synth.fp8_awq(rows, dim, seed=7)
        d = _d(w, dev)
        out = ap.awq_ada_layer_norm_quant_fp8_bf16(d["x"], d["scale"], d["shift"], d["inv_s"], d["act_scale"])
        u = {k: synth.u16(w.inputs[k]) for k in ("x", "scale", "shift", "inv_s")}
        ref = oracle.ln_quant_fp8(u["x"], _act(w), oracle.MOD_AWQ, scale=u["scale"], shift=u["shift"],
                                  inv_s=u["inv_s"])
    check_fp8(_codes(out), ref, _act(w))


@pytest.mark.parametrize("op", ["ln", "bcast"])
def test_blk_many_rows_per_group(ap, dev, op, monkeypatch):
    # block-per-lane kernels with one CTA per SM: every row group walks many
    # rows (prefetch buffer, parity slots); 17 and 192 blocks per row
    monkeypatch.setenv("NVFP4AP_KERNEL", "5:1")  # one CTA per SM: ~16 rows per row group
    for ctas, (rows, dim) in enumerate(((40000, 272), (20000, 3072))):
        if op == "bcast":
            w = synth.fp8_broadcast(rows, dim, seed=ctas)
            d = _d(w, dev)
            out = ap.ada_layer_norm_quant_fp8_bf16(d["x"], d["scale"], d["shift"], d["act_scale"])
            u = {k: synth.u16(w.inputs[k]) for k in ("x", "scale", "shift")}
            ref = oracle.ln_quant_fp8(u["x"], _act(w), oracle.MOD_BCAST, scale=u["scale"], shift=u["shift"])
        else:
            w = synth.fp8_ln(rows, dim, seed=ctas)
            d = _d(w, dev)
            out = ap.layer_norm_no_affine_quant_fp8_static_bf16(d["x"], d["act_scale"])
            ref = oracle.ln_quant_fp8(synth.u16(w.inputs["x"]), _act(w), oracle.MOD_NONE)
        check_fp8(_codes(out), ref, _act(w))


@pytest.mark.parametrize("op", ["ln", "bcast", "ptok", "table"])
def test_tma_pipeline_many_rows_per_cta(ap, dev, op, monkeypatch):
    # one and two CTAs per SM: each CTA walks ~20-40 rows, so every stage's
    # mbarrier goes through many phases and refills
    rows, dim = 6000, 1024
    for ctas in (1, 2):
        monkeypatch.setenv("NVFP4AP_KERNEL", f"4:{ctas}")
        seed = 40 + ctas
        if op == "table":
            w = synth.fp8_table(rows, dim, seed=seed, shift_idx=4, scale_idx=2)
            d = _d(w, dev)
            out = ap.ada_layer_norm_quant_fp8_ptok_table_bf16(d["x"], d["temb"], d["table"], d["act_scale"], 4, 2)
            ref = oracle.ln_quant_fp8(synth.u16(w.inputs["x"]), _act(w), oracle.MOD_TABLE,
                                      temb=synth.u16(w.inputs["temb"]), table=w.inputs["table"].numpy(),
                                      shift_idx=4, scale_idx=2)
        elif op == "ptok":
            w = synth.fp8_ptok(rows, dim, seed=seed)
            d = _d(w, dev)
            out = ap.ada_layer_norm_quant_fp8_ptok_bf16(d["x"], d["scale"], d["shift"], d["act_scale"])
            u = {k: synth.u16(w.inputs[k]) for k in ("x", "scale", "shift")}
            ref = oracle.ln_quant_fp8(u["x"], _act(w), oracle.MOD_PTOK, scale=u["scale"], shift=u["shift"])
        elif op == "bcast":
            w = synth.fp8_broadcast(rows, dim, seed=seed)
            d = _d(w, dev)
            out = ap.ada_layer_norm_quant_fp8_bf16(d["x"], d["scale"], d["shift"], d["act_scale"])
            u = {k: synth.u16(w.inputs[k]) for k in ("x", "scale", "shift")}
            ref = oracle.ln_quant_fp8(u["x"], _act(w), oracle.MOD_BCAST, scale=u["scale"], shift=u["shift"])
        else:
            w = synth.fp8_ln(rows, dim, seed=seed)
            d = _d(w, dev)
            out = ap.layer_norm_no_affine_quant_fp8_static_bf16(d["x"], d["act_scale"])
            ref = oracle.ln_quant_fp8(synth.u16(w.inputs["x"]), _act(w), oracle.MOD_NONE)
        check_fp8(_codes(out), ref, _act(w))
    ap.take_device_fault()
