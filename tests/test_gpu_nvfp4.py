"""GPU parity of the NVFP4 producers against the oracle (through the C ABI).

Tolerance: tests/parity.py.  Cases span ragged rows (padding rows of the
last 128-row scale tile), dims whose block count is not a multiple of 4
(padding columns), one to several thread groups per row, the largest dim,
and adversarial blocks built from constant rows (y = shift exactly): every
e2m1 midpoint tie at many scales, signed zeros, all-zero blocks, subnormal
and saturated block scales.  The scale buffer is pre-filled with 0xFF so that
padding must be written, and is surrounded by guard bands.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import check_nvfp4, padding_mask

pytestmark = pytest.mark.gpu

SHAPES = [(1, 16), (3, 48), (127, 64), (129, 80), (300, 3072), (64, 5376), (128, 7168), (33, 14336),
          (5, 32768), (257, 1536), (51, 1152)]


def _run(ap, fn_kind, w, dev, guard=4096, sf_shift=0):
    rows, dim = w.rows, w.dim
    n = ap.swizzled_sf_size(rows, dim)
    sfbuf = torch.full((n + 2 * guard + sf_shift,), 0xFF, dtype=torch.uint8, device=dev)[sf_shift:]
    pkbuf = torch.full((rows * dim // 2 + 2 * guard,), 0xEE, dtype=torch.uint8, device=dev)
    sf = sfbuf[guard:guard + n]
    packed = pkbuf[guard:guard + rows * dim // 2].view(rows, dim // 2)
    x = w.inputs["x"].to(dev)
    if fn_kind == "bcast":
        ap.ada_layer_norm_quant_nvfp4_swizzled_bf16(x, w.inputs["scale"].to(dev), w.inputs["shift"].to(dev),
                                                    eps=w.params["eps"], packed=packed, sf_swizzled=sf)
    else:
        ap.layer_norm_no_affine_quant_nvfp4_swizzled_bf16(x, eps=w.params["eps"], packed=packed, sf_swizzled=sf)
    sb, pb = sfbuf.cpu().numpy(), pkbuf.cpu().numpy()
    assert np.all(sb[:guard] == 0xFF) and np.all(sb[-guard:] == 0xFF)
    assert np.all(pb[:guard] == 0xEE) and np.all(pb[-guard:] == 0xEE)
    return pb[guard:-guard].reshape(rows, dim // 2), sb[guard:-guard]


def _oracle(w, kind):
    x = synth.u16(w.inputs["x"])
    if kind == "bcast":
        mod = dict(scale=synth.u16(w.inputs["scale"]), shift=synth.u16(w.inputs["shift"]))
        k = oracle.MOD_BCAST
    else:
        mod, k = {}, oracle.MOD_NONE
    packed, sf = oracle.ln_quant_nvfp4(x, k, eps=w.params["eps"], **mod)
    y = oracle.modulated(x, k, eps=w.params["eps"], **mod)
    v = torch.from_numpy(y.astype(np.float32)).to(torch.bfloat16).double().numpy()
    return packed, sf, v


@pytest.mark.parametrize("rows,dim", SHAPES)
@pytest.mark.parametrize("kind", ["ln", "bcast"])
def test_nvfp4_parity(ap, dev, path, kind, rows, dim):
    w = (synth.nvfp4_broadcast if kind == "bcast" else synth.nvfp4_ln)(rows, dim, seed=rows * 3 + dim)
    gp, gs = _run(ap, kind, w, dev)
    op, os_, v = _oracle(w, kind)
    check_nvfp4(gp, gs, op, os_, rows, dim, v_orc=v)


def _crafted_rows():
    """Shift rows whose values are exact e2m1 ties and edge cases for many block scales."""
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    blocks = []
    # every midpoint at scales 1, 2^-9 (smallest subnormal e4m3), 0.375, 448 (largest)
    for s in (1.0, 2.0 ** -9, 0.375, 3.5, 448.0):
        b = np.concatenate([[6 * s], mids * s, -mids * s, [-6 * s]])
        blocks.append(b)
    blocks.append(np.zeros(16))                                          # all-zero block: scale 0
    blocks.append(np.array([-2.0 ** -100, 2.0 ** -100] + [0.0] * 14))    # underflowing block: signed zeros
    blocks.append(np.array([4000.0, -4000.0, 2560.0, 1.0] + [0.0] * 12))  # scale saturates at 448
    blocks.append(np.array([6.0, -0.125, 0.125, -2.875, 2.875, 2.0 ** -10] + [0.5] * 10))  # small values round to +-0
    # amax/6 = 1.0625 lies halfway between e4m3 1.0 and 1.125: the scale is 1.0
    blocks.append(np.array([6.375, 1, -1, 2, -3, 0.5, -0.5, 4, -4, 1.5, -1.5, 3, 0.25, 0.75, -5, 5.0]))
    v = np.concatenate(blocks)
    dim = int(np.ceil(v.size / 64) * 64)
    return np.concatenate([v, np.zeros(dim - v.size)]).astype(np.float32)


def test_nvfp4_exact_ties_and_edges(ap, dev, path):
    shift = _crafted_rows()
    dim = shift.size
    rows = 130  # ragged: two rows in the second 128-row tile
    x = synth.bf16(np.full((rows, dim), -2.5, dtype=np.float32))
    sh = synth.bf16(shift)
    assert np.array_equal(sh.float().numpy(), shift)  # every crafted value is exact in bf16
    sc = synth.bf16(np.zeros(dim, dtype=np.float32))
    w = synth.Workload("crafted", rows, dim, {"x": x, "scale": sc, "shift": sh}, {"eps": 1e-5})
    gp, gs = _run(ap, "bcast", w, dev)
    op, os_, _ = _oracle(w, "bcast")
    assert np.array_equal(gp, op), "crafted ties must be bit-exact"
    assert np.array_equal(gs, os_)
    assert not gs[padding_mask(rows, dim)].any()


def test_zero_modulation_equals_plain(ap, dev, path):
    w = synth.nvfp4_broadcast(200, 3072, seed=4)
    x = w.inputs["x"].to(dev)
    z = torch.zeros(3072, dtype=torch.bfloat16, device=dev)
    a = ap.ada_layer_norm_quant_nvfp4_swizzled_bf16(x, z, z)
    b = ap.layer_norm_no_affine_quant_nvfp4_swizzled_bf16(x)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_batch_invariance(ap, dev, path):
    w = synth.nvfp4_broadcast(640, 3072, seed=12)
    x, sc, sh = (w.inputs[k].to(dev) for k in ("x", "scale", "shift"))
    pk, sf = ap.ada_layer_norm_quant_nvfp4_swizzled_bf16(x, sc, sh)
    from parity import unswizzle
    full_p = pk.cpu().numpy()
    full_s = unswizzle(sf.cpu().numpy(), 640, 3072)
    for start, n in ((0, 1), (128, 128), (256, 300), (5, 77)):
        p2, s2 = ap.ada_layer_norm_quant_nvfp4_swizzled_bf16(x[start:start + n].contiguous(), sc, sh)
        assert np.array_equal(p2.cpu().numpy(), full_p[start:start + n])
        assert np.array_equal(unswizzle(s2.cpu().numpy(), n, 3072), full_s[start:start + n])


def test_misaligned_input_takes_the_element_wise_kernel(ap, dev):
    w = synth.nvfp4_ln(16, 64, seed=8)
    x = w.inputs["x"]
    ref_p, ref_s = oracle.ln_quant_nvfp4(synth.u16(x))
    for off in (8, 4, 1):  # 16-byte aligned (vector kernels), 8-byte, 2-byte (element-wise kernel)
        y = torch.zeros(16 * 64 + off, dtype=torch.bfloat16, device=dev)[off:].view(16, 64)
        y.copy_(x.to(dev))
        pk, sf = ap.layer_norm_no_affine_quant_nvfp4_swizzled_bf16(y)
        check_nvfp4(pk.cpu().numpy(), sf.cpu().numpy(), ref_p, ref_s, 16, 64, what=f"x offset {off}")


@pytest.mark.parametrize("kind", ["ln", "bcast"])
def test_tma_pipeline_many_rows_per_cta(ap, dev, kind, monkeypatch):
    rows, dim = 3000, 272   # 17 blocks per row: column padding; 3000 rows: row padding
    for ctas in (1, 2):  # persistent CTAs per SM: each walks many rows through its stages
        monkeypatch.setenv("NVFP4AP_KERNEL", f"4:{ctas}")
        w = (synth.nvfp4_broadcast if kind == "bcast" else synth.nvfp4_ln)(rows, dim, seed=ctas)
        gp, gs = _run(ap, kind, w, dev)
        op, os_, v = _oracle(w, kind)
        check_nvfp4(gp, gs, op, os_, rows, dim, v_orc=v)
    ap.take_device_fault()


@pytest.mark.parametrize("rows,dim", [(131, 2048), (3001, 4096), (257, 6144), (129, 8192), (77, 4608), (130, 3072)])
@pytest.mark.parametrize("kind", ["ln", "bcast"])
def test_rowblk_shapes(ap, dev, kind, rows, dim, monkeypatch):
    # the one-row-per-CTA block-per-lane kernel (the default where a row is
    # exactly 64-128 threads x 2-4 blocks): 2 (dims 2048, 4096), 3 (3072, 4608,
    # 6144) and 4 (8192) blocks per lane, 64-128 threads per row, ragged row
    # counts (padding rows of the last scale tile)
    monkeypatch.delenv("NVFP4AP_KERNEL", raising=False)
    w = (synth.nvfp4_broadcast if kind == "bcast" else synth.nvfp4_ln)(rows, dim, seed=rows + dim)
    gp, gs = _run(ap, kind, w, dev)
    op, os_, v = _oracle(w, kind)
    check_nvfp4(gp, gs, op, os_, rows, dim, v_orc=v)


@pytest.mark.parametrize("kind", ["ln", "bcast"])
def test_blk_many_rows_per_group(ap, dev, kind, monkeypatch):
    # block-per-lane kernels with one CTA per SM: every row group walks many
    # rows (prefetch buffer, parity slots); 17 and 192 blocks per row (one idle
    # lane range and an exact fit); 20000 rows (row padding of the last scale
    # tile)
    monkeypatch.setenv("NVFP4AP_KERNEL", "5:1")  # one CTA per SM: ~16 rows per row group
    for rows, dim in ((40000, 272), (20000, 3072)):
        w = (synth.nvfp4_broadcast if kind == "bcast" else synth.nvfp4_ln)(rows, dim, seed=dim)
        gp, gs = _run(ap, kind, w, dev)
        op, os_, v = _oracle(w, kind)
        check_nvfp4(gp, gs, op, os_, rows, dim, v_orc=v)


@pytest.mark.parametrize("kind", ["ln", "bcast"])
def test_unaligned_scale_buffer(ap, dev, kind):
    # a scale buffer off 16-byte alignment takes the byte-store path
    w = (synth.nvfp4_broadcast if kind == "bcast" else synth.nvfp4_ln)(300, 3072, seed=17)
    gp, gs = _run(ap, kind, w, dev, sf_shift=4)
    op, os_, v = _oracle(w, kind)
    check_nvfp4(gp, gs, op, os_, 300, 3072, v_orc=v)
