"""The NVFP4 producers' outputs feed a block-scaled GEMM unchanged.

The producers write e2m1 codes two per byte and e4m3 16-element block scales
in the 128x4 tiled layout (adaptive-layernorm-producers README, "Tensor
Contract": the "FlashRT/CUTLASS 128x4 swizzled uint8 scale layout").  Here
the packed codes and the swizzled scale buffers of two producer calls -- an
activation (rows, K) and a weight-like matrix (N, K) -- go straight into
cuBLASLt's NVFP4 block-scaled GEMM (through torch._scaled_mm, which takes
the scales in that tiled layout), and the product is compared with a float64
GEMM of the same codes and scales decoded by the oracle and placed by the
oracle's own offset formula.  A wrong nibble order, swizzle permutation or
padding would give O(1) errors; the bound below only allows the GEMM's fp32
accumulation and bf16 output rounding.

The same pair also runs as one CUDA graph (producer, then GEMM on the same
stream), the form in which the producer precedes its consumer in a model.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import unswizzle

pytestmark = pytest.mark.gpu


def _need_fp4():
    if not hasattr(torch, "float4_e2m1fn_x2"):
        pytest.skip("this torch build has no float4_e2m1fn_x2 dtype (no NVFP4 scaled GEMM)")


def _decode(packed: np.ndarray, sf: np.ndarray, rows: int, dim: int) -> np.ndarray:
    codes = oracle.unpack_e2m1(packed)
    scales = unswizzle(sf, rows, dim)
    return (oracle.e2m1_table()[codes].reshape(rows, dim // 16, 16) *
            oracle.e4m3_table()[scales][..., None]).reshape(rows, dim)


def _gemm(a_pk, a_sf, b_pk, b_sf):
    a = a_pk.view(torch.float4_e2m1fn_x2)
    b = b_pk.view(torch.float4_e2m1fn_x2)
    return torch._scaled_mm(a, b.t(), a_sf.view(torch.float8_e4m3fn), b_sf.view(torch.float8_e4m3fn),
                            out_dtype=torch.bfloat16)


@pytest.mark.parametrize("m,n,k", [(256, 384, 3072), (129, 256, 2048), (512, 128, 1536)])
def test_block_scaled_gemm_consumes_producer_layout(ap, dev, m, n, k):
    _need_fp4()
    wa = synth.nvfp4_broadcast(m, k, seed=m + k)
    wb = synth.nvfp4_ln(n, k, seed=n + 7 * k)
    a_pk, a_sf = ap.ada_layer_norm_quant_nvfp4_swizzled_bf16(wa.inputs["x"].to(dev), wa.inputs["scale"].to(dev),
                                                             wa.inputs["shift"].to(dev))
    b_pk, b_sf = ap.layer_norm_no_affine_quant_nvfp4_swizzled_bf16(wb.inputs["x"].to(dev))
    d = _gemm(a_pk, a_sf, b_pk, b_sf).float().cpu().numpy()
    A = _decode(a_pk.cpu().numpy(), a_sf.cpu().numpy(), m, k)
    B = _decode(b_pk.cpu().numpy(), b_sf.cpu().numpy(), n, k)
    ref = A @ B.T
    mag = np.abs(A) @ np.abs(B).T
    err = np.abs(d - ref)
    # bf16 output rounding (2^-9 relative) plus fp32 accumulation over k terms
    assert np.all(err <= 2.0 ** -8 * np.abs(ref) + 1e-5 * mag + 1e-30), float((err / (mag + 1e-30)).max())
    rel = np.linalg.norm(d - ref) / np.linalg.norm(ref)
    assert rel < 5e-3, rel


def test_producer_then_gemm_in_one_graph(ap, dev):
    _need_fp4()
    m, n, k = 256, 256, 3072
    wa = synth.nvfp4_broadcast(m, k, seed=31)
    wb = synth.nvfp4_ln(n, k, seed=32)
    x, sc, sh = (wa.inputs[key].to(dev) for key in ("x", "scale", "shift"))
    b_pk, b_sf = ap.layer_norm_no_affine_quant_nvfp4_swizzled_bf16(wb.inputs["x"].to(dev))
    a_pk = torch.empty((m, k // 2), dtype=torch.uint8, device=dev)
    a_sf = torch.empty((ap.swizzled_sf_size(m, k),), dtype=torch.uint8, device=dev)
    st = torch.cuda.Stream(dev)
    with torch.cuda.stream(st):
        ap.ada_layer_norm_quant_nvfp4_swizzled_bf16(x, sc, sh, packed=a_pk, sf_swizzled=a_sf)
        eager = _gemm(a_pk, a_sf, b_pk, b_sf)
        st.synchronize()
        a_pk.zero_()
        a_sf.fill_(0xFF)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            ap.ada_layer_norm_quant_nvfp4_swizzled_bf16(x, sc, sh, packed=a_pk, sf_swizzled=a_sf)
            out = _gemm(a_pk, a_sf, b_pk, b_sf)
        g.replay()
    st.synchronize()
    assert torch.equal(out, eager)


def test_other_scale_layouts_are_rejected_by_the_bound(ap, dev):
    # the same scale bytes placed row-major (unswizzled, padded) or with the
    # 32-row groups of each tile exchanged must break the bound above: the
    # GEMM really reads the tiled layout the producers write
    _need_fp4()
    m, n, k = 256, 256, 3072
    wa = synth.nvfp4_broadcast(m, k, seed=41)
    wb = synth.nvfp4_ln(n, k, seed=42)
    a_pk, a_sf = ap.ada_layer_norm_quant_nvfp4_swizzled_bf16(wa.inputs["x"].to(dev), wa.inputs["scale"].to(dev),
                                                             wa.inputs["shift"].to(dev))
    b_pk, b_sf = ap.layer_norm_no_affine_quant_nvfp4_swizzled_bf16(wb.inputs["x"].to(dev))
    A = _decode(a_pk.cpu().numpy(), a_sf.cpu().numpy(), m, k)
    B = _decode(b_pk.cpu().numpy(), b_sf.cpu().numpy(), n, k)
    ref = A @ B.T
    logical = unswizzle(a_sf.cpu().numpy(), m, k)                       # (m, k/16)
    row_major = np.zeros(a_sf.numel(), dtype=np.uint8)
    row_major[:logical.size] = logical.reshape(-1)
    tiles = a_sf.cpu().numpy().reshape(-1, 32, 4, 4)                     # [tile][r%32][group][col]
    swapped = tiles[:, :, [1, 0, 3, 2], :].reshape(-1)
    for wrong in (row_major, swapped):
        d = _gemm(a_pk, torch.from_numpy(np.ascontiguousarray(wrong)).to(dev), b_pk, b_sf).float().cpu().numpy()
        rel = np.linalg.norm(d - ref) / np.linalg.norm(ref)
        assert rel > 0.1, rel
