"""GPU parity of the SwiGLU producers (C ABI).

v = bf16(bf16(silu(gate)) * up) (h3-blackwell-runtime compare page,
NVFP4_SWIGLU_FUSION_DESIGN.md), then the two-level NVFP4 contract.  The
staged values must equal the oracle's bit for bit (swiglu_bf16): every
finite bf16 gate pattern (times one and times random ups), random gates,
gates whose binary32 silu lies within 16 ulp of a bf16 rounding midpoint,
gates beyond the fp32 exponential's range, both memory layouts (two tensors,
halves of one).  The two-level outputs follow tests/parity.py with the
tensor scale exact.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import check_nvfp4

pytestmark = pytest.mark.gpu


def _bits(t):
    return synth.u16(t.cpu())


def _near_midpoint_gates() -> np.ndarray:
    """bf16 gates in (-100, 100) whose binary32 silu is within 16 ulp of a bf16 midpoint."""
    b = np.arange(0, 0x10000, dtype=np.uint32)
    g32 = (b << 16).view(np.float32)
    g = g32[np.isfinite(g32)].astype(np.float64)
    g = g[np.abs(g) < 100]
    with np.errstate(over="ignore"):
        s = (g / (1.0 + np.exp(-g))).astype(np.float32)
    low = s.view(np.uint32) & 0xFFFF
    return g[(low > 0x8000 - 16) & (low < 0x8000 + 16)].astype(np.float32)


def _values_case(ap, dev, g, u, fused):
    rows, dim = g.shape
    if fused:
        x = torch.cat([g, u], dim=1).to(dev)
        gate, up = x[:, :dim], x[:, dim:]
    else:
        gate, up = g.to(dev), u.to(dev)
    out = ap.swiglu_bf16(gate, up)
    ref = oracle.swiglu_values(_bits(g), _bits(u))
    got = _bits(out)
    bad = np.argwhere(got != ref)[:8]
    detail = [(int(r), int(c), hex(_bits(g)[r, c]), hex(_bits(u)[r, c]), hex(got[r, c]), hex(ref[r, c])) for r, c in bad]
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} differ (row, col, gate, up, got, oracle): {detail}"


@pytest.mark.parametrize("rows,dim", [(1, 8), (37, 1536), (129, 5376), (64, 14336)])
@pytest.mark.parametrize("fused", [False, True])
def test_swiglu_values_bit_exact(ap, dev, rows, dim, fused):
    g = synth.bf16(synth.normal(rows + dim, 0, (rows, dim), 3.0))
    u = synth.bf16(synth.normal(rows + dim, 1, (rows, dim), 1.0))
    _values_case(ap, dev, g, u, fused)


def test_swiglu_values_every_gate_pattern(ap, dev):
    b = np.arange(0, 0x10000, dtype=np.uint32)
    g32 = (b << 16).view(np.float32)
    pats = b[np.isfinite(g32)].astype(np.uint16)
    dim = 256
    n = (pats.size + dim - 1) // dim * dim
    gb = np.zeros(n, dtype=np.uint16)
    gb[:pats.size] = pats
    g = torch.from_numpy(gb.view(np.int16).reshape(-1, dim)).view(torch.bfloat16)
    _values_case(ap, dev, g, synth.bf16(np.ones(g.shape, dtype=np.float32)), False)
    _values_case(ap, dev, g, synth.bf16(synth.normal(9, 1, g.shape, 1.0)), True)


def test_swiglu_values_near_bf16_midpoints_and_extremes(ap, dev):
    near = _near_midpoint_gates()
    assert near.size > 20
    extreme = np.array([-80.5, -87.5, -88.5, -95.0, -100.0, -104.0, -110.0, -300.0, -1e30, 80.0, 100.0, 3e4,
                        1e30, 0.0, -0.0], dtype=np.float32)
    vals = np.concatenate([near, extreme])
    dim = 64
    n = (len(vals) + dim - 1) // dim * dim
    g = np.zeros(n, dtype=np.float32)
    g[:len(vals)] = vals
    g = synth.bf16(g.reshape(-1, dim))
    one = synth.bf16(np.ones(g.shape, dtype=np.float32))
    _values_case(ap, dev, g, one, False)
    u = synth.bf16(synth.normal(5, 1, g.shape, 1.0))
    _values_case(ap, dev, g, u, False)


@pytest.mark.parametrize("rows,dim", [(1, 16), (3, 48), (129, 80), (300, 3072), (64, 5376), (130, 14336),
                                      (5, 32768)])
@pytest.mark.parametrize("fused", [False, True])
def test_swiglu_two_level(ap, dev, rows, dim, fused):
    g = synth.bf16(synth.normal(rows * 7 + dim, 0, (rows, dim), 2.0))
    u = synth.bf16(synth.normal(rows * 7 + dim, 1, (rows, dim), 1.0))
    if fused:
        x = torch.cat([g, u], dim=1).to(dev)
        gate, up = x[:, :dim], x[:, dim:]
    else:
        gate, up = g.to(dev), u.to(dev)
    n = ap.swizzled_sf_size(rows, dim)
    guard = 256
    sfbuf = torch.full((n + 2 * guard,), 0xFF, dtype=torch.uint8, device=dev)
    pk, _, ts = ap.swiglu_quant_nvfp4_2level_bf16(gate, up, sf_swizzled=sfbuf[guard:guard + n])
    sb = sfbuf.cpu().numpy()
    assert np.all(sb[:guard] == 0xFF) and np.all(sb[-guard:] == 0xFF)
    opk, osf, ots = oracle.swiglu_quant_nvfp4_2level(_bits(g), _bits(u))
    assert float(ts.cpu()[0]) == ots
    v = torch.from_numpy(oracle.swiglu_values(_bits(g), _bits(u)).view(np.int16)).view(torch.bfloat16).double()
    check_nvfp4(pk.cpu().numpy(), sb[guard:guard + n], opk, osf, rows, dim, v.numpy(), "swiglu two-level", ts=ots)


def test_swiglu_two_level_16_byte_aligned_inputs(ap, dev):
    # gate and up 16- but not 32-byte aligned: the two-load path of the kernels
    rows, dim = 131, 1040
    g = synth.bf16(synth.normal(31, 0, (rows, dim), 2.0))
    u = synth.bf16(synth.normal(31, 1, (rows, dim), 1.0))
    buf = torch.zeros((rows * 2 * dim + 8,), dtype=torch.bfloat16, device=dev)
    x = buf[8:].view(rows, 2 * dim)
    x[:, :dim] = g.to(dev)
    x[:, dim:] = u.to(dev)
    gate, up = x[:, :dim], x[:, dim:]
    assert gate.data_ptr() % 32 == 16
    pk, sf, ts = ap.swiglu_quant_nvfp4_2level_bf16(gate, up)
    opk, osf, ots = oracle.swiglu_quant_nvfp4_2level(_bits(g), _bits(u))
    assert float(ts.cpu()[0]) == ots
    v = torch.from_numpy(oracle.swiglu_values(_bits(g), _bits(u)).view(np.int16)).view(torch.bfloat16).double()
    check_nvfp4(pk.cpu().numpy(), sf.cpu().numpy(), opk, osf, rows, dim, v.numpy(), "swiglu 16-byte aligned", ts=ots)
    _values_case(ap, dev, g, u, True)


def test_swiglu_two_level_graph_and_workspace_reuse(ap, dev):
    rows, dim = 257, 7168
    g = synth.bf16(synth.normal(21, 0, (rows, dim), 2.0)).to(dev)
    u = synth.bf16(synth.normal(21, 1, (rows, dim), 1.0)).to(dev)
    ws = torch.zeros(4, dtype=torch.uint8, device=dev)
    a = ap.swiglu_quant_nvfp4_2level_bf16(g, u, workspace=ws)
    b = ap.swiglu_quant_nvfp4_2level_bf16(g, u, workspace=ws)
    assert all(torch.equal(x, y) for x, y in zip(a, b))
    pk = torch.zeros((rows, dim // 2), dtype=torch.uint8, device=dev)
    sf = torch.zeros((ap.swizzled_sf_size(rows, dim),), dtype=torch.uint8, device=dev)
    ts = torch.zeros((1,), dtype=torch.float32, device=dev)
    st = torch.cuda.Stream(dev)
    with torch.cuda.stream(st):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=st):
            ap.swiglu_quant_nvfp4_2level_bf16(g, u, packed=pk, sf_swizzled=sf, tensor_scale=ts, workspace=ws)
        gr.replay()
        gr.replay()
    st.synchronize()
    assert torch.equal(pk, a[0]) and torch.equal(sf, a[1]) and torch.equal(ts, a[2])


@pytest.mark.parametrize("rows,dim", [(129, 80), (300, 3072)])
def test_swiglu_two_level_tiny_tensor(ap, dev, rows, dim):
    # gate and up of order 2^-40: v = bf16(bf16(silu(g)) * u) near 2^-81, the
    # tensor scale near 2^-92 and every code divisor s * ts below 2^-64 (the
    # rescaled code path)
    g = synth.bf16(synth.normal(rows + dim, 0, (rows, dim), 2.0 ** -40))
    u = synth.bf16(synth.normal(rows + dim, 1, (rows, dim), 2.0 ** -40))
    pk, sf, ts = ap.swiglu_quant_nvfp4_2level_bf16(g.to(dev), u.to(dev))
    opk, osf, ots = oracle.swiglu_quant_nvfp4_2level(_bits(g), _bits(u))
    assert 0.0 < ots < 2.0 ** -80
    assert float(ts.cpu()[0]) == ots
    v = torch.from_numpy(oracle.swiglu_values(_bits(g), _bits(u)).view(np.int16)).view(torch.bfloat16).double()
    check_nvfp4(pk.cpu().numpy(), sf.cpu().numpy(), opk, osf, rows, dim, v.numpy(), "swiglu two-level tiny", ts=ots)
