"""GPU parity at the exact benchmark configurations, on the default kernels.

The five workloads of the producers' benchmark (adaptive-layernorm-producers
README, "Available Functions" with the shapes of benchmarks/RESULTS.md and the
H3/Wan activations), each with its own seed (synth.CONFIGS), through the
default dispatch with no NVFP4AP_* setting:
  - FP8 broadcast 16x2048;
  - FP8 per-token 2520x3072 with 1% of the rows scaled by 8;
  - FP8 table 4096x3072 (two of six temb chunks plus fp32 table rows);
  - NVFP4 broadcast and layer norm 5070x3072;
  - six-way modulation 1x5070x6x3072 (bit-exact);
plus the modfp8 and AWQ sources at the shapes of their broadcast
counterparts, and the table form's staged kernel held to one CTA per SM so
that each CTA walks ~27 rows through its ring of stages at dim 3072.
FP8/NVFP4 tolerance: tests/parity.py.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import check_fp8, check_nvfp4

pytestmark = pytest.mark.gpu

KNOBS = ("NVFP4AP_KERNEL",)


@pytest.fixture
def default(monkeypatch):
    for k in KNOBS:
        monkeypatch.delenv(k, raising=False)
    return monkeypatch


def _d(w, dev):
    return {k: v.to(dev) for k, v in w.inputs.items()}


def _act(w):
    return float(w.inputs["act_scale"][0])


def _u(w, *keys):
    return {k: synth.u16(w.inputs[k]) for k in keys}


def _codes(t):
    return t.view(torch.uint8).cpu().numpy()


def test_c1_fp8_broadcast_16x2048(ap, dev, default):
    w = synth.CONFIGS["fp8_broadcast_16x2048"]()
    d = _d(w, dev)
    out = ap.ada_layer_norm_quant_fp8_bf16(d["x"], d["scale"], d["shift"], d["act_scale"])
    u = _u(w, "x", "scale", "shift")
    ref = oracle.ln_quant_fp8(u["x"], _act(w), oracle.MOD_BCAST, scale=u["scale"], shift=u["shift"])
    check_fp8(_codes(out), ref, _act(w), "C1")


def test_c2_fp8_per_token_2520x3072_outliers(ap, dev, default):
    w = synth.CONFIGS["fp8_ptok_2520x3072"]()
    assert len(synth.outlier_rows(1002, 2520)) == 25
    d = _d(w, dev)
    out = ap.ada_layer_norm_quant_fp8_ptok_bf16(d["x"], d["scale"], d["shift"], d["act_scale"])
    u = _u(w, "x", "scale", "shift")
    ref = oracle.ln_quant_fp8(u["x"], _act(w), oracle.MOD_PTOK, scale=u["scale"], shift=u["shift"])
    check_fp8(_codes(out), ref, _act(w), "C2")


def _table(ap, dev, what):
    w = synth.CONFIGS["fp8_table_4096x3072"]()
    d = _d(w, dev)
    out = ap.ada_layer_norm_quant_fp8_ptok_table_bf16(d["x"], d["temb"], d["table"], d["act_scale"], 0, 1)
    ref = oracle.ln_quant_fp8(synth.u16(w.inputs["x"]), _act(w), oracle.MOD_TABLE,
                              temb=synth.u16(w.inputs["temb"]), table=w.inputs["table"].numpy(),
                              shift_idx=0, scale_idx=1)
    check_fp8(_codes(out), ref, _act(w), what)


def test_c3_fp8_table_4096x3072(ap, dev, default):
    _table(ap, dev, "C3")


def test_c3_table_kernel_one_cta_per_sm(ap, dev, default):
    # the staged (TMA) kernel of the table form, full-row instance at dim
    # 3072, one persistent CTA per SM: every CTA walks its rows through the
    # stage ring many times over
    default.setenv("NVFP4AP_KERNEL", "4:1")
    _table(ap, dev, "C3 one CTA per SM")


@pytest.mark.parametrize("kind", ["bcast", "ln"])
def test_c4_nvfp4_5070x3072(ap, dev, default, kind):
    w = synth.CONFIGS["nvfp4_broadcast_5070x3072" if kind == "bcast" else "nvfp4_ln_5070x3072"]()
    x = w.inputs["x"].to(dev)
    if kind == "bcast":
        pk, sf = ap.ada_layer_norm_quant_nvfp4_swizzled_bf16(x, w.inputs["scale"].to(dev), w.inputs["shift"].to(dev))
        mod, mk = _u(w, "scale", "shift"), oracle.MOD_BCAST
    else:
        pk, sf = ap.layer_norm_no_affine_quant_nvfp4_swizzled_bf16(x)
        mod, mk = {}, oracle.MOD_NONE
    xu = synth.u16(w.inputs["x"])
    op, os_ = oracle.ln_quant_nvfp4(xu, mk, **mod)
    y = oracle.modulated(xu, mk, **mod)
    v = torch.from_numpy(y.astype(np.float32)).to(torch.bfloat16).double().numpy()
    check_nvfp4(pk.cpu().numpy(), sf.cpu().numpy(), op, os_, 5070, 3072, v_orc=v, what=f"C4 {kind}")


def test_c5_modulation6_1x5070x3072_bit_exact(ap, dev, default):
    w = synth.CONFIGS["modulation6_1x5070x3072"]()
    p, m = w.inputs["params"], w.inputs["modulation"]
    outs = ap.adaln_modulation6_bf16(p.to(dev), m.to(dev))
    ref = oracle.adaln_modulation6(p.numpy(), m.numpy())
    for i in range(6):
        got = outs[i].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got, ref[i]), f"C5 output {i}"


def _modfp8_src(w):
    return dict(scale_fp8=w.inputs["scale_fp8"].view(torch.uint8).numpy(),
                shift_fp8=w.inputs["shift_fp8"].view(torch.uint8).numpy(),
                scale_deq=float(w.inputs["scale_deq"][0]), shift_deq=float(w.inputs["shift_deq"][0]))


def test_fp8_modfp8_and_awq_4096x3072(ap, dev, default):
    w = synth.fp8_modfp8(4096, 3072, 2006)
    d = _d(w, dev)
    out = ap.ada_layer_norm_quant_fp8_modfp8_bf16(d["x"], d["scale_fp8"], d["shift_fp8"], d["scale_deq"],
                                                  d["shift_deq"], d["act_scale"])
    ref = oracle.ln_quant_fp8(synth.u16(w.inputs["x"]), _act(w), oracle.MOD_MODFP8, **_modfp8_src(w))
    check_fp8(_codes(out), ref, _act(w), "FP8 modfp8 4096x3072")
    w = synth.fp8_awq(4096, 3072, 2007)
    d = _d(w, dev)
    out = ap.awq_ada_layer_norm_quant_fp8_bf16(d["x"], d["scale"], d["shift"], d["inv_s"], d["act_scale"])
    u = _u(w, "x", "scale", "shift", "inv_s")
    ref = oracle.ln_quant_fp8(u["x"], _act(w), oracle.MOD_AWQ, scale=u["scale"], shift=u["shift"], inv_s=u["inv_s"])
    check_fp8(_codes(out), ref, _act(w), "FP8 AWQ 4096x3072")


def test_nvfp4_modfp8_5070x3072(ap, dev, default):
    w = synth.nvfp4_modfp8(5070, 3072, 2008)
    d = _d(w, dev)
    pk, sf = ap.ada_layer_norm_quant_nvfp4_swizzled_modfp8_bf16(d["x"], d["scale_fp8"], d["shift_fp8"],
                                                                d["scale_deq"], d["shift_deq"])
    xu = synth.u16(w.inputs["x"])
    src = _modfp8_src(w)
    op, os_ = oracle.ln_quant_nvfp4(xu, oracle.MOD_MODFP8, **src)
    y = oracle.modulated(xu, oracle.MOD_MODFP8, **src)
    v = torch.from_numpy(y.astype(np.float32)).to(torch.bfloat16).double().numpy()
    check_nvfp4(pk.cpu().numpy(), sf.cpu().numpy(), op, os_, 5070, 3072, v_orc=v, what="NVFP4 modfp8 5070x3072")
