"""The producers give the same bytes through the C marshalling module and
through ctypes (GPU), and the C module is the one in use where it was built.

The marshalling paths only convert arguments (csrc/pycall.c; the ctypes
declarations in the binding), so every output byte must agree between them;
the six-way producer's output pointers travel as a sequence on both.
"""
import os

import pytest
import torch

import synth
from nvfp4_activation_producer_gb300 import build as b

pytestmark = pytest.mark.gpu


def _fresh(monkeypatch, pycall: str):
    import nvfp4_activation_producer_gb300 as ap
    monkeypatch.setenv("NVFP4AP_PYCALL", pycall)
    monkeypatch.setattr(ap, "_lib", None)
    return ap


def _run_all(ap, dev):
    out = []
    w = synth.fp8_broadcast(300, 3072, seed=4)
    d = {k: v.to(dev) for k, v in w.inputs.items()}
    out.append(ap.ada_layer_norm_quant_fp8_bf16(d["x"], d["scale"], d["shift"], d["act_scale"]).view(torch.uint8))
    out.append(ap.layer_norm_no_affine_quant_fp8_static_bf16(d["x"], d["act_scale"]).view(torch.uint8))
    out.extend(ap.ada_layer_norm_quant_nvfp4_swizzled_bf16(d["x"], d["scale"], d["shift"]))
    out.extend(ap.layer_norm_no_affine_quant_nvfp4_2level_bf16(d["x"])[:2])
    w6 = synth.modulation6(1, 257, 1536, seed=5)
    d6 = {k: v.to(dev) for k, v in w6.inputs.items()}
    out.extend(ap.adaln_modulation6_bf16(d6["params"], d6["modulation"]))
    torch.cuda.synchronize()
    return [t.clone() for t in out]


def test_c_marshalling_in_use_where_built(monkeypatch):
    ap = _fresh(monkeypatch, "1")
    expected = "c" if (b.pycall_command() is not None and os.path.exists(b.PYCALL)) else "ctypes"
    assert ap.marshalling() == expected


def test_both_paths_give_the_same_bytes(monkeypatch, dev):
    ap = _fresh(monkeypatch, "0")
    assert ap.marshalling() == "ctypes"
    via_ctypes = _run_all(ap, dev)
    ap = _fresh(monkeypatch, "1")
    via_c = _run_all(ap, dev)
    assert len(via_c) == len(via_ctypes)
    for i, (x, y) in enumerate(zip(via_c, via_ctypes)):
        assert torch.equal(x, y), f"output {i} differs between the marshalling paths"
