"""Programmatic dependent launch keeps dependent chains correct.

The row and six-way kernels are launched so that a kernel may be dispatched
while the previous one on the stream drains; each waits for its predecessor
before reading memory.  Here every producer reads what the previous launch
wrote (six-way outputs -> FP8 / NVFP4 producers -> ...), back to back on one
stream, with inputs changed between rounds; the results must equal those of
the same chain run with NVFP4AP_PDL=0 (plain stream order), bit for bit.
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def _chain(ap, params, mod, scale, shift, act):
    outs = ap.adaln_modulation6_bf16(params, mod)
    S, D = outs[0].shape[1], outs[0].shape[2]
    x = outs[0].view(S, D)
    q1 = ap.ada_layer_norm_quant_fp8_bf16(x, scale, shift, act)
    q2 = ap.layer_norm_no_affine_quant_fp8_static_bf16(outs[1].view(S, D), act)
    pk, sf = ap.ada_layer_norm_quant_nvfp4_swizzled_bf16(outs[2].view(S, D), scale, shift)
    # feed a producer's output back into the next six-way call
    params2 = params.clone()
    params2[0, :, 3, :] += q1.view(torch.uint8)[:, :].float() * 1e-3
    outs2 = ap.adaln_modulation6_bf16(params2, mod)
    q3 = ap.layer_norm_no_affine_quant_fp8_static_bf16(outs2[3].view(S, D), act)
    return [t.view(torch.uint8).cpu().numpy() if t.dtype != torch.bfloat16 else t.view(torch.int16).cpu().numpy()
            for t in (q1, q2, pk, sf, outs2[3], q3)]


def test_dependent_chain_equals_plain_stream_order(ap, dev, monkeypatch):
    S, D = 2520, 3072
    res = {}
    for pdl in ("1", "0"):
        monkeypatch.setenv("NVFP4AP_PDL", pdl)
        got = []
        for r in range(3):
            w = synth.modulation6(1, S, D, seed=70 + r)
            b = synth.fp8_broadcast(1, D, seed=80 + r)
            params, mod = w.inputs["params"].to(dev), w.inputs["modulation"].to(dev)
            scale, shift = b.inputs["scale"].to(dev), b.inputs["shift"].to(dev)
            act = b.inputs["act_scale"].to(dev)
            got.append(_chain(ap, params, mod, scale, shift, act))
        torch.cuda.synchronize()
        res[pdl] = got
    for r in range(3):
        for a, b in zip(res["1"][r], res["0"][r]):
            assert np.array_equal(a, b)
