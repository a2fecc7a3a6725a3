"""GPU parity of adaln_modulation6_bf16 against the oracle: bit-exact.

Covers the 16-byte vector path (dim a multiple of 8, aligned pointers), the
element path (odd dim, or outputs off 16-byte alignment), six separate
output tensors vs one (6, B, S, D) buffer, zero tokens, and guard bands.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("b,s,d", [(1, 1, 8), (1, 51, 1536), (2, 37, 3072), (1, 333, 1152), (3, 7, 1000),
                                   (1, 5, 13), (2, 64, 5376)])
def test_modulation6_bit_exact(ap, dev, b, s, d):
    w = synth.modulation6(b, s, d, seed=b * 100 + s + d)
    p, m = w.inputs["params"], w.inputs["modulation"]
    outs = ap.adaln_modulation6_bf16(p.to(dev), m.to(dev))
    ref = oracle.adaln_modulation6(p.numpy(), m.numpy())
    assert len(outs) == 6
    for i in range(6):
        assert outs[i].shape == (b, s, d) and outs[i].dtype == torch.bfloat16
        assert np.array_equal(_bits(outs[i]), ref[i])


def test_separate_and_misaligned_outputs(ap, dev):
    b, s, d = 1, 100, 3072
    w = synth.modulation6(b, s, d, seed=3)
    p, m = w.inputs["params"].to(dev), w.inputs["modulation"].to(dev)
    ref = oracle.adaln_modulation6(w.inputs["params"].numpy(), w.inputs["modulation"].numpy())
    guard = 1024
    bufs = [torch.full((b * s * d + 2 * guard + 1,), -7, dtype=torch.int16, device=dev) for _ in range(6)]
    # output 3 sits 2 bytes off 16-byte alignment: the element path must take it
    outs = [bufs[i][guard + (1 if i == 3 else 0):guard + (1 if i == 3 else 0) + b * s * d].view(torch.bfloat16).view(b, s, d)
            for i in range(6)]
    ap.adaln_modulation6_bf16(p, m, out=outs)
    for i in range(6):
        assert np.array_equal(_bits(outs[i]), ref[i])
        raw = bufs[i].cpu().numpy()
        assert np.all(raw[:guard] == -7) and np.all(raw[-guard:] == -7)


def test_zero_tokens(ap, dev):
    p = torch.empty((1, 0, 6, 64), dtype=torch.float32, device=dev)
    m = torch.zeros((6, 64), dtype=torch.float32, device=dev)
    outs = ap.adaln_modulation6_bf16(p, m)
    assert all(o.shape == (1, 0, 64) for o in outs)


def test_one_buffer_output(ap, dev):
    w = synth.modulation6(2, 10, 256, seed=9)
    buf = torch.empty((6, 2, 10, 256), dtype=torch.bfloat16, device=dev)
    outs = ap.adaln_modulation6_bf16(w.inputs["params"].to(dev), w.inputs["modulation"].to(dev), out=buf)
    ref = oracle.adaln_modulation6(w.inputs["params"].numpy(), w.inputs["modulation"].numpy())
    assert np.array_equal(_bits(buf).reshape(6, 2, 10, 256), ref)
    assert outs[0].data_ptr() == buf.data_ptr()
