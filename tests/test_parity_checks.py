"""CPU checks of the acceptance rules in tests/parity.py themselves.

Mistakes are planted in a copy of the oracle's output (never in a kernel):
the rules must reject a single row whose every code is one step off (which
the whole-tensor rules alone would let through in a large tensor), a code two
steps off, and a scale byte without an amax explanation; the unmodified
output must pass.
"""
import numpy as np
import pytest

import oracle
import synth
from parity import check_fp8, check_nvfp4


def _bump(codes: np.ndarray, sign_bit: int) -> np.ndarray:
    """Each code one step up in magnitude (saturating codes left alone)."""
    c = codes.astype(np.int64)
    mag = c & (sign_bit - 1)
    top = 0x7E if sign_bit == 0x80 else 0x7
    out = np.where(mag < top, c + 1, c)
    return out.astype(codes.dtype)


def test_fp8_rules_catch_one_shifted_row(orc):
    w = synth.fp8_broadcast(2000, 2048, 77)
    u = {k: synth.u16(w.inputs[k]) for k in ("x", "scale", "shift")}
    ref = oracle.ln_quant_fp8(u["x"], 0.025, oracle.MOD_BCAST, scale=u["scale"], shift=u["shift"])
    check_fp8(ref.copy(), ref, 0.025, "unmodified")
    bad = ref.copy()
    bad[1234] = _bump(bad[1234], 0x80)  # 0.05% of the tensor, every code one step off
    assert (bad != ref).mean() < 0.001
    with pytest.raises(AssertionError, match="mismatched codes"):
        check_fp8(bad, ref, 0.025, "one row shifted")
    two = ref.copy()
    two[5, 7] = _bump(_bump(two[5:6, 7:8], 0x80), 0x80)[0, 0]
    with pytest.raises(AssertionError, match="step off"):
        check_fp8(two, ref, 0.025, "two steps")


def test_nvfp4_rules_catch_a_shifted_row_and_a_wrong_scale(orc):
    rows, dim = 2000, 2048
    w = synth.nvfp4_ln(rows, dim, 78)
    xu = synth.u16(w.inputs["x"])
    pk, sf = oracle.ln_quant_nvfp4(xu)
    check_nvfp4(pk.copy(), sf.copy(), pk, sf, rows, dim, what="unmodified")
    codes = oracle.unpack_e2m1(pk)
    codes[77] = _bump(codes[77], 0x8)
    bad = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    with pytest.raises(AssertionError, match="mismatched codes"):
        check_nvfp4(bad, sf.copy(), pk, sf, rows, dim, what="one row shifted")
    sf_bad = sf.copy()
    from parity import _offsets
    sf_bad[_offsets(rows, dim)[10]] ^= 0x08
    y = oracle.modulated(xu)
    import torch
    v = torch.from_numpy(y.astype(np.float32)).to(torch.bfloat16).double().numpy()
    with pytest.raises(AssertionError, match="scale bytes differ"):
        check_nvfp4(pk.copy(), sf_bad, pk, sf, rows, dim, v_orc=v, what="wrong scale")
