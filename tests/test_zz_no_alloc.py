"""The allocation-free FP8 broadcast entry point, through the C ABI.

ada_layer_norm_quant_fp8_bf16_noalloc is for callers that cannot allocate
device memory (a device-memory budget fixed at start-up, or a framework region
whose allocator must not grow): its kernel's per-CTA scratch words live in a
fixed array inside the library.  Two calls in a row, on different inputs, must
each agree with the oracle and with ada_layer_norm_quant_fp8_bf16 within the
parity tolerance of these tests (tests/parity.py), and each call's per-CTA
progress words (read back with nvfp4ap_noalloc_progress) must account for
every row with no timeout bit -- the second call also shows that the scratch
left behind by the first one does not leak into it.

This file is collected last so that a run stopping at the first failure has
run every other test before it; it passes alone in a fresh process too (the
first call does the library's one-time set-up, outside any stream capture).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import check_codes, check_fp8

pytestmark = pytest.mark.gpu


def _c_call(L, w, out, stream):
    d = w["d"]
    return L.ada_layer_norm_quant_fp8_bf16_noalloc(
        d["x"].data_ptr(), d["scale"].data_ptr(), d["shift"].data_ptr(), d["act_scale"].data_ptr(),
        ctypes.c_float(1e-5), out.data_ptr(), d["x"].shape[0], d["x"].shape[1], stream)


@pytest.mark.parametrize("rows,dim", [(4096, 3072), (129, 1536)])
def test_noalloc_matches_allocating_entry_point_twice(ap, dev, rows, dim):
    L = ap._load()
    stream = torch.cuda.current_stream(dev).cuda_stream
    for call, seed in enumerate((31, 32)):
        w = synth.fp8_broadcast(rows, dim, seed=seed + rows)
        d = {k: v.to(dev) for k, v in w.inputs.items()}
        out = torch.full((rows, dim), 0x7F, dtype=torch.uint8, device=dev)  # NaN codes until written
        assert _c_call(L, {"d": d}, out, stream) == 0, f"call {call}"
        ref = ap.ada_layer_norm_quant_fp8_bf16(d["x"], d["scale"], d["shift"], d["act_scale"])
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        exp = ref.view(torch.uint8).cpu().numpy()
        assert not (got == 0x7F).any(), f"call {call}: output not fully written"
        check_codes(got, exp, 0x80, f"noalloc call {call}")
        t = np.nan_to_num(torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy())
        dg, de = t[got], t[exp]
        assert np.sqrt(((dg - de) ** 2).sum()) / np.sqrt((de ** 2).sum()) < 1e-2
        # against the oracle directly, with the bounds every parity test uses
        u = {k: synth.u16(w.inputs[k]) for k in ("x", "scale", "shift")}
        act = float(w.inputs["act_scale"][0])
        ref_o = oracle.ln_quant_fp8(u["x"], act, oracle.MOD_BCAST, scale=u["scale"], shift=u["shift"])
        check_fp8(got, ref_o, act, f"noalloc call {call} vs oracle")
        # the scratch words of this call: every row finished, no wait ran out
        words = ap.noalloc_progress()
        assert len(words) > 0, f"call {call}: no progress words"
        assert all(wd & 0x80000000 == 0 for wd in words), f"call {call}: a wait ran out"
        assert sum(wd & 0x7FFFFFFF for wd in words) == rows, f"call {call}: progress words do not sum to rows"
    ap.take_device_fault()
