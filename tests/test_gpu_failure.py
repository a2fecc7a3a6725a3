"""GPU failure path of the bounded waits (no GPU fault is involved).

The kernels that stage rows through shared memory with bulk copies (the
table form's default kernel, the allocation-free producer's ring kernel and
the single-read two-level NVFP4 kernel) bound every wait on a copy.
nvfp4ap_set_wait_limit shrinks that bound to a few SM clock cycles, so the
first wait of each CTA gives up before its copy lands: the kernel must then
wait for every copy it has in flight (with the default bound), stop, and
report through nvfp4ap_take_device_fault (NVFP4AP_ERR_TIMEOUT) -- the call
itself returns normally.  A normal call right after (default bound restored)
must match the oracle within the parity tolerance of tests/parity.py.
"""
import pytest
import torch

import oracle
import synth
from parity import check_fp8, check_nvfp4

pytestmark = pytest.mark.gpu


@pytest.fixture
def tiny_wait(ap, monkeypatch):
    monkeypatch.delenv("NVFP4AP_KERNEL", raising=False)
    ap.take_device_fault()  # start from a clear word
    ap.set_wait_limit(4)
    try:
        yield ap
    finally:
        ap.set_wait_limit(0)
        torch.cuda.synchronize()


def _act(w):
    return float(w.inputs["act_scale"][0])


def _table_ref(w, si, ci):
    return oracle.ln_quant_fp8(synth.u16(w.inputs["x"]), _act(w), oracle.MOD_TABLE, temb=synth.u16(w.inputs["temb"]),
                               table=w.inputs["table"].numpy(), shift_idx=si, scale_idx=ci)


def test_table_kernel_wait_runs_out_then_recovers(tiny_wait, dev):
    ap = tiny_wait
    rows, dim = 2048, 3072
    w = synth.fp8_table(rows, dim, seed=4242)
    d = {k: v.to(dev) for k, v in w.inputs.items()}
    ap.ada_layer_norm_quant_fp8_ptok_table_bf16(d["x"], d["temb"], d["table"], d["act_scale"], 0, 1)
    torch.cuda.synchronize()
    with pytest.raises(ap.NvFp4ApError) as e:
        ap.take_device_fault()
    assert e.value.status == ap.ERR_TIMEOUT
    ap.take_device_fault()  # the word was cleared by the read above
    ap.set_wait_limit(0)
    out = ap.ada_layer_norm_quant_fp8_ptok_table_bf16(d["x"], d["temb"], d["table"], d["act_scale"], 0, 1)
    torch.cuda.synchronize()
    ap.take_device_fault()
    check_fp8(out.view(torch.uint8).cpu().numpy(), _table_ref(w, 0, 1), _act(w), "table after a timeout")


def test_noalloc_wait_runs_out_then_recovers(tiny_wait, dev):
    ap = tiny_wait
    rows, dim = 2048, 3072
    w = synth.fp8_broadcast(rows, dim, seed=4243)
    d = {k: v.to(dev) for k, v in w.inputs.items()}
    L = ap._load()
    stream = torch.cuda.current_stream(dev).cuda_stream
    out = torch.empty((rows, dim), dtype=torch.uint8, device=dev)
    import ctypes

    def call():
        return L.ada_layer_norm_quant_fp8_bf16_noalloc(
            d["x"].data_ptr(), d["scale"].data_ptr(), d["shift"].data_ptr(), d["act_scale"].data_ptr(),
            ctypes.c_float(1e-5), out.data_ptr(), rows, dim, stream)

    assert call() == 0
    torch.cuda.synchronize()
    with pytest.raises(ap.NvFp4ApError) as e:
        ap.take_device_fault()
    assert e.value.status == ap.ERR_TIMEOUT
    words = ap.noalloc_progress()
    assert any(wd & 0x80000000 for wd in words), "no CTA recorded its timeout"
    assert sum(wd & 0x7FFFFFFF for wd in words) < rows
    ap.set_wait_limit(0)
    assert call() == 0
    torch.cuda.synchronize()
    ap.take_device_fault()
    words = ap.noalloc_progress()
    assert all(wd & 0x80000000 == 0 for wd in words) and sum(words) == rows
    u = {k: synth.u16(w.inputs[k]) for k in ("x", "scale", "shift")}
    ref = oracle.ln_quant_fp8(u["x"], _act(w), oracle.MOD_BCAST, scale=u["scale"], shift=u["shift"])
    check_fp8(out.cpu().numpy(), ref, _act(w), "noalloc after a timeout")


def test_two_level_single_read_wait_runs_out_then_recovers(tiny_wait, dev):
    # 2048 x 3072 fits the single-read kernel (14 rows per SM); a CTA whose row
    # wait gives up still arrives at the grid barrier, so the others do not wait
    ap = tiny_wait
    rows, dim = 2048, 3072
    w = synth.nvfp4_ln(rows, dim, seed=4244)
    x = w.inputs["x"].to(dev)
    ap.layer_norm_no_affine_quant_nvfp4_2level_bf16(x)
    torch.cuda.synchronize()
    with pytest.raises(ap.NvFp4ApError) as e:
        ap.take_device_fault()
    assert e.value.status == ap.ERR_TIMEOUT
    ap.set_wait_limit(0)
    pk, sf, ts = ap.layer_norm_no_affine_quant_nvfp4_2level_bf16(x)
    torch.cuda.synchronize()
    ap.take_device_fault()
    u = synth.u16(w.inputs["x"])
    opk, osf, ots = oracle.ln_quant_nvfp4_2level(u)
    assert float(ts.cpu()[0]) == ots
    v = torch.from_numpy(oracle.staged(u, oracle.MOD_NONE).view("int16")).view(torch.bfloat16).double().numpy()
    check_nvfp4(pk.cpu().numpy(), sf.cpu().numpy(), opk, osf, rows, dim, v, "two-level after a timeout", ts=ots)
