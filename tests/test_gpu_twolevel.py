"""GPU parity of the segmented and two-level NVFP4 producers (C ABI).

Segmented modulation: row r takes row seg_idx[r] of (nseg, dim) tables
(h3-blackwell-runtime compare page).  Two-level NVFP4 (same page,
"Numerical Constraint" and the P1 checkpoint's numerical contract): global
bf16 amax -> tensor scale ts = bf16(amax / 2688); block scales e4m3(min((amax_b
/ 6) / ts, 448)); codes e2m1(v / (s * ts)).  Tolerance: tests/parity.py; the
tensor scale must equal the oracle's exactly.  Cases: ragged rows (padding of
the last scale tile), several dims (capped and uncapped kernels), the page's
segment layout and random segment assignments, an all-zero tensor, a tensor
whose maximum is 2688 (ts = 1), an out-of-range segment index (zero
modulation for that row plus the device fault word), workspace reuse, a CUDA
graph capture of the three operations.  Every case runs on the default
kernels (block-per-lane for the two-level forms, register row kernels for the
single-level segmented forms), on the register row kernels
(NVFP4AP_KERNEL=3), on the block-per-lane kernels (NVFP4AP_KERNEL=5) and with
the warp-per-row kernels forced at every size (NVFP4AP_KERNEL=6: the two-level
maximum pass and the FP8 segmented producer; the row held in registers where a
lane's share fits, dims up to 6144, else read twice, dim 8192).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import check_fp8, check_nvfp4

pytestmark = pytest.mark.gpu

SHAPES = [(1, 16), (3, 48), (127, 64), (129, 80), (300, 3072), (64, 5376), (130, 4096), (5, 32768), (257, 1536),
          (41, 8192)]


@pytest.fixture(autouse=True, params=["auto", "rows", "blk", "warp"])
def family(request, monkeypatch):
    kernel = {"auto": None, "rows": "3", "blk": "5", "warp": "6"}[request.param]
    if kernel is None:
        monkeypatch.delenv("NVFP4AP_KERNEL", raising=False)
    else:
        monkeypatch.setenv("NVFP4AP_KERNEL", kernel)
    return request.param


def _u(t):
    return synth.u16(t)


def _seg_src(w):
    return dict(seg_idx=w.inputs["seg_idx"].numpy(), seg_scale=_u(w.inputs["seg_scale"]),
                seg_shift=_u(w.inputs["seg_shift"]))


def _v(x, kind, **mod):
    """The oracle's staged bf16 values as float64 (explains scale-byte mismatches)."""
    return torch.from_numpy(oracle.staged(x, kind, **mod).view(np.int16)).view(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("rows,dim", [(1, 32), (40, 16), (127, 1536), (129, 3072), (300, 2048), (5, 32768),
                                      (33, 6144)])
def test_fp8_segmented(ap, dev, rows, dim):
    w = synth.segmented(rows, dim, seed=rows + dim)
    d = {k: v.to(dev) for k, v in w.inputs.items()}
    out = ap.ada_layer_norm_quant_fp8_seg_bf16(d["x"], d["seg_idx"], d["seg_scale"], d["seg_shift"],
                                               d["act_scale"])
    ref = oracle.ln_quant_fp8(_u(w.inputs["x"]), 0.025, oracle.MOD_SEG, **_seg_src(w))
    check_fp8(out.view(torch.uint8).cpu().numpy(), ref, 0.025, "fp8 seg")


@pytest.mark.parametrize("rows,dim", SHAPES)
def test_nvfp4_segmented(ap, dev, rows, dim):
    w = synth.segmented(rows, dim, seed=3 * rows + dim)
    d = {k: v.to(dev) for k, v in w.inputs.items()}
    pk, sf = ap.ada_layer_norm_quant_nvfp4_swizzled_seg_bf16(d["x"], d["seg_idx"], d["seg_scale"], d["seg_shift"])
    x, src = _u(w.inputs["x"]), _seg_src(w)
    opk, osf = oracle.ln_quant_nvfp4(x, oracle.MOD_SEG, **src)
    check_nvfp4(pk.cpu().numpy(), sf.cpu().numpy(), opk, osf, rows, dim, _v(x, oracle.MOD_SEG, **src), "nvfp4 seg")


def _two_level(ap, dev, kind, w):
    d = {k: v.to(dev) for k, v in w.inputs.items()}
    rows, dim = w.rows, w.dim
    n = ap.swizzled_sf_size(rows, dim)
    guard = 256
    sfbuf = torch.full((n + 2 * guard,), 0xFF, dtype=torch.uint8, device=dev)
    sf = sfbuf[guard:guard + n]
    if kind == "none":
        pk, _, ts = ap.layer_norm_no_affine_quant_nvfp4_2level_bf16(d["x"], sf_swizzled=sf)
        mk, mod = oracle.MOD_NONE, {}
    elif kind == "bcast":
        pk, _, ts = ap.ada_layer_norm_quant_nvfp4_2level_bf16(d["x"], d["scale"], d["shift"], sf_swizzled=sf)
        mk, mod = oracle.MOD_BCAST, dict(scale=_u(w.inputs["scale"]), shift=_u(w.inputs["shift"]))
    else:
        pk, _, ts = ap.ada_layer_norm_quant_nvfp4_2level_seg_bf16(d["x"], d["seg_idx"], d["seg_scale"],
                                                                  d["seg_shift"], sf_swizzled=sf)
        mk, mod = oracle.MOD_SEG, _seg_src(w)
    sb = sfbuf.cpu().numpy()
    assert np.all(sb[:guard] == 0xFF) and np.all(sb[-guard:] == 0xFF)
    x = _u(w.inputs["x"])
    opk, osf, ots = oracle.ln_quant_nvfp4_2level(x, mk, **mod)
    return pk.cpu().numpy(), sb[guard:guard + n], float(ts.cpu()[0]), opk, osf, ots, _v(x, mk, **mod)


@pytest.mark.parametrize("rows,dim", SHAPES)
@pytest.mark.parametrize("kind", ["none", "bcast", "seg"])
def test_nvfp4_two_level(ap, dev, kind, rows, dim):
    seed = 5 * rows + dim
    w = synth.segmented(rows, dim, seed) if kind == "seg" else \
        (synth.nvfp4_broadcast(rows, dim, seed) if kind == "bcast" else synth.nvfp4_ln(rows, dim, seed))
    gpk, gsf, gts, opk, osf, ots, v = _two_level(ap, dev, kind, w)
    assert gts == ots, (gts, ots)
    check_nvfp4(gpk, gsf, opk, osf, rows, dim, v, f"two-level {kind}", ts=ots)


def test_two_level_zero_tensor(ap, dev):
    rows, dim = 130, 96
    x = torch.zeros((rows, dim), dtype=torch.bfloat16, device=dev)
    pk, sf, ts = ap.layer_norm_no_affine_quant_nvfp4_2level_bf16(x)
    opk, osf, ots = oracle.ln_quant_nvfp4_2level(np.zeros((rows, dim), dtype=np.uint16))
    assert float(ts.cpu()[0]) == ots == 0.0
    assert np.array_equal(pk.cpu().numpy(), opk) and np.array_equal(sf.cpu().numpy(), osf)


def test_two_level_tensor_scale_one(ap, dev):
    # shift 2688 in one column with scale 0 there: the global maximum is 2688, ts = 1
    rng = np.random.default_rng(8)
    rows, dim = 77, 3072
    x = synth.bf16(rng.standard_normal((rows, dim)).astype(np.float32))
    sc = rng.normal(0, 0.1, dim).astype(np.float32)
    sh = rng.normal(0, 0.1, dim).astype(np.float32)
    sc[7], sh[7] = 0.0, 2688.0
    scale, shift = synth.bf16(sc), synth.bf16(sh)
    pk, sf, ts = ap.ada_layer_norm_quant_nvfp4_2level_bf16(x.to(dev), scale.to(dev), shift.to(dev))
    mod = dict(scale=_u(scale), shift=_u(shift))
    opk, osf, ots = oracle.ln_quant_nvfp4_2level(_u(x), oracle.MOD_BCAST, **mod)
    assert ots == 1.0 and float(ts.cpu()[0]) == 1.0
    check_nvfp4(pk.cpu().numpy(), sf.cpu().numpy(), opk, osf, rows, dim, _v(_u(x), oracle.MOD_BCAST, **mod),
                "two-level ts=1", ts=1.0)


def test_out_of_range_segment_index(ap, dev):
    import nvfp4_activation_producer_gb300 as m
    assert m._load().nvfp4ap_take_device_fault() == 0
    w = synth.segmented(64, 1536, seed=9)
    idx = w.inputs["seg_idx"].clone()
    idx[5], idx[40] = 3, -1                      # nseg = 3: both out of range
    d = {k: v.to(dev) for k, v in w.inputs.items()}
    out = ap.ada_layer_norm_quant_fp8_seg_bf16(d["x"], idx.to(dev), d["seg_scale"], d["seg_shift"], d["act_scale"])
    assert m._load().nvfp4ap_take_device_fault() == m.ERR_FAULT
    assert m._load().nvfp4ap_take_device_fault() == 0          # read and cleared
    # the two rows carry no modulation; the others the oracle's segmented output
    x = _u(w.inputs["x"])
    got = out.view(torch.uint8).cpu().numpy()
    plain = oracle.ln_quant_fp8(x, 0.025, oracle.MOD_NONE)
    check_fp8(got[[5, 40]], plain[[5, 40]], 0.025, "zero modulation rows")
    keep = np.setdiff1d(np.arange(64), [5, 40])
    src = _seg_src(w)
    src["seg_idx"] = src["seg_idx"][keep]
    check_fp8(got[keep], oracle.ln_quant_fp8(x[keep], 0.025, oracle.MOD_SEG, **src), 0.025, "valid rows")


def test_two_level_workspace_too_small_is_rejected(ap, dev):
    # the binding checks the statistics slots' size (the C ABI cannot)
    w = synth.nvfp4_ln(64, 256, seed=2)
    x = w.inputs["x"].to(dev)
    small = torch.zeros(ap.workspace_2level_bytes(63), dtype=torch.uint8, device=dev)
    with pytest.raises(ValueError):
        ap.layer_norm_no_affine_quant_nvfp4_2level_bf16(x, workspace=small)
    ok = torch.zeros(ap.workspace_2level_bytes(64), dtype=torch.uint8, device=dev)
    a = ap.layer_norm_no_affine_quant_nvfp4_2level_bf16(x, workspace=ok)
    b = ap.layer_norm_no_affine_quant_nvfp4_2level_bf16(x)
    assert all(torch.equal(u, v) for u, v in zip(a, b))


def test_two_level_workspace_reuse_and_graph(ap, dev):
    w = synth.segmented(515, 5376, seed=11)
    d = {k: v.to(dev) for k, v in w.inputs.items()}
    rows, dim = w.rows, w.dim
    ws = torch.zeros(ap.workspace_2level_bytes(rows), dtype=torch.uint8, device=dev)
    outs = []
    for _ in range(2):
        outs.append(ap.ada_layer_norm_quant_nvfp4_2level_seg_bf16(d["x"], d["seg_idx"], d["seg_scale"],
                                                                  d["seg_shift"], workspace=ws))
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    pk = torch.empty((rows, dim // 2), dtype=torch.uint8, device=dev)
    sf = torch.empty((ap.swizzled_sf_size(rows, dim),), dtype=torch.uint8, device=dev)
    ts = torch.empty((1,), dtype=torch.float32, device=dev)
    st = torch.cuda.Stream(dev)
    with torch.cuda.stream(st):
        ap.ada_layer_norm_quant_nvfp4_2level_seg_bf16(d["x"], d["seg_idx"], d["seg_scale"], d["seg_shift"],
                                                      packed=pk, sf_swizzled=sf, tensor_scale=ts, workspace=ws)
        st.synchronize()
        pk.zero_(); sf.zero_(); ts.zero_()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            ap.ada_layer_norm_quant_nvfp4_2level_seg_bf16(d["x"], d["seg_idx"], d["seg_scale"], d["seg_shift"],
                                                          packed=pk, sf_swizzled=sf, tensor_scale=ts, workspace=ws)
        g.replay()
        g.replay()
    st.synchronize()
    assert torch.equal(pk, outs[0][0]) and torch.equal(sf, outs[0][1]) and torch.equal(ts, outs[0][2])


@pytest.mark.parametrize("kind", ["none", "bcast", "seg"])
def test_two_level_many_rows_per_group(ap, dev, family, kind, monkeypatch):
    # block-per-lane kernels with one CTA per SM: each row group walks ~16 rows
    # and the maximum pass reduces them in one atomic per CTA
    if family != "blk":
        pytest.skip("runs once")
    monkeypatch.setenv("NVFP4AP_KERNEL", "5:1")
    for dim, rows in ((272, 40000), (3072, 20000)):
        w = synth.segmented(rows, dim, seed=dim + 7)
        d = {k: v.to(dev) for k, v in w.inputs.items()}
        x = _u(w.inputs["x"])
        if kind == "seg":
            src = _seg_src(w)
            pk, sf, ts = ap.ada_layer_norm_quant_nvfp4_2level_seg_bf16(d["x"], d["seg_idx"], d["seg_scale"],
                                                                       d["seg_shift"])
            mk = oracle.MOD_SEG
        elif kind == "bcast":
            sc, sh = d["seg_scale"][1].contiguous(), d["seg_shift"][1].contiguous()
            src = dict(scale=_u(w.inputs["seg_scale"][1]), shift=_u(w.inputs["seg_shift"][1]))
            pk, sf, ts = ap.ada_layer_norm_quant_nvfp4_2level_bf16(d["x"], sc, sh)
            mk = oracle.MOD_BCAST
        else:
            src = {}
            pk, sf, ts = ap.layer_norm_no_affine_quant_nvfp4_2level_bf16(d["x"])
            mk = oracle.MOD_NONE
        opk, osf, ots = oracle.ln_quant_nvfp4_2level(x, mk, **src)
        assert float(ts.cpu()[0]) == ots
        check_nvfp4(pk.cpu().numpy(), sf.cpu().numpy(), opk, osf, rows, dim, _v(x, mk, **src),
                    f"two-level {kind} {rows}x{dim}, one CTA per SM", ts=ots)


def test_register_warp_path_from_the_element_threshold(ap, dev, family, monkeypatch):
    # the register-resident warp kernels take a tensor from sms * 128 * 3072
    # elements (fewer rows than the two-sweep kernel's sms * 128 at wide dims):
    # just above it, the default gives the forced warp path's bytes, within the
    # oracle's tolerance
    if family != "auto":
        pytest.skip("runs once")
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    dim = 6144
    rows = -(-sms * 128 * 3072 // dim) + 8
    assert rows < sms * 128
    w = synth.segmented(rows, dim, seed=77)
    d = {k: v.to(dev) for k, v in w.inputs.items() if isinstance(v, torch.Tensor)}
    q = ap.ada_layer_norm_quant_fp8_seg_bf16(d["x"], d["seg_idx"], d["seg_scale"], d["seg_shift"], d["act_scale"])
    pk, sf, ts = ap.ada_layer_norm_quant_nvfp4_2level_seg_bf16(d["x"], d["seg_idx"], d["seg_scale"], d["seg_shift"])
    default = (q.view(torch.uint8).clone(), pk.clone(), sf.clone(), ts.clone())
    monkeypatch.setenv("NVFP4AP_KERNEL", "6")
    q = ap.ada_layer_norm_quant_fp8_seg_bf16(d["x"], d["seg_idx"], d["seg_scale"], d["seg_shift"], d["act_scale"])
    pk, sf, ts = ap.ada_layer_norm_quant_nvfp4_2level_seg_bf16(d["x"], d["seg_idx"], d["seg_scale"], d["seg_shift"])
    for a, b in zip(default, (q.view(torch.uint8), pk, sf, ts)):
        assert torch.equal(a, b)
    ref = oracle.ln_quant_fp8(_u(w.inputs["x"]), 0.025, oracle.MOD_SEG, **_seg_src(w))
    check_fp8(default[0].cpu().numpy(), ref, 0.025, "fp8 segmented above the element threshold")


def _kernel_names(fn):
    """Names of the CUDA kernels that fn() launches (torch profiler), or None."""
    from torch.profiler import ProfilerActivity, profile
    torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        fn()
        torch.cuda.synchronize()
    names = {e.name for e in prof.events() if e.device_type == torch.autograd.DeviceType.CUDA}
    return names or None


# (rows, dim, single read expected): several rows per row group (1300 x 1040,
# dim / 8 not a multiple of 32), the largest share of rows one CTA takes
# (128 rows of 32 bytes), the largest tensor at dim 3072 whose rows fit in the
# SMs' shared memory and the first that does not
ONCHIP_SHAPES = [(1300, 1040, True), (19456, 16, True), (5320, 3072, True), (5321, 3072, False)]


@pytest.mark.parametrize("rows,dim,onchip", ONCHIP_SHAPES)
@pytest.mark.parametrize("kind", ["none", "bcast", "seg"])
def test_two_level_single_read_path(ap, dev, family, kind, rows, dim, onchip):
    if family != "auto":
        pytest.skip("default dispatch only")
    if torch.cuda.get_device_properties(dev).multi_processor_count != 152:
        pytest.skip("the shapes are chosen for 152 SMs")
    seed = 3 * rows + dim
    w = synth.segmented(rows, dim, seed) if kind == "seg" else \
        (synth.nvfp4_broadcast(rows, dim, seed) if kind == "bcast" else synth.nvfp4_ln(rows, dim, seed))
    gpk, gsf, gts, opk, osf, ots, v = _two_level(ap, dev, kind, w)
    assert gts == ots, (gts, ots)
    check_nvfp4(gpk, gsf, opk, osf, rows, dim, v, f"two-level {kind} {rows}x{dim}", ts=ots)
    if kind == "none":
        x = w.inputs["x"].to(dev)
        names = _kernel_names(lambda: ap.layer_norm_no_affine_quant_nvfp4_2level_bf16(x))
        if names is None:
            pytest.skip("the profiler recorded no CUDA kernels")
        assert any("nv2l_onchip" in n for n in names) == onchip, sorted(names)


@pytest.mark.parametrize("rows,dim", [(300, 3072), (20000, 64)])
@pytest.mark.parametrize("e", [-60, -110])
def test_two_level_tiny_tensor(ap, dev, rows, dim, e):
    # scale = -1 makes 1 + scale = 0, so v = bf16(shift) exactly; shifts of
    # order 2^e put the tensor scale near the bottom of the fp32 range and the
    # code divisors s * ts below 2^-64 (the rescaled code path; at 2^-60 both
    # sides of that bound occur in one tensor)
    rng = np.random.default_rng(17 + rows - e)
    x = synth.bf16(rng.standard_normal((rows, dim)).astype(np.float32))
    sc = np.full(dim, -1.0, dtype=np.float32)
    sh = (rng.standard_normal(dim) * 2.0 ** e).astype(np.float32)
    scale, shift = synth.bf16(sc), synth.bf16(sh)
    pk, sf, ts = ap.ada_layer_norm_quant_nvfp4_2level_bf16(x.to(dev), scale.to(dev), shift.to(dev))
    mod = dict(scale=_u(scale), shift=_u(shift))
    opk, osf, ots = oracle.ln_quant_nvfp4_2level(_u(x), oracle.MOD_BCAST, **mod)
    assert 0.0 < ots < 2.0 ** (e - 8)
    assert float(ts.cpu()[0]) == ots
    check_nvfp4(pk.cpu().numpy(), sf.cpu().numpy(), opk, osf, rows, dim, _v(_u(x), oracle.MOD_BCAST, **mod),
                f"two-level tiny 2^{e}", ts=ots)


@pytest.mark.parametrize("rows,dim", [(300, 3072), (20000, 64)])
def test_two_level_out_of_range_segment_index(ap, dev, rows, dim):
    # rows whose segment index is outside [0, nseg) take zero modulation and set
    # the fault word; the expected output is the oracle's with those rows
    # pointed at an appended all-zero table row (the tensor maximum couples
    # every row, so the whole tensor is compared)
    import nvfp4_activation_producer_gb300 as m
    ap.take_device_fault()
    w = synth.segmented(rows, dim, seed=rows + 5)
    nseg = int(w.inputs["seg_scale"].shape[0])
    idx = w.inputs["seg_idx"].clone()
    bad_rows = [5, rows // 2, rows - 1]
    idx[bad_rows[0]], idx[bad_rows[1]], idx[bad_rows[2]] = nseg, -1, 1 << 20
    d = {k: v.to(dev) for k, v in w.inputs.items()}
    pk, sf, ts = ap.ada_layer_norm_quant_nvfp4_2level_seg_bf16(d["x"], idx.to(dev), d["seg_scale"], d["seg_shift"])
    torch.cuda.synchronize()
    with pytest.raises(ap.NvFp4ApError) as e:
        ap.take_device_fault()
    assert e.value.status == m.ERR_FAULT
    oidx = idx.numpy().astype(np.int32).copy()
    oidx[bad_rows] = nseg
    zero = np.zeros((1, dim), dtype=np.uint16)
    src = dict(seg_idx=oidx, seg_scale=np.concatenate([_u(w.inputs["seg_scale"]), zero]),
               seg_shift=np.concatenate([_u(w.inputs["seg_shift"]), zero]))
    x = _u(w.inputs["x"])
    opk, osf, ots = oracle.ln_quant_nvfp4_2level(x, oracle.MOD_SEG, **src)
    assert float(ts.cpu()[0]) == ots
    check_nvfp4(pk.cpu().numpy(), sf.cpu().numpy(), opk, osf, rows, dim, _v(x, oracle.MOD_SEG, **src),
                "two-level, out-of-range segment rows", ts=ots)
