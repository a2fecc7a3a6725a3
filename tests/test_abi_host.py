"""Host-side checks of the C-ABI library (CPU only, nothing is launched).

- libnvfp4ap.so builds, loads and exports exactly the entry points that
  include/nvfp4ap.h declares;
- every argument error is reported with its status code before anything is
  launched (the pointers below are never dereferenced);
- swizzled_sf_size agrees with the oracle's size and the pages' byte counts.
"""
import ctypes
import json
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4ap.h")


@pytest.fixture(scope="module")
def lib():
    from nvfp4_activation_producer_gb300 import build as b
    path = b.build()
    import nvfp4_activation_producer_gb300 as ap
    return ap._load(), path


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\**\s+\**([A-Za-z_][A-Za-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_exports_match_header(lib):
    _, path = lib
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout
    exported = sorted(l.split()[-1] for l in out.splitlines() if re.search(r" T ", l))
    declared = declared_functions()
    assert declared == exported, (declared, exported)
    assert len(declared) == 27


def test_status_strings_and_version(lib):
    L, _ = lib
    for s in range(11):
        assert L.nvfp4ap_status_string(s) != b"unknown status"
    assert L.nvfp4ap_status_string(99) == b"unknown status"
    # the status values of the boundary's contract
    import nvfp4_activation_producer_gb300 as ap
    assert (ap.ERR_NULL, ap.ERR_SHAPE, ap.ERR_DIM, ap.ERR_INDEX, ap.ERR_ALIGN, ap.ERR_LAUNCH, ap.ERR_TIMEOUT) == tuple(
        range(1, 8))
    assert b"wait ran out" in L.nvfp4ap_status_string(ap.ERR_TIMEOUT)
    assert b"segment index" in L.nvfp4ap_status_string(ap.ERR_FAULT)
    assert L.nvfp4ap_version() >= 100


def test_two_level_single_read_query_arguments(lib):
    # argument errors come before any device query; *single_read stays 0
    L, _ = lib
    flag = ctypes.c_int(7)
    assert L.nvfp4ap_2level_single_read(10, 3072, 0, None) == 1              # NVFP4AP_ERR_NULL
    assert L.nvfp4ap_2level_single_read(-1, 3072, 0, ctypes.byref(flag)) == 2 and flag.value == 0
    flag.value = 7
    assert L.nvfp4ap_2level_single_read(10, 0, 0, ctypes.byref(flag)) == 2 and flag.value == 0
    assert L.nvfp4ap_2level_single_read(10, 40, 0, ctypes.byref(flag)) == 3    # dim % 16
    assert L.nvfp4ap_2level_single_read(10, 65536, 0, ctypes.byref(flag)) == 3
    assert L.nvfp4ap_2level_single_read(10, 3072, 3, ctypes.byref(flag)) == 8  # modulation
    flag.value = 7
    assert L.nvfp4ap_2level_single_read(0, 3072, 1, ctypes.byref(flag)) == 0 and flag.value == 0


def test_wait_limit_setting(lib):
    # the bound of the TMA kernels' waits: set, read back, default restored
    L, _ = lib
    assert L.nvfp4ap_set_wait_limit(1000) == 0
    assert L.nvfp4ap_wait_limit() == 1000
    assert L.nvfp4ap_set_wait_limit(0) == 0
    assert L.nvfp4ap_wait_limit() == 2000000000
    assert L.nvfp4ap_set_wait_limit(-5) == 0
    assert L.nvfp4ap_wait_limit() == 2000000000


def test_argument_statuses_raise_value_errors():
    import nvfp4_activation_producer_gb300 as ap
    for rc in (ap.ERR_NULL, ap.ERR_SHAPE, ap.ERR_DIM, ap.ERR_INDEX, ap.ERR_ALIGN, ap.ERR_VALUE, ap.ERR_SCRATCH):
        with pytest.raises(ValueError):
            ap._raise("f", rc)
    for rc in (ap.ERR_LAUNCH, ap.ERR_TIMEOUT, ap.ERR_FAULT):
        with pytest.raises(RuntimeError) as e:
            ap._raise("f", rc)
        assert not isinstance(e.value, ValueError)


def test_swizzled_sf_size_matches_oracle_and_pages(lib, orc, golden_dir):
    L, _ = lib
    for rows, dim in [(0, 16), (1, 16), (5070, 3072), (129, 80), (127, 48), (4096, 7168), (3, 32768)]:
        assert L.swizzled_sf_size(rows, dim) == orc.swizzled_sf_size(rows, dim)
    for bad in [(1, 8), (1, 0), (-1, 16), (4, 17)]:
        assert L.swizzled_sf_size(*bad) == -1
    g = json.load(open(os.path.join(golden_dir, "nvfp4_ring_sizes.json")))
    for rec in g["records"]:
        assert L.swizzled_sf_size(rec["row_capacity"], rec["K"]) == rec["sfa_bytes"]


A = 0x100000  # a 16-byte aligned fake device address, never dereferenced
NULL = None


def test_fp8_argument_errors(lib):
    L, _ = lib
    f = L.ada_layer_norm_quant_fp8_bf16
    assert f(A, A, A, A, 1e-5, A, -1, 64, NULL) == 2          # negative rows
    assert f(A, A, A, A, 1e-5, A, 4, 0, NULL) == 2            # dim 0
    assert f(A, A, A, A, 1e-5, A, 4, 63, NULL) == 3           # odd dim
    assert f(A, A, A, A, 1e-5, A, 4, 32770, NULL) == 3        # above the maximum dim
    assert f(A, A, A, A, -1.0, A, 4, 64, NULL) == 8           # negative eps
    assert f(A, A, A, A, float("nan"), A, 4, 64, NULL) == 8   # NaN eps
    assert f(NULL, A, A, A, 1e-5, A, 4, 64, NULL) == 1        # null x
    assert f(A, NULL, A, A, 1e-5, A, 4, 64, NULL) == 1        # null scale
    assert f(A, A, A, NULL, 1e-5, A, 4, 64, NULL) == 1        # null act_scale
    assert f(A + 1, A, A, A, 1e-5, A, 4, 64, NULL) == 5       # bf16 x at an odd address (not element-aligned)
    assert f(A, A, A, A + 2, 1e-5, A, 4, 64, NULL) == 5       # act_scale misaligned
    assert f(A, A + 1, A, A, 1e-5, A, 4, 64, NULL) == 5       # bf16 scale at an odd address
    assert f(NULL, NULL, NULL, NULL, 1e-5, NULL, 0, 64, NULL) == 0  # rows == 0: no-op
    g = L.ada_layer_norm_quant_fp8_ptok_bf16
    assert g(A, A, NULL, A, 1e-5, A, 4, 64, NULL) == 1
    h = L.layer_norm_no_affine_quant_fp8_static_bf16
    assert h(A, A, 1e-5, NULL, 4, 64, NULL) == 1
    assert h(A, A, 1e-5, A, 4, 7, NULL) == 3


def test_table_index_errors(lib):
    L, _ = lib
    t = L.ada_layer_norm_quant_fp8_ptok_table_bf16
    assert t(A, A, A, 6, 6, 1, A, 1e-5, A, 4, 64, NULL) == 4   # shift_idx == chunks
    assert t(A, A, A, 6, 0, -1, A, 1e-5, A, 4, 64, NULL) == 4  # negative scale_idx
    assert t(A, A, A, 0, 0, 0, A, 1e-5, A, 4, 64, NULL) == 4   # no chunks
    assert t(A, NULL, A, 6, 0, 1, A, 1e-5, A, 4, 64, NULL) == 1
    assert t(A, A, A + 2, 6, 0, 1, A, 1e-5, A, 4, 64, NULL) == 5  # fp32 table not 4-byte aligned


def test_nvfp4_argument_errors(lib):
    L, _ = lib
    f = L.ada_layer_norm_quant_nvfp4_swizzled_bf16
    assert f(A, A, A, 1e-5, A, A, 4, 40, NULL) == 3            # dim % 16
    assert f(A, A, A, 1e-5, A, A, 4, 32784, NULL) == 3         # above the maximum dim
    assert f(A, A, A, 1e-5, NULL, A, 4, 64, NULL) == 1         # null packed
    assert f(A, A, A, 1e-5, A, NULL, 4, 64, NULL) == 1         # null scales
    assert f(A + 1, A, A, 1e-5, A, A, 4, 64, NULL) == 5        # x at an odd address
    assert f(A, A, A + 1, 1e-5, A, A, 4, 64, NULL) == 5        # shift at an odd address
    assert f(A, A, A, 1e-5, A, A, 0, 64, NULL) == 0
    g = L.layer_norm_no_affine_quant_nvfp4_swizzled_bf16
    assert g(A, 1e-5, A, A, -3, 64, NULL) == 2
    assert g(A, float("inf"), A, A, 3, 64, NULL) == 8


def test_modfp8_and_awq_argument_errors(lib):
    L, _ = lib
    m = L.ada_layer_norm_quant_fp8_modfp8_bf16  # x, s8, h8, sdeq, hdeq, act, eps, out, rows, dim
    assert m(A, NULL, A, A, A, A, 1e-5, A, 4, 64, NULL) == 1      # null scale_fp8
    assert m(A, A, A, A, NULL, A, 1e-5, A, 4, 64, NULL) == 1      # null shift_deq
    assert m(A, A, A, A + 2, A, A, 1e-5, A, 4, 64, NULL) == 5     # scale_deq misaligned
    assert m(A + 1, A, A, A, A, A, 1e-5, A, 4, 64, NULL) == 5     # x at an odd address
    assert m(A, A, A, A, A, A, 1e-5, A, 4, 63, NULL) == 3         # odd dim
    assert m(A, A, A, A, A, A, -2.0, A, 4, 64, NULL) == 8
    assert m(NULL, NULL, NULL, NULL, NULL, NULL, 1e-5, NULL, 0, 64, NULL) == 0
    w = L.awq_ada_layer_norm_quant_fp8_bf16  # x, scale, shift, inv_s, act, eps, out, rows, dim
    assert w(A, A, A, NULL, A, 1e-5, A, 4, 64, NULL) == 1         # null inv_s
    assert w(A, A, NULL, A, A, 1e-5, A, 4, 64, NULL) == 1         # null shift
    assert w(A, A, A, A + 1, A, 1e-5, A, 4, 64, NULL) == 5        # inv_s at an odd address
    assert w(A, A, A, A, A, float("nan"), A, 4, 64, NULL) == 8
    assert w(A, A, A, A, A, 1e-5, A, 4, 32770, NULL) == 3
    n = L.ada_layer_norm_quant_nvfp4_swizzled_modfp8_bf16  # x, s8, h8, sdeq, hdeq, eps, packed, sf, rows, dim
    assert n(A, A, A, A, A, 1e-5, A, A, 4, 40, NULL) == 3         # dim % 16
    assert n(A, A, A, A, NULL, 1e-5, A, A, 4, 64, NULL) == 1      # null shift_deq
    assert n(A + 1, A, A, A, A, 1e-5, A, A, 4, 64, NULL) == 5     # x at an odd address
    assert n(A, A, A, A + 1, A, 1e-5, A, A, 4, 64, NULL) == 5     # scale_deq misaligned
    assert n(NULL, NULL, NULL, NULL, NULL, 1e-5, NULL, NULL, 0, 64, NULL) == 0


def test_seg_and_two_level_argument_errors(lib):
    L, _ = lib
    f = L.ada_layer_norm_quant_fp8_seg_bf16  # x, seg_idx, seg_scale, seg_shift, nseg, act, eps, out, rows, dim
    assert f(A, A, A, A, 0, A, 1e-5, A, 4, 64, NULL) == 4          # no segments
    assert f(A, NULL, A, A, 3, A, 1e-5, A, 4, 64, NULL) == 1       # null index
    assert f(A, A, A, A + 1, 3, A, 1e-5, A, 4, 64, NULL) == 5      # shift table at an odd address
    assert f(A, A + 2, A, A, 3, A, 1e-5, A, 4, 64, NULL) == 5      # index not 4-byte aligned
    assert f(A, A, A, A, 3, A, 1e-5, A, 4, 63, NULL) == 3          # odd dim
    assert f(NULL, NULL, NULL, NULL, 0, NULL, 1e-5, NULL, 0, 64, NULL) == 0
    g = L.ada_layer_norm_quant_nvfp4_swizzled_seg_bf16  # x, idx, s, h, nseg, eps, packed, sf, rows, dim
    assert g(A, A, A, A, 3, 1e-5, A, A, 4, 40, NULL) == 3          # dim % 16
    assert g(A, A, A, A, 3, 1e-5, A, NULL, 4, 64, NULL) == 1
    n = L.layer_norm_no_affine_quant_nvfp4_2level_bf16  # x, eps, packed, sf, ts, ws, rows, dim
    assert n(A, 1e-5, A, A, NULL, A, 4, 64, NULL) == 1             # null tensor scale
    assert n(A, 1e-5, A, A, A, NULL, 4, 64, NULL) == 1             # null workspace
    assert n(A, 1e-5, A, A, A + 2, A, 4, 64, NULL) == 5            # tensor scale misaligned
    assert n(A, 1e-5, A, A, A, A + 1, 4, 64, NULL) == 5            # workspace misaligned
    assert n(A, 1e-5, A, A, A, A + 8, 4, 64, NULL) == 5            # workspace not 16-byte aligned
    ws = L.nvfp4ap_2level_workspace_bytes
    assert ws(0) == 16 and ws(37810) == 16 + 16 * 37810 and ws(-1) == -1 and ws(1 << 62) == -1
    assert n(A, 1e-5, A, A, A, A, 4, 72, NULL) == 3
    assert n(NULL, 1e-5, NULL, NULL, NULL, NULL, 0, 64, NULL) == 0
    b = L.ada_layer_norm_quant_nvfp4_2level_bf16  # x, scale, shift, eps, packed, sf, ts, ws, rows, dim
    assert b(A, NULL, A, 1e-5, A, A, A, A, 4, 64, NULL) == 1
    assert b(A, A, A + 4, 1e-5, A, A, A, A, 4, 64, NULL) == 5
    w = L.swiglu_quant_nvfp4_2level_bf16  # gate, up, ld, packed, sf, ts, ws, rows, dim
    assert w(A, A, 64, A, A, A, A, 4, 40, NULL) == 3               # dim % 16
    assert w(A, A, 32, A, A, A, A, 4, 64, NULL) == 2               # ld < dim
    assert w(A, A, 68, A, A, A, A, 4, 64, NULL) == 2               # ld % 8
    assert w(A + 8, A, 64, A, A, A, A, 4, 64, NULL) == 5           # gate not 16-byte aligned
    assert w(A, A, 64, A, A, NULL, A, 4, 64, NULL) == 1
    assert w(NULL, NULL, 64, NULL, NULL, NULL, NULL, 0, 64, NULL) == 0
    assert w(A, A, 64, A, A, A, A, 1 << 29, 64, NULL) == 2         # rows * dim/8 >= 2^32 work items
    v = L.swiglu_bf16  # gate, up, ld, out, rows, dim
    assert v(A, A, 64, A, 1 << 29, 64, NULL) == 2
    assert v(A, A, 64, A, 4, 60, NULL) == 3                        # dim % 8
    assert v(A, A, 64, A + 2, 4, 64, NULL) == 5                    # out not 16-byte aligned
    assert v(A, A, 64, NULL, 4, 64, NULL) == 1
    c = L.ada_layer_norm_quant_nvfp4_2level_seg_bf16  # x, idx, s, h, nseg, eps, packed, sf, ts, ws, rows, dim
    assert c(A, A, A, A, -1, 1e-5, A, A, A, A, 4, 64, NULL) == 4
    assert c(A, A, A, A, 2, float("nan"), A, A, A, A, 4, 64, NULL) == 8


def test_modulation6_argument_errors(lib):
    L, _ = lib
    f = L.adaln_modulation6_bf16
    six = lambda *p: (ctypes.c_void_p * 6)(*p)
    outs = six(A, A, A, A, A, A)
    assert f(A, A, outs, -1, 4, 64, NULL) == 2
    assert f(A, A, outs, 1, 4, 0, NULL) == 2
    assert f(NULL, A, outs, 1, 4, 64, NULL) == 1
    assert f(A, A, six(A, A, A, NULL, A, A), 1, 4, 64, NULL) == 1
    assert f(A + 2, A, outs, 1, 4, 64, NULL) == 5              # params not 4-byte aligned
    assert f(A, A, six(A, A, A, A, A + 1, A), 1, 4, 64, NULL) == 5
    assert f(NULL, NULL, outs, 0, 4, 64, NULL) == 0            # no tokens: no-op


def test_noalloc_argument_errors(lib):
    L, _ = lib
    f = L.ada_layer_norm_quant_fp8_bf16_noalloc
    f.restype = ctypes.c_int
    p, i64, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float
    f.argtypes = [p, p, p, p, f32, p, i64, i64, p]
    assert f(A, A, A, A, 1e-5, A, 4, 60, NULL) == 3            # dim not a multiple of 8
    assert f(A, A, A, A, 1e-5, A, -4, 64, NULL) == 2
    assert f(A + 4, A, A, A, 1e-5, A, 4, 64, NULL) == 5        # x not 16-byte aligned
    assert f(A, A, A, A, 1e-5, NULL, 4, 64, NULL) == 1
    assert f(NULL, NULL, NULL, NULL, 1e-5, NULL, 0, 64, NULL) == 0


def test_two_level_single_read_binding(lib):
    # the binding's checks before any device query; without a device a valid
    # query reports NVFP4AP_ERR_LAUNCH (on a GPU machine it answers)
    import torch
    import nvfp4_activation_producer_gb300 as ap
    with pytest.raises(ValueError):
        ap.two_level_single_read(10, 3072, "diagonal")
    with pytest.raises(ap.NvFp4ApArgumentError):
        ap.two_level_single_read(10, 40)
    assert ap.two_level_single_read(0, 3072, "segmented") is False
    if not torch.cuda.is_available():
        with pytest.raises(ap.NvFp4ApError) as e:
            ap.two_level_single_read(5070, 3072)
        assert e.value.status == ap.ERR_LAUNCH
