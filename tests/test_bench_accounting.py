"""bench.py's accounting, on the CPU: the algorithmic bytes every GB/s and
roofline figure divides by (the per-op formulas: each input element the
producer uses read once, each output byte written once), and the kernel
launches per call that the JSON line's gpu_launches counts."""
import sys
import types

import pytest

sys.argv = sys.argv[:1]
import bench  # noqa: E402


def _w(R, D):
    # the shape is all the formulas read for these producers
    return types.SimpleNamespace(rows=R, dim=D, inputs={})


def _sf(R, D):
    return ((R + 127) // 128 * 128) * ((D // 16 + 3) // 4 * 4)


@pytest.mark.parametrize("name,make,expect", [
    # x read, codes written, plus the broadcast vectors and the act_scale word
    ("fp8_broadcast", lambda: _w(4096, 3072), 4096 * 3072 * 3 + 4 * 3072 + 4),
    ("fp8_layer_norm", lambda: _w(4096, 3072), 4096 * 3072 * 3 + 4),
    # per-token: x and the two (R, D) bf16 tensors read
    ("fp8_per_token", lambda: _w(2520, 3072), 2520 * 3072 * 7 + 4),
    # table: x, two of the six temb chunks, two fp32 table rows
    ("fp8_table", lambda: _w(4096, 3072), 4096 * 3072 * 7 + 8 * 3072 + 4),
    # NVFP4: x read, half a byte per element, the padded swizzled scale buffer
    ("nvfp4_layer_norm", lambda: _w(5070, 3072), 5070 * 3072 * 2 + 5070 * 1536 + _sf(5070, 3072)),
    ("nvfp4_broadcast", lambda: _w(5070, 3072),
     5070 * 3072 * 2 + 4 * 3072 + 5070 * 1536 + _sf(5070, 3072)),
    # six-way: fp32 params and modulation read, six bf16 outputs written
    ("modulation6", lambda: _w(5070, 3072), 5070 * 3072 * 36 + 24 * 3072),
])
def test_alg_bytes(name, make, expect):
    assert bench.alg_bytes(name, make()) == expect


def test_swizzled_buffer_size_matches_the_library_formula():
    # the 128x4 layout: rows padded to 128, 16-element blocks padded to 4 columns
    assert _sf(5070, 3072) == 5120 * 192 == 983040


@pytest.mark.parametrize("name,n", [("nvfp4_2level_layer_norm", 3), ("nvfp4_2level_seg_h3", 3),
                                    ("nvfp4_2level_swiglu_h3", 3), ("swiglu_values_h3", 1), ("fp8_broadcast", 1),
                                    ("modulation6", 1), ("fp8_seg_h3", 1)])
def test_launches_per_call(name, n):
    assert bench.launches_per_call(name) == n


def test_shape_suffixed_lines_count_as_their_producer():
    # per_op lines of a producer at another shape (the pages' FP8 shapes)
    assert bench.op_kind("fp8_broadcast_16x2048") == "fp8_broadcast"
    assert bench.op_kind("fp8_layer_norm_32768x3072") == "fp8_layer_norm"
    assert bench.op_kind("nvfp4_2level_seg_h3") == "nvfp4_2level_seg_h3"
    assert bench.alg_bytes("fp8_broadcast_16x2048", _w(16, 2048)) == 16 * 2048 * 3 + 4 * 2048 + 4
    assert bench.alg_bytes("fp8_layer_norm_2520x3072", _w(2520, 3072)) == 2520 * 3072 * 3 + 4
    names = [n for n, _ in bench.page_shape_workloads()]
    for R, D, _, _ in bench.PAGE_FP8_SHAPES:
        if (R, D) != (4096, 3072):
            assert f"fp8_broadcast_{R}x{D}" in names and f"fp8_layer_norm_{R}x{D}" in names
    assert bench.page_context("fp8_broadcast_16x2048", 16, 2048)["us"] == 4.117
    assert bench.page_context("fp8_layer_norm", 4096, 3072)["us"] == 16.412
    assert bench.page_context("nvfp4_broadcast", 5070, 3072) is None


@pytest.mark.parametrize("passes", [1, 2])
def test_two_level_layer_norm_bytes_follow_the_passes(monkeypatch, passes):
    # the input is counted once per pass the library makes over it
    monkeypatch.setattr(bench, "two_level_passes", lambda name, w: passes)
    R, D = 5070, 3072
    assert bench.alg_bytes("nvfp4_2level_layer_norm", _w(R, D)) == passes * 2 * R * D + R * D // 2 + _sf(R, D) + 4
    assert bench.launches_per_call("nvfp4_2level_layer_norm", _w(R, D)) == 1 + passes


def test_two_level_passes_without_a_device():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device answers the query")
    assert bench.two_level_passes("nvfp4_2level_layer_norm", _w(5070, 3072)) == 2
