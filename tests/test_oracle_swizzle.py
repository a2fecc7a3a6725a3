"""Pins of the oracle's swizzled scale layout (CPU only).

- The size formula reproduces every qdata/sfa byte count of the NVFP4 ring
  records on the h3-blackwell-runtime compare page.
- The offset map is a bijection onto the non-padding bytes.
- The layout equals an independent formulation of the 128x4 block-scale tile
  layout as tensor reshapes/permutes (the form in which public block-scaled
  GEMM documentation describes it): pad to (128*Rt, 4*Ct), view as
  (Rt, 4, 32, Ct, 4) [row = 128*rt + 32*g + i], permute to (Rt, Ct, i, g, c).
"""
import json
import os

import numpy as np
import pytest
import torch


def test_sizes_match_page_ring_records(orc, golden_dir):
    g = json.load(open(os.path.join(golden_dir, "nvfp4_ring_sizes.json")))
    for rec in g["records"]:
        rows, k = rec["row_capacity"], rec["K"]
        assert orc.swizzled_sf_size(rows, k) == rec["sfa_bytes"]
        assert rows * k // 2 == rec["qdata_bytes"]


def test_size_padding_and_invalid(orc):
    assert orc.swizzled_sf_size(0, 64) == 0
    assert orc.swizzled_sf_size(1, 16) == 128 * 4
    assert orc.swizzled_sf_size(129, 80) == 256 * 8          # 5 blocks -> 8 columns
    assert orc.swizzled_sf_size(5070, 3072) == 5120 * 192    # 983,040 bytes
    assert orc.swizzled_sf_size(10, 24) == -1
    assert orc.swizzled_sf_size(-1, 64) == -1
    assert orc.swizzled_sf_size(10, 0) == -1


@pytest.mark.parametrize("rows,dim", [(1, 16), (127, 48), (128, 64), (129, 80), (300, 1040), (257, 3072)])
def test_offsets_bijective(orc, rows, dim):
    nblk = dim // 16
    r, c = np.meshgrid(np.arange(rows), np.arange(nblk), indexing="ij")
    off = orc.sf_offsets(r.ravel(), c.ravel(), dim)
    size = orc.swizzled_sf_size(rows, dim)
    assert off.min() >= 0 and off.max() < size
    assert np.unique(off).size == off.size


def _blocked_reference(logical: np.ndarray) -> np.ndarray:
    rows, cols = logical.shape
    rt, ct = -(-rows // 128), -(-cols // 4)
    pad = torch.zeros((rt * 128, ct * 4), dtype=torch.uint8)
    pad[:rows, :cols] = torch.from_numpy(logical)
    t = pad.view(rt, 4, 32, ct, 4).permute(0, 3, 2, 1, 4)
    return t.contiguous().view(-1).numpy()


@pytest.mark.parametrize("rows,dim", [(1, 16), (128, 64), (200, 96), (257, 3072), (5, 1040)])
def test_layout_equals_reshape_formulation(orc, rows, dim):
    rng = np.random.default_rng(rows * 7 + dim)
    logical = rng.integers(1, 256, size=(rows, dim // 16), dtype=np.uint8)
    got = orc.swizzle_scales(logical, rows, dim)
    assert np.array_equal(got, _blocked_reference(logical))


def test_padding_is_zero_and_every_scale_once(orc):
    rows, dim = 130, 80  # ragged in both rows (130 % 128) and columns (5 % 4)
    logical = np.arange(1, rows * 5 + 1, dtype=np.int64).reshape(rows, 5)
    logical = (logical % 255 + 1).astype(np.uint8)  # never zero
    buf = orc.swizzle_scales(logical, rows, dim)
    assert buf.size == 256 * 8
    assert np.count_nonzero(buf) == rows * 5
    assert sorted(buf[buf != 0].tolist()) == sorted(logical.ravel().tolist())
