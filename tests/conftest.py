"""Test configuration: the ``gpu`` marker and the shared fixtures.

Tests marked ``gpu`` need a CUDA device and the compiled CUDA library; all
others run on the CPU (the oracle's pins, host-side argument checks, the
library's exported symbols, the multi-rank host logic over gloo).
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the compiled CUDA library")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="session")
def dev():
    """cuda:0 with the CUDA library built; a gpu test fails (not skips) without them."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for a gpu-marked test")
    from nvfp4_activation_producer_gb300 import build as b
    b.build()
    import nvfp4_activation_producer_gb300 as ap
    ap.library_path()
    return torch.device("cuda:0")


@pytest.fixture(scope="session")
def ap(dev):
    import nvfp4_activation_producer_gb300 as ap
    return ap


@pytest.fixture(params=["auto", "rows", "rows_flat", "tile4", "tma", "ring", "legacy", "blk"])
def path(request, monkeypatch):
    """Run a LayerNorm-producer test on each kernel family: the default choice
    (TMA pipeline for the table form, register row kernels otherwise), the
    register row kernels for every form (NVFP4AP_KERNEL=3) with and without
    the persistent broadcast variant and the register-capped NVFP4 instance
    (NVFP4AP_PERSIST=-1, NVFP4AP_FULL=0), the NVFP4
    four-row-tile variant (NVFP4AP_TILE4=1), the TMA pipeline
    for every form (4), the warp-per-row TMA ring (1), the first register
    kernels (2) and the block-per-lane persistent kernels (5)."""
    kernel = {"auto": None, "rows": "3", "rows_flat": "3", "tile4": "3", "tma": "4", "ring": "1",
              "legacy": "2", "blk": "5"}[request.param]
    if kernel is None:
        monkeypatch.delenv("NVFP4AP_KERNEL", raising=False)
    else:
        monkeypatch.setenv("NVFP4AP_KERNEL", kernel)
    if request.param == "rows_flat":
        monkeypatch.setenv("NVFP4AP_PERSIST", "-1")
        monkeypatch.setenv("NVFP4AP_FULL", "0")
    else:
        monkeypatch.delenv("NVFP4AP_PERSIST", raising=False)
        monkeypatch.delenv("NVFP4AP_FULL", raising=False)
    if request.param == "tile4":
        monkeypatch.setenv("NVFP4AP_TILE4", "1")
    else:
        monkeypatch.delenv("NVFP4AP_TILE4", raising=False)
    return request.param
