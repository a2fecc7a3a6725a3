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


@pytest.fixture(params=["auto", "rows", "rows_c1", "tma", "blk", "rowblk"])
def path(request, monkeypatch):
    """Run a LayerNorm-producer test on each kernel family through the one
    selection setting the library reads (NVFP4AP_KERNEL=F[:C]): the default
    choice, the register row kernels for every form (3; the persistent
    broadcast kernel for the broadcast sources, the register-capped NVFP4
    instance where a row fills the CTA exactly), the same with one persistent
    CTA per SM (3:1, so every CTA walks many rows), the TMA pipeline wherever
    it applies (4), the block-per-lane persistent kernels (5) and the
    one-row-per-CTA block-per-lane kernels (8); a family that does not take a
    form or shape falls back to the register row kernels."""
    kernel = {"auto": None, "rows": "3", "rows_c1": "3:1", "tma": "4", "blk": "5", "rowblk": "8"}[request.param]
    if kernel is None:
        monkeypatch.delenv("NVFP4AP_KERNEL", raising=False)
    else:
        monkeypatch.setenv("NVFP4AP_KERNEL", kernel)
    return request.param
