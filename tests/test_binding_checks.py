"""The Python binding's tensor-contract checks, on the CPU (no library call).

The binding (README "Tensor Contract": bf16 (rows, dim) x, (dim,) vectors,
one-element fp32 scalars, contiguous CUDA tensors on one device) takes a fast
path for well-formed tensors and falls back to checks that name what is
wrong.  Every malformed argument must still be rejected with the same error as
before the fast path existed.
"""
import pytest
import torch

import nvfp4_activation_producer_gb300 as ap

CUDA0 = torch.device("cuda", 0)


@pytest.mark.parametrize("make,exc,msg", [
    (lambda: torch.empty(4, 4, dtype=torch.bfloat16), ValueError, "CUDA"),
    (lambda: torch.empty(4, dtype=torch.bfloat16), ValueError, "2-D"),
    (lambda: torch.empty(4, 4), TypeError, "bfloat16"),
    (lambda: [[1.0]], ValueError, "2-D"),
    (lambda: torch.nn.Parameter(torch.empty(4, 4, dtype=torch.bfloat16), requires_grad=False), ValueError, "CUDA"),
])
def test_x_rejected(make, exc, msg):
    with pytest.raises(exc, match=msg):
        ap._x(make())


@pytest.mark.parametrize("t,dtype,shape,device,exc,msg", [
    (torch.empty(3, dtype=torch.bfloat16), torch.bfloat16, (3,), CUDA0, ValueError, "CUDA"),
    (torch.empty(3, dtype=torch.bfloat16), torch.bfloat16, (3,), None, ValueError, "CUDA"),
    (torch.empty(3), torch.bfloat16, (3,), None, TypeError, "bfloat16"),
    ([1, 2, 3], torch.bfloat16, (3,), None, TypeError, "torch.Tensor"),
    (torch.empty(3, dtype=torch.float8_e4m3fn), torch.bfloat16, (3,), None, TypeError, "bfloat16"),
])
def test_need_rejected(t, dtype, shape, device, exc, msg):
    with pytest.raises(exc, match=msg):
        ap._need(t, "v", dtype, shape, device)


@pytest.mark.parametrize("t", [torch.tensor([1.0]), torch.tensor([1.0, 2.0]), torch.tensor([1], dtype=torch.int32),
                               1.0])
def test_scalar_rejected(t):
    with pytest.raises(TypeError, match="CUDA float32 tensor with one element"):
        ap._scalar(t, "act_scale", CUDA0)

