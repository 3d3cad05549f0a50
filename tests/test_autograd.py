"""The autograd contract of "support for pytorch autograd" (SageAttention issue 60):
for q, k, v of shape (2, 4, 8, 64) with requires_grad, the attention output must carry
requires_grad and back-propagate non-None, finite gradients -- here the straight-through
gradients of the high-precision output, checked against torch float64 autograd."""

import math

import pytest
import torch

from quantization_aware_attention_gb300 import attention
from quantization_aware_attention_gb300 import build as qbuild

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    qbuild.build()


def test_page_autograd_contract():
    torch.manual_seed(0)
    q = torch.randn((2, 4, 8, 64), device="cuda", dtype=torch.bfloat16, requires_grad=True)
    k = torch.randn_like(q, requires_grad=True)
    v = torch.randn_like(q, requires_grad=True)
    out = attention(q, k, v)
    assert out.requires_grad
    sdpa = torch.nn.functional.scaled_dot_product_attention(q, k, v)
    assert sdpa.requires_grad
    do = torch.randn_like(out)
    out.backward(do)
    for t in (q, k, v):
        assert t.grad is not None and torch.isfinite(t.grad).all()
    # straight-through: gradients are those of plain softmax attention
    q64, k64, v64 = (t.detach().double().requires_grad_(True) for t in (q, k, v))
    ref = torch.softmax(q64 @ k64.transpose(-1, -2) / math.sqrt(64), -1) @ v64
    ref.backward(do.double())
    for t, r in ((q, q64), (k, k64), (v, v64)):
        err = (t.grad.double() - r.grad).norm() / r.grad.norm()
        assert err < 1e-2, float(err)
    # the returned output is the quantized one
    assert (out.double() - ref.detach()).norm() / ref.norm() < 5e-2
