"""GPU parity of quant_mode 2, the page's default backward ("attn_qat_train.py",
_attn_bwd_dkdv with use_high_prec_o = False): dV from the quantized P, Delta from O_q,
dS from the unquantized P -- against the oracle's head_backward_page."""

import numpy as np
import pytest
import torch

from oracle import qat_oracle as orc
from quantization_aware_attention_gb300 import attention
from quantization_aware_attention_gb300 import build as qbuild
from quantization_aware_attention_gb300 import capi
from quantization_aware_attention_gb300.attention import (qat_attention_backward,
                                                          qat_attention_forward)
from quantization_aware_attention_gb300.capi import Status
from quantization_aware_attention_gb300.inputs import WORKLOADS, custom_inputs, make_inputs

from gpu_util import TOL_Q, dev_bf16, host_f64, oracle_f64, rel_l2

pytestmark = pytest.mark.gpu
MODE = capi.QUANT_P_FP8E4M3_ROW_TILE64_PAGE_BWD


@pytest.fixture(scope="module", autouse=True)
def built():
    qbuild.build()


def _check(inp, causal, sc, heads):
    q, k, v, do = (dev_bf16(inp[n]) for n in ("q", "k", "v", "do"))
    o_q, o_hp, lse = qat_attention_forward(q, k, v, causal, sc, MODE)
    dq, dk, dv = qat_attention_backward(q, k, v, o_q, lse, do, causal, sc, MODE)
    torch.cuda.synchronize()
    assert capi.qat_attn_device_status() == Status.OK
    f = oracle_f64(inp)
    got = {n: [] for n in ("dq", "dk", "dv")}
    want = {n: [] for n in got}
    for b, h in heads:
        w = orc.head_backward_page(f["q"][b, h], f["k"][b, h], f["v"][b, h], f["do"][b, h],
                                   sc, causal)
        for n, g, x in zip(("dq", "dk", "dv"), (dq, dk, dv), w):
            got[n].append(host_f64(g[b, h]))
            want[n].append(x)
    e = {n: rel_l2(np.stack(got[n]), np.stack(want[n])) for n in got}
    assert all(x <= TOL_Q for x in e.values()), e
    # and it really is the other variant: dV differs from the straight-through one
    _, _, dv_ste = qat_attention_backward(q, k, v, o_hp, lse, do, causal, sc)
    assert rel_l2(host_f64(dv), host_f64(dv_ste)) > 1e-3
    return e


def test_page_backward_c1():
    w = WORKLOADS["c1"]
    _check(make_inputs(w), False, w.sm_scale, [(0, 0), (0, 1)])


@pytest.mark.parametrize("B,H,N,D,causal", [(1, 2, 200, 128, True), (2, 1, 130, 64, False),
                                            (1, 1, 65, 128, True),
                                            (1, 1, 2048, 64, False)])  # dK/dV stream-K: 64 ranges of 4 blocks
def test_page_backward_edges(B, H, N, D, causal):
    inp = custom_inputs(1200 + N, B, H, N, N, D)
    _check(inp, causal, 1.0 / np.sqrt(D), [(b, h) for b in range(B) for h in range(H)])


def test_page_backward_autograd():
    inp = custom_inputs(1300, 1, 2, 96, 96, 128)
    q, k, v = (dev_bf16(inp[n]).requires_grad_(True) for n in ("q", "k", "v"))
    attention(q, k, v, quant_mode=MODE).backward(dev_bf16(inp["do"]))
    for t in (q, k, v):
        assert t.grad is not None and torch.isfinite(t.grad).all()
