"""The failure path of the kernels' bounded waits in the real forward and backward, made
to happen without a fault: the test entry qat_debug_set_wait_limit_us lowers the wait
limit, so the kernels give up at their first slow wait, set the device error word, let
every copy and MMA they issued complete, and return.  The torch path must report it
(check=True raises QatError), and the next normal call must match the oracle."""

import numpy as np
import pytest
import torch

from oracle import qat_oracle as orc
from quantization_aware_attention_gb300 import attention
from quantization_aware_attention_gb300 import build as qbuild
from quantization_aware_attention_gb300 import capi
from quantization_aware_attention_gb300.attention import (qat_attention_backward,
                                                          qat_attention_forward)
from quantization_aware_attention_gb300.capi import QatError, Status
from quantization_aware_attention_gb300.inputs import custom_inputs

from gpu_util import TOL_Q, dev_bf16, host_f64, oracle_f64, rel_l2

pytestmark = pytest.mark.gpu

DEFAULT_LIMIT_US = 4000000


@pytest.fixture(scope="module", autouse=True)
def built():
    qbuild.build()


@pytest.fixture()
def low_limit():
    assert capi.qat_debug_set_wait_limit_us(0) == Status.OK
    try:
        yield
    finally:
        assert capi.qat_debug_set_wait_limit_us(DEFAULT_LIMIT_US) == Status.OK
        capi.qat_attn_device_status()  # leave the error word clear


def _inputs():
    inp = custom_inputs(270, 1, 8, 2048, 2048, 128)
    return inp, [dev_bf16(inp[n]) for n in ("q", "k", "v", "do")]


def test_expired_wait_raises_on_the_torch_path(low_limit):
    _, (q, k, v, do) = _inputs()
    raised = None
    for _ in range(5):          # a wait slower than a few hundred polls comes at once
        try:
            attention(q, k, v, check=True)
        except QatError as e:
            raised = e
            break
    assert raised is not None and raised.status == Status.TIMEOUT
    assert capi.qat_attn_device_status() == Status.OK   # the raise read and cleared it


def test_expired_wait_in_the_backward_sets_the_error_word(low_limit):
    _, (q, k, v, do) = _inputs()
    assert capi.qat_debug_set_wait_limit_us(DEFAULT_LIMIT_US) == Status.OK
    _, o_hp, lse = qat_attention_forward(q, k, v)
    assert capi.qat_attn_device_status() == Status.OK
    assert capi.qat_debug_set_wait_limit_us(0) == Status.OK
    seen = False
    for _ in range(5):
        qat_attention_backward(q, k, v, o_hp, lse, do)
        if capi.qat_attn_device_status() == Status.TIMEOUT:
            seen = True
            break
    assert seen
    # without check the autograd path does not synchronize; the word waits for a reader
    qq = q.clone().requires_grad_(True)
    attention(qq, k, v, check=False).backward(do)
    torch.cuda.synchronize()
    assert capi.qat_attn_device_status() in (Status.TIMEOUT, Status.OK)


def test_context_usable_after_expired_waits():
    """After the tests above: default limit, clean error word, and a forward + backward
    that matches the oracle."""
    assert capi.qat_attn_device_status() == Status.OK
    inp = custom_inputs(271, 1, 2, 200, 200, 128)
    q, k, v = (dev_bf16(inp[n]).requires_grad_(True) for n in ("q", "k", "v"))
    sc = 1.0 / np.sqrt(128)
    out = attention(q, k, v, True, sc, check=True)
    out.backward(dev_bf16(inp["do"]))
    torch.cuda.synchronize()
    f = oracle_f64(inp)
    wq, _, _ = orc.forward(f["q"], f["k"], f["v"], sc, True, quant=True)
    gq, gk, gv = orc.backward(f["q"], f["k"], f["v"], f["do"], sc, True)
    assert rel_l2(host_f64(out), wq) <= TOL_Q
    for g, w in ((q.grad, gq), (k.grad, gk), (v.grad, gv)):
        assert rel_l2(host_f64(g), w) <= TOL_Q
    assert capi.qat_attn_device_status() == Status.OK
