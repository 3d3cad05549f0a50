"""GPU parity of the Q/K/V fake-quantization path ("attn_qat_train.py",
_attention.forward with IS_QAT and smooth_k): the token-block FP8 rule bit for bit, the
channel mean, and attention on fake-quantized inputs against the fp64 oracle, which
builds its own quantized inputs with the same fp32 rule."""

import numpy as np
import pytest
import torch

from oracle import qat_oracle as orc
from quantization_aware_attention_gb300 import attention, qat_prepare_qkv
from quantization_aware_attention_gb300 import build as qbuild
from quantization_aware_attention_gb300 import capi
from quantization_aware_attention_gb300.attention import (qat_attention_backward,
                                                          qat_attention_forward)
from quantization_aware_attention_gb300.capi import Status
from quantization_aware_attention_gb300.inputs import WORKLOADS, custom_inputs, make_inputs

from gpu_util import TOL_HP, TOL_Q, dev_bf16, host_f64, oracle_f64, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    qbuild.build()


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("B,H,N,D,with_mean", [(2, 3, 100, 128, True), (1, 2, 100, 128, False),
                                               (2, 2, 33, 64, True), (1, 1, 7, 64, False)])
def test_fake_quant_tokens_bit_exact(B, H, N, D, with_mean):
    inp = custom_inputs(300 + N + D, B, H, N, N, D)
    x = inp["k"].copy()
    xf = orc.bf16_bits_to_f64(x).astype(np.float32)
    xf[..., 5] *= 40.0                                  # an outlier channel
    if N > 64:
        xf[:, :, 32:64] = 0.0                           # an all-zero block
    x = (xf.view(np.uint32) >> 16).astype(np.uint16)    # truncated to bf16; both sides use these bits
    mean = (np.random.default_rng(7).standard_normal(D) * 3).astype(np.float32) if with_mean else None
    dx = dev_bf16(x)
    out = torch.empty_like(dx)
    nb = (N + 31) // 32
    scales = torch.empty((B, H, nb), dtype=torch.float32, device="cuda")
    dm = torch.from_numpy(mean).cuda() if with_mean else None
    assert capi.qat_fake_quant_tokens(dx, dm, out, scales, B, H, N, D) == Status.OK
    torch.cuda.synchronize()
    got_bits, got_sc = _bits(out), scales.cpu().numpy()
    xv = orc.bf16_bits_to_f64(x).astype(np.float32)
    for b in range(B):
        for h in range(H):
            w_out, w_sc, _ = orc.fake_quant_tokens_fp32(xv[b, h], mean)
            w_bits = (w_out.view(np.uint32) >> 16).astype(np.uint16)
            assert np.array_equal(got_bits[b, h], w_bits), (b, h)
            assert np.array_equal(got_sc[b, h].view(np.uint32), w_sc.view(np.uint32)), (b, h)


def test_channel_mean():
    w = WORKLOADS["c3"]
    inp = make_inputs(w, with_do=False)
    k = dev_bf16(inp["k"])
    mean = torch.empty(w.D, dtype=torch.float32, device="cuda")
    assert capi.qat_channel_mean(k, mean, w.B, w.H, w.Nkv, w.D) == Status.OK
    want = orc.channel_mean(orc.bf16_bits_to_f64(inp["k"]))
    assert np.allclose(mean.cpu().numpy(), want, rtol=1e-5, atol=1e-5)


def test_qkv_quant_attention_c3_outlier_channels():
    """The full IS_QAT path on the DiT workload with per-channel K offsets: smooth_k,
    Q/K/V fake quantization, QAT attention forward and the straight-through backward."""
    w = WORKLOADS["c3"]
    inp = make_inputs(w)
    q, k, v, do = (dev_bf16(inp[n]) for n in ("q", "k", "v", "do"))
    qf, kf, vf, k_mean = qat_prepare_qkv(q, k, v, smooth_k=True)
    o_q, o_hp, lse = qat_attention_forward(qf, kf, vf, False, w.sm_scale)
    dq, dk, dv = qat_attention_backward(qf, kf, vf, o_hp, lse, do, False, w.sm_scale)
    torch.cuda.synchronize()
    assert capi.qat_attn_device_status() == Status.OK
    f = oracle_f64(inp)
    mu = orc.channel_mean(f["k"]).astype(np.float32)
    assert np.allclose(k_mean.cpu().numpy(), mu, rtol=1e-5, atol=1e-5)
    errs = {n: [] for n in ("o_q", "o_hp", "lse", "dq", "dk", "dv")}
    got = dict(o_q=o_q, o_hp=o_hp, lse=lse, dq=dq, dk=dk, dv=dv)
    for b, h in ((0, 0), (0, 11), (0, 23)):
        fq = orc.fake_quant_tokens_fp32(f["q"][b, h].astype(np.float32))[0].astype(np.float64)
        fk = orc.fake_quant_tokens_fp32(f["k"][b, h].astype(np.float32), mu)[0].astype(np.float64)
        fv = orc.fake_quant_tokens_fp32(f["v"][b, h].astype(np.float32))[0].astype(np.float64)
        r = orc.head_forward(fq, fk, fv, w.sm_scale, False, True)
        g = orc.head_backward(fq, fk, fv, f["do"][b, h], w.sm_scale, False)
        for n, val in (("o_q", r["o_q"]), ("o_hp", r["o_hp"]), ("lse", r["lse"]),
                       ("dq", g[0]), ("dk", g[1]), ("dv", g[2])):
            errs[n].append((host_f64(got[n][b, h]), val))
    e = {n: rel_l2(np.stack([a for a, _ in x]), np.stack([c for _, c in x])) for n, x in errs.items()}
    print("errors", {n: f"{v:.2e}" for n, v in e.items()})
    assert e["o_hp"] <= TOL_HP and e["lse"] <= TOL_HP, e
    for n in ("o_q", "dq", "dk", "dv"):
        assert e[n] <= TOL_Q, (n, e)
    # smooth_k is what keeps K's quantization error small under outlier channels
    kf_plain = qat_prepare_qkv(q, k, v, smooth_k=False)[1]
    k64 = host_f64(k)
    err_smooth = rel_l2(host_f64(kf) + k_mean.cpu().numpy().astype(np.float64), k64)
    err_plain = rel_l2(host_f64(kf_plain), k64)
    assert err_smooth < err_plain


def test_qkv_quant_autograd():
    inp = custom_inputs(808, 2, 4, 40, 40, 64)
    q, k, v = (dev_bf16(inp[n]).requires_grad_(True) for n in ("q", "k", "v"))
    out = attention(q, k, v, qkv_quant=True, smooth_k=True)
    assert out.requires_grad
    out.backward(dev_bf16(inp["do"]))
    for t in (q, k, v):
        assert t.grad is not None and torch.isfinite(t.grad).all()
    with pytest.raises(ValueError):
        attention(q, k, v, smooth_k=True)
