"""GPU parity of smooth_k in the backward ("attn_qat_train.py"): the SMOOTH_K dQ term of
_attn_bwd_dq (dq += rowsum(ds) k_mean) under the page's default backward (quant_mode 2,
Delta from O_q, where the term is not zero) and under the straight-through one, and the
backward on the unquantized inputs (_attention.forward with use_qat_qkv_backward =
False keeps q, k - k_mean and v).  The oracle builds its own fake-quantized inputs with
the same fp32 rule and rematerializes P from the saved lse as the page does."""

import numpy as np
import pytest
import torch

from oracle import qat_oracle as orc
from quantization_aware_attention_gb300 import attention
from quantization_aware_attention_gb300 import build as qbuild
from quantization_aware_attention_gb300 import capi
from quantization_aware_attention_gb300.attention import qat_subtract_mean
from quantization_aware_attention_gb300.capi import Status
from quantization_aware_attention_gb300.inputs import WORKLOADS, custom_inputs, make_inputs

from gpu_util import TOL_Q, dev_bf16, host_f64, oracle_f64, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    qbuild.build()


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def test_subtract_mean_bit_exact():
    inp = custom_inputs(260, 2, 3, 70, 70, 128)
    x = dev_bf16(inp["k"])
    mu = (np.random.default_rng(261).standard_normal(128) * 2).astype(np.float32)
    out = qat_subtract_mean(x, torch.from_numpy(mu).cuda())
    torch.cuda.synchronize()
    want = orc.subtract_mean_bf16(orc.bf16_bits_to_f64(inp["k"]).astype(np.float32), mu)
    assert np.array_equal(_bits(out), (want.view(np.uint32) >> 16).astype(np.uint16))


def _grads(inp, quant_mode, use_qat_qkv_backward, causal, sm_scale):
    q, k, v = (dev_bf16(inp[n]).requires_grad_(True) for n in ("q", "k", "v"))
    out = attention(q, k, v, causal, sm_scale, quant_mode, qkv_quant=True, smooth_k=True,
                    use_qat_qkv_backward=use_qat_qkv_backward, check=True)
    out.backward(dev_bf16(inp["do"]))
    torch.cuda.synchronize()
    assert capi.qat_attn_device_status() == Status.OK
    return q.grad, k.grad, v.grad


def _oracle_head(f, b, h, mu32, quant_mode, use_qat_qkv_backward, causal, sm_scale):
    q32, k32, v32 = (f[n][b, h].astype(np.float32) for n in ("q", "k", "v"))
    fq = orc.fake_quant_tokens_fp32(q32)[0].astype(np.float64)
    fk = orc.fake_quant_tokens_fp32(k32, mu32)[0].astype(np.float64)
    fv = orc.fake_quant_tokens_fp32(v32)[0].astype(np.float64)
    page = quant_mode == capi.QUANT_P_FP8E4M3_ROW_TILE64_PAGE_BWD
    mu = mu32.astype(np.float64)
    if use_qat_qkv_backward:
        if page:
            return orc.head_backward_page(fq, fk, fv, f["do"][b, h], sm_scale, causal, k_mean=mu)
        return orc.head_backward(fq, fk, fv, f["do"][b, h], sm_scale, causal, k_mean=mu)
    r = orc.head_forward(fq, fk, fv, sm_scale, causal, True)
    ks = orc.subtract_mean_bf16(k32, mu32).astype(np.float64)
    return orc.head_backward_from_stats(f["q"][b, h], ks, f["v"][b, h], f["do"][b, h],
                                        r["o_q"] if page else r["o_hp"], r["lse"], sm_scale,
                                        causal, quant_dv=page, k_mean=mu)


@pytest.mark.parametrize("quant_mode,use_qat_qkv_backward", [
    (capi.QUANT_P_FP8E4M3_ROW_TILE64_PAGE_BWD, True),
    (capi.QUANT_P_FP8E4M3_ROW_TILE64_PAGE_BWD, False),
    (capi.QUANT_P_FP8E4M3_ROW_TILE64, False),
])
def test_smooth_k_backward_c3_outlier_channels(quant_mode, use_qat_qkv_backward):
    """The DiT workload with per-channel K offsets through attention(qkv_quant=True,
    smooth_k=True): dQ, dK, dV of three heads against the oracle."""
    w = WORKLOADS["c3"]
    inp = make_inputs(w)
    dq, dk, dv = _grads(inp, quant_mode, use_qat_qkv_backward, w.causal, w.sm_scale)
    f = oracle_f64(inp)
    mu32 = orc.channel_mean(f["k"]).astype(np.float32)
    got, want = {n: [] for n in "qkv"}, {n: [] for n in "qkv"}
    for b, h in ((0, 0), (0, 11), (0, 23)):
        g = _oracle_head(f, b, h, mu32, quant_mode, use_qat_qkv_backward, w.causal, w.sm_scale)
        for n, gt, val in zip("qkv", (dq, dk, dv), g):
            got[n].append(host_f64(gt[b, h]))
            want[n].append(val)
    e = {n: rel_l2(np.stack(got[n]), np.stack(want[n])) for n in got}
    print("errors", {n: f"{x:.2e}" for n, x in e.items()})
    assert all(x <= TOL_Q for x in e.values()), e


def test_smooth_k_term_changes_page_dq_only():
    """The SMOOTH_K term is what separates the two dQ: without it dQ under quant_mode 2
    moves away from the oracle; dK and dV do not change (the same kernels, bit for bit)."""
    inp = custom_inputs(262, 1, 2, 300, 300, 128)
    f = oracle_f64(inp)
    # channel offsets ~ N(0, 2^2) as in the DiT workload.  (The term multiplies
    # rowsum(dS) = Delta(O_hp) - Delta(O_q), whose error is set by the bf16 rounding of the
    # stored O_q; larger offsets scale that error up.)
    kk = f["k"] + (np.random.default_rng(263).standard_normal(128) * 2)[None, None, None, :]
    k_bits = (orc.f32_to_bf16_rn(kk.astype(np.float32)).view(np.uint32) >> 16).astype(np.uint16)
    q, k, v, do = dev_bf16(inp["q"]), dev_bf16(k_bits), dev_bf16(inp["v"]), dev_bf16(inp["do"])
    from quantization_aware_attention_gb300 import qat_prepare_qkv
    from quantization_aware_attention_gb300.attention import (qat_attention_backward,
                                                              qat_attention_forward)
    qf, kf, vf, k_mean = qat_prepare_qkv(q, k, v, smooth_k=True)
    sc, page = 1.0 / np.sqrt(128), capi.QUANT_P_FP8E4M3_ROW_TILE64_PAGE_BWD
    o_q, _, lse = qat_attention_forward(qf, kf, vf, False, sc, page)
    with_t = qat_attention_backward(qf, kf, vf, o_q, lse, do, False, sc, page, k_mean=k_mean)
    without = qat_attention_backward(qf, kf, vf, o_q, lse, do, False, sc, page)
    torch.cuda.synchronize()
    assert torch.equal(with_t[1], without[1]) and torch.equal(with_t[2], without[2])
    mu32 = k_mean.cpu().numpy()
    want = []
    for h in range(2):
        fq = orc.fake_quant_tokens_fp32(f["q"][0, h].astype(np.float32))[0].astype(np.float64)
        fk = orc.fake_quant_tokens_fp32(orc.bf16_bits_to_f64(k_bits)[0, h].astype(np.float32),
                                        mu32)[0].astype(np.float64)
        fv = orc.fake_quant_tokens_fp32(f["v"][0, h].astype(np.float32))[0].astype(np.float64)
        want.append(orc.head_backward_page(fq, fk, fv, f["do"][0, h], sc, False,
                                           k_mean=mu32.astype(np.float64))[0])
    want = np.stack(want)
    e_with = rel_l2(host_f64(with_t[0][0]), want)
    e_without = rel_l2(host_f64(without[0][0]), want)
    print(f"dq error with the term {e_with:.2e}, without {e_without:.2e}")
    assert e_with <= TOL_Q < e_without
