"""GPU parity of the key-chunk forward and the lse merge (the single-GPU building block
of ring attention, "usp: differentiable operators for training (Ulysses/Ring/local
attention)"): chunks starting at multiples of 64 keys, merged, reproduce the one-pass
forward and the oracle."""

import numpy as np
import pytest
import torch

from oracle import qat_oracle as orc
from quantization_aware_attention_gb300 import build as qbuild
from quantization_aware_attention_gb300 import capi
from quantization_aware_attention_gb300.attention import qat_attention_forward
from quantization_aware_attention_gb300.capi import Status
from quantization_aware_attention_gb300.inputs import custom_inputs

from gpu_util import TOL_HP, TOL_Q, dev_bf16, host_f64, oracle_f64, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    qbuild.build()


def chunked_forward(q, k, v, edges, sm_scale, quant=1):
    B, H, Nq, D = q.shape
    Nkv = k.shape[2]
    acc = part = None
    out_q = torch.empty_like(q)
    out_h = torch.empty_like(q)
    for i, (lo, hi) in enumerate(zip(edges[:-1], edges[1:])):
        buf = (torch.empty(B, H, Nq, D, device="cuda"), torch.empty(B, H, Nq, D, device="cuda"),
               torch.empty(B, H, Nq, device="cuda"))
        st = capi.qat_attn_fwd_chunk(q, k, v, *buf, B, H, Nq, Nkv, lo, hi - lo, D, sm_scale, quant)
        assert st == Status.OK
        if acc is None:
            acc = buf
        else:
            last = i == len(edges) - 2
            st = capi.qat_attn_merge(*acc, *buf, out_q if last else None, out_h if last else None,
                                     B, H, Nq, D)
            assert st == Status.OK
    torch.cuda.synchronize()
    return out_q, out_h, acc[2]


@pytest.mark.parametrize("B,H,Nq,Nkv,D,edges", [
    (1, 3, 200, 600, 128, (0, 192, 448, 600)),
    (2, 2, 130, 512, 64, (0, 256, 512)),
    (1, 4, 257, 320, 128, (0, 64, 128, 320)),
])
def test_chunks_merge_to_one_pass(B, H, Nq, Nkv, D, edges):
    inp = custom_inputs(900 + Nkv, B, H, Nq, Nkv, D)
    q, k, v = (dev_bf16(inp[n]) for n in ("q", "k", "v"))
    sc = 1.0 / np.sqrt(D)
    oq, oh, lse = chunked_forward(q, k, v, edges, sc)
    r_q, r_h, r_l = qat_attention_forward(q, k, v, False, sc)
    torch.cuda.synchronize()
    assert capi.qat_attn_device_status() == Status.OK
    # against the one-pass kernel: both round P to bf16 for the MMA, relative to different
    # running maxima, so each carries its own ~2e-3 of rounding noise (about sqrt(2) x
    # that between them); the oracle comparisons below are the parity checks
    assert rel_l2(host_f64(oh), host_f64(r_h)) < 6e-3
    assert rel_l2(host_f64(oq), host_f64(r_q)) < 8e-3
    assert float((lse - r_l).abs().max()) < 1e-4
    # against the oracle
    f = oracle_f64(inp)
    w_q, w_h, w_l = orc.forward(f["q"], f["k"], f["v"], sc, False, quant=True)
    assert rel_l2(host_f64(oh), w_h) <= TOL_HP
    assert rel_l2(host_f64(lse), w_l) <= TOL_HP
    assert rel_l2(host_f64(oq), w_q) <= TOL_Q


def test_merge_with_empty_partial_is_identity():
    B, H, Nq, D = 1, 2, 70, 128
    g = torch.Generator(device="cuda").manual_seed(3)
    acc = [torch.randn(B, H, Nq, D, device="cuda", generator=g) for _ in range(2)]
    acc.append(torch.randn(B, H, Nq, device="cuda", generator=g))
    keep = [t.clone() for t in acc]
    part = [torch.randn_like(acc[0]), torch.randn_like(acc[1]),
            torch.full((B, H, Nq), float("-inf"), device="cuda")]
    assert capi.qat_attn_merge(*acc, *part, None, None, B, H, Nq, D) == Status.OK
    torch.cuda.synchronize()
    for a, b in zip(acc, keep):
        assert torch.allclose(a, b, rtol=1e-6, atol=1e-6)
