"""qat_attn_bwd_noalloc: the backward for callers that cannot allocate device memory
(their device memory belongs to another runtime's pool, or they must not allocate once
running).  Its scratch is a fixed array inside the library, so these tests check that
it gives the same gradients as qat_attn_bwd with a caller workspace, on two calls in a
row (the second call must not see the first call's leftovers), and that it refuses
sizes whose scratch would not fit.

This file is named to be collected last."""

import numpy as np
import pytest
import torch

from quantization_aware_attention_gb300 import build as qbuild
from quantization_aware_attention_gb300 import capi
from quantization_aware_attention_gb300.attention import (qat_attention_backward,
                                                          qat_attention_forward)
from quantization_aware_attention_gb300.capi import Status
from quantization_aware_attention_gb300.inputs import custom_inputs

pytestmark = pytest.mark.gpu

TOL = 1e-2  # the gradients' relative-L2 tolerance used by the parity tests


@pytest.fixture(scope="module", autouse=True)
def built():
    qbuild.build()


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _rel(a, b):
    a, b = a.double(), b.double()
    return float((a - b).norm() / b.norm().clamp_min(1e-30))


def test_noalloc_matches_workspace_entry_on_two_calls():
    problems = [((1, 3, 200, 200, 128), True, 11), ((2, 2, 77, 150, 64), False, 12),
                ((1, 1, 2000, 130, 64), False, 13)]  # the last splits its dK/dV items
    for (B, H, Nq, Nkv, D), causal, seed in problems:
        inp = custom_inputs(seed, B, H, Nq, Nkv, D)
        q, k, v, do = (_dev(inp[n]) for n in ("q", "k", "v", "do"))
        sc = 1.0 / np.sqrt(D)
        _, o_hp, lse = qat_attention_forward(q, k, v, causal, sc)
        want = qat_attention_backward(q, k, v, o_hp, lse, do, causal, sc)
        got = [torch.full_like(t, float("nan")) for t in want]
        st = capi.qat_attn_bwd_noalloc(q, k, v, o_hp, lse, do, *got, B, H, Nq, Nkv, D, sc,
                                       int(causal), capi.QUANT_P_FP8E4M3_ROW_TILE64)
        assert st == Status.OK
        torch.cuda.synchronize()
        for g, w in zip(got, want):
            assert torch.isfinite(g).all()
            assert _rel(g, w) <= TOL


def test_noalloc_rejects_sizes_beyond_its_scratch():
    fake = 0x100000  # never dereferenced: the size check comes first
    st = capi.qat_attn_bwd_noalloc(*([fake] * 9), 1, 128, 65537, 65537, 128, 0.088, 0, 1)
    assert st == Status.WORKSPACE
