"""CPU tests of the C-ABI library: it loads, exports every declared symbol, and its
host-side validation rejects bad arguments before anything reaches a device.
Every call here fails validation (or has no work), so nothing is ever launched."""

import ctypes
import os
import re

import pytest

from quantization_aware_attention_gb300 import build as qbuild
from quantization_aware_attention_gb300 import capi
from quantization_aware_attention_gb300.capi import Status

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "qat_attn.h")
A = 0x100000  # a 256-byte-aligned fake address: never dereferenced by these tests


@pytest.fixture(scope="module", autouse=True)
def built():
    qbuild.build()


def declared_functions():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return sorted(set(re.findall(r"\b(qat_\w+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    names = declared_functions()
    assert names == sorted(capi.EXPORTED)
    L = ctypes.CDLL(capi.LIB_PATH)
    for n in names:
        assert getattr(L, n) is not None


def test_status_strings():
    for s in Status:
        assert capi.qat_status_string(s).startswith("QAT_")
    assert "UNKNOWN" in capi.qat_status_string(99)


def fwd(**kw):
    args = dict(q=A, k=A, v=A, o_q=A, o_hp=A, lse=A, B=1, H=1, Nq=8, Nkv=8, D=64,
                sm_scale=0.125, causal=0, quant_mode=1, stream=0)
    args.update(kw)
    return capi.qat_attn_fwd(**args)


def bwd(**kw):
    args = dict(q=A, k=A, v=A, o_hp=A, lse=A, dO=A, dq=A, dk=A, dv=A, B=1, H=1, Nq=8, Nkv=8,
                D=64, sm_scale=0.125, causal=0, quant_mode=1, workspace=None,
                workspace_bytes=0, stream=0)
    args.update(kw)
    return capi.qat_attn_bwd(**args)


@pytest.mark.parametrize("kw,want", [
    (dict(D=96), Status.INVALID_ARG),
    (dict(D=256), Status.INVALID_ARG),
    (dict(B=-1), Status.INVALID_ARG),
    (dict(Nkv=0), Status.INVALID_ARG),
    (dict(sm_scale=0.0), Status.INVALID_ARG),
    (dict(sm_scale=float("nan")), Status.INVALID_ARG),
    (dict(sm_scale=float("inf")), Status.INVALID_ARG),
    (dict(causal=2), Status.INVALID_ARG),
    (dict(quant_mode=7), Status.INVALID_ARG),
    (dict(quant_mode=3), Status.INVALID_ARG),
    (dict(q=None), Status.INVALID_ARG),
    (dict(lse=None), Status.INVALID_ARG),
    (dict(o_hp=A + 8), Status.INVALID_ARG),
    (dict(causal=1, Nkv=9), Status.UNSUPPORTED),
    (dict(B=70000), Status.UNSUPPORTED),
    (dict(B=65536, H=65536, Nq=1, Nkv=1), Status.INVALID_ARG),
    (dict(B=0, q=None, k=None), Status.OK),
    (dict(Nq=0, q=None), Status.OK),
])
def test_forward_validation(kw, want):
    assert fwd(**kw) == want


@pytest.mark.parametrize("kw,want", [
    (dict(D=32), Status.INVALID_ARG),
    (dict(dq=None), Status.INVALID_ARG),
    (dict(dO=A + 4), Status.INVALID_ARG),
    (dict(workspace=None, workspace_bytes=0), Status.WORKSPACE),
    (dict(workspace=A, workspace_bytes=16), Status.WORKSPACE),
    (dict(workspace=A + 16, workspace_bytes=1 << 20), Status.INVALID_ARG),
    (dict(causal=1, Nq=16), Status.UNSUPPORTED),
    (dict(quant_mode=3), Status.INVALID_ARG),
    (dict(H=0, q=None), Status.OK),
    (dict(Nq=0, dk=None), Status.INVALID_ARG),
])
def test_backward_validation(kw, want):
    assert bwd(**kw) == want


def _base_workspace(B, H, Nq):
    """The workspace without dK/dV segment sums: lse and Delta (fp32), the two 16-element
    bf16 extension rows per padded query row, and the 128 x 16 bf16 ones tile."""
    up = lambda x: (x + 255) // 256 * 256
    rows = B * H * ((Nq + 127) // 128 * 128)
    return 2 * up(rows * 4) + 2 * up(rows * 32) + up(128 * 32)


def test_workspace_holds_segment_sums_only_for_few_key_items():
    # c4: 10240 (head, key block) items, 67 per SM: one CTA per item, no partial sums
    assert capi.qat_attn_bwd_workspace_bytes(1, 40, 32768, 32768, 128) == _base_workspace(1, 40, 32768)
    # c5b: 160 items of 128 query blocks on 152 SMs -> stream-K over 152 CTAs, two
    # 128-row slots of fp32 dV and dK per CTA
    extra = capi.qat_attn_bwd_workspace_bytes(1, 40, 16384, 512, 128) - _base_workspace(1, 40, 16384)
    assert extra == 152 * 2 * 2 * 128 * 128 * 4
    # one item of 7 query blocks: two CTAs would not pay for their partial sums
    assert capi.qat_attn_bwd_workspace_bytes(1, 1, 896, 100, 64) == _base_workspace(1, 1, 896)
    # 2 items x 16 query blocks: 8 CTAs of 4 blocks (at least 4 per range)
    extra = capi.qat_attn_bwd_workspace_bytes(1, 1, 2000, 130, 64) - _base_workspace(1, 1, 2000)
    assert extra == 8 * 2 * 2 * 128 * 64 * 4


def test_workspace_bytes():
    assert capi.qat_attn_bwd_workspace_bytes(1, 40, 32768, 32768, 128) >= 40 * 32768 * 4
    assert capi.qat_attn_bwd_workspace_bytes(2, 4, 8, 8, 64) % 256 == 0
    assert capi.qat_attn_bwd_workspace_bytes(1, 1, 8, 8, 96) == 0
    assert capi.qat_attn_bwd_workspace_bytes(-1, 1, 8, 8, 64) == 0


def test_debug_quant_validation():
    assert capi.qat_debug_quant_tiles(None, -1, 4, A, A, A, stream=0) == Status.INVALID_ARG
    assert capi.qat_debug_quant_tiles(None, 4, 64, A, A, A, stream=0) == Status.INVALID_ARG
    assert capi.qat_debug_quant_tiles(None, 0, 64, None, None, None, stream=0) == Status.OK


def test_wait_timeout_validation():
    # rejected before anything touches the device
    assert capi.qat_debug_wait_timeout(0, stream=0) == Status.INVALID_ARG
    assert capi.qat_debug_wait_timeout(4001, stream=0) == Status.INVALID_ARG


def test_chunk_and_merge_validation():
    base = dict(q=A, k=A, v=A, o_q=A, o_hp=A, lse=A, B=1, H=1, Nq=8, Nkv_total=256, D=128,
                sm_scale=0.1, quant_mode=1, stream=0)
    assert capi.qat_attn_fwd_chunk(kv_begin=32, kv_len=64, **base) == Status.UNSUPPORTED
    assert capi.qat_attn_fwd_chunk(kv_begin=192, kv_len=128, **base) == Status.INVALID_ARG
    assert capi.qat_attn_fwd_chunk(kv_begin=-64, kv_len=64, **base) == Status.INVALID_ARG
    assert capi.qat_attn_fwd_chunk(kv_begin=0, kv_len=0, **base) == Status.INVALID_ARG
    assert capi.qat_attn_merge(A, A, None, A, A, A, None, None, 1, 1, 8, 128, 0) == Status.INVALID_ARG
    assert capi.qat_attn_merge(A, A, A, A, A, A, None, None, 1, 1, 8, 96, 0) == Status.INVALID_ARG
    assert capi.qat_attn_merge(None, None, None, None, None, None, None, None, 0, 1, 8, 128, 0) == Status.OK


def noalloc(**kw):
    args = dict(q=A, k=A, v=A, o_hp=A, lse=A, dO=A, dq=A, dk=A, dv=A, B=1, H=128, Nq=65537,
                Nkv=65537, D=128, sm_scale=0.088, causal=0, quant_mode=1, stream=0)
    args.update(kw)
    return capi.qat_attn_bwd_noalloc(**args)


@pytest.mark.parametrize("kw,want", [
    (dict(), Status.WORKSPACE),                       # valid, but its scratch would not fit
    (dict(causal=1, Nkv=65536), Status.UNSUPPORTED),  # argument errors come first, as in
    (dict(sm_scale=-1.0), Status.INVALID_ARG),        # qat_attn_bwd
    (dict(quant_mode=5), Status.INVALID_ARG),
    (dict(D=80), Status.INVALID_ARG),
    (dict(dv=None), Status.INVALID_ARG),
    (dict(q=A + 8), Status.INVALID_ARG),
    (dict(H=0, q=None), Status.OK),
    (dict(Nq=0, dk=None), Status.INVALID_ARG),
])
def test_noalloc_validation_order(kw, want):
    """The no-alloc backward checks its arguments exactly as qat_attn_bwd does, before the
    size of its fixed scratch: an oversize call with a bad mode or shape reports that."""
    assert noalloc(**kw) == want


def test_smooth_k_backward_validation():
    args = dict(q=A, k=A, v=A, o_hp=A, lse=A, dO=A, dq=A, dk=A, dv=A, k_mean=A, B=1, H=1, Nq=8,
                Nkv=8, D=64, sm_scale=0.125, causal=0, quant_mode=2, workspace=None,
                workspace_bytes=0, stream=0)
    assert capi.qat_attn_bwd_smooth_k(**{**args, "k_mean": None}) == Status.INVALID_ARG
    assert capi.qat_attn_bwd_smooth_k(**{**args, "k_mean": A + 4}) == Status.INVALID_ARG
    assert capi.qat_attn_bwd_smooth_k(**args) == Status.WORKSPACE
    assert capi.qat_attn_bwd_smooth_k(**{**args, "D": 96}) == Status.INVALID_ARG


def test_subtract_mean_and_wait_limit_validation():
    assert capi.qat_subtract_mean(A, A, A, 1, 1, 8, 96, stream=0) == Status.INVALID_ARG
    assert capi.qat_subtract_mean(A, None, A, 1, 1, 8, 64, stream=0) == Status.INVALID_ARG
    assert capi.qat_subtract_mean(A, A + 4, A, 1, 1, 8, 64, stream=0) == Status.INVALID_ARG
    assert capi.qat_subtract_mean(None, None, None, 0, 1, 8, 64, stream=0) == Status.OK
    assert capi.qat_debug_set_wait_limit_us(-1, stream=0) == Status.INVALID_ARG
    assert capi.qat_debug_set_wait_limit_us(4000001, stream=0) == Status.INVALID_ARG
