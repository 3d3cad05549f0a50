"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the same
seeded inputs.  Full tensors where the oracle finishes in seconds; sampled heads, rows
and keys at the full workload sizes."""

import numpy as np
import pytest
import torch

from oracle import qat_oracle as orc
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


def run_gpu(inp, causal, sm_scale, quant=1):
    q, k, v, do = (dev_bf16(inp[n]) for n in ("q", "k", "v", "do"))
    o_q, o_hp, lse = qat_attention_forward(q, k, v, causal, sm_scale, quant)
    dq, dk, dv = qat_attention_backward(q, k, v, o_hp, lse, do, causal, sm_scale, quant)
    torch.cuda.synchronize()
    assert capi.qat_attn_device_status() == Status.OK
    return dict(o_q=o_q, o_hp=o_hp, lse=lse, dq=dq, dk=dk, dv=dv)


def check_full(inp, causal, sm_scale, heads=None):
    """Compare every output of the listed (b, h) heads (default all) with the oracle."""
    g = run_gpu(inp, causal, sm_scale)
    f = oracle_f64(inp)
    B, H = inp["q"].shape[:2]
    heads = heads or [(b, h) for b in range(B) for h in range(H)]
    want = {n: [] for n in ("o_q", "o_hp", "lse", "dq", "dk", "dv")}
    got = {n: [] for n in want}
    for b, h in heads:
        r = orc.head_forward(f["q"][b, h], f["k"][b, h], f["v"][b, h], sm_scale, causal, True)
        dq, dk, dv = orc.head_backward(f["q"][b, h], f["k"][b, h], f["v"][b, h], f["do"][b, h],
                                       sm_scale, causal)
        for n, val in (("o_q", r["o_q"]), ("o_hp", r["o_hp"]), ("lse", r["lse"]),
                       ("dq", dq), ("dk", dk), ("dv", dv)):
            want[n].append(val)
            got[n].append(host_f64(g[n][b, h]))
    errs = {n: rel_l2(np.stack(got[n]), np.stack(want[n])) for n in want}
    lse_abs = float(np.max(np.abs(np.stack(got["lse"]) - np.stack(want["lse"]))))
    assert errs["o_hp"] <= TOL_HP and errs["lse"] <= TOL_HP, errs
    assert lse_abs < 1e-3, lse_abs
    for n in ("o_q", "dq", "dk", "dv"):
        assert errs[n] <= TOL_Q, (n, errs)
    # O_q really is quantized: with more than a few keys per row it differs from O_hp
    # by the FP8 error (with one key P = 1 quantizes exactly and the two are equal)
    if inp["k"].shape[2] >= 16:
        assert rel_l2(np.stack(got["o_q"]), np.stack(got["o_hp"])) > 1e-4
    print("errors", {n: f"{e:.2e}" for n, e in errs.items()})
    return errs


# ------------------------------------------------------------------ quant primitive

def test_quant_primitive_bit_exact():
    rng = np.random.default_rng(11)
    rows, cols = 3000, 200                          # 3 full tiles + a ragged tile of 8
    p = np.exp(rng.standard_normal((rows, cols)) * 4).astype(np.float32)
    p[0] = 0.0                                      # all-zero tiles
    p[1, 64:128] = 0.0
    p[2] *= np.float32(1e-36)                       # tiny (some subnormal) values
    p[3] = np.float32(1.0)
    p[4, :] = np.float32(2.0 ** -20)
    p[5] = np.minimum(p[5], np.float32(1e30))
    tiles = (cols + 63) // 64
    dp = torch.from_numpy(p).cuda()
    deq = torch.empty_like(dp)
    scales = torch.empty((rows, tiles), dtype=torch.float32, device="cuda")
    codes = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    assert capi.qat_debug_quant_tiles(dp, rows, cols, deq, scales, codes) == Status.OK
    torch.cuda.synchronize()
    deq, scales, codes = deq.cpu().numpy(), scales.cpu().numpy(), codes.cpu().numpy()
    for t in range(tiles):
        sl = slice(t * 64, min(cols, (t + 1) * 64))
        w_deq, w_scale, w_codes = orc.quant_tiles_fp32(p[:, sl])
        assert np.array_equal(codes[:, sl], w_codes), t
        assert np.array_equal(scales[:, t].view(np.uint32), w_scale.view(np.uint32)), t
        assert np.array_equal(deq[:, sl].view(np.uint32), w_deq.view(np.uint32)), t


# ------------------------------------------------------------------ workloads

@pytest.mark.parametrize("name", ["c1", "c2"])
def test_small_workloads_full(name):
    w = WORKLOADS[name]
    check_full(make_inputs(w), w.causal, w.sm_scale)


def test_c3_dit_outlier_channels_sampled_heads():
    w = WORKLOADS["c3"]
    check_full(make_inputs(w), w.causal, w.sm_scale, heads=[(0, 0), (0, 13), (0, 23)])


def test_c5b_cross_attention_sampled_heads():
    w = WORKLOADS["c5b"]
    check_full(make_inputs(w), w.causal, w.sm_scale, heads=[(0, 0), (0, 39)])


@pytest.mark.parametrize("B,H,Nq,Nkv,D,causal", [
    (1, 1, 1, 1, 64, False),
    (1, 1, 1, 1, 128, True),
    (1, 2, 63, 63, 128, True),
    (1, 1, 65, 65, 64, True),
    (1, 1, 129, 129, 128, False),
    (1, 1, 129, 200, 128, False),
    (2, 1, 100, 37, 64, False),
    (1, 1, 200, 200, 128, True),
    (1, 1, 7, 300, 128, False),
    (1, 2, 1100, 300, 128, False),  # few (head, key block) items, one CTA each
    (1, 1, 2000, 130, 64, False),   # stream-K, items in 4 segments, D = 64
])
def test_edge_shapes(B, H, Nq, Nkv, D, causal):
    inp = custom_inputs(500 + Nq + Nkv, B, H, Nq, Nkv, D)
    check_full(inp, causal, 1.0 / np.sqrt(D))


def test_large_scale_and_quant_off():
    inp = custom_inputs(77, 1, 2, 130, 130, 128)
    check_full(inp, False, 0.5)  # sharper softmax: many tiles with tiny amax
    q, k, v = (dev_bf16(inp[n]) for n in ("q", "k", "v"))
    o_q, o_hp, _ = qat_attention_forward(q, k, v, False, 0.5, capi.QUANT_NONE)
    assert torch.equal(o_q, o_hp)


def test_backward_without_queries_zeroes_key_grads():
    k = torch.randn(1, 2, 70, 64, device="cuda").to(torch.bfloat16)
    q = torch.empty(1, 2, 0, 64, device="cuda", dtype=torch.bfloat16)
    lse = torch.empty(1, 2, 0, device="cuda")
    dk = torch.full_like(k, 3.0)
    dv = torch.full_like(k, 3.0)
    st = capi.qat_attn_bwd(q, k, k, q, lse, q, q, dk, dv, 1, 2, 0, 70, 64, 0.125, 0, 1, None, 0)
    torch.cuda.synchronize()
    assert st == Status.OK and not dk.any() and not dv.any()


@pytest.mark.parametrize("causal", [False, True])
def test_deterministic(causal):
    """Every output is bit-identical run to run: each CTA sums its own rows in a fixed
    order (dQ per query block in TMEM, dK/dV per key block), with no atomics."""
    inp = custom_inputs(91, 1, 2, 300, 300, 128)
    a = run_gpu(inp, causal, 0.088)
    b = run_gpu(inp, causal, 0.088)
    for n in ("o_q", "o_hp", "lse", "dq", "dk", "dv"):
        assert torch.equal(a[n], b[n]), n


def test_deterministic_stream_k():
    """With few (head, key block) items the dK/dV kernel runs stream-K: equal ranges of
    the items' query blocks per CTA, cut items storing fp32 partial sums that a second
    kernel adds in CTA order, so dK and dV stay bit-identical run to run."""
    inp = custom_inputs(93, 1, 1, 2000, 130, 64)
    a = run_gpu(inp, False, 0.125)
    b = run_gpu(inp, False, 0.125)
    for n in ("dq", "dk", "dv"):
        assert torch.equal(a[n], b[n]), n


def _at_16_byte_offset(t):
    """A copy of t whose storage starts 16 bytes past a 256-byte boundary: aligned as the
    C ABI requires (16 bytes) but not to 32 bytes."""
    buf = torch.empty(t.numel() + 8, dtype=t.dtype, device=t.device)
    view = buf[8:].view(t.shape)
    view.copy_(t)
    assert view.data_ptr() % 32 == 16
    return view


def test_inputs_16_byte_aligned_match_aligned():
    """Q (and the other inputs) at 16-byte but not 32-byte aligned addresses give bit-
    identical outputs: the dQ kernel's 32-byte row loads are used only on 32-byte aligned
    q, and every other access needs 16 bytes."""
    inp = custom_inputs(95, 1, 2, 300, 700, 128)
    a = run_gpu(inp, False, 0.088)
    q, k, v, do = (_at_16_byte_offset(dev_bf16(inp[n])) for n in ("q", "k", "v", "do"))
    o_q, o_hp, lse = qat_attention_forward(q, k, v, False, 0.088)
    dq, dk, dv = qat_attention_backward(q, k, v, o_hp, lse, do, False, 0.088)
    torch.cuda.synchronize()
    assert capi.qat_attn_device_status() == Status.OK
    for n, t in (("o_q", o_q), ("o_hp", o_hp), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert torch.equal(a[n], t), n


def test_stream_k_without_room_for_its_sums_runs_one_cta_per_item():
    """A workspace that holds everything but the dK/dV segments' partial sums (as the
    no-alloc scratch may) runs the backward with one CTA per item instead of stream-K:
    the same gradients up to the fp32 summation order.  One byte less than that is
    refused."""
    B, H, Nq, Nkv, D, sc = 1, 1, 2000, 130, 64, 0.125
    inp = custom_inputs(94, B, H, Nq, Nkv, D)
    q, k, v, do = (dev_bf16(inp[n]) for n in ("q", "k", "v", "do"))
    _, o_hp, lse = qat_attention_forward(q, k, v, False, sc)
    full = capi.qat_attn_bwd_workspace_bytes(B, H, Nq, Nkv, D)
    # 2 items x 16 query blocks: 8 stream-K CTAs of 4 blocks, two 128-row slots of fp32
    # dV and dK each
    base = full - 8 * 2 * 2 * 128 * D * 4
    outs = {}
    for name, nbytes in (("split", full), ("unsplit", base)):
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        g = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
        st = capi.qat_attn_bwd(q, k, v, o_hp, lse, do, *g, B, H, Nq, Nkv, D, sc, 0, 1, ws, nbytes)
        torch.cuda.synchronize()
        assert st == Status.OK and capi.qat_attn_device_status() == Status.OK
        outs[name] = g
    for a, b in zip(outs["split"], outs["unsplit"]):
        assert rel_l2(host_f64(a), host_f64(b)) <= 2e-3
    ws = torch.empty(base, dtype=torch.uint8, device="cuda")
    g = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
    st = capi.qat_attn_bwd(q, k, v, o_hp, lse, do, *g, B, H, Nq, Nkv, D, sc, 0, 1, ws, base - 1)
    assert st == Status.WORKSPACE


def test_expired_wait_is_reported_then_cleared():
    """The failure path of the kernels' bounded waits: the test entry waits on a barrier
    nothing arrives on, gives up after 50 ms and sets the device error word; the next
    status read reports QAT_ERR_TIMEOUT and clears it, and the context stays usable."""
    assert capi.qat_debug_wait_timeout(50) == Status.OK
    assert capi.qat_attn_device_status() == Status.TIMEOUT
    assert capi.qat_attn_device_status() == Status.OK
    inp = custom_inputs(123, 1, 2, 200, 200, 128)
    check_full(inp, True, 1.0 / np.sqrt(128))


def test_forward_deterministic_causal_many_items():
    """The c5a shape, causal: thousands of items of 1 to 64 key blocks over 152 CTAs.
    Every output must be bit-identical across runs.  (An epilogue that waited on a
    per-block barrier could pass while the last two PV products were still running;
    at this size that showed as a few dozen query tiles differing run to run.)"""
    B, H, N, D = 4, 32, 8192, 128
    gen = torch.Generator(device="cuda").manual_seed(5)
    q, k, v = (torch.randn(B, H, N, D, device="cuda", generator=gen).to(torch.bfloat16)
               for _ in range(3))
    outs = []
    for _ in range(3):
        o_q, o_hp = torch.empty_like(q), torch.empty_like(q)
        lse = torch.empty(B, H, N, device="cuda")
        st = capi.qat_attn_fwd(q, k, v, o_q, o_hp, lse, B, H, N, N, D, 1.0 / np.sqrt(D), 1, 1)
        assert st == Status.OK
        torch.cuda.synchronize()
        outs.append((o_q, o_hp, lse))
    assert capi.qat_attn_device_status() == Status.OK
    for o in outs[1:]:
        for a_, b_ in zip(outs[0], o):
            assert torch.equal(a_, b_)


def test_forward_deterministic_short_kv_many_items():
    """Cross-attention with 4 key blocks per item (the c5b shape, 34 items per CTA): the
    forward instance that stores an item's outputs after the next item's first block of
    P.  Every output must be bit-identical across runs, and every row finite (each
    CTA's last item is stored after its loop)."""
    B, H, Nq, Nkv, D = 1, 40, 16384, 512, 128
    gen = torch.Generator(device="cuda").manual_seed(6)
    q = torch.randn(B, H, Nq, D, device="cuda", generator=gen).to(torch.bfloat16)
    k, v = (torch.randn(B, H, Nkv, D, device="cuda", generator=gen).to(torch.bfloat16)
            for _ in range(2))
    outs = []
    for _ in range(3):
        o_q = torch.full_like(q, float("nan"))
        o_hp = torch.full_like(q, float("nan"))
        lse = torch.full((B, H, Nq), float("nan"), device="cuda")
        st = capi.qat_attn_fwd(q, k, v, o_q, o_hp, lse, B, H, Nq, Nkv, D, 1.0 / np.sqrt(D), 0, 1)
        assert st == Status.OK
        torch.cuda.synchronize()
        outs.append((o_q, o_hp, lse))
    assert capi.qat_attn_device_status() == Status.OK
    for t in outs[0]:
        assert torch.isfinite(t).all()
    for o in outs[1:]:
        for a_, b_ in zip(outs[0], o):
            assert torch.equal(a_, b_)


def test_backward_deterministic_causal_many_items():
    """The c5a shape, causal, through the backward: dQ, dK and dV bit-identical across
    runs (each CTA sums its own rows in a fixed order; no atomics)."""
    B, H, N, D = 4, 32, 8192, 128
    gen = torch.Generator(device="cuda").manual_seed(6)
    q, k, v, do = (torch.randn(B, H, N, D, device="cuda", generator=gen).to(torch.bfloat16)
                   for _ in range(4))
    sm = 1.0 / np.sqrt(D)
    o_q, o_hp = torch.empty_like(q), torch.empty_like(q)
    lse = torch.empty(B, H, N, device="cuda")
    assert capi.qat_attn_fwd(q, k, v, o_q, o_hp, lse, B, H, N, N, D, sm, 1, 1) == Status.OK
    wsb = capi.qat_attn_bwd_workspace_bytes(B, H, N, N, D)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(3):
        g = [torch.empty_like(q) for _ in range(3)]
        st = capi.qat_attn_bwd(q, k, v, o_hp, lse, do, *g, B, H, N, N, D, sm, 1, 1, ws, wsb)
        assert st == Status.OK
        torch.cuda.synchronize()
        outs.append(g)
    assert capi.qat_attn_device_status() == Status.OK
    for o in outs[1:]:
        for a_, b_ in zip(outs[0], o):
            assert torch.equal(a_, b_)


# ------------------------------------------------------------------ full-size, sampled
#
# The full workloads are checked on sampled rows and keys, stratified so that every
# 128-row query block and every 128-key block is hit: n of each per block.  Beside the
# tolerance on the whole sample, every 128-block's own relative L2 must stay within
# BLOCK_FACTOR times it, so one wrong tile (a bad mask, a stale buffer, a padding
# block) cannot hide under the average.

BLOCK_FACTOR = 3.0


def _stratified(rng, n_total, per_block, blk=128):
    """per_block distinct indices from every blk-wide block of [0, n_total), sorted."""
    out = []
    for b0 in range(0, n_total, blk):
        size = min(blk, n_total - b0)
        out.append(b0 + rng.choice(size, min(per_block, size), replace=False))
    return np.sort(np.concatenate(out))


def _per_block(got, want, idx, blk=128):
    """Worst relative L2 over the 128-blocks of the sampled indices (rows of got/want)."""
    worst, where = 0.0, -1
    for b in np.unique(idx // blk):
        m = idx // blk == b
        e = rel_l2(got[m], want[m])
        if e > worst:
            worst, where = e, int(b)
    return worst, where


def _check_sampled(name, got, want, idx, tol):
    e = rel_l2(got, want)
    wb, where = _per_block(got, want, idx)
    print(f"{name}: {e:.2e} (worst 128-block {where}: {wb:.2e})")
    assert e <= tol, (name, e)
    assert wb <= BLOCK_FACTOR * tol, (name, where, wb)


def _sampled_full_size(name, fwd_heads, bwd_heads, per_block=2):
    w = WORKLOADS[name]
    inp = make_inputs(w)
    g = run_gpu(inp, w.causal, w.sm_scale)
    for n in ("o_q", "o_hp", "dq", "dk", "dv"):
        assert torch.isfinite(g[n]).all(), n
    rng = np.random.default_rng(w.idx)
    f = oracle_f64(inp)
    for b, h in fwd_heads:
        rows = _stratified(rng, w.Nq, per_block)
        r = orc.head_forward(f["q"][b, h], f["k"][b, h], f["v"][b, h], w.sm_scale, w.causal,
                             True, rows=rows)
        for n, tol in (("o_q", TOL_Q), ("o_hp", TOL_HP), ("lse", TOL_HP)):
            _check_sampled(f"{n} head {(b, h)}", host_f64(g[n][b, h])[rows], r[n], rows, tol)
    for b, h in bwd_heads:
        rows = _stratified(rng, w.Nq, per_block)
        keys = _stratified(rng, w.Nkv, per_block)
        dq, dk, dv = orc.head_backward_sampled(f["q"][b, h], f["k"][b, h], f["v"][b, h],
                                               f["do"][b, h], w.sm_scale, w.causal, rows, keys)
        _check_sampled(f"dq head {(b, h)}", host_f64(g["dq"][b, h])[rows], dq, rows, TOL_Q)
        _check_sampled(f"dk head {(b, h)}", host_f64(g["dk"][b, h])[keys], dk, keys, TOL_Q)
        _check_sampled(f"dv head {(b, h)}", host_f64(g["dv"][b, h])[keys], dv, keys, TOL_Q)


def test_c4_video_dit_full_size_sampled():
    _sampled_full_size("c4", fwd_heads=[(0, 0), (0, 17), (0, 39)], bwd_heads=[(0, 21), (0, 38)])


def test_c5a_causal_full_size_sampled():
    _sampled_full_size("c5a", fwd_heads=[(0, 0), (3, 31)], bwd_heads=[(2, 5), (3, 30)])


def test_c3_every_head_sampled_rows():
    """c3 (outlier K channels): the forward of all 24 heads on stratified rows, and the
    backward of two heads on stratified rows and keys."""
    w = WORKLOADS["c3"]
    _sampled_full_size("c3", fwd_heads=[(0, h) for h in range(w.H)],
                       bwd_heads=[(0, 5), (0, 18)])
