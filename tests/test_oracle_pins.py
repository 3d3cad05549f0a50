"""Pins for the fp64 oracle, checked against facts outside the oracle itself:
the OCP E4M3 table, brute-force nearest-value search, closed forms, invariants,
torch's own float64 SDPA / autograd (library routines) and finite differences.
CPU only."""

import math
import os

import numpy as np
import pytest
import torch

from oracle import qat_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers (test side)

def _all_finite_codes():
    """Every non-negative finite E4M3 code and its value, decoded here bit by bit."""
    codes, vals = [], []
    for c in range(0x7F):                     # 0x7F is NaN
        e, m = (c >> 3) & 0xF, c & 7
        v = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
        codes.append(c)
        vals.append(v)
    return np.array(codes), np.array(vals)


def nearest_e4m3(x):
    """Brute force: the finite E4M3 value nearest to x >= 0, ties to the even code,
    values above the largest finite value saturate."""
    codes, vals = _all_finite_codes()
    if x >= vals.max():
        return int(codes[np.argmax(vals)]), float(vals.max())
    d = np.abs(vals - x)
    best = np.flatnonzero(d == d.min())
    if best.size > 1:
        best = [b for b in best if codes[b] % 2 == 0]
    b = best[0]
    return int(codes[b]), float(vals[b])


def rng_f64(seed, *shape, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def rel_l2(a, b):
    return float(np.linalg.norm(np.ravel(a - b)) / np.linalg.norm(np.ravel(b)))


# ---------------------------------------------------------------- E4M3

def test_e4m3_golden_table():
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "e4m3_ocp_values.txt"))
            if ln.strip() and not ln.startswith("#")]
    codes = np.array([int(c, 16) for c, _ in rows])
    want = np.array([float(v) for _, v in rows])
    got = orc.e4m3_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    fin = ~np.isnan(want)
    assert np.array_equal(got[fin], want[fin])
    # encoding the finite values gives back their codes
    c2, v2 = orc.e4m3_rne_satfinite(want[fin])
    assert np.array_equal(c2, codes[fin].astype(np.uint8))
    assert np.array_equal(v2, want[fin])


def test_e4m3_rne_matches_bruteforce_nearest():
    codes, vals = _all_finite_codes()
    vals_sorted = np.sort(vals)
    mids = (vals_sorted[1:] + vals_sorted[:-1]) / 2          # exact ties
    rnd = np.abs(np.random.default_rng(7).standard_normal(3000)) * 40
    tiny = np.abs(np.random.default_rng(8).standard_normal(500)) * 2 ** -8
    big = np.array([448.0, 455.9, 464.0, 470.0, 479.9, 480.0, 1e6])
    xs = np.concatenate([vals, mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9),
                         rnd, tiny, big, [0.0, 2.0 ** -10, 2.0 ** -10 * 1.0001]])
    got_c, got_v = orc.e4m3_rne_satfinite(xs)
    for x, c, v in zip(xs, got_c, got_v):
        wc, wv = nearest_e4m3(float(x))
        assert (int(c), float(v)) == (wc, wv), x
    # decode/encode round trip over every finite code, both signs
    allc = np.concatenate([codes, codes[1:] | 0x80])
    dec = orc.e4m3_decode(allc)
    c3, v3 = orc.e4m3_rne_satfinite(dec)
    assert np.array_equal(c3, allc.astype(np.uint8)) and np.array_equal(v3, dec)


# ---------------------------------------------------------------- fp32 quant primitive

def _bf16_rn_scalar(x32):
    u = int(np.float32(x32).view(np.uint32))
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return float(np.uint32(u).view(np.float32))


def test_quant_primitive_matches_scalar_loop():
    rng = np.random.default_rng(3)
    p = np.exp(rng.standard_normal((40, 64)) * 3).astype(np.float32)
    p[5] = 0.0                                   # empty tile
    p[6, :10] = 0.0
    p[7] = np.float32(1e-30) * p[7]              # tiny but normal amax
    deq, scale, codes = orc.quant_tiles_fp32(p)
    for r in range(p.shape[0]):
        amax = np.float32(max(p[r]))
        if amax == 0:
            assert scale[r] == 0 and not codes[r].any() and not deq[r].any()
            continue
        inv = np.float32(448.0) / amax
        s = amax / np.float32(448.0)
        assert scale[r] == s
        for c in range(64):
            x = np.float32(p[r, c] * inv)
            wc, wv = nearest_e4m3(float(x))
            assert codes[r, c] == wc
            assert deq[r, c] == _bf16_rn_scalar(np.float32(np.float32(wv) * s))


def test_quant_primitive_max_maps_to_448_and_scale_invariance():
    rng = np.random.default_rng(4)
    p = np.exp(rng.standard_normal((32, 64)) * 2).astype(np.float32)
    deq, scale, codes = orc.quant_tiles_fp32(p)
    am = p.argmax(axis=1)
    assert np.all(codes[np.arange(32), am] == 0x7E)
    for k in (-20, -3, 1, 7):
        d2, s2, c2 = orc.quant_tiles_fp32(p * np.float32(2.0 ** k))
        assert np.array_equal(c2, codes)
        assert np.array_equal(s2, scale * np.float32(2.0 ** k))
        assert np.array_equal(d2, deq * np.float32(2.0 ** k))


def test_quant_primitive_idempotent_codes():
    rng = np.random.default_rng(5)
    p = np.exp(rng.standard_normal((64, 64)) * 2).astype(np.float32)
    deq, _, codes = orc.quant_tiles_fp32(p)
    _, _, codes2 = orc.quant_tiles_fp32(deq)
    assert np.array_equal(codes, codes2)


# ---------------------------------------------------------------- forward

def _sdpa64(q, k, v, scale, causal):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    return torch.nn.functional.scaled_dot_product_attention(
        t(q), t(k), t(v), scale=scale, is_causal=causal).numpy()


@pytest.mark.parametrize("nq,nkv,d,causal", [(37, 37, 16, False), (37, 37, 16, True),
                                              (20, 150, 8, False), (130, 9, 32, False)])
def test_forward_hp_equals_library_sdpa_and_lse(nq, nkv, d, causal):
    q, k, v = rng_f64(1, 2, 3, nq, d), rng_f64(2, 2, 3, nkv, d), rng_f64(3, 2, 3, nkv, d)
    sc = 1 / math.sqrt(d)
    _, o_hp, lse = orc.forward(q, k, v, sc, causal, quant=False, row_chunk=16)
    assert np.allclose(o_hp, _sdpa64(q, k, v, sc, causal), rtol=1e-12, atol=1e-12)
    s = torch.from_numpy(q) @ torch.from_numpy(k).transpose(-1, -2) * sc
    if causal:
        s = s.masked_fill(torch.ones(nq, nkv, dtype=torch.bool).triu(1), -math.inf)
    want = (torch.logsumexp(s, dim=-1) / math.log(2)).numpy()
    assert np.allclose(lse, want, rtol=1e-12, atol=1e-12)


def test_forward_rows_of_p_sum_to_one_and_causal_zeros():
    q, k, v = rng_f64(4, 50, 8), rng_f64(5, 50, 8), rng_f64(6, 50, 8)
    r = orc.head_forward(q, k, v, 0.4, True, quant=True, return_p=True)
    assert np.allclose(r["p"].sum(axis=1), 1.0, atol=1e-13)
    upper = np.triu(np.ones((50, 50), dtype=bool), 1)
    assert not r["p"][upper].any() and not r["pq"][upper].any()


def test_forward_identical_keys_closed_form():
    nkv, d = 200, 16
    q, v = rng_f64(7, 9, d), rng_f64(8, nkv, d)
    k = np.tile(rng_f64(9, 1, d), (nkv, 1))
    sc = 0.3
    r = orc.head_forward(q, k, v, sc, False, quant=True)
    assert np.allclose(r["o_hp"], v.mean(axis=0)[None], rtol=0, atol=1e-13)
    assert np.allclose(r["o_q"], v.mean(axis=0)[None], rtol=0, atol=1e-13)
    want_lse = sc * (q @ k[0]) / math.log(2) + math.log2(nkv)
    assert np.allclose(r["lse"], want_lse, rtol=0, atol=1e-12)


def test_forward_causal_ignores_future_keys():
    n, d = 70, 8
    q, k, v = rng_f64(10, n, d), rng_f64(11, n, d), rng_f64(12, n, d)
    a = orc.head_forward(q, k, v, 0.5, True, quant=True)
    k2, v2 = k.copy(), v.copy()
    k2[40:] += 5.0
    v2[40:] -= 3.0
    b = orc.head_forward(q, k2, v2, 0.5, True, quant=True)
    for key in ("o_q", "o_hp", "lse"):
        assert np.array_equal(a[key][:40], b[key][:40])
        assert not np.allclose(a[key][41:], b[key][41:])


@pytest.mark.parametrize("causal", [False, True])
def test_forward_quantized_output_bruteforce(causal):
    """O_q from a pure-Python loop: per row, per absolute 64-key tile, code by
    brute-force nearest search, weight exp(T - m) / 448 / l."""
    n, d = 150, 4                              # 3 tiles, ragged tail of 22 keys
    q, k, v = rng_f64(13, n, d, scale=2.0), rng_f64(14, n, d), rng_f64(15, n, d)
    sc = 0.7
    r = orc.head_forward(q, k, v, sc, causal, quant=True)
    want = np.zeros((n, d))
    for i in range(n):
        keys = [j for j in range(n) if (j <= i or not causal)]
        s = {j: sc * float(q[i] @ k[j]) for j in keys}
        m = max(s.values())
        l = sum(math.exp(s[j] - m) for j in keys)
        for t in range(3):
            tk = [j for j in keys if j // 64 == t]
            if not tk:
                continue
            T = max(s[j] for j in tk)
            for j in tk:
                _, c = nearest_e4m3(448.0 * math.exp(s[j] - T))
                want[i] += c * math.exp(T - m) / 448.0 / l * v[j]
    assert np.allclose(r["o_q"], want, rtol=1e-12, atol=1e-12)
    assert rel_l2(r["o_q"], r["o_hp"]) < 0.05


def _quant_p_exact(p, tile=64):
    """The quantization of an already-normalized P row block, step by step (fp64)."""
    out = np.zeros_like(p)
    for lo in range(0, p.shape[1], tile):
        blk = p[:, lo:lo + tile]
        amax = blk.max(axis=1, keepdims=True)
        _, c = orc.e4m3_rne_satfinite(448.0 * blk / np.where(amax > 0, amax, 1))
        out[:, lo:lo + tile] = c * amax / 448.0
    return out


def test_forward_quant_idempotent_and_matches_p_form():
    n, d = 130, 8
    q, k, v = rng_f64(16, n, d, scale=1.5), rng_f64(17, n, d), rng_f64(18, n, d)
    r = orc.head_forward(q, k, v, 0.6, False, quant=True, return_p=True)
    pq = _quant_p_exact(r["p"])
    assert np.allclose(r["pq"], pq, rtol=1e-12, atol=0)
    assert np.allclose(_quant_p_exact(pq), pq, rtol=1e-13, atol=0)


def test_forward_row_chunking_is_transparent():
    q, k, v = rng_f64(19, 1, 2, 77, 8), rng_f64(20, 1, 2, 77, 8), rng_f64(21, 1, 2, 77, 8)
    a = orc.forward(q, k, v, 0.3, True, quant=True, row_chunk=5)
    b = orc.forward(q, k, v, 0.3, True, quant=True, row_chunk=1000)
    for x, y in zip(a, b):
        assert np.allclose(x, y, rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------- backward (STE)

@pytest.mark.parametrize("nq,nkv,causal", [(23, 23, False), (23, 23, True), (9, 70, False)])
def test_backward_matches_torch_autograd_fp64(nq, nkv, causal):
    d = 16
    q, k, v = rng_f64(22, 2, 2, nq, d), rng_f64(23, 2, 2, nkv, d), rng_f64(24, 2, 2, nkv, d)
    do = rng_f64(25, 2, 2, nq, d)
    sc = 1 / math.sqrt(d)
    tq, tk, tv = (torch.from_numpy(a).requires_grad_(True) for a in (q, k, v))
    s = tq @ tk.transpose(-1, -2) * sc
    if causal:
        s = s.masked_fill(torch.ones(nq, nkv, dtype=torch.bool).triu(1), -math.inf)
    o = torch.softmax(s, dim=-1) @ tv
    o.backward(torch.from_numpy(do))
    dq, dk, dv = orc.backward(q, k, v, do, sc, causal)
    for got, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        assert np.allclose(got, ref.numpy(), rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_finite_differences(causal):
    n, d = 6, 5
    q, k, v, do = (rng_f64(30 + i, n, d) for i in range(4))
    sc = 0.45
    dq, dk, dv = orc.head_backward(q, k, v, do, sc, causal)

    def loss(qq, kk, vv):
        return float((do * orc.head_forward(qq, kk, vv, sc, causal, quant=False)["o_hp"]).sum())

    h = 1e-6
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        num = np.zeros_like(grad)
        for idx in np.ndindex(*grad.shape):
            args_p = [q.copy(), k.copy(), v.copy()]
            args_m = [q.copy(), k.copy(), v.copy()]
            args_p[which][idx] += h
            args_m[which][idx] -= h
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        assert np.allclose(grad, num, rtol=1e-6, atol=1e-8)


def test_backward_sampled_equals_full():
    n, d = 90, 8
    q, k, v, do = (rng_f64(40 + i, n, d) for i in range(4))
    for causal in (False, True):
        dq, dk, dv = orc.head_backward(q, k, v, do, 0.35, causal)
        rows, keys = np.array([0, 7, 63, 64, 89]), np.array([1, 30, 88])
        sq, sk, sv = orc.head_backward_sampled(q, k, v, do, 0.35, causal, rows, keys, row_chunk=17)
        assert np.allclose(sq, dq[rows], rtol=1e-12, atol=1e-13)
        assert np.allclose(sk, dk[keys], rtol=1e-12, atol=1e-13)
        assert np.allclose(sv, dv[keys], rtol=1e-12, atol=1e-13)
        m, l = orc.head_row_stats(q, k, 0.35, causal, row_chunk=13)
        f = orc.head_forward(q, k, v, 0.35, causal, quant=False)
        assert np.allclose(f["m"], m) and np.allclose(f["l"], l)


# ---------------------------------------------------------------- Q/K/V fake quantization

def _nearest_signed(x):
    c, v = nearest_e4m3(abs(x))
    return (c | 0x80, -v) if (x < 0 and v > 0) else (c, v)


def test_qkv_fake_quant_matches_scalar_loop():
    rng = np.random.default_rng(50)
    x = (rng.standard_normal((70, 8)) * 3).astype(np.float32)      # 3 blocks, ragged tail
    x[40:64] = 0.0                                                   # an all-zero block
    mean = (rng.standard_normal(8) * 2).astype(np.float32)
    out, scales, codes = orc.fake_quant_tokens_fp32(x, mean)
    xs = (x - mean[None, :]).astype(np.float32)
    for b in range(3):
        blk = xs[32 * b:32 * b + 32]
        amax = np.float32(np.abs(blk).max())
        inv = np.float32(448.0) / amax
        s = amax / np.float32(448.0)
        assert scales[b] == s
        for (i, j), val in np.ndenumerate(blk):
            wc, wv = _nearest_signed(float(np.float32(val * inv)))
            assert codes[32 * b + i, j] == wc
            assert out[32 * b + i, j] == _bf16_rn_scalar(np.float32(np.float32(wv) * s))


def test_qkv_fake_quant_invariants():
    rng = np.random.default_rng(51)
    x = (rng.standard_normal((96, 16)) * 2).astype(np.float32)
    out, scales, codes = orc.fake_quant_tokens_fp32(x)
    o2, s2, c2 = orc.fake_quant_tokens_fp32(-x)                     # sign symmetry
    assert np.array_equal(o2, -out) and np.array_equal(s2, scales)
    assert np.array_equal(c2 & 0x7F, codes & 0x7F)
    o3, s3, c3 = orc.fake_quant_tokens_fp32(x * np.float32(8.0))    # scale invariance
    assert np.array_equal(c3, codes) and np.array_equal(o3, out * np.float32(8.0))
    for b in range(3):                                               # block max -> +-448
        blk = np.abs(x[32 * b:32 * b + 32])
        i, j = np.unravel_index(np.argmax(blk), blk.shape)
        assert codes[32 * b + i, j] & 0x7F == 0x7E
    _, _, c4 = orc.fake_quant_tokens_fp32(out)                       # idempotent codes
    assert np.array_equal(c4, codes)
    exact = orc.fake_quant_tokens_exact(x.astype(np.float64))
    assert np.allclose(out, exact, rtol=2 ** -7, atol=0)             # bf16 rounding only


def test_smooth_k_is_a_softmax_shift():
    """Subtracting the per-channel K mean shifts each score row by a constant, so the
    unquantized outputs and the normalized P are unchanged."""
    q, k, v = rng_f64(52, 2, 3, 40, 8), rng_f64(53, 2, 3, 40, 8), rng_f64(54, 2, 3, 40, 8)
    k = k + np.array([5.0, -3.0, 0.5, 9.0, 0.0, -7.0, 2.0, 1.0])
    mu = orc.channel_mean(k)
    assert np.allclose(mu, k.mean(axis=(0, 1, 2)))
    assert np.allclose(orc.channel_mean(k - mu), 0.0, atol=1e-12)
    a = orc.forward(q, k, v, 0.3, False, quant=False)
    b = orc.forward(q, k - mu, v, 0.3, False, quant=False)
    assert np.allclose(a[1], b[1], rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- key-chunk partials and merge

@pytest.mark.parametrize("cuts", [(64,), (128, 192), (64, 128, 256)])
def test_merge_of_chunks_equals_one_pass(cuts):
    """Forward over key chunks starting at multiples of 64, merged by lse, equals the
    one-pass forward for O_hp, lse and O_q (the quantization tiles stay whole)."""
    n, d = 300, 8
    q, k, v = rng_f64(60, 1, 2, 20, d), rng_f64(61, 1, 2, n, d), rng_f64(62, 1, 2, n, d)
    full = orc.forward(q, k, v, 0.4, False, quant=True)
    edges = (0,) + tuple(cuts) + (n,)
    acc_q = acc_h = acc_l = None
    for lo, hi in zip(edges[:-1], edges[1:]):
        oq, oh, lse = orc.forward(q, k[:, :, lo:hi], v[:, :, lo:hi], 0.4, False, quant=True)
        if acc_l is None:
            acc_q, acc_h, acc_l = oq, oh, lse
        else:
            acc_q, _ = orc.merge_partials(acc_q, acc_l, oq, lse)
            acc_h, acc_l = orc.merge_partials(acc_h, acc_l, oh, lse)
    assert np.allclose(acc_h, full[1], rtol=1e-12, atol=1e-13)
    assert np.allclose(acc_l, full[2], rtol=1e-12, atol=1e-13)
    assert np.allclose(acc_q, full[0], rtol=1e-12, atol=1e-13)


def test_merge_identity_and_symmetry():
    o = rng_f64(63, 5, 4)
    lse = rng_f64(64, 5)
    o2, l2 = orc.merge_partials(o, lse, rng_f64(65, 5, 4), np.full(5, -np.inf))
    assert np.allclose(o2, o) and np.allclose(l2, lse)
    a = orc.merge_partials(o, lse, o * 2, lse + 1)
    b = orc.merge_partials(o * 2, lse + 1, o, lse)
    assert np.allclose(a[0], b[0]) and np.allclose(a[1], b[1])


def test_chunk_not_aligned_to_quant_tiles_differs():
    """A cut inside a 64-key tile splits that tile's quantization, so O_q changes (this
    is why chunked calls require starts at multiples of 64); O_hp still merges."""
    n, d = 200, 8
    q, k, v = rng_f64(66, 1, 1, 10, d, scale=2.0), rng_f64(67, 1, 1, n, d), rng_f64(68, 1, 1, n, d)
    full = orc.forward(q, k, v, 0.6, False, quant=True)
    a = orc.forward(q, k[:, :, :100], v[:, :, :100], 0.6, False, quant=True)
    b = orc.forward(q, k[:, :, 100:], v[:, :, 100:], 0.6, False, quant=True)
    oh, _ = orc.merge_partials(a[1], a[2], b[1], b[2])
    oq, _ = orc.merge_partials(a[0], a[2], b[0], b[2])
    assert np.allclose(oh, full[1], rtol=1e-12)
    assert not np.allclose(oq, full[0], rtol=1e-9)


# ---------------------------------------------------------------- the page's backward variant

def test_page_backward_terms():
    """dV uses the quantized P, Delta the quantized output, dS the unquantized P: checked
    term by term against direct products of the oracle's own P, Pq and O_q, and against
    the straight-through gradients where quantization leaves P unchanged."""
    n, d = 90, 8
    q, k, v, do = (rng_f64(70 + i, n, d) for i in range(4))
    sc = 0.5
    dq, dk, dv = orc.head_backward_page(q, k, v, do, sc, False)
    f = orc.head_forward(q, k, v, sc, False, quant=True, return_p=True)
    assert np.allclose(dv, f["pq"].T @ do, rtol=1e-12)
    delta = (do * f["o_q"]).sum(axis=1)
    ds = f["p"] * (do @ v.T - delta[:, None])
    assert np.allclose(dk, sc * ds.T @ q, rtol=1e-12) and np.allclose(dq, sc * ds @ k, rtol=1e-12)
    _, _, dv_ste = orc.head_backward(q, k, v, do, sc, False)
    assert not np.allclose(dv, dv_ste, rtol=1e-6)          # the variants differ ...
    assert rel_l2(dv, dv_ste) < 0.05                         # ... by the FP8 error only
    # identical keys: every code is 448, Pq = P, so both variants agree exactly
    kk = np.tile(rng_f64(75, 1, d), (n, 1))
    a = orc.head_backward_page(q, kk, v, do, sc, False)
    b = orc.head_backward(q, kk, v, do, sc, False)
    for x, y in zip(a, b):
        assert np.allclose(x, y, rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- bf16 conversions vs torch

def _torch_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """torch's own float32 -> bfloat16 conversion (a library routine), as bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x32, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_bf16_rounding_matches_torch():
    """f32_to_bf16_rn against torch's conversion: exact ties with an even and an odd kept
    bit, the neighbours of ties, subnormals, the largest finite values (which round to
    infinity), signed zeros, infinities and NaNs."""
    rng = np.random.default_rng(31)
    hi = rng.integers(0, 1 << 16, 4000, dtype=np.uint64)
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF], np.uint64)
    pats = (hi[:, None] << 16 | lows[None, :]).ravel()
    even_tie = (np.arange(0, 1 << 16, 2, dtype=np.uint64) << 16) | 0x8000   # kept bit 0
    odd_tie = (np.arange(1, 1 << 16, 2, dtype=np.uint64) << 16) | 0x8000    # kept bit 1
    special = np.array([0x00000000, 0x80000000, 0x00000001, 0x00008000, 0x00018000,
                        0x007FFFFF, 0x807F8000, 0x7F7FFFFF, 0x7F7F7FFF, 0x7F7F8000,
                        0xFF7FFFFF, 0x7F800000, 0xFF800000, 0x7FC00000, 0xFFC00000,
                        0x7F800001, 0x7F807FFF, 0xFF800001, 0x7FFFFFFF], np.uint64)
    u = np.concatenate([pats, even_tie, odd_tie, special]).astype(np.uint32)
    x = u.view(np.float32)
    got = (orc.f32_to_bf16_rn(x).view(np.uint32) >> 16).astype(np.uint16)
    want = _torch_bf16_bits(x)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], want[~nan])
    # NaN stays NaN with its sign (torch's NaN payload is its own choice)
    g32 = (got[nan].astype(np.uint32) << 16).view(np.float32)
    assert np.isnan(g32).all() and np.array_equal(np.signbit(g32), np.signbit(x[nan]))
    # the finite tie cases really go to the even kept pattern, both ways (a carry out
    # of the largest finite pattern gives infinity, as it should)
    for ties, up in ((even_tie, 0), (odd_tie, 1)):
        t32 = ties.astype(np.uint32).view(np.float32)
        fin = np.isfinite(t32)
        g = (orc.f32_to_bf16_rn(t32[fin]).view(np.uint32) >> 16).astype(np.uint64)
        assert np.array_equal(g, (ties[fin] >> 16) + up)
        assert fin.sum() > 32000


def test_bf16_widening_matches_torch():
    """bf16_bits_to_f64 against torch's bfloat16 -> float64 on every bit pattern."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):        # NaN patterns widen to NaN
        got = orc.bf16_bits_to_f64(bits)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


# ---------------------------------------------------------------- Delta source and smooth_k

def _torch_ste_grads(q, k, v, do, sc, causal):
    """float64 autograd of <dO, softmax(sc Q K^T) V> (torch, a library routine)."""
    tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(
        tq[None, None], tk[None, None], tv[None, None], is_causal=causal, scale=sc)[0, 0]
    (o * torch.tensor(do)).sum().backward()
    return o.detach().numpy(), tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


def _torch_softmax(q, k, sc, causal):
    s = torch.tensor(q) @ torch.tensor(k).T * sc
    if causal:
        n = s.shape[0]
        s = s.masked_fill(torch.ones(n, n, dtype=torch.bool).triu(1), float("-inf"))
    return torch.softmax(s, dim=1).numpy()


@pytest.mark.parametrize("causal", [False, True])
def test_page_backward_delta_source_closed_forms(causal):
    """The page's backward forms Delta from O_q.  Then dS = dS_ste + c_i P_ij with
    c_i = <dO_i, O_hp,i - O_q,i>, so against the straight-through gradients (torch
    float64 autograd) dQ_page - dQ_ste = sm_scale c (P K) and dK_page - dK_ste =
    sm_scale P^T diag(c) Q.  dV_page = Pq^T dO is pinned by its adjoint: for any V',
    <dV_page, V'> = <dO, O_q(Q, K, V')>.  A Delta taken from O_hp, a dropped or
    sign-flipped term, or a transposed dV product fails one of these."""
    n, d, sc = 150, 8, 0.9
    q, k, v, do = (rng_f64(200 + i, n, d, scale=1.5) for i in range(4))
    dq, dk, dv = orc.head_backward_page(q, k, v, do, sc, causal)
    o_hp, dq_s, dk_s, dv_s = _torch_ste_grads(q, k, v, do, sc, causal)
    o_q = orc.head_forward(q, k, v, sc, causal, quant=True)["o_q"]
    c = (do * (o_hp - o_q)).sum(axis=1)
    assert np.abs(c).max() > 1e-3 * np.abs((do * o_hp).sum(axis=1)).max()  # O_q != O_hp
    p = _torch_softmax(q, k, sc, causal)
    assert np.allclose(dq - dq_s, sc * c[:, None] * (p @ k), rtol=1e-9, atol=1e-12)
    assert np.allclose(dk - dk_s, sc * p.T @ (c[:, None] * q), rtol=1e-9, atol=1e-12)
    v2 = rng_f64(209, n, d)
    o_q2 = orc.head_forward(q, k, v2, sc, causal, quant=True)["o_q"]
    assert np.isclose((dv * v2).sum(), (do * o_q2).sum(), rtol=1e-10)
    assert not np.allclose(dq, dq_s, rtol=1e-4)   # the Delta source matters here


def test_smooth_k_dq_term_closed_forms():
    """SMOOTH_K adds sm_scale rowsum(dS) k_mean to dQ.  Straight-through: rowsum(dS) = 0,
    and dQ equals torch's gradient through the unsmoothed K = K_s + k_mean.  The page's
    backward: dQ = dQ_ste(K_s) + sm_scale c (P K_s + k_mean) with c as above."""
    n, d, sc = 120, 8, 0.8
    q, ks, v, do = (rng_f64(220 + i, n, d) for i in range(4))
    mu = rng_f64(225, d, scale=3.0)
    dq0, dk0, dv0 = orc.head_backward(q, ks, v, do, sc, False)
    dq1, dk1, dv1 = orc.head_backward(q, ks, v, do, sc, False, k_mean=mu)
    _, dq_t, _, _ = _torch_ste_grads(q, ks + mu[None, :], v, do, sc, False)
    assert np.allclose(dq1, dq_t, rtol=1e-9, atol=1e-12)
    assert np.allclose(dq1, dq0, rtol=1e-9, atol=1e-12)
    assert np.array_equal(dk1, dk0) and np.array_equal(dv1, dv0)
    dqp, dkp, dvp = orc.head_backward_page(q, ks, v, do, sc, False, k_mean=mu)
    o_hp, dq_s, _, _ = _torch_ste_grads(q, ks, v, do, sc, False)
    o_q = orc.head_forward(q, ks, v, sc, False, quant=True)["o_q"]
    c = (do * (o_hp - o_q)).sum(axis=1)
    p = _torch_softmax(q, ks, sc, False)
    assert np.allclose(dqp, dq_s + sc * c[:, None] * (p @ ks + mu[None, :]), rtol=1e-9, atol=1e-12)
    dqp0, dkp0, dvp0 = orc.head_backward_page(q, ks, v, do, sc, False)
    assert np.array_equal(dkp, dkp0) and np.array_equal(dvp, dvp0)
    assert not np.allclose(dqp, dqp0, rtol=1e-4)


def test_quant_rows_exact_matches_forward_quantization():
    """Quantizing the forward's P per row x tile gives the forward's Pq (the code depends
    only on p / amax; the scale carries exp(T - m) / l); the codes are idempotent."""
    n, d = 70, 8
    q, k, v = (rng_f64(230 + i, n, d, scale=2.0) for i in range(3))
    for causal in (False, True):
        f = orc.head_forward(q, k, v, 0.7, causal, quant=True, return_p=True)
        assert np.allclose(orc.quant_rows_exact(f["p"]), f["pq"], rtol=1e-12, atol=1e-15)
    pq = orc.quant_rows_exact(f["p"])
    assert np.allclose(orc.quant_rows_exact(pq), pq, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_from_stats(causal):
    """With (o, lse) from a forward on the same inputs the literal page form equals the
    straight-through and the page's backward.  It rematerializes P from the SAVED lse:
    shifting lse by an integer delta scales P by 2^-delta, and with o fixed every
    gradient scales the same way, dV exactly so also when it is quantized (the E4M3 code
    depends only on p / amax)."""
    n, d, sc = 100, 8, 0.6
    q, k, v, do = (rng_f64(240 + i, n, d) for i in range(4))
    mu = rng_f64(245, d)
    f = orc.head_forward(q, k, v, sc, causal, quant=True)
    a = orc.head_backward_from_stats(q, k, v, do, f["o_hp"], f["lse"], sc, causal, k_mean=mu)
    b = orc.head_backward(q, k, v, do, sc, causal, k_mean=mu)
    for x, y in zip(a, b):
        assert np.allclose(x, y, rtol=1e-9, atol=1e-12)
    a = orc.head_backward_from_stats(q, k, v, do, f["o_q"], f["lse"], sc, causal, quant_dv=True,
                                     k_mean=mu)
    b = orc.head_backward_page(q, k, v, do, sc, causal, k_mean=mu)
    for x, y in zip(a, b):
        assert np.allclose(x, y, rtol=1e-9, atol=1e-12)
    for qd in (False, True):
        base = orc.head_backward_from_stats(q, k, v, do, f["o_q"], f["lse"], sc, causal, quant_dv=qd)
        shift = orc.head_backward_from_stats(q, k, v, do, f["o_q"], f["lse"] + 3.0, sc, causal,
                                             quant_dv=qd)
        for x, y in zip(shift, base):
            assert np.allclose(x, y / 8.0, rtol=1e-12, atol=1e-15)


def test_subtract_mean_bf16_matches_torch():
    """bf16(fl32(x - mean)) against torch's float32 subtraction and bf16 conversion."""
    rng = np.random.default_rng(250)
    x = orc.f32_to_bf16_rn(rng.standard_normal((40, 64)).astype(np.float32) * 3)
    mu = (rng.standard_normal(64) * 2).astype(np.float32)
    got = orc.subtract_mean_bf16(x, mu)
    want = (torch.from_numpy(x) - torch.from_numpy(mu)).to(torch.bfloat16).float().numpy()
    assert np.array_equal(got, want)
    assert np.array_equal(orc.subtract_mean_bf16(x, np.zeros(64, np.float32)), x)
