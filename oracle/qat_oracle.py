"""Plain, slow fp64 CPU oracle for quantization-aware attention (QAT attention).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference arm of ``bench.py`` may import this module.  The product
path (the CUDA library and its Python binding) never imports, calls or links it,
and this module imports nothing from the product package.

What it computes, per (batch b, head h, query row i), over the valid keys
V_i = {j < Nkv, and j <= i when causal}:

  s_ij   = sm_scale * <q_i, k_j>
  m_i    = max_j s_ij,  e_ij = exp(s_ij - m_i),  l_i = sum_j e_ij,  P_ij = e_ij / l_i
  O_hp,i = sum_j P_ij v_j                       (the straight-through output)
  lse_i  = (m_i + ln l_i) / ln 2                (base-2 log-sum-exp)
  quant tile t of row i = {j in V_i : floor(j / 64) = t}, T_it = max_{j in t} s_ij
  c_ij   = E4M3_RNE_SATFINITE(448 * exp(s_ij - T_it))
  Pq_ij  = c_ij * exp(T_it - m_i) / 448 / l_i
  O_q,i  = sum_j Pq_ij v_j                      (the returned output)

Sources (page titles and sections):
  * "attn_qat_train.py" (FastVideo fastvideo-kernel), ``_attn_fwd_inner``: online
    base-2 softmax with qk_scale = sm_scale * log2(e), exp2 of the shifted scores,
    ``fake_quantize`` of P per (query rows x KV tile), the row sum l taken from the
    *unquantized* P, and two accumulators (quantized and high precision).
  * same page, ``_attn_fwd`` epilogue: ``m_i += log2(l_i)`` stored as M (base 2), and
    both accumulators divided by l_i.
  * same page, ``_attn_bwd_preprocess``: Delta_i = sum_d O_id dO_id.
  * same page, ``_attn_bwd_dkdv`` / ``_attn_bwd_dq``: P rematerialized from the saved
    statistic, dP = dO V^T, dS = P o (dP - Delta), dK = sm_scale dS^T Q,
    dQ = sm_scale dS K, dV = P^T dO.
  * "support for pytorch autograd" (SageAttention issue 60): the backward is built by
    rematerialization, as for FlashAttention.

Readings where the pages are silent (``quant_utils`` is imported but not shown):
  * FP8 format: OCP E4M3 (bias 7, max 448, subnormal step 2^-9), round to nearest
    even, saturating to +-448.
  * Scale: absmax / 448 per (query row x 64-key tile); tiles aligned to absolute key 0.
  * Masked / padded keys are excluded from the tile max, from l and from O.
  * Straight-through estimator: the backward differentiates L = <dO, O_hp>, i.e.
    quantization is treated as the identity; Delta uses O_hp; dV uses unquantized P.

The fp32 quantization primitive (``quant_tiles_fp32``) is the bit-level rule the
CUDA kernels follow for one row x 64-key tile of fp32 probabilities:
  amax = max p; if amax == 0: scale 0, codes 0, values 0;
  else inv = fl32(448 / amax), scale = fl32(amax / 448) (IEEE round-to-nearest),
  code = E4M3_RNE_SATFINITE(fl32(p * inv)), value = bf16_rn(fl32(decode(code) * scale)).
In exact arithmetic code depends only on p / amax, so it equals the definition above.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, invariants, brute force, library routines, finite differences):
the bf16 conversions against torch's own conversions over tie, subnormal, overflow,
infinity and NaN patterns; the page's backward through the closed forms its Delta
source implies (dQ_page - dQ_ste = sm_scale c P K with c = <dO, O_hp - O_q>, torch
autograd for the straight-through part) and the adjoint identity of its dV; the
SMOOTH_K dQ term by the same closed forms.  The one exception is fidelity to the
pages' own ``fake_quantize`` — parity unpinned, because its source (``quant_utils``)
is not on the pages.
"""

from __future__ import annotations

import math

import numpy as np

E4M3_MAX = 448.0          # largest finite OCP E4M3 value: 2^8 * 1.75
E4M3_MIN_NORMAL_EXP = -6  # exponent of the smallest normal E4M3 value (2^-6)
E4M3_MANT_BITS = 3
QUANT_TILE = 64           # keys per quantization tile (absolute key alignment)
LN2 = math.log(2.0)


# ---------------------------------------------------------------------------
# OCP FP8 E4M3
# ---------------------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    """Value of each E4M3 byte (OCP OFP8): sign bit 7, exponent bits 6..3 (bias 7),
    mantissa bits 2..0; exponent 0 is subnormal (2^-6 * m / 8); 0x7F / 0xFF are NaN."""
    c = np.asarray(codes, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64))
    sub = np.ldexp(m / 8.0, np.full_like(e, E4M3_MIN_NORMAL_EXP))
    val = sign * np.where(e == 0, sub, normal)
    return np.where((c & 0x7F) == 0x7F, np.nan, val)


def e4m3_rne_satfinite(x) -> tuple[np.ndarray, np.ndarray]:
    """Round finite reals to E4M3 with round-to-nearest-even, saturating to +-448.

    Returns (code bytes as uint8, value as float64).  The rounding quantum of a value
    with binary exponent e is 2^(max(e, -6) - 3); dividing by a power of two and
    ``np.rint`` (ties to even) are exact, so the result is the correctly rounded one.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, ex = np.frexp(a)                      # a = f * 2^ex, f in [0.5, 1)
    e = np.maximum(ex - 1, E4M3_MIN_NORMAL_EXP)
    quantum = np.ldexp(1.0, e - E4M3_MANT_BITS)
    q = np.rint(a / quantum) * quantum
    q = np.minimum(q, E4M3_MAX)
    # encode q (exactly representable by construction)
    _, qex = np.frexp(q)
    qe = qex - 1
    is_norm = q >= 2.0 ** E4M3_MIN_NORMAL_EXP
    mant_norm = np.rint(np.ldexp(q, -qe) * 8.0 - 8.0)
    code_norm = ((qe + 7) << 3) + mant_norm.astype(np.int64)
    code_sub = np.rint(q / 2.0 ** -9).astype(np.int64)
    code = np.where(is_norm, code_norm, code_sub)
    code = np.where(np.signbit(x) & (q > 0), code | 0x80, code)
    return code.astype(np.uint8), np.copysign(q, x)


# ---------------------------------------------------------------------------
# bf16 helpers (the oracle's own; nothing shared with the product)
# ---------------------------------------------------------------------------

def bf16_bits_to_f64(bits) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) exactly to float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def f32_to_bf16_rn(x) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns float32 values.

    On the bit pattern u: adding 0x7FFF plus the lowest kept bit and truncating the low
    16 bits rounds to nearest with ties to the even kept pattern; a carry out of the
    mantissa raises the exponent (the largest finite values round up to infinity), and
    infinities are unchanged.  NaN stays NaN: the carry could turn a NaN whose payload
    sits in the low 16 bits into infinity, so NaNs take the quiet NaN of their sign.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    r = np.where(np.isnan(x), (u & 0x80000000) | 0x7FC00000, r)
    return r.astype(np.uint32).view(np.float32)


# ---------------------------------------------------------------------------
# The fp32 quantization primitive for row x 64-key tiles
# ---------------------------------------------------------------------------

def quant_tiles_fp32(p) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Fake-quantize fp32 tiles row by row: p has shape [rows, cols] (one tile per row).
    amax is the largest magnitude, so signed data (Q, K, V) use the same rule as P.

    Returns (deq float32 [rows, cols] = bf16-rounded quantized values,
             scale float32 [rows] = amax / 448,
             codes uint8 [rows, cols]).
    All arithmetic is IEEE float32 with round-to-nearest, as the rule states.
    """
    p = np.ascontiguousarray(p, dtype=np.float32)
    amax = np.abs(p).max(axis=1)
    nz = amax > 0
    safe = np.where(nz, amax, np.float32(1.0)).astype(np.float32)
    inv = (np.float32(E4M3_MAX) / safe).astype(np.float32)
    scale = (safe / np.float32(E4M3_MAX)).astype(np.float32)
    x = (p * inv[:, None]).astype(np.float32)
    codes, vals = e4m3_rne_satfinite(x.astype(np.float64))
    deq32 = (vals.astype(np.float32) * scale[:, None]).astype(np.float32)
    deq = f32_to_bf16_rn(deq32)
    codes = np.where(nz[:, None], codes, np.uint8(0)).astype(np.uint8)
    deq = np.where(nz[:, None], deq, np.float32(0)).astype(np.float32)
    scale = np.where(nz, scale, np.float32(0)).astype(np.float32)
    return deq, scale, codes


# ---------------------------------------------------------------------------
# Forward (fp64) for one (b, h) head
# ---------------------------------------------------------------------------

def _valid_mask(rows: np.ndarray, nkv: int, causal: bool) -> np.ndarray:
    cols = np.arange(nkv)
    if causal:
        return cols[None, :] <= rows[:, None]
    return np.ones((rows.size, nkv), dtype=bool)


def head_forward(q, k, v, sm_scale: float, causal: bool, quant: bool,
                 rows=None, return_p: bool = False):
    """fp64 forward of one head.

    q [Nq, D], k/v [Nkv, D] (float64).  ``rows`` selects query rows (default all);
    rows are independent, so a subset is the same definition applied to fewer i.
    Returns dict with o_hp, o_q (if quant), lse (base 2), and optionally p / pq.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    nq, nkv = q.shape[0], k.shape[0]
    rows = np.arange(nq) if rows is None else np.asarray(rows)
    valid = _valid_mask(rows, nkv, causal)
    s = sm_scale * (q[rows] @ k.T)                              # s_ij
    s_m = np.where(valid, s, -np.inf)
    m = s_m.max(axis=1)                                         # m_i
    e = np.where(valid, np.exp(s_m - m[:, None]), 0.0)          # e_ij
    l = e.sum(axis=1)                                           # l_i (unquantized)
    p = e / l[:, None]                                          # P_ij
    out = {"o_hp": p @ v, "lse": (m + np.log(l)) / LN2, "m": m, "l": l}
    if return_p:
        out["p"] = p
    if quant:
        pq = np.zeros_like(p)
        ntiles = (nkv + QUANT_TILE - 1) // QUANT_TILE
        for t in range(ntiles):
            lo, hi = t * QUANT_TILE, min(nkv, (t + 1) * QUANT_TILE)
            st = s_m[:, lo:hi]
            vt = valid[:, lo:hi]
            has = vt.any(axis=1)
            T = np.where(has, st.max(axis=1), 0.0)              # T_it
            ratio = np.where(vt, np.exp(st - T[:, None]), 0.0)  # exp(s_ij - T_it)
            _, c = e4m3_rne_satfinite(E4M3_MAX * ratio)         # c_ij (values)
            w = np.where(has, np.exp(T - m) / E4M3_MAX / l, 0.0)
            pq[:, lo:hi] = c * w[:, None]                       # Pq_ij
        out["o_q"] = pq @ v
        if return_p:
            out["pq"] = pq
    return out


def forward(q, k, v, sm_scale: float, causal: bool, quant: bool, row_chunk: int = 2048):
    """fp64 forward over [B, H, N, D] arrays; returns (o_q, o_hp, lse) (o_q None if not quant)."""
    B, H, nq, D = q.shape
    o_hp = np.zeros((B, H, nq, D))
    o_q = np.zeros((B, H, nq, D)) if quant else None
    lse = np.zeros((B, H, nq))
    for b in range(B):
        for h in range(H):
            for r0 in range(0, nq, row_chunk):
                rows = np.arange(r0, min(nq, r0 + row_chunk))
                r = head_forward(q[b, h], k[b, h], v[b, h], sm_scale, causal, quant, rows)
                o_hp[b, h, rows] = r["o_hp"]
                lse[b, h, rows] = r["lse"]
                if quant:
                    o_q[b, h, rows] = r["o_q"]
    return o_q, o_hp, lse


# ---------------------------------------------------------------------------
# Backward (fp64, straight-through estimator) for one (b, h) head
# ---------------------------------------------------------------------------

def _smooth_k_dq_term(ds, k_mean, sm_scale: float):
    """The page's SMOOTH_K correction of dQ ("attn_qat_train.py", _attn_bwd_dq, the
    ``if SMOOTH_K`` branch): every key block adds rowsum(dS) k_mean to dQ, so in all
    sm_scale * rowsum_j(dS_ij) * k_mean.  K went into the scores with its channel mean
    subtracted; the term gives dQ as if the mean had stayed in (dS (K + 1 k_mean^T))."""
    if k_mean is None:
        return 0.0
    return sm_scale * ds.sum(axis=1)[:, None] * np.asarray(k_mean, np.float64)[None, :]


def head_backward(q, k, v, do, sm_scale: float, causal: bool, k_mean=None):
    """Gradients of L = <dO, O_hp> with respect to q, k, v for one head (fp64).

    Delta_i = sum_d dO_id O_hp,id ; dP = dO V^T ; dS = P o (dP - Delta) ;
    dQ = sm_scale dS K ; dK = sm_scale dS^T Q ; dV = P^T dO.
    With ``k_mean`` (smooth_k: K is the smoothed key) dQ also gets the page's SMOOTH_K
    term sm_scale rowsum(dS) k_mean, which is zero in exact arithmetic here because
    Delta comes from the same O_hp that P and V form.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    do = np.asarray(do, np.float64)
    f = head_forward(q, k, v, sm_scale, causal, quant=False, return_p=True)
    p, o_hp = f["p"], f["o_hp"]
    delta = (do * o_hp).sum(axis=1)
    dp = do @ v.T
    ds = p * (dp - delta[:, None])
    dq = sm_scale * (ds @ k) + _smooth_k_dq_term(ds, k_mean, sm_scale)
    return dq, sm_scale * (ds.T @ q), p.T @ do


def backward(q, k, v, do, sm_scale: float, causal: bool):
    """fp64 STE backward over [B, H, N, D] arrays; returns (dq, dk, dv)."""
    dq = np.zeros(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            dq[b, h], dk[b, h], dv[b, h] = head_backward(
                q[b, h], k[b, h], v[b, h], do[b, h], sm_scale, causal)
    return dq, dk, dv


# ---------------------------------------------------------------------------
# Sampled checks for long sequences (same definitions, fewer outputs)
# ---------------------------------------------------------------------------

def head_row_stats(q, k, sm_scale: float, causal: bool, row_chunk: int = 1024):
    """m_i and l_i for every query row of one head, rows taken in independent chunks."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    nq, nkv = q.shape[0], k.shape[0]
    m = np.empty(nq)
    l = np.empty(nq)
    for r0 in range(0, nq, row_chunk):
        rows = np.arange(r0, min(nq, r0 + row_chunk))
        valid = _valid_mask(rows, nkv, causal)
        s = np.where(valid, sm_scale * (q[rows] @ k.T), -np.inf)
        m[rows] = s.max(axis=1)
        l[rows] = np.exp(s - m[rows][:, None]).sum(axis=1)
    return m, l


def head_backward_sampled(q, k, v, do, sm_scale: float, causal: bool,
                          q_rows, kv_rows, row_chunk: int = 1024):
    """dQ at rows ``q_rows`` and dK / dV at key rows ``kv_rows`` of one head (fp64).

    Uses the same formulas as ``head_backward``; O_hp and Delta are needed for every
    query row because dK_j and dV_j sum over all i, so they are formed chunk by chunk.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    do = np.asarray(do, np.float64)
    nq, nkv = q.shape[0], k.shape[0]
    q_rows = np.asarray(q_rows)
    kv_rows = np.asarray(kv_rows)
    m, l = head_row_stats(q, k, sm_scale, causal, row_chunk)
    delta = np.empty(nq)
    p_cols = np.empty((nq, kv_rows.size))      # P[:, kv_rows]
    for r0 in range(0, nq, row_chunk):
        rows = np.arange(r0, min(nq, r0 + row_chunk))
        valid = _valid_mask(rows, nkv, causal)
        s = np.where(valid, sm_scale * (q[rows] @ k.T), -np.inf)
        p = np.exp(s - m[rows][:, None]) / l[rows][:, None]
        delta[rows] = (do[rows] * (p @ v)).sum(axis=1)
        p_cols[rows] = p[:, kv_rows]
    dp_cols = do @ v[kv_rows].T                                 # dP[:, kv_rows]
    ds_cols = p_cols * (dp_cols - delta[:, None])
    dk = sm_scale * (ds_cols.T @ q)
    dv = p_cols.T @ do
    valid = _valid_mask(q_rows, nkv, causal)
    s = np.where(valid, sm_scale * (q[q_rows] @ k.T), -np.inf)
    p = np.exp(s - m[q_rows][:, None]) / l[q_rows][:, None]
    ds = p * (do[q_rows] @ v.T - delta[q_rows][:, None])
    dq = sm_scale * (ds @ k)
    return dq, dk, dv


# ---------------------------------------------------------------------------
# Q / K / V fake quantization and smooth_k (the page's IS_QAT input path)
# ---------------------------------------------------------------------------
# Sources: "attn_qat_train.py", _attention.forward: with IS_QAT the inputs are replaced
# by fake-quantized copies (fake_quantize_q with BLOCK_M = 32 tokens, fake_quantize_kv
# with BLOCK_N = 32 tokens, one program per 32-token block of one (batch, head)), the
# backward uses those copies (use_qat_qkv_backward), and smooth_k first subtracts
# k.mean(dim=(0, 1, 2)), the per-channel mean over batch, heads and tokens.
# Readings (quant_utils is not on the pages): one FP8 E4M3 absmax scale per 32-token x D
# block, tokens beyond N excluded; the smoothed value is fl32(k - mean) and is quantized
# directly (no intermediate bf16 rounding); the stored result is bf16.

QKV_TOKEN_BLOCK = 32


def fake_quant_tokens_fp32(x, mean=None):
    """fp32 rule for one head: x [N, D] (float32 values), optional fp32 mean [D] subtracted
    first; one scale per 32-token block over all D values.  Returns (out float32 values
    of the bf16 result [N, D], scales float32 [ceil(N/32)], codes uint8 [N, D])."""
    x = np.asarray(x, dtype=np.float32)
    if mean is not None:
        x = (x - np.asarray(mean, dtype=np.float32)[None, :]).astype(np.float32)
    n, d = x.shape
    nb = (n + QKV_TOKEN_BLOCK - 1) // QKV_TOKEN_BLOCK
    out = np.zeros((n, d), np.float32)
    codes = np.zeros((n, d), np.uint8)
    scales = np.zeros(nb, np.float32)
    for b in range(nb):
        lo, hi = b * QKV_TOKEN_BLOCK, min(n, (b + 1) * QKV_TOKEN_BLOCK)
        deq, sc, cd = quant_tiles_fp32(x[lo:hi].reshape(1, -1))
        out[lo:hi] = deq.reshape(hi - lo, d)
        codes[lo:hi] = cd.reshape(hi - lo, d)
        scales[b] = sc[0]
    return out, scales, codes


def fake_quant_tokens_exact(x):
    """Exact-arithmetic form for one head (fp64): per 32-token block,
    value = E4M3(448 x / amax) amax / 448 (zero block -> zero)."""
    x = np.asarray(x, np.float64)
    out = np.zeros_like(x)
    for lo in range(0, x.shape[0], QKV_TOKEN_BLOCK):
        blk = x[lo:lo + QKV_TOKEN_BLOCK]
        amax = np.abs(blk).max()
        if amax > 0:
            _, c = e4m3_rne_satfinite(448.0 * blk / amax)
            out[lo:lo + QKV_TOKEN_BLOCK] = c * amax / 448.0
    return out


def subtract_mean_bf16(x, mean):
    """smooth_k's subtraction without the quantization, as stored: bf16_rn(fl32(x - mean))
    per element (x float32 values [..., D], mean float32 [D]); returns float32 values."""
    x = np.asarray(x, np.float32)
    d = (x - np.asarray(mean, np.float32)).astype(np.float32)
    return f32_to_bf16_rn(d)


def channel_mean(x):
    """smooth_k's offset: the mean of x [B, H, N, D] over B, H and N, per channel (fp64)."""
    x = np.asarray(x, np.float64)
    return x.reshape(-1, x.shape[-1]).mean(axis=0)


# ---------------------------------------------------------------------------
# Partial results over key chunks and their merge (ring / context-parallel block)
# ---------------------------------------------------------------------------
# A forward over keys [c0, c1) of each head gives O_q, O_hp (each normalized by its own
# l) and lse (base 2).  Two partials over disjoint key sets merge exactly:
#   lse = log2(2^lse_a + 2^lse_b),  O = 2^(lse_a - lse) O_a + 2^(lse_b - lse) O_b
# for O_hp; for O_q the same holds when every chunk starts at a multiple of 64 keys, so
# each 64-key quantization tile lies inside one chunk (the per-tile codes and amax are
# then the same as in a one-pass forward, and O_q carries the same weights as O_hp).
# Source of the setting: "usp: differentiable operators for training (Ulysses/Ring/local
# attention)" (ring attention passes partial outputs between ranks and merges them).

def merge_partials(o_a, lse_a, o_b, lse_b):
    """Merge two partial attention results (fp64): o [..., rows, D], lse [..., rows]."""
    lse_a = np.asarray(lse_a, np.float64)
    lse_b = np.asarray(lse_b, np.float64)
    hi = np.maximum(lse_a, lse_b)
    hi = np.where(np.isfinite(hi), hi, 0.0)
    wa = np.exp2(lse_a - hi)
    wb = np.exp2(lse_b - hi)
    lse = hi + np.log2(wa + wb)
    tot = wa + wb
    o = (wa[..., None] * np.asarray(o_a, np.float64) + wb[..., None] * np.asarray(o_b, np.float64))
    return o / tot[..., None], lse


# ---------------------------------------------------------------------------
# The page's own backward variant (quant_mode 2)
# ---------------------------------------------------------------------------
# "attn_qat_train.py", _attn_bwd_dkdv: dv += dot(trans(p_quant), do) with
# p_quant = fake_quantize(p) (the same per query row x KV tile quantization as the
# forward), while ds = p * (dp - Di) uses the unquantized p; _attention.forward passes
# o_for_bwd = O (the quantized output) to _attn_bwd_preprocess when use_high_prec_o is
# False (its default), so Delta = rowsum(dO * O_q).

def head_backward_page(q, k, v, do, sm_scale: float, causal: bool, k_mean=None):
    """dQ, dK, dV of the page's default backward for one head (fp64).  With ``k_mean``
    dQ gets the SMOOTH_K term, which is not zero here: sum_j dS_ij = Delta(O_hp)_i -
    Delta(O_q)_i."""
    do = np.asarray(do, np.float64)
    f = head_forward(q, k, v, sm_scale, causal, quant=True, return_p=True)
    p, pq, o_q = f["p"], f["pq"], f["o_q"]
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    q = np.asarray(q, np.float64)
    delta = (do * o_q).sum(axis=1)
    ds = p * (do @ v.T - delta[:, None])
    dq = sm_scale * (ds @ k) + _smooth_k_dq_term(ds, k_mean, sm_scale)
    return dq, sm_scale * (ds.T @ q), pq.T @ do


def quant_rows_exact(p):
    """Exact-arithmetic fake quantization of probabilities p [rows, Nkv] (fp64) per row x
    absolute 64-key tile: code = E4M3(448 p / amax), value = code amax / 448; a tile with
    amax = 0 stays zero.  (The same rule as the forward's, applied to a given P.)"""
    p = np.asarray(p, np.float64)
    out = np.zeros_like(p)
    for lo in range(0, p.shape[1], QUANT_TILE):
        t = p[:, lo:lo + QUANT_TILE]
        amax = t.max(axis=1)
        safe = np.where(amax > 0, amax, 1.0)
        _, c = e4m3_rne_satfinite(E4M3_MAX * t / safe[:, None])
        out[:, lo:lo + QUANT_TILE] = np.where((amax > 0)[:, None], c * (safe / E4M3_MAX)[:, None], 0.0)
    return out


def head_backward_from_stats(q, k, v, do, o, lse, sm_scale: float, causal: bool,
                             quant_dv: bool = False, k_mean=None):
    """The page's backward kernels taken literally for one head (fp64): P is
    rematerialized from the SAVED base-2 lse ("attn_qat_train.py", _attn_bwd_dkdv and
    _attn_bwd_dq: p = exp2(qk * qk_scale - m)), Delta from the given output o
    (_attn_bwd_preprocess), dV from P or, with ``quant_dv``, from fake_quantize(P) per
    query row x 64-key tile, and dQ with the SMOOTH_K term when ``k_mean`` is given.

    When (o, lse) come from a forward on the same q, k, v this is ``head_backward``
    (o = O_hp) or ``head_backward_page`` (o = O_q, quant_dv).  The page also runs it on
    other inputs: with use_qat_qkv_backward = False the backward gets the unquantized
    q, k, v while o and lse come from the forward on their fake-quantized copies, and
    then the rows of P need not sum to 1."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    do = np.asarray(do, np.float64)
    nq, nkv = q.shape[0], k.shape[0]
    valid = _valid_mask(np.arange(nq), nkv, causal)
    s = sm_scale * (q @ k.T)
    p = np.where(valid, np.exp2(s / LN2 - np.asarray(lse, np.float64)[:, None]), 0.0)
    delta = (do * np.asarray(o, np.float64)).sum(axis=1)
    ds = p * (do @ v.T - delta[:, None])
    dq = sm_scale * (ds @ k) + _smooth_k_dq_term(ds, k_mean, sm_scale)
    pv = quant_rows_exact(p) if quant_dv else p
    return dq, sm_scale * (ds.T @ q), pv.T @ do
