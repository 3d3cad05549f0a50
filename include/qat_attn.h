/*
 * qat_attn.h -- C ABI of the GB300 (sm_103a) quantization-aware attention library.
 *
 * The library computes training-time scaled-dot-product attention whose softmax
 * probabilities P are fake-quantized to FP8 E4M3 with an absmax scale per
 * (query row x 64-key tile), keeping a straight-through high-precision output beside
 * the quantized one, and the matching backward.
 *
 * Sources (page titles and sections):
 *   "attn_qat_train.py" (FastVideo fastvideo-kernel):
 *     _attn_fwd_inner   online base-2 softmax, fake_quantize(P), l from unquantized P,
 *                       two accumulators (quantized and high precision);
 *     _attn_fwd         epilogue: M = m + log2(l) (base 2), both outputs divided by l;
 *     _attn_bwd_preprocess  Delta = rowsum(O * dO);
 *     _attn_bwd_dkdv, _attn_bwd_dq, _attn_bwd  dV, dP, dS, dK, dQ with P rematerialized;
 *     _attention.forward / .backward  the host contract (save q, k, v, O, M).
 *   "support for pytorch autograd" (SageAttention issue 60): backward by
 *     rematerialization, as for FlashAttention.
 *
 * Conventions shared by every entry point
 *   - Tensors are dense, contiguous, row-major; bf16 tensors are [B, H, N, D] with D
 *     innermost.  "bf16" buffers hold IEEE bfloat16 bit patterns.
 *   - All pointers are DEVICE pointers unless stated otherwise, 16-byte aligned.
 *   - The caller owns every buffer.  The library allocates no device memory on these
 *     paths and keeps no per-call state; it caches only its loaded kernels and the
 *     SM count of each device.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  A QAT_OK return means the work was enqueued.
 *   - Nothing throws across the ABI; every failure is a status code.  Arguments are
 *     validated on the host before anything is enqueued.
 */
#ifndef QAT_ATTN_H
#define QAT_ATTN_H

#include <stddef.h>

#if defined(__GNUC__)
#define QAT_API __attribute__((visibility("default")))
#else
#define QAT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QAT_OK = 0,
  QAT_ERR_INVALID_ARG = 1, /* null / misaligned pointer, bad size, bad D or mode   */
  QAT_ERR_UNSUPPORTED = 2, /* valid request this library does not implement       */
  QAT_ERR_CUDA = 3,        /* a CUDA runtime / launch error (see cudaGetLastError) */
  QAT_ERR_TIMEOUT = 4,     /* a bounded device-side wait expired (kernel returned)  */
  QAT_ERR_WORKSPACE = 5    /* workspace missing or smaller than required            */
} qat_status_t;

/* quant_mode values */
enum {
  QAT_QUANT_NONE = 0,                 /* O_q is computed with P unquantized (= O_hp)  */
  QAT_QUANT_P_FP8E4M3_ROW_TILE64 = 1, /* P fake-quantized per row x 64-key tile;
                                         straight-through backward                     */
  QAT_QUANT_P_FP8E4M3_ROW_TILE64_PAGE_BWD = 2 /* forward as mode 1; the page's default
                                         backward ("attn_qat_train.py", _attn_bwd_dkdv,
                                         use_high_prec_o = False): dV from the quantized
                                         P, Delta from O_q (pass O_q as `o_hp`), dS from
                                         the unquantized P                               */
};

/*
 * qat_attn_fwd -- forward pass.
 *   ("attn_qat_train.py", _attn_fwd and _attn_fwd_inner.)
 *
 *   q      bf16 [B, H, Nq,  D]   queries
 *   k, v   bf16 [B, H, Nkv, D]   keys, values
 *   o_q    bf16 [B, H, Nq,  D]   OUT: sum_j quant(P)_ij v_j  (the returned output)
 *   o_hp   bf16 [B, H, Nq,  D]   OUT: sum_j P_ij v_j         (straight-through output)
 *   lse    fp32 [B, H, Nq]       OUT: m_i + log2(l_i) in base-2 units of the scaled
 *                                logits s_ij * log2(e); kept for the backward.
 *   sm_scale   finite, > 0; scores are s_ij = sm_scale * <q_i, k_j>.
 *   causal     0 or 1; 1 masks keys j > i (top-left aligned); requires Nq == Nkv.
 *   quant_mode QAT_QUANT_NONE or QAT_QUANT_P_FP8E4M3_ROW_TILE64.  Quantization:
 *              per row i and tile t = {j : floor(j/64) = t}, amax = max_j p_ij,
 *              code = E4M3_RNE_SATFINITE(p_ij * (448 / amax)),
 *              quant(P)_ij = code * (amax / 448) / l_i, l_i summed from unquantized p.
 *   D          64 or 128.   B, H, Nq >= 0 (any zero: nothing to do, returns QAT_OK);
 *              Nkv >= 1 whenever there is work.
 * Errors: QAT_ERR_INVALID_ARG (null or non-16-byte-aligned pointer, negative size,
 *   Nkv < 1, D not in {64, 128}, bad sm_scale / causal / quant_mode, or a tensor of
 *   more than 2^31 rows), QAT_ERR_UNSUPPORTED (causal with Nq != Nkv),
 *   QAT_ERR_CUDA (launch failure).
 */
QAT_API qat_status_t qat_attn_fwd(const void* q, const void* k, const void* v,
                          void* o_q, void* o_hp, float* lse,
                          int B, int H, int Nq, int Nkv, int D,
                          float sm_scale, int causal, int quant_mode,
                          void* stream);

/*
 * qat_attn_bwd_workspace_bytes -- device workspace qat_attn_bwd needs for these sizes,
 * with Nq rounded up to a multiple of 128 per head (Nq_pad), each piece 256-byte
 * aligned: fp32 lse and Delta [B, H, Nq_pad]; bf16 [B, H, Nq_pad, 16] rows holding
 * -lse / (sm_scale log2 e) and -Delta, each as a sum of three bf16 terms, which the
 * dK/dV kernel adds to its score products through one extra MMA step; and a 4 KB
 * bf16 ones tile.  About 72 bytes per padded query row.  When the sizes give few
 * (head, 128-key block) pairs for the GPU's SMs, the dK/dV kernel cuts the pairs' query
 * blocks into one equal range per CTA (stream-K) and the workspace also holds fp32
 * partial sums of dV and dK for the pairs the ranges cut: two 128-row slots per CTA,
 * CTAs x 2 x 2 x 128 x D x 4 bytes (152 CTAs at B1 H40 Nq16384 Nkv512 D128, 40 MB).
 * The rule depends on the sizes only; it is also applied for causal calls, which do
 * not split, so a causal caller may get more workspace than it uses.
 * Returns 0 for invalid sizes.  Host-only; never touches the device.
 */
QAT_API size_t qat_attn_bwd_workspace_bytes(int B, int H, int Nq, int Nkv, int D);

/*
 * qat_attn_bwd -- backward pass through the straight-through estimator: gradients of
 * L = <dO, O_hp>, i.e. quantization of P is treated as the identity.
 *   ("attn_qat_train.py", _attn_bwd_preprocess, _attn_bwd_dkdv, _attn_bwd_dq.)
 *
 *   q, k, v  bf16        the forward's inputs
 *   o_hp     bf16 [B, H, Nq, D]  the forward's straight-through output
 *   lse      fp32 [B, H, Nq]     the forward's lse output
 *   dO       bf16 [B, H, Nq, D]  upstream gradient of o_q
 *   dq       bf16 [B, H, Nq, D]  OUT
 *   dk, dv   bf16 [B, H, Nkv, D] OUT
 *   Delta_i = sum_d dO_id O_hp,id;  P_ij = exp2(s_ij log2(e) - lse_i);
 *   dP = dO V^T;  dS = P o (dP - Delta);  dQ = sm_scale dS K;  dK = sm_scale dS^T Q;
 *   dV = P^T dO.
 *   quant_mode 0 and 1: the straight-through estimator, as above.  quant_mode 2: the
 *   page's default backward instead: pass the forward's O_q as `o_hp` (Delta =
 *   rowsum(dO o O_q)) and dV = quant(P)^T dO with the forward's per-tile rule.
 *   workspace  device buffer of at least qat_attn_bwd_workspace_bytes(...) bytes,
 *              256-byte aligned, owned by the caller; its contents on entry are
 *              ignored and on exit unspecified.
 *              A buffer that holds everything but the dK/dV partial sums (see
 *              qat_attn_bwd_workspace_bytes) is accepted and runs with one CTA per
 *              (head, key block) pair instead.
 * Errors: as qat_attn_fwd, plus QAT_ERR_WORKSPACE when workspace is NULL or
 *   workspace_bytes is below the workspace without the partial sums.  Nq == 0 with
 *   Nkv >= 1 writes zero dk, dv.
 */
QAT_API qat_status_t qat_attn_bwd(const void* q, const void* k, const void* v,
                          const void* o_hp, const float* lse, const void* dO,
                          void* dq, void* dk, void* dv,
                          int B, int H, int Nq, int Nkv, int D,
                          float sm_scale, int causal, int quant_mode,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * qat_attn_bwd_smooth_k -- qat_attn_bwd for keys smoothed by smooth_k (the channel mean
 * of K subtracted before attention, see qat_channel_mean): dQ also gets the page's
 * SMOOTH_K term.  ("attn_qat_train.py", _attn_bwd_dq, the `if SMOOTH_K` branch: every key
 * block adds rowsum(dS) k_mean to dq.)
 *   k        the SMOOTHED keys the forward used (k - k_mean, or their fake-quantized copy)
 *   k_mean   fp32 [D] (device, 16-byte aligned): the mean that was subtracted
 *   dQ_i = sm_scale (sum_j dS_ij k_j + (sum_j dS_ij) k_mean), the fp32 dS summed over all
 *   valid keys; dK and dV as qat_attn_bwd.  The term is zero in exact arithmetic under the
 *   straight-through estimator (quant_mode 0 / 1: sum_j dS_ij = 0 when Delta comes from
 *   O_hp) and not under quant_mode 2, where Delta comes from O_q.
 *   Every other argument as qat_attn_bwd.
 * Errors: as qat_attn_bwd; QAT_ERR_INVALID_ARG for a NULL or misaligned k_mean.
 */
QAT_API qat_status_t qat_attn_bwd_smooth_k(const void* q, const void* k, const void* v,
                          const void* o_hp, const float* lse, const void* dO,
                          void* dq, void* dk, void* dv, const float* k_mean,
                          int B, int H, int Nq, int Nkv, int D,
                          float sm_scale, int causal, int quant_mode,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * qat_attn_bwd_noalloc -- the same backward as qat_attn_bwd for callers that cannot
 * allocate device memory: for example a program whose device memory all belongs to
 * another runtime's pool, or one that must not allocate once running (an allocation
 * can block on the device or fail under memory pressure mid-step).  The paper has no
 * counterpart; this entry exists for such callers only.
 *   Arguments as qat_attn_bwd, without workspace / workspace_bytes.  The scratch lives
 *   in a fixed 32 MiB device array inside the library, held on every GPU that loads
 *   the library until the process exits.  It allocates nothing (no cudaMalloc,
 *   cudaFree or allocating library call).
 *   Every call looks up that array's device address with the device current (a host-side
 *   lookup that allocates nothing); the first call on a device also loads the library's
 *   device code there, so make that first call before any stream capture.
 *   All calls share the array and it keeps the last call's contents; calls that overlap
 *   on the GPU race on it and must be ordered by the caller.
 * Errors: as qat_attn_bwd, checked in the same order (sizes and modes, then pointers);
 *   then QAT_ERR_WORKSPACE when the sizes need more scratch than the array holds, not
 *   counting the dK/dV partial sums (the workspace without them above 32 MiB).  When the
 *   partial sums do not fit as well, the call runs with one CTA per (head, key block).
 */
QAT_API qat_status_t qat_attn_bwd_noalloc(const void* q, const void* k, const void* v,
                          const void* o_hp, const float* lse, const void* dO,
                          void* dq, void* dk, void* dv,
                          int B, int H, int Nq, int Nkv, int D,
                          float sm_scale, int causal, int quant_mode, void* stream);

/*
 * qat_attn_fwd_chunk -- forward over one chunk of keys, returning a partial result to be
 * merged with qat_attn_merge: the single-GPU building block of ring / context-parallel
 * attention ("usp: differentiable operators for training (Ulysses/Ring/local attention)":
 * ring attention rotates K/V chunks and merges partial outputs).
 *   q           bf16 [B, H, Nq, D]
 *   k, v        bf16 [B, H, Nkv_total, D]; keys [kv_begin, kv_begin + kv_len) are used
 *   o_q, o_hp   fp32 [B, H, Nq, D] OUT: the chunk's outputs, each normalized by the
 *               chunk's own row sum
 *   lse         fp32 [B, H, Nq] OUT: the chunk's base-2 log-sum-exp
 *   Non-causal only.  kv_begin must be a multiple of 64 so that no quantization tile is
 *   split between chunks; then merging all chunks reproduces the one-pass O_q exactly
 *   in real arithmetic, as it does O_hp and lse.
 * Errors: as qat_attn_fwd; QAT_ERR_INVALID_ARG for a chunk outside [0, Nkv_total);
 *   QAT_ERR_UNSUPPORTED when kv_begin % 64 != 0.
 */
QAT_API qat_status_t qat_attn_fwd_chunk(const void* q, const void* k, const void* v,
                                        float* o_q, float* o_hp, float* lse,
                                        int B, int H, int Nq, int Nkv_total, int kv_begin,
                                        int kv_len, int D, float sm_scale, int quant_mode,
                                        void* stream);

/*
 * qat_attn_merge -- merges a partial result into an accumulator (both fp32, same
 * layout as qat_attn_fwd_chunk's outputs), in place:
 *   lse_acc <- log2(2^lse_acc + 2^lse_part)
 *   O_acc   <- 2^(lse_acc_old - lse_acc) O_acc + 2^(lse_part - lse_acc) O_part
 * for O_q and O_hp.  If o_q_out / o_hp_out (bf16 [B, H, Nq, D]) are not NULL, the merged
 * outputs are also written there.  An lse of -inf marks an empty partial.
 * Errors: QAT_ERR_INVALID_ARG (null / misaligned pointer, bad size or D), QAT_ERR_CUDA.
 */
QAT_API qat_status_t qat_attn_merge(float* o_q_acc, float* o_hp_acc, float* lse_acc,
                                    const float* o_q_part, const float* o_hp_part,
                                    const float* lse_part, void* o_q_out, void* o_hp_out,
                                    int B, int H, int Nq, int D, void* stream);

/*
 * qat_channel_mean -- smooth_k's offset: mean[c] = mean of x[b, h, n, c] over b, h and n.
 *   ("attn_qat_train.py", _attention.forward: k.mean(dim=(0, 1, 2)).)
 *   x     bf16 [B, H, N, D] (device)
 *   mean  fp32 [D] (device) OUT.  Summed with fp32 atomics, so its last bits may vary
 *         from run to run.
 *   D 64 or 128; B, H, N >= 0 (an empty x gives mean = 0).
 * Errors: QAT_ERR_INVALID_ARG (null / misaligned pointer, bad size or D), QAT_ERR_CUDA.
 */
QAT_API qat_status_t qat_channel_mean(const void* x, float* mean, int B, int H, int N, int D,
                                      void* stream);

/*
 * qat_fake_quant_tokens -- fake-quantizes Q, K or V to FP8 E4M3 with one absmax scale
 * per (head, 32-token block) over all D channels, as the page's IS_QAT path does before
 * attention.  ("attn_qat_train.py", _attention.forward: fake_quantize_q with
 * BLOCK_M = 32, fake_quantize_kv with BLOCK_N = 32.)
 *   x       bf16 [B, H, N, D] (device)
 *   mean    fp32 [D] or NULL: subtracted from every token first (smooth_k for K)
 *   out     bf16 [B, H, N, D] OUT (may be x itself)
 *   scales  fp32 [B, H, ceil(N / 32)] OUT or NULL: amax / 448 per block
 *   Rule per block: x' = fl32(x - mean), amax = max |x'|,
 *   code = E4M3_RNE_SATFINITE(fl32(x' * fl32(448 / amax))),
 *   out = bf16(fl32(decode(code) * fl32(amax / 448))); an all-zero block stays zero.
 *   Tokens beyond N are excluded.
 * Errors: QAT_ERR_INVALID_ARG (null / misaligned x or out, bad size or D), QAT_ERR_CUDA.
 */
QAT_API qat_status_t qat_fake_quant_tokens(const void* x, const float* mean, void* out,
                                           float* scales, int B, int H, int N, int D,
                                           void* stream);

/*
 * qat_subtract_mean -- out = bf16_RN(fl32(x - mean_c)): smooth_k's subtraction without the
 * quantization.  The page's backward runs on the unquantized (but smoothed) keys when
 * use_qat_qkv_backward is False ("attn_qat_train.py", _attention.forward keeps
 * q_orig / k_orig / v_orig, taken after k = k - k_mean).
 *   x     bf16 [B, H, N, D] (device)
 *   mean  fp32 [D] (device, 16-byte aligned)
 *   out   bf16 [B, H, N, D] OUT (may be x itself)
 * Errors: QAT_ERR_INVALID_ARG (null / misaligned pointer, bad size or D), QAT_ERR_CUDA.
 */
QAT_API qat_status_t qat_subtract_mean(const void* x, const float* mean, void* out, int B, int H,
                                       int N, int D, void* stream);

/* Static, human-readable name of a status code (never NULL). */
QAT_API const char* qat_status_string(qat_status_t status);

/*
 * qat_attn_device_status -- synchronizes `stream`, then reads and clears the
 * library's device-side error word on the current device.  Kernels whose waits are
 * bounded set it when a wait expires (they then return early instead of hanging).
 * Returns QAT_OK, QAT_ERR_TIMEOUT, or QAT_ERR_CUDA if the synchronization failed.
 */
QAT_API qat_status_t qat_attn_device_status(void* stream);

/*
 * qat_debug_quant_tiles -- test entry: applies the kernels' own per-tile FP8 rule to
 * given fp32 data.  ("attn_qat_train.py", fake_quantize call in _attn_fwd_inner.)
 *   p       fp32 [rows, cols]  device, row-major; each row is split into tiles of 64
 *                              columns aligned at column 0 (the last may be shorter)
 *   deq     fp32 [rows, cols]  OUT: bf16-rounded quantized values, widened to fp32
 *   scales  fp32 [rows, ceil(cols/64)]  OUT: amax / 448 (0 for an all-zero tile)
 *   codes   u8   [rows, cols]  OUT: E4M3 code bytes
 * Inputs must be finite and >= 0 (probabilities).  rows, cols >= 0.
 * Errors: QAT_ERR_INVALID_ARG (null pointer with work to do, negative size).
 */
QAT_API qat_status_t qat_debug_quant_tiles(const float* p, int rows, int cols, float* deq,
                                   float* scales, unsigned char* codes, void* stream);

/*
 * qat_debug_wait_timeout -- test entry for the failure path of the kernels' bounded
 * waits: one thread waits, with the same bounded mbarrier wait the attention kernels use,
 * on a barrier nothing arrives on.  After limit_ms milliseconds the wait gives up, sets
 * the device error word and the kernel returns normally (no fault, trap or hang), so the
 * next qat_attn_device_status(stream) returns QAT_ERR_TIMEOUT and clears the word.  The
 * page has no counterpart; this entry exists for the tests.
 *   limit_ms  1 .. 4000
 * Errors: QAT_ERR_INVALID_ARG (limit out of range), QAT_ERR_CUDA (launch error).
 */
QAT_API qat_status_t qat_debug_wait_timeout(int limit_ms, void* stream);

/*
 * qat_debug_set_wait_limit_us -- test entry: sets the limit of the kernels' bounded waits
 * on the current device (default 4,000,000 us = 4 s; 0 makes every wait that is not
 * satisfied within its first few hundred polls expire).  With a lowered limit a real
 * forward or backward gives up at its first slow wait: it sets the device error word,
 * lets every copy and MMA it issued complete (those waits keep the 4 s limit), frees its
 * TMEM and returns, leaving its outputs partly written; nothing faults or hangs.  The
 * next qat_attn_device_status then reports QAT_ERR_TIMEOUT.  Synchronizes `stream` and
 * the device first.  The page has no counterpart; this entry exists for the tests of the
 * failure path.
 *   limit_us  0 .. 4000000
 * Errors: QAT_ERR_INVALID_ARG (limit out of range), QAT_ERR_CUDA.
 */
QAT_API qat_status_t qat_debug_set_wait_limit_us(int limit_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QAT_ATTN_H */
