// qat_internal.h -- declarations shared by the library's translation units (not ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#include "qat_attn.h"

namespace qat {

constexpr long long kMaxRows = 2147483647LL;  // rows of a [B*H*N, D] view
constexpr int kMaxBH = 65535;                   // grid y dimension

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Size and mode checks shared by the forward and backward entry points.  Sets *empty
// when there is no query work (B, H or Nq is zero).
inline qat_status_t check_sizes(int B, int H, int Nq, int Nkv, int D, float sm_scale, int causal,
                                int quant_mode, bool* empty) {
  *empty = false;
  if (B < 0 || H < 0 || Nq < 0 || Nkv < 0) return QAT_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return QAT_ERR_INVALID_ARG;
  if (!(sm_scale > 0.f) || !isfinite(sm_scale)) return QAT_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return QAT_ERR_INVALID_ARG;
  if (quant_mode != QAT_QUANT_NONE && quant_mode != QAT_QUANT_P_FP8E4M3_ROW_TILE64 &&
      quant_mode != QAT_QUANT_P_FP8E4M3_ROW_TILE64_PAGE_BWD)
    return QAT_ERR_INVALID_ARG;
  if (B == 0 || H == 0) {
    *empty = true;
    return QAT_OK;
  }
  if (Nkv < 1) return QAT_ERR_INVALID_ARG;
  const long long bh = static_cast<long long>(B) * H;
  if (bh * Nq > kMaxRows || bh * Nkv > kMaxRows) return QAT_ERR_INVALID_ARG;
  if (bh > kMaxBH) return QAT_ERR_UNSUPPORTED;
  if (causal && Nq != Nkv) return QAT_ERR_UNSUPPORTED;
  if (Nq == 0) *empty = true;
  return QAT_OK;
}

// Backward workspace, each piece 256-byte aligned; query rows are padded per head to a
// multiple of 128:
//   lse_pad, delta   fp32 [B, H, Nq_pad]
//   lse_ext, d_ext   bf16 [B, H, Nq_pad, 16]: -lse / qk_scale and -Delta of each row as
//                    the exact sum of three bf16 terms (elements 0-2, the rest zero)
//   ones             bf16 [128, 16]: 1 in elements 0-2 of every row
// The dK/dV kernel multiplies ones by lse_ext (d_ext) in one extra MMA k-step, so its
// score accumulators come out as S^T - lse / qk_scale and dP^T - Delta.
// With the non-causal dK/dV work cut into ranges (bwd_stream_k_ctas returns G > 0), the
// layout ends with the segments' partial sums, two slots per CTA:
//   part             fp32 [2G][2][128][D], [slot][0] = dV and [slot][1] = dK / sm_scale
struct BwdWorkspace {
  size_t nq_pad, off_lse, off_delta, off_lse_ext, off_d_ext, off_ones, off_part, total;
};

inline BwdWorkspace bwd_workspace_layout(int B, int H, int Nq, int Nkv, int D, int sk_ctas) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  BwdWorkspace w;
  w.nq_pad = (static_cast<size_t>(Nq) + 127) / 128 * 128;
  const size_t rows_pad = static_cast<size_t>(B) * H * w.nq_pad;
  w.off_lse = 0;
  w.off_delta = up(rows_pad * sizeof(float));
  w.off_lse_ext = w.off_delta + up(rows_pad * sizeof(float));
  w.off_d_ext = w.off_lse_ext + up(rows_pad * 32);
  w.off_ones = w.off_d_ext + up(rows_pad * 32);
  w.off_part = w.off_ones + up(128 * 32);
  const size_t part = sk_ctas > 0 ? static_cast<size_t>(sk_ctas) * 2 * 2 * 128 * D * sizeof(float) : 0;
  w.total = w.off_part + up(part);
  if (w.total == 0) w.total = 256;
  return w;
}

// Work split of the non-causal dK/dV kernel.  One CTA runs per SM, so with few (head,
// 128-key block) items the last wave runs ragged: B1 H40 Nkv512 has 160 items of 128
// query blocks each, and 8 CTAs ran two while the rest idled half the time.  Then the
// kernel runs stream-K: the items' (key block, query block) units, in head-major item
// order, are cut into G equal contiguous ranges, one per CTA.  A CTA walks its range
// item by item; an item cut by a range boundary is done in segments, each of which
// stores fp32 partial sums of dV and dK (the CTA's first segment in slot 2c, its last in
// 2c + 1), and one more kernel adds an item's segments in CTA order, so the result stays
// deterministic.  Each range has at least 4 units.  The choice compares estimated
// makespans for 152 SMs, from the sizes alone, so the workspace size is a function of
// the sizes too: ~2 blocks of fixed cost per item without the split, ~5 per segment with
// it (measured: B1 H24 N4608 ran 9% and B2 H8 Nq4096 Nkv1024 17% slower split, where ~2
// per segment had predicted a gain).  With many items the
// ragged wave costs little and the head-major item order, which keeps the CTAs running
// together on one head's Q and dO in L2, is kept: returns 0.
inline int bwd_stream_k_ctas(int B, int H, int Nq, int Nkv) {
  constexpr long long kSms = 152, kMinSeg = 4;
  const long long items = static_cast<long long>(B) * H * ((Nkv + 127) / 128);
  const long long M = (Nq + 127) / 128;
  if (items <= 0 || M < 2) return 0;
  const long long W = items * M;
  if (W > (1ll << 30)) return 0;  // the kernel's range arithmetic is 32-bit
  long long G = W / kMinSeg;
  if (G > kSms) G = kSms;
  if (G < 1) return 0;
  const double classic = static_cast<double>((items + kSms - 1) / kSms) * (M + 2);
  const double per_cta = static_cast<double>(W) / G;
  const double split = per_cta + 5.0 * (per_cta / M + 2.0);
  return split < 0.95 * classic ? static_cast<int>(G) : 0;
}

// [BH, N, D] bf16 viewed as a 3-D TMA tensor (D innermost), 64 x 128 x 1 boxes,
// 128-byte swizzle, zero fill out of bounds.
bool make_bf16_map_3d(CUtensorMap* m, const void* ptr, int D, int N, int BH,
                      int head_rows = -1);
// [BH, N, 16] bf16 as a 3-D TMA tensor with 16 x 128 x 1 boxes, 32-byte swizzle.
bool make_ext_map_3d(CUtensorMap* m, const void* ptr, int N, int BH);

// Arguments of one forward launch (device pointers, validated by the ABI layer).
struct FwdArgs {
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  uint16_t* o_q;
  uint16_t* o_hp;
  float* lse;
  int B, H, Nq, Nkv, D;
  float sm_scale;
  float qk_scale;  // sm_scale * log2(e)
  int causal;
  int quant;
  int kv_head_rows;  // rows between consecutive heads in K/V memory (Nkv unless a chunk)
  float* o_q_f32;    // when set (with o_hp_f32), fp32 outputs replace the bf16 ones
  float* o_hp_f32;
};

// Arguments of one backward launch.
struct BwdArgs {
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  const uint16_t* o_hp;
  const float* lse;
  const uint16_t* dO;
  uint16_t* dq;
  uint16_t* dk;
  uint16_t* dv;
  float* delta;     // fp32 [B, H, Nq_pad] in the workspace (0 in padding rows)
  float* lse_pad;   // fp32 [B, H, Nq_pad] copy of lse (+inf in padding rows)
  uint16_t* lse_ext;  // bf16 [B, H, Nq_pad, 16] (see BwdWorkspace)
  uint16_t* d_ext;    // bf16 [B, H, Nq_pad, 16]
  uint16_t* ones;     // bf16 [128, 16]
  float* part;        // dK/dV segment sums (BwdWorkspace::off_part) when sk_ctas > 0
  const float* k_mean;  // fp32 [D] or null: smooth_k's channel mean (dQ's SMOOTH_K term)
  int sk_ctas;        // 0, or the stream-K CTA bound of bwd_stream_k_ctas (non-causal)
  int B, H, Nq, Nkv, D;
  float sm_scale;
  float qk_scale;
  int causal;
  int page_bwd;     // 1: dV from quantized P and Delta from the O passed (O_q)
};

// Kernel launchers (return cudaGetLastError() after the launches).
cudaError_t launch_fwd_tc(const FwdArgs& a, unsigned int* err, int num_sms, cudaStream_t s);
// prep + dK/dV + dQ kernels
cudaError_t launch_bwd_tc(const BwdArgs& a, unsigned int* err, int num_sms, cudaStream_t s);
cudaError_t launch_bwd_dq(const BwdArgs& a, unsigned int* err, int num_sms, cudaStream_t s);
cudaError_t launch_channel_mean(const uint16_t* x, float* mean, long long rows, int D,
                                int num_sms, cudaStream_t s);
cudaError_t launch_fake_quant_tokens(const uint16_t* x, const float* mean, uint16_t* out,
                                     float* scales, int BH, int N, int D, cudaStream_t s);
cudaError_t launch_subtract_mean(const uint16_t* x, const float* mean, uint16_t* out,
                                 long long rows, int D, int num_sms, cudaStream_t s);
cudaError_t launch_merge(float* o_q_acc, float* o_hp_acc, float* lse_acc, const float* o_q_part,
                         const float* o_hp_part, const float* lse_part, uint16_t* o_q_out,
                         uint16_t* o_hp_out, long long rows, int D, int num_sms, cudaStream_t s);
cudaError_t launch_debug_quant(const float* p, int rows, int cols, float* deq,
                               float* scales, uint8_t* codes, cudaStream_t s);

// Causal work order.  A causal item (one head x one 128-row block) has between 1 and M
// blocks of work, so the persistent kernels take the longest items first.  Heads are
// taken in groups: inside a group the length classes descend and the group's heads
// alternate within a class, so the CTAs running together touch only a group or two of
// heads and the K/V (or Q/dO) blocks they all stream stay in L2.  With every head in
// one group the order is pure longest-first, which leaves a wave on as many heads as
// there are CTAs and has each CTA fetch its head's blocks from DRAM.
inline int causal_head_group(long long bytes_per_head, int BH) {
  constexpr long long kGroupBytes = 32ll << 20;  // a wave spans about two groups of L2
  long long g = kGroupBytes / (bytes_per_head > 0 ? bytes_per_head : 1);
  if (g < 1) g = 1;
  if (g > BH) g = BH;
  return static_cast<int>(g);
}

#ifdef __CUDACC__
// Item idx of that order -> head bh and length class cls (0 = the longest, M blocks).
__device__ __forceinline__ void causal_item(int idx, int BH, int M, int hgroup, int& bh,
                                            int& cls) {
  const int per = hgroup * M;
  const int gi = idx / per;
  const int h0 = gi * hgroup;
  const int hs = min(hgroup, BH - h0);
  const int j = idx - gi * per;
  cls = j / hs;
  bh = h0 + (j - cls * hs);
}
#endif

// Device-side error word (bounded waits set it); defined in qat_api.cu.
cudaError_t read_and_clear_device_error(unsigned int* out, cudaStream_t s);
// Device address of that word (the first member of the library's device state, looked
// up on every call, so a context created after cudaDeviceReset gets its own) and the SM
// count of the current device (cached).
cudaError_t device_context(unsigned int** err, int* num_sms);

}  // namespace qat
