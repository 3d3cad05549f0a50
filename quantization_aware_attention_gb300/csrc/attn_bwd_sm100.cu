// attn_bwd_sm100.cu -- QAT attention backward (straight-through estimator) on the
// Blackwell tensor core (tcgen05 + TMEM + TMA): the preprocessing kernel and dK, dV.
// dQ comes from its own kernel (attn_bwd_dq_sm100.cu), as in the page's split into a
// dK/dV program and a dQ program.
//
// Gradients of L = <dO, O_hp> ("attn_qat_train.py", _attn_bwd_preprocess,
// _attn_bwd_dkdv; P rematerialized from the saved base-2 lse as "support for pytorch
// autograd" suggests):
//   Delta_i = sum_d dO_id O_hp,id
//   P^T = exp2(S^T qk_scale - lse)     S^T = K Q^T
//   dP^T = V dO^T,   dS^T = P^T o (dP^T - Delta)
//   dV += P^T dO,    dK += dS^T Q     (dK scaled by sm_scale at the end)
//
// Kernels, in launch order on the caller's stream:
//   bwd_prep_kernel       Delta and a copy of lse padded to 128-row blocks (+inf in the
//                         padding, so P = 0 there).
//   attn_bwd_dkdv_kernel  one CTA per SM, persistent over (head, 128-key block) items;
//                         with few such items (non-causal), over equal ranges of the
//                         items' query blocks, whose cut items store fp32 partial sums
//                         (stream-K, bwd_stream_k_ctas).
//   bwd_segment_sum_kernel  only then: adds a cut item's segments in order -> bf16.
//   attn_bwd_dq_kernel    one CTA per SM, persistent over (head, 128-row query block).
//
// attn_bwd_dkdv_kernel, 352 threads:
//   warp 0      TMA producer: the ones tile once; K, V once per item; per 128-row query
//               block Q with its lse_ext rows and dO with its d_ext rows (2 stages each).
//   warps 1, 2  MMA issuers (lane 0 of each); warp 1 also owns TMEM:
//                 warp 1:  dV  += P^T_b dO    TS  (A = P^T bf16 in TMEM [0,32) + [64,96),
//                                                  B = dO MN-major), then
//                          S^T_{b+1} = K Q^T  SS  -> TMEM [0,128)   (A = K, B = Q, K-major)
//                 warp 2:  dK  += dS^T_b Q    TS  (A = dS^T bf16 in TMEM [128,160) +
//                                                  [192,224), B = Q MN-major), then
//                          dP^T_{b+1} = V dO^T SS -> TMEM [128,256)
//               Each score product takes one more k-step: a constant ones tile times the
//               query block's lse_ext (d_ext) rows, so TMEM receives S^T - lse / qk_scale
//               and dP^T - Delta and the compute warps read no per-query values at all.
//               Each stream only overwrites TMEM its own earlier MMAs read (S^T over P^T,
//               dP^T over dS^T); operands both read (Q, dO, K/V) are released by one
//               commit from each.  Each issuer waits for the next block's Q (dO) tile
//               before the compute warps' barrier, so the next score product follows
//               without a wait.  What bounds the kernel is the loop this in-place reuse
//               makes: P^T_b written -> dV_b -> S^T_{b+1} -> its completion -> the next
//               P phase (TMEM has no room for a second S^T buffer).
//   warps 3-10  two compute warpgroups, each owning 64 of a block's 128 query columns:
//               P phase (P^T = exp2(qk_scale (S^T - lse / qk_scale)), bf16 over the
//               group's S^T columns), dS phase (dS^T = P^T o (dP^T - Delta), bf16 over the
//               group's dP^T columns), and per item one of dV / dK -> bf16 global
//               (fp32 partial sums in the workspace for a segment of a cut item).
// TMEM (512 columns): S^T [0,128), dP^T [128,256), dV [256,256+D), dK [256+D,256+2D).
// Shared memory: K, V (one tile each), Q and dO (2 stages each, 128-byte swizzle), the
// ones tile and the lse_ext / d_ext rows (128 x 16 bf16, 32-byte swizzle).
#include "qat_internal.h"
#include "qat_quant.cuh"
#include "sm100.cuh"

#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

namespace qat {
namespace {

using namespace sm100;

constexpr int kBlk = 128;       // keys per item, queries per block
constexpr int kThreads = 352;
constexpr int kPrefetch = 3;    // query blocks between an L2 prefetch and the block's load
constexpr int kMaxSkCtas = 160; // stream-K CTAs at most (bwd_stream_k_ctas caps them at 152)

template <int D>
struct BwdTc {
  static constexpr int kChunks = D / 64;
  static constexpr uint32_t kChunkBytes = kBlk * 128;      // 16 KB box: 128 rows x 128 B
  static constexpr uint32_t kTileBytes = kChunks * kChunkBytes;
  static constexpr uint32_t kOffK = 0;
  static constexpr uint32_t kOffV = kOffK + kTileBytes;
  static constexpr uint32_t kOffQ = kOffV + kTileBytes;     // 2 stages
  static constexpr uint32_t kOffDO = kOffQ + 2 * kTileBytes;  // 2 stages
  static constexpr uint32_t kExtBytes = kBlk * 32;            // 128 rows x 16 bf16 (SW32)
  static constexpr uint32_t kOffOnes = kOffDO + 2 * kTileBytes;  // ones tile
  static constexpr uint32_t kOffQX = kOffOnes + kExtBytes;    // lse_ext, 2 stages with Q
  static constexpr uint32_t kOffDX = kOffQX + 2 * kExtBytes;  // d_ext, 2 stages with dO
  static constexpr uint32_t kOffPx = kOffDX + 2 * kExtBytes;  // quant_mode 2: tile maxima, scales
  static constexpr uint32_t kOffBar = kOffPx + 8192;
  static constexpr uint32_t kOffMisc = kOffBar + 256;
  static constexpr uint32_t kUsed = kOffMisc + 64;
  static constexpr uint32_t kSmemBytes = (kUsed + 1024 > 118784u ? kUsed + 1024 : 118784u);
  static constexpr uint32_t kTmemS = 0, kTmemDP = 128, kTmemDV = 256, kTmemDK = 256 + D;
};

enum : uint32_t {
  B_ONES_FULL = 0, B_KV_FULL, B_KV_EMPTY, B_Q_FULL0, B_Q_FULL1, B_Q_EMPTY0, B_Q_EMPTY1,
  B_DO_FULL0, B_DO_FULL1, B_DO_EMPTY0, B_DO_EMPTY1, B_S_FULL, B_DP_FULL, B_P_FULL, B_DS_FULL,
  B_DKDV_FULL, B_DKDV_EMPTY, B_DRAIN, B_DRAIN_B, B_PX0, B_PX1, B_PX2, B_PX3, B_COUNT
};

struct BwdTcParams {
  BwdArgs a;
  unsigned int* err;
  int mtiles;   // query blocks per head
  int ktiles;   // key blocks per head
  int items;    // B * H * ktiles
  int nq_pad;   // mtiles * 128
  int hgroup;   // heads per group of the causal order (causal_head_group)
  int streamk;  // 1: CTA c walks units [work c / G, work (c + 1) / G), G = gridDim.x
  int work;     // items * mtiles (key block, query block) units (stream-K only)
};

// One dK/dV item (or segment of one): key block kb of head bh over `count` query blocks
// starting at q0.  Whole non-causal items walk their range from a rotated start (rot),
// so that the CTAs of one head do not all read the same query block at once.  slot: -1
// stores bf16 dV and dK; else the segment's fp32 partial sums go to that workspace slot.
struct BwdItem {
  int bh, kb, q0, count, rot, slot;
};

// First unit of CTA c's stream-K range.
__device__ __forceinline__ int sk_start(int work, int c, int G) {
  return static_cast<int>(static_cast<long long>(work) * c / G);
}

// The CTA's items: idx runs from bwd_first to bwd_end in steps of bwd_step.  kSK false,
// one CTA per item: idx is the item, stepping by gridDim.x.  kSK true (stream-K): idx is
// the first unit of a segment of the CTA's range, which ends at the next item boundary
// or the range end.  (The two are separate kernel instances: with the range arithmetic
// in it, the one-CTA-per-item loop kept its item values out of the uniform registers
// and ran 5% slower.)
template <bool kSK>
__device__ __forceinline__ int bwd_first(const BwdTcParams& p) {
  if constexpr (kSK) return sk_start(p.work, blockIdx.x, gridDim.x);
  else return static_cast<int>(blockIdx.x);
}

template <bool kSK>
__device__ __forceinline__ int bwd_end(const BwdTcParams& p) {
  if constexpr (kSK) return sk_start(p.work, blockIdx.x + 1, gridDim.x);
  else return p.items;
}

template <bool kSK>
__device__ __forceinline__ BwdItem bwd_item(int idx, const BwdTcParams& p) {
  BwdItem t;
  t.slot = -1;
  if constexpr (!kSK) {
    if (p.a.causal) {  // longest first (small key blocks see the most queries), heads in groups
      causal_item(idx, p.a.B * p.a.H, p.ktiles, p.hgroup, t.bh, t.kb);
      t.q0 = t.kb;
      t.count = p.mtiles - t.kb;
      t.rot = 0;
    } else {           // head-major: the CTAs running together share one head's Q/dO in L2
      t.bh = idx / p.ktiles;
      t.kb = idx - t.bh * p.ktiles;
      t.q0 = 0;
      t.count = p.mtiles;
      t.rot = t.kb % t.count;
    }
  } else {
    const int M = p.mtiles;
    const int item = idx / M;
    t.bh = item / p.ktiles;
    t.kb = item - t.bh * p.ktiles;
    t.q0 = idx - item * M;
    t.count = min((item + 1) * M, bwd_end<true>(p)) - idx;
    t.rot = 0;
    if (t.q0 != 0 || t.count != M)
      t.slot = 2 * static_cast<int>(blockIdx.x) + (idx == bwd_first<true>(p) ? 0 : 1);
  }
  return t;
}

template <bool kSK>
__device__ __forceinline__ int bwd_step(int idx, const BwdItem& t) {
  if constexpr (kSK) return idx + t.count;
  else return idx + static_cast<int>(gridDim.x);
}

// query block of the item's ii-th step.  Stream-K segments are walked from their last
// query block down: a CTA's first segment usually runs to its item's end, so the CTAs
// that start the key blocks of one head part-way through its query blocks (their ranges
// begin 134.7 units apart at B1 H40 Nq16384 Nkv512) then read the same blocks together
// and share them in L2.
template <bool kSK>
__device__ __forceinline__ int block_at(const BwdItem& t, int ii) {
  if constexpr (kSK) {
    return t.q0 + t.count - 1 - ii;
  } else {
    int b = t.rot + ii;
    if (b >= t.count) b -= t.count;
    return t.q0 + b;
  }
}

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Bounds of 384 threads cap registers at 168 per thread: with 11 warps, three share a
// sub-partition's 16K registers, so a 352-thread CTA cannot launch with more.
template <int D, bool kSK>
__global__ void __launch_bounds__(384, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmDO,
                         const __grid_constant__ CUtensorMap tmQX,
                         const __grid_constant__ CUtensorMap tmDX,
                         const __grid_constant__ CUtensorMap tmOnes, const BwdTcParams p) {
  using C = BwdTc<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kOffMisc);
  volatile WaitCtl* abort_flag = reinterpret_cast<volatile WaitCtl*>(gbase + C::kOffMisc + 8);
  const uint32_t bars = base + C::kOffBar;
  auto bar = [&](uint32_t i) { return bars + 8u * i; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    wait_ctl_init(abort_flag, p.err);
    for (uint32_t i = 0; i < B_COUNT; ++i) {
      // released by one commit from each MMA issuer
      const bool both = i == B_KV_EMPTY || i == B_Q_EMPTY0 || i == B_Q_EMPTY1 ||
                        i == B_DO_EMPTY0 || i == B_DO_EMPTY1 || i == B_DKDV_FULL;
      const uint32_t cnt = (i == B_P_FULL || i == B_DS_FULL || i == B_DKDV_EMPTY)
                               ? 256u : (i >= B_PX0 ? 64u : (both ? 2u : 1u));
      mbar_init(bar(i), cnt);
    }
    fence_barrier_init();
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    prefetch_tmap(&tmDO);
    prefetch_tmap(&tmQX);
    prefetch_tmap(&tmDX);
    prefetch_tmap(&tmOnes);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t qc = 0, dc = 0;  // Q loads, dO loads issued
      int it = 0;
      bool ok = true;
      // the ones tile, once per CTA
      mbar_arrive_expect_tx(bar(B_ONES_FULL), C::kExtBytes);
      tma_load_3d(base + C::kOffOnes, &tmOnes, bar(B_ONES_FULL), 0, 0, 0);
      // Q_blk with its lse_ext rows
      auto load_q = [&](int bh, int blk) -> bool {
        const uint32_t st = qc & 1, use = qc >> 1;
        if (!mbar_wait(bar(B_Q_EMPTY0 + st), (use & 1) ^ 1, abort_flag, p.err)) return false;
        const uint32_t fb = bar(B_Q_FULL0 + st);
        mbar_arrive_expect_tx(fb, C::kTileBytes + C::kExtBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(base + C::kOffQ + st * C::kTileBytes + c * C::kChunkBytes, &tmQ, fb, 64 * c,
                      blk * kBlk, bh);
        tma_load_3d(base + C::kOffQX + st * C::kExtBytes, &tmQX, fb, 0, blk * kBlk, bh);
        ++qc;
        return true;
      };
      for (int idx = bwd_first<kSK>(p), end = bwd_end<kSK>(p), nx; idx < end && ok; idx = nx, ++it) {
        const BwdItem t = bwd_item<kSK>(idx, p);
        nx = bwd_step<kSK>(idx, t);
        const int bh = t.bh, kb = t.kb, count = t.count;
        ok = mbar_wait(bar(B_KV_EMPTY), (it & 1) ^ 1, abort_flag, p.err);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(B_KV_FULL), 2 * C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_3d(base + C::kOffK + c * C::kChunkBytes, &tmK, bar(B_KV_FULL), 64 * c,
                      kb * kBlk, bh);
          tma_load_3d(base + C::kOffV + c * C::kChunkBytes, &tmV, bar(B_KV_FULL), 64 * c,
                      kb * kBlk, bh);
        }
        ok = load_q(bh, block_at<kSK>(t, 0));
        for (int ii = 0; ii < count && ok; ++ii) {
          const int blk = block_at<kSK>(t, ii);
          const uint32_t dst = dc & 1, duse = dc >> 1;
          ok = mbar_wait(bar(B_DO_EMPTY0 + dst), (duse & 1) ^ 1, abort_flag, p.err);
          if (!ok) break;
          const uint32_t fb = bar(B_DO_FULL0 + dst);
          mbar_arrive_expect_tx(fb, C::kTileBytes + C::kExtBytes);
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(base + C::kOffDO + dst * C::kTileBytes + c * C::kChunkBytes, &tmDO, fb,
                        64 * c, blk * kBlk, bh);
          tma_load_3d(base + C::kOffDX + dst * C::kExtBytes, &tmDX, fb, 0, blk * kBlk, bh);
          ++dc;
          // Q and dO of the block kPrefetch ahead into L2: when the CTAs running together
          // stream different heads (stream-K ranges), a block's first read comes from
          // DRAM, which the two-stage rings alone do not cover.  (With one CTA per item
          // the CTAs share one head and the prefetches only add L2 traffic: 5% slower.)
          if (kSK && ii + kPrefetch < count) {
            const int pb = block_at<kSK>(t, ii + kPrefetch) * kBlk;
            for (int c = 0; c < C::kChunks; ++c) {
              tma_prefetch_l2_3d(&tmQ, 64 * c, pb, bh);
              tma_prefetch_l2_3d(&tmDO, 64 * c, pb, bh);
            }
            tma_prefetch_l2_3d(&tmQX, 0, pb, bh);
            tma_prefetch_l2_3d(&tmDX, 0, pb, bh);
          }
          if (ii + 1 < count) ok = load_q(bh, block_at<kSK>(t, ii + 1));
        }
      }
      // drain: every issued load lands before the CTA exits
      if (it > 0) mbar_wait_drain(bar(B_KV_FULL), (it - 1) & 1, p.err);
      for (uint32_t i = (qc > 2 ? qc - 2 : 0); i < qc; ++i)
        mbar_wait_drain(bar(B_Q_FULL0 + (i & 1)), (i >> 1) & 1, p.err);
      for (uint32_t i = (dc > 2 ? dc - 2 : 0); i < dc; ++i)
        mbar_wait_drain(bar(B_DO_FULL0 + (i & 1)), (i >> 1) & 1, p.err);
      mbar_wait_drain(bar(B_ONES_FULL), 0, p.err);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer A: S^T, dV
    if (lane == 0) {
      constexpr uint32_t idSS = idesc_bf16_f32(kBlk, kBlk, false, false);  // S^T
      constexpr uint32_t idKM = idesc_bf16_f32(kBlk, D, true, false);      // dV
      const uint32_t sK = base + C::kOffK;
      uint32_t qc = 0;  // query blocks processed (global)
      int it = 0;
      bool ok = true, issued = false;
      auto w = [&](uint32_t b_, uint32_t par) { return mbar_wait(b_, par, abort_flag, p.err); };
      auto wait_q = [&](uint32_t c) { return w(bar(B_Q_FULL0 + (c & 1)), (c >> 1) & 1); };
      auto issue_s = [&](uint32_t c) {  // S^T_c = K Q_c^T (Q_c has landed)
        const uint32_t st = c & 1;
        tc_fence_after();
        const uint32_t sQ = base + C::kOffQ + st * C::kTileBytes;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * C::kChunkBytes + (ks & 3) * 32;
          mma_ss(tbase + C::kTmemS, smem_desc_sw128(sK + off, 16, 1024),
                 smem_desc_sw128(sQ + off, 16, 1024), idSS, ks > 0 ? 1u : 0u);
        }
        // one more k-step: ones x lse_ext adds -lse / qk_scale to every key row
        mma_ss(tbase + C::kTmemS, smem_desc_sw32(base + C::kOffOnes),
               smem_desc_sw32(base + C::kOffQX + st * C::kExtBytes), idSS, 1u);
        mma_commit(bar(B_S_FULL));
        issued = true;
      };
      ok = w(bar(B_ONES_FULL), 0);
      for (int idx = bwd_first<kSK>(p), end = bwd_end<kSK>(p), nx; idx < end && ok; idx = nx, ++it) {
        const BwdItem t = bwd_item<kSK>(idx, p);
        nx = bwd_step<kSK>(idx, t);
        const int count = t.count;
        ok = w(bar(B_KV_FULL), it & 1) && wait_q(qc);
        if (ok) issue_s(qc);
        for (int ii = 0; ii < count && ok; ++ii, ++qc) {
          const uint32_t dst = qc & 1;
          // the next block's Q is waited for first (it has almost always landed), so that
          // S^T_{c+1} follows dV_c without a wait in between
          if (ii + 1 < count && !(ok = wait_q(qc + 1))) break;
          // dV += P^T dO (TS: P^T halves at TMEM columns [0,32) and [64,96)), once the
          // compute warps have written P^T of this block over its S^T
          if (!(ok = w(bar(B_P_FULL), qc & 1) && w(bar(B_DO_FULL0 + dst), (qc >> 1) & 1))) break;
          if (ii == 0 && !(ok = w(bar(B_DKDV_EMPTY), (it & 1) ^ 1))) break;
          tc_fence_after();
          const uint32_t sDO = base + C::kOffDO + dst * C::kTileBytes;
#pragma unroll
          for (int ks = 0; ks < kBlk / 16; ++ks)
            mma_ts(tbase + C::kTmemDV, tbase + C::kTmemS + (ks < 4 ? 8 * ks : 32 + 8 * ks),
                   smem_desc_sw128(sDO + ks * 2048, C::kChunkBytes, 1024), idKM,
                   (ii > 0 || ks > 0) ? 1u : 0u);
          mma_commit(bar(B_DO_EMPTY0 + dst));     // dO_c: read by dP^T_c (B) and dV_c
          mma_commit(bar(B_Q_EMPTY0 + (qc & 1)));  // Q_c: read by S^T_c and dK_c (B)
          // S^T_{c+1} overwrites P^T_c after dV_c, in this stream's order.  (Issuing it
          // before the two commits above delays the producer's refill of the two-stage
          // Q / dO rings and measured 10% slower.)
          if (ii + 1 < count) issue_s(qc + 1);
        }
        if (!ok) break;
        mma_commit(bar(B_KV_EMPTY));
        mma_commit(bar(B_DKDV_FULL));
      }
      if (issued) {
        mma_commit(bar(B_DRAIN));
        mbar_wait_drain(bar(B_DRAIN), 0, p.err);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ MMA issuer B: dK, dP^T
    if (lane == 0) {
      constexpr uint32_t idSS = idesc_bf16_f32(kBlk, kBlk, false, false);  // dP^T
      constexpr uint32_t idKM = idesc_bf16_f32(kBlk, D, true, false);      // dK
      const uint32_t sV = base + C::kOffV;
      uint32_t qc = 0;
      int it = 0;
      bool ok = true, issued = false;
      auto w = [&](uint32_t b_, uint32_t par) { return mbar_wait(b_, par, abort_flag, p.err); };
      auto wait_do = [&](uint32_t c) { return w(bar(B_DO_FULL0 + (c & 1)), (c >> 1) & 1); };
      // dP^T_c = V dO_c^T (dO_c has landed); it overwrites dS^T_{c-1}, which dK_{c-1}
      // (issued before) reads
      auto issue_dp = [&](uint32_t c) {
        tc_fence_after();
        const uint32_t sDO = base + C::kOffDO + (c & 1) * C::kTileBytes;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * C::kChunkBytes + (ks & 3) * 32;
          mma_ss(tbase + C::kTmemDP, smem_desc_sw128(sV + off, 16, 1024),
                 smem_desc_sw128(sDO + off, 16, 1024), idSS, ks > 0 ? 1u : 0u);
        }
        // one more k-step: ones x d_ext subtracts Delta from every key row
        mma_ss(tbase + C::kTmemDP, smem_desc_sw32(base + C::kOffOnes),
               smem_desc_sw32(base + C::kOffDX + (c & 1) * C::kExtBytes), idSS, 1u);
        mma_commit(bar(B_DP_FULL));
        mma_commit(bar(B_DO_EMPTY0 + (c & 1)));
        issued = true;
      };
      ok = w(bar(B_ONES_FULL), 0);
      for (int idx = bwd_first<kSK>(p), end = bwd_end<kSK>(p), nx; idx < end && ok; idx = nx, ++it) {
        const BwdItem t = bwd_item<kSK>(idx, p);
        nx = bwd_step<kSK>(idx, t);
        const int count = t.count;
        ok = w(bar(B_KV_FULL), it & 1) && wait_do(qc);
        if (ok) issue_dp(qc);
        for (int ii = 0; ii < count && ok; ++ii, ++qc) {
          const uint32_t st = qc & 1;
          if (ii + 1 < count && !(ok = wait_do(qc + 1))) break;  // the next dO, first
          // dK += dS^T Q  (dS^T halves at columns [128,160) and [192,224))
          if (!(ok = w(bar(B_DS_FULL), qc & 1) && w(bar(B_Q_FULL0 + st), (qc >> 1) & 1))) break;
          if (ii == 0 && !(ok = w(bar(B_DKDV_EMPTY), (it & 1) ^ 1))) break;
          tc_fence_after();
          const uint32_t sQ = base + C::kOffQ + st * C::kTileBytes;
#pragma unroll
          for (int ks = 0; ks < kBlk / 16; ++ks)
            mma_ts(tbase + C::kTmemDK, tbase + C::kTmemDP + (ks < 4 ? 8 * ks : 32 + 8 * ks),
                   smem_desc_sw128(sQ + ks * 2048, C::kChunkBytes, 1024), idKM,
                   (ii > 0 || ks > 0) ? 1u : 0u);
          mma_commit(bar(B_Q_EMPTY0 + st));
          if (ii + 1 < count) issue_dp(qc + 1);
        }
        if (!ok) break;
        mma_commit(bar(B_KV_EMPTY));
        mma_commit(bar(B_DKDV_FULL));
      }
      if (issued) {
        mma_commit(bar(B_DRAIN_B));
        mbar_wait_drain(bar(B_DRAIN_B), 0, p.err);
      }
    }
  } else {
    // ------------------------------------------------------------ compute warpgroups
    // Two warpgroups, h = 0 (warps 3-6) and h = 1 (warps 7-10); each thread owns one key
    // row (TMEM lane) and query columns [64h, 64h + 64) of every block:
    //   P phase   P^T = exp2(S^T qk_scale - lse) -> bf16 into TMEM columns [64h, 64h+32)
    //   dS phase  dS^T = P^T o (dP^T - Delta) -> bf16 into TMEM columns [128+64h, +32)
    //   epilogue  h = 0 stores dV, h = 1 stores dK (x sm_scale) for the item's key rows.
    const int h = (warp - 3) >> 2;
    const int quarter = warp & 3;
    const int r = 32 * quarter + lane;               // key row (TMEM lane)
    const uint32_t lrow = (32u * quarter) << 16;
    const float qk = p.a.qk_scale;
    auto wwait = [&](uint32_t b_, uint32_t par) {
      const bool okw = mbar_wait(b_, par, abort_flag, p.err);
      return __all_sync(0xffffffffu, okw) != 0;
    };
    uint32_t Pp[32];                                  // P^T of the current block, bf16 pairs
    // this thread's row of P^T (64 queries, bf16 pairs) over its S^T columns [64h, 64h+32):
    // the A operand of the dV MMA
    auto store_pt = [&](const uint32_t (&v)[32]) -> bool {
      tmem_st16(tbase + lrow + C::kTmemS + 64 * h, *reinterpret_cast<const uint32_t(*)[16]>(&v[0]));
      tmem_st16(tbase + lrow + C::kTmemS + 64 * h + 16,
                *reinterpret_cast<const uint32_t(*)[16]>(&v[16]));
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_P_FULL));
      return true;
    };
    // P phase of block `blk` (global index c): P^T -> TMEM for the dV MMA
    auto p_phase = [&](uint32_t c, int blk, int kb, bool key_ok, int key) -> bool {
      if (!wwait(bar(B_S_FULL), c & 1)) return false;
      tc_fence_after();
      const bool diag = p.a.causal && blk == kb;
      const int qh = blk * kBlk + 64 * h;             // first query of this thread's columns
      {
        uint32_t sr[64];
        tmem_ld32(tbase + lrow + C::kTmemS + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        tmem_ld32(tbase + lrow + C::kTmemS + 64 * h + 32,
                  *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 64; i += 2) {           // TMEM holds S^T - lse / qk_scale
          const float2 x = mul_rn_f32x2(make_float2(__uint_as_float(sr[i]), __uint_as_float(sr[i + 1])),
                                        make_float2(qk, qk));
          Pp[i / 2] = pack_bf16x2(ex2f(x.x), ex2f(x.y));
        }
        // keys past Nkv (whole rows) and queries before the key on the causal diagonal
        // get P = 0; a separate pass, taken only by the few rows and blocks that need it
        if (__any_sync(0xffffffffu, !key_ok) || diag) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const bool m0 = !key_ok || (diag && qh + 2 * i < key);
            const bool m1 = !key_ok || (diag && qh + 2 * i + 1 < key);
            Pp[i] &= (m0 ? 0xffff0000u : 0xffffffffu) & (m1 ? 0x0000ffffu : 0xffffffffu);
          }
        }
      }
      return store_pt(Pp);
    };
    // quant_mode 2 (the page's backward, "attn_qat_train.py" _attn_bwd_dkdv): the dV MMA
    // consumes P^T quantized per (query, 64-key tile) with the forward's rule.  The 64
    // keys of a tile are the lanes of a warp pair (quarters 0-1 or 2-3 of this group):
    // column maxima by redux within each warp, exchanged through shared memory.
    float* px = reinterpret_cast<float*>(gbase + C::kOffPx);          // [4][2 parity][2][64]
    float* psc = reinterpret_cast<float*>(gbase + C::kOffPx + 4096);  // [8 warps][128]
    const int pair = 2 * h + (quarter >> 1);
    const int wip = quarter & 1;
    auto p_phase_page = [&](uint32_t c, int blk, int kb, bool key_ok, int key) -> bool {
      if (!wwait(bar(B_S_FULL), c & 1)) return false;
      tc_fence_after();
      const bool diag = p.a.causal && blk == kb;
      const int qh = blk * kBlk + 64 * h;
      uint32_t pf[64];                                 // P^T of this row, fp32 bits
      tmem_ld32(tbase + lrow + C::kTmemS + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&pf[0]));
      tmem_ld32(tbase + lrow + C::kTmemS + 64 * h + 32, *reinterpret_cast<uint32_t(*)[32]>(&pf[32]));
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 64; i += 2) {             // TMEM holds S^T - lse / qk_scale
        const float2 x = mul_rn_f32x2(make_float2(__uint_as_float(pf[i]), __uint_as_float(pf[i + 1])),
                                      make_float2(qk, qk));
        pf[i] = __float_as_uint(ex2f(x.x));
        pf[i + 1] = __float_as_uint(ex2f(x.y));
      }
      if (__any_sync(0xffffffffu, !key_ok) || diag) {
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if (!key_ok || (diag && qh + i < key)) pf[i] = 0u;
      }
#pragma unroll
      for (int i = 0; i < 64; i += 2)
        Pp[i / 2] = pack_bf16x2(__uint_as_float(pf[i]), __uint_as_float(pf[i + 1]));
      // column maxima over this warp's 32 keys (non-negative floats order as their bits)
      uint32_t mine0 = 0u, mine1 = 0u;
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        const uint32_t mx = __reduce_max_sync(0xffffffffu, pf[i]);
        if ((i & 31) == lane) {
          if (i < 32) mine0 = mx; else mine1 = mx;
        }
      }
      float* slot = px + ((pair * 2 + (c & 1)) * 2) * 64;
      slot[wip * 64 + lane] = __uint_as_float(mine0);
      slot[wip * 64 + 32 + lane] = __uint_as_float(mine1);
      mbar_arrive(bar(B_PX0 + pair));
      if (!wwait(bar(B_PX0 + pair), c & 1)) return false;
      const float a0 = fmaxf(__uint_as_float(mine0), slot[(wip ^ 1) * 64 + lane]);
      const float a1 = fmaxf(__uint_as_float(mine1), slot[(wip ^ 1) * 64 + 32 + lane]);
      const TileScale t0 = tile_scale(a0), t1 = tile_scale(a1);
      float* ws = psc + (warp - 3) * 128;              // inv [0,64), scale [64,128)
      ws[lane] = t0.inv;
      ws[32 + lane] = t1.inv;
      ws[64 + lane] = t0.scale;
      ws[96 + lane] = t1.scale;
      __syncwarp();
      uint32_t pq[32];
#pragma unroll
      for (int i = 0; i < 64; i += 2) {
        const float2 inv = *reinterpret_cast<const float2*>(ws + i);
        const float2 scl = *reinterpret_cast<const float2*>(ws + 64 + i);
        const float2 x = mul_rn_f32x2(make_float2(__uint_as_float(pf[i]), __uint_as_float(pf[i + 1])), inv);
        const float2 d = mul_rn_f32x2(e4m3x2_decode(e4m3x2_rn_satfinite(x.x, x.y)), scl);
        pq[i / 2] = pack_bf16x2(d.x, d.y);
      }
      __syncwarp();                                    // ws is rewritten next block
      return store_pt(pq);
    };
    // dS phase of block c: dS^T = P^T o (dP^T - Delta) -> bf16 over this group's dP^T
    // columns (each 32-column load is consumed before the 16 packed columns it becomes
    // are written; dP^T_{c+1} overwrites them only after dK_c has read them)
    auto ds_phase = [&](uint32_t c) -> bool {
      if (!wwait(bar(B_DP_FULL), c & 1)) return false;
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t dr[32];
        tmem_ld32(tbase + lrow + C::kTmemDP + 64 * h + 32 * cc, dr);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {           // TMEM holds dP^T - Delta
          const uint32_t pa = Pp[16 * cc + i / 2];
          const float2 d = mul_rn_f32x2(
              make_float2(__uint_as_float(pa << 16), __uint_as_float(pa & 0xffff0000u)),
              make_float2(__uint_as_float(dr[i]), __uint_as_float(dr[i + 1])));
          pk[i / 2] = pack_bf16x2(d.x, d.y);
        }
        tmem_st16(tbase + lrow + C::kTmemDP + 64 * h + 16 * cc, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_DS_FULL));
      return true;
    };
    uint32_t qc = 0;
    int it = 0;
    bool ok = true;
    for (int idx = bwd_first<kSK>(p), end = bwd_end<kSK>(p), nx; idx < end && ok; idx = nx, ++it) {
      const BwdItem t = bwd_item<kSK>(idx, p);
      nx = bwd_step<kSK>(idx, t);
      const int bh = t.bh, kb = t.kb, count = t.count;
      const int key = kb * kBlk + r;
      const bool key_ok = key < p.a.Nkv;
      // order per block b: dS_b, then P_{b+1}, which is ready before dV_{b+1} is issued
      auto pp = [&](uint32_t c_, int blk_) {
        return p.a.page_bwd ? p_phase_page(c_, blk_, kb, key_ok, key)
                            : p_phase(c_, blk_, kb, key_ok, key);
      };
      ok = pp(qc, block_at<kSK>(t, 0));
      for (int ii = 0; ii < count && ok; ++ii, ++qc) {
        ok = ds_phase(qc);
        if (ok && ii + 1 < count) ok = pp(qc + 1, block_at<kSK>(t, ii + 1));
      }
      if (!ok) break;
      // ---- epilogue: h = 0 stores dV, h = 1 stores dK for this item's key rows
      ok = wwait(bar(B_DKDV_FULL), it & 1);
      if (!ok) break;
      tc_fence_after();
      const size_t grow = (static_cast<size_t>(bh) * p.a.Nkv + (key_ok ? key : 0)) * D;
      const uint32_t tcol = h ? C::kTmemDK : C::kTmemDV;
      uint16_t* out = h ? p.a.dk : p.a.dv;
      const float scale = h ? p.a.sm_scale : 1.0f;
      // a segment of a cut item stores its fp32 partial sums (dK unscaled) in its slot;
      // bwd_segment_sum_kernel adds an item's segments in order and converts
      float* part = kSK && t.slot >= 0
                        ? p.a.part + ((static_cast<size_t>(t.slot) * 2 + h) * kBlk + r) * D
                        : nullptr;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(tbase + lrow + tcol + 32 * c, ov);
        tmem_wait_ld();
        if (part != nullptr) {
          if (key_ok) {
            uint4* dst = reinterpret_cast<uint4*>(part + 32 * c);
#pragma unroll
            for (int v = 0; v < 8; ++v) dst[v] = make_uint4(ov[4 * v], ov[4 * v + 1], ov[4 * v + 2], ov[4 * v + 3]);
          }
          continue;
        }
        uint32_t wv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          wv[i] = pack_bf16x2(__uint_as_float(ov[2 * i]) * scale,
                              __uint_as_float(ov[2 * i + 1]) * scale);
        if (key_ok) {
          uint4* dst = reinterpret_cast<uint4*>(out + grow + 32 * c);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v] = make_uint4(wv[4 * v], wv[4 * v + 1], wv[4 * v + 2], wv[4 * v + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(bar(B_DKDV_EMPTY));
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

// ------------------------------------------------------------------ small kernels

// x as the sum of three bf16 terms (exact to about 2^-27 relative): each term rounds
// what the previous ones left, and each difference is exact in fp32.
__device__ __forceinline__ void bf16_split3(float x, uint16_t (&t)[3]) {
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const __nv_bfloat16 b = __float2bfloat16_rn(x);
    t[i] = *reinterpret_cast<const uint16_t*>(&b);
    x = x - __bfloat162float(b);
  }
}

// Per padded query row: Delta, the lse copy (+inf in padding rows), and the row's
// lse_ext / d_ext entries (-lse / qk_scale and -Delta as three bf16 terms; padding rows
// get -1e30 and 0, so P = 0 there).  D / 8 lanes cover a row with 16-byte loads, so a
// warp has 32 / (D / 8) rows in flight per pass.  Block 0 also writes the ones tile.
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(BwdArgs a, int nq_pad) {
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < 128 * 16; i += blockDim.x)
      a.ones[i] = (i & 15) < 3 ? 0x3F80u : 0u;   // bf16 1.0 in elements 0-2
  constexpr int kLanesPerRow = D / 8;          // 8 bf16 per lane
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  const long long rows = static_cast<long long>(a.B) * a.H * nq_pad;
  const long long warp0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane % kLanesPerRow, slot = lane / kLanesPerRow;
  for (long long first = warp0 * kRowsPerWarp; first < rows; first += nw * kRowsPerWarp) {
    const long long rw = first + slot;
    const bool valid = rw < rows;
    const long long bh = valid ? rw / nq_pad : 0;
    const int q = valid ? static_cast<int>(rw % nq_pad) : 0;
    const bool in = valid && q < a.Nq;
    float acc = 0.f;
    // the row's lse is loaded with its O_hp and dO, not after the sum: one memory
    // latency per pass instead of two
    const float lse = in ? a.lse[bh * a.Nq + q] : 0.f;
    if (in) {
      const long long src = (bh * a.Nq + q) * D + 8 * sub;
      const uint4 ov = *reinterpret_cast<const uint4*>(a.o_hp + src);
      const uint4 dv = *reinterpret_cast<const uint4*>(a.dO + src);
      const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
      const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&dv);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 of = __bfloat1622float2(o2[i]);
        const float2 df = __bfloat1622float2(d2[i]);
        acc = fmaf(of.x, df.x, acc);
        acc = fmaf(of.y, df.y, acc);
      }
    }
#pragma unroll
    for (int off = kLanesPerRow / 2; off > 0; off >>= 1)   // within the row's lanes
      acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (!valid) continue;
    if (sub == 0) {
      a.delta[rw] = in ? acc : 0.f;
      a.lse_pad[rw] = in ? lse : INFINITY;
    }
    if (sub < 2) {                    // elements 8 sub .. 8 sub + 7 of both ext rows
      uint4 el = make_uint4(0u, 0u, 0u, 0u), ed = make_uint4(0u, 0u, 0u, 0u);
      if (sub == 0) {
        uint16_t tl[3], td[3];
        bf16_split3(in ? -lse / a.qk_scale : -1e30f, tl);
        bf16_split3(in ? -acc : 0.f, td);
        el = make_uint4(tl[0] | (static_cast<uint32_t>(tl[1]) << 16), tl[2], 0u, 0u);
        ed = make_uint4(td[0] | (static_cast<uint32_t>(td[1]) << 16), td[2], 0u, 0u);
      }
      *reinterpret_cast<uint4*>(a.lse_ext + rw * 16 + 8 * sub) = el;
      *reinterpret_cast<uint4*>(a.d_ext + rw * 16 + 8 * sub) = ed;
    }
  }
}

// Stream-K fix-up, blockIdx.x = item: for an item that range boundaries cut, adds its
// segments' fp32 partial sums in CTA order (the CTAs c0..c1 whose ranges meet the item;
// a segment sits in slot 2c when it is CTA c's first, else 2c + 1) and stores bf16 dV
// and dK (x sm_scale).  Items inside one range were stored by the dK/dV kernel directly.
template <int D>
__global__ void __launch_bounds__(256) bwd_segment_sum_kernel(const float4* __restrict__ part,
                                                              int work, int G, int mtiles,
                                                              int ktiles, int Nkv, float sm_scale,
                                                              uint2* dv, uint2* dk) {
  constexpr int kD4 = D / 4;
  __shared__ int slot_of[kMaxSkCtas];
  const int item = blockIdx.x;
  const long long first = static_cast<long long>(item) * mtiles, last = first + mtiles - 1;
  // CTA whose range holds unit u: the last c with work c / G <= u (64-bit products)
  const int c0 = static_cast<int>(((first + 1) * G - 1) / work);
  const int c1 = static_cast<int>(((last + 1) * G - 1) / work);
  if (c0 == c1) return;
  for (int c = c0 + static_cast<int>(threadIdx.x); c <= c1; c += blockDim.x)
    slot_of[c - c0] = 2 * c + (sk_start(work, c, G) >= first ? 0 : 1);
  __syncthreads();
  const int kb = item % ktiles;
  const long long bh = item / ktiles;
  const int rows = min(kBlk, Nkv - kb * kBlk);
  // blockIdx.y takes every gridDim.y-th group of 256 of the item's 2 x 128 x D/4 float4s
  for (int i = blockIdx.y * blockDim.x + threadIdx.x; i < 2 * kBlk * kD4;
       i += gridDim.y * blockDim.x) {
    const int t = i / (kBlk * kD4);                    // 0: dV, 1: dK
    const int row = (i / kD4) % kBlk;
    const int c4 = i % kD4;
    if (row >= rows) continue;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c = 0; c <= c1 - c0; ++c) {
      const float4 x = part[((static_cast<long long>(slot_of[c]) * 2 + t) * kBlk + row) * kD4 + c4];
      acc.x += x.x;
      acc.y += x.y;
      acc.z += x.z;
      acc.w += x.w;
    }
    const float sc = t ? sm_scale : 1.0f;
    const long long o = ((bh * Nkv) + kb * kBlk + row) * kD4 + c4;
    (t ? dk : dv)[o] = make_uint2(pack_bf16x2(acc.x * sc, acc.y * sc), pack_bf16x2(acc.z * sc, acc.w * sc));
  }
}

template <int D>
cudaError_t launch_bwd_tc_d(const BwdArgs& a, unsigned int* err, int num_sms, cudaStream_t s) {
  using C = BwdTc<D>;
  const int BH = a.B * a.H;
  BwdTcParams p;
  p.a = a;
  p.err = err;
  p.mtiles = (a.Nq + kBlk - 1) / kBlk;
  p.ktiles = (a.Nkv + kBlk - 1) / kBlk;
  p.items = BH * p.ktiles;
  // stream-K: at most the CTAs the workspace has slots for, each with >= 4 units
  const long long work = static_cast<long long>(p.items) * p.mtiles;
  int G = a.causal || a.part == nullptr ? 0 : a.sk_ctas;
  if (G > num_sms) G = num_sms;
  if (G > kMaxSkCtas) G = kMaxSkCtas;  // the fix-up's shared slot table
  if (G > 0 && (work < 4ll * G || work > (1ll << 30))) G = 0;
  p.work = G > 0 ? static_cast<int>(work) : 0;
  p.streamk = G > 0;
  p.nq_pad = p.mtiles * kBlk;
  // a causal item streams its head's Q and dO blocks
  p.hgroup = causal_head_group(4ll * a.Nq * D, BH);

  const long long prow = static_cast<long long>(BH) * p.nq_pad;
  constexpr long long kPrepRowsPerBlock = 8 * (256 / D);  // 8 warps of 32 / (D / 8) rows
  long long pblocks = (prow + kPrepRowsPerBlock - 1) / kPrepRowsPerBlock;
  if (pblocks > static_cast<long long>(num_sms) * 64) pblocks = static_cast<long long>(num_sms) * 64;
  bwd_prep_kernel<D><<<static_cast<unsigned>(pblocks), 256, 0, s>>>(a, p.nq_pad);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  CUtensorMap mq, mk, mv, mdo, mqx, mdx, mones;
  if (!make_bf16_map_3d(&mq, a.q, D, a.Nq, BH) || !make_bf16_map_3d(&mk, a.k, D, a.Nkv, BH) ||
      !make_bf16_map_3d(&mv, a.v, D, a.Nkv, BH) || !make_bf16_map_3d(&mdo, a.dO, D, a.Nq, BH) ||
      !make_ext_map_3d(&mqx, a.lse_ext, p.nq_pad, BH) ||
      !make_ext_map_3d(&mdx, a.d_ext, p.nq_pad, BH) || !make_ext_map_3d(&mones, a.ones, 128, 1))
    return cudaErrorInvalidValue;
  auto kern = p.streamk ? attn_bwd_dkdv_kernel<D, true> : attn_bwd_dkdv_kernel<D, false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(C::kSmemBytes));
  if (e != cudaSuccess) return e;
  const int grid = p.streamk ? G : (p.items < num_sms ? p.items : num_sms);
  kern<<<grid, kThreads, C::kSmemBytes, s>>>(mq, mk, mv, mdo, mqx, mdx, mones, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.streamk) {
    bwd_segment_sum_kernel<D><<<dim3(p.items, 2 * kBlk * (D / 4) / 512), 256, 0, s>>>(
        reinterpret_cast<const float4*>(a.part), p.work, G, p.mtiles, p.ktiles, a.Nkv, a.sm_scale,
        reinterpret_cast<uint2*>(a.dv), reinterpret_cast<uint2*>(a.dk));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return launch_bwd_dq(a, err, num_sms, s);
}

}  // namespace

cudaError_t launch_bwd_tc(const BwdArgs& a, unsigned int* err, int num_sms, cudaStream_t s) {
  return a.D == 64 ? launch_bwd_tc_d<64>(a, err, num_sms, s)
                   : launch_bwd_tc_d<128>(a, err, num_sms, s);
}

}  // namespace qat
