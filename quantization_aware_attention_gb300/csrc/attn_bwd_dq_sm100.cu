// attn_bwd_dq_sm100.cu -- dQ of the QAT attention backward on the Blackwell tensor core
// (tcgen05 + TMEM + TMA), warp-specialized and persistent.  One CTA owns a 128-row query
// block and walks the key blocks, so dQ is summed in TMEM and written once: no atomics,
// and the result does not depend on the order the CTAs run in.
//
// Per query row i and key block j ("attn_qat_train.py", _attn_bwd_dq; P rematerialized
// from the saved base-2 lse):
//   S = Q K_j^T,  P = exp2(S qk_scale - lse_i),  dP = dO V_j^T,
//   dS = P o (dP - Delta_i),  dQ += dS K_j       (dQ scaled by sm_scale at the end)
// P is the unquantized probability in every quant mode: the straight-through estimator
// passes the gradient of O_q through the quantizer as the identity.
// With smooth_k's channel mean (BwdArgs::k_mean) dQ also gets the page's SMOOTH_K term
// (_attn_bwd_dq, "if SMOOTH_K": dq += rowsum(ds) k_mean per key block): each thread sums
// its fp32 dS over the item, the two warpgroups exchange their row sums through shared
// memory, and the epilogue adds rowsum x k_mean before scaling.
//
// CTA layout (352 threads, one CTA per SM, persistent over (head, 128-row query block)):
//   warp 0      TMA producer: per item K_0 and V_0, the item's dO tile (once the
//               previous item's last dP has read the buffer), then the other K_j (4-stage
//               ring) and V_j (2-stage ring), 128 rows x D in 128-byte-swizzled boxes.
//   warp 1      TMEM owner; lane 0 issues, per block j, S_{j+1} then dQ_{j-1}:
//                 S  = Q K^T      TS  (A = Q bf16 in TMEM, B = K_j K-major)   -> TMEM S
//                 dQ += dS K      TS  (A = dS bf16 in TMEM, B = K_j MN-major) -> TMEM dQ
//   warp 2      lane 0 issues dP = dO V^T (SS, A = dO K-major, B = V_j K-major) -> TMEM dP
//               as soon as the compute warps have read the previous dP.
//               Two issuers let the dP stream run ahead independently of the S / dQ
//               stream.  S, dP and dS each have their own TMEM columns, so no product
//               waits for another block's dQ.
//   warps 3-10  two compute warpgroups; group h owns keys [64h, 64h + 64) of every block,
//               each thread one query row (TMEM lane): P from S, dS from P and dP, held
//               in registers and written to the dS columns after the next block's P,
//               and at the end half of dQ's columns to global memory.  Per item they
//               also copy their half of each Q row into TMEM.
// TMEM (512 columns for D = 128): S [0,128), dP [128,256), dQ [256,256+D),
// Q [256+D, 256+3D/2), dS [256+3D/2, 256+3D/2+64).
#include "qat_internal.h"
#include "qat_quant.cuh"
#include "sm100.cuh"

#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

namespace qat {
namespace {

using namespace sm100;

constexpr int kBlk = 128;       // queries per item, keys per block
constexpr int kThreads = 352;
constexpr int kKStages = 4;  // K_j stays until dQ_j, issued a block after S_{j+1}
constexpr int kVStages = 2;

template <int D>
struct BwdDq {
  static constexpr int kChunks = D / 64;
  static constexpr uint32_t kChunkBytes = kBlk * 128;      // 16 KB box: 128 rows x 128 B
  static constexpr uint32_t kTileBytes = kChunks * kChunkBytes;
  static constexpr uint32_t kOffDO = 0;
  static constexpr uint32_t kOffK = kOffDO + kTileBytes;
  static constexpr uint32_t kOffV = kOffK + kKStages * kTileBytes;
  static constexpr uint32_t kOffBar = kOffV + kVStages * kTileBytes;
  static constexpr uint32_t kOffMisc = kOffBar + 256;
  static constexpr uint32_t kOffRs = kOffMisc + 64;       // dS row sums [2 groups][128]
  static constexpr uint32_t kUsed = kOffRs + 2 * 128 * 4;
  // at least 116 KB so that no two CTAs share an SM (each holds all 512 TMEM columns)
  static constexpr uint32_t kSmemBytes = (kUsed + 1024 > 118784u ? kUsed + 1024 : 118784u);
  static constexpr uint32_t kTmemS = 0, kTmemDP = 128, kTmemDQ = 256;
  static constexpr uint32_t kTmemQ = 256 + D, kTmemDS = 256 + D + D / 2;
};
static_assert(BwdDq<128>::kSmemBytes <= 232448u, "shared memory budget");
static_assert(BwdDq<128>::kTmemDS + 64 <= 512u, "TMEM budget");

enum : uint32_t {
  Q_K_FULL = 0, Q_K_EMPTY = Q_K_FULL + kKStages, Q_V_FULL = Q_K_EMPTY + kKStages,
  Q_V_EMPTY = Q_V_FULL + kVStages, Q_DO_FULL = Q_V_EMPTY + kVStages, Q_DO_EMPTY, Q_S_FULL,
  Q_S_EMPTY, Q_DP_FULL, Q_DP_EMPTY, Q_DS_FULL, Q_DS_FREE, Q_QR_FULL, Q_QR_EMPTY, Q_DQ_FULL,
  Q_DQ_EMPTY, Q_DRAIN_A, Q_DRAIN_B, Q_RS, Q_COUNT
};
static_assert(Q_COUNT <= 32, "barrier block");

struct DqParams {
  BwdArgs a;
  unsigned int* err;
  int mtiles;   // query blocks per head
  int ntiles;   // key blocks per head
  int items;    // B * H * mtiles
  int nq_pad;   // mtiles * 128
  int hgroup;   // heads per group of the causal order (causal_head_group)
};

__device__ __forceinline__ void dq_item(int idx, const DqParams& p, int& bh, int& mt, int& J) {
  const int BH = p.a.B * p.a.H;
  if (p.a.causal) {  // longest first (late query blocks see the most keys), heads in groups
    int cls;
    causal_item(idx, BH, p.mtiles, p.hgroup, bh, cls);
    mt = p.mtiles - 1 - cls;
    J = min(p.ntiles, mt + 1);
  } else {           // head-major: the CTAs running together share one head's K/V in L2
    bh = idx / p.mtiles;
    mt = idx % p.mtiles;
    J = p.ntiles;
  }
}

// 32 bytes from global memory (32-byte aligned) into r[0..7]
__device__ __forceinline__ void load32(const uint16_t* ptr, uint32_t* r) {
  asm volatile("ld.global.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "l"(ptr));
}

__device__ __forceinline__ void prefetch_l2(const void* ptr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
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
// kSmooth: a k_mean is passed (the SMOOTH_K term); a separate instance, so that the
// hot loop of the plain backward carries no row-sum register or add.
template <int D, bool kSmooth>
__global__ void __launch_bounds__(384, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmDO, const DqParams p) {
  using C = BwdDq<D>;
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
    for (uint32_t i = 0; i < Q_COUNT; ++i) {
      const bool wg = i == Q_S_EMPTY || i == Q_DP_EMPTY || i == Q_DS_FULL || i == Q_QR_FULL ||
                      i == Q_DQ_EMPTY || i == Q_RS;
      mbar_init(bar(i), wg ? 256u : 1u);
    }
    fence_barrier_init();
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    prefetch_tmap(&tmDO);
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
      uint32_t kc = 0, vc = 0;
      int it = 0;
      bool ok = true;
      for (int idx = blockIdx.x; idx < p.items && ok; idx += gridDim.x, ++it) {
        int bh, mt, J;
        dq_item(idx, p, bh, mt, J);
        // the item's dO waits for the previous item's last dP; its first K and V tiles
        // only for ring stages, so they go first and the item's first S can follow the
        // previous item's last one without waiting for that dP
        auto load_do = [&]() -> bool {
          if (!mbar_wait(bar(Q_DO_EMPTY), (it & 1) ^ 1, abort_flag, p.err)) return false;
          mbar_arrive_expect_tx(bar(Q_DO_FULL), C::kTileBytes);
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(base + C::kOffDO + c * C::kChunkBytes, &tmDO, bar(Q_DO_FULL), 64 * c,
                        mt * kBlk, bh);
          // the next item's dO tile into L2 (each dO tile is read once, so from DRAM)
          if (idx + static_cast<int>(gridDim.x) < p.items) {
            int nbh, nmt, nJ;
            dq_item(idx + gridDim.x, p, nbh, nmt, nJ);
            for (int c = 0; c < C::kChunks; ++c)
              tma_prefetch_l2_3d(&tmDO, 64 * c, nmt * kBlk, nbh);
          }
          return true;
        };
        for (int j = 0; j < J && ok; ++j) {
          if (j == 1 && !(ok = load_do())) break;
          {
            const uint32_t st = kc % kKStages, use = kc / kKStages;
            ok = mbar_wait(bar(Q_K_EMPTY + st), (use & 1) ^ 1, abort_flag, p.err);
            if (!ok) break;
            mbar_arrive_expect_tx(bar(Q_K_FULL + st), C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_3d(base + C::kOffK + st * C::kTileBytes + c * C::kChunkBytes, &tmK,
                          bar(Q_K_FULL + st), 64 * c, j * kBlk, bh);
            ++kc;
          }
          {
            const uint32_t st = vc % kVStages, use = vc / kVStages;
            ok = mbar_wait(bar(Q_V_EMPTY + st), (use & 1) ^ 1, abort_flag, p.err);
            if (!ok) break;
            mbar_arrive_expect_tx(bar(Q_V_FULL + st), C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_3d(base + C::kOffV + st * C::kTileBytes + c * C::kChunkBytes, &tmV,
                          bar(Q_V_FULL + st), 64 * c, j * kBlk, bh);
            ++vc;
          }
        }
        if (ok && J == 1) ok = load_do();
      }
      // drain: every issued load lands before the CTA exits
      if (it > 0) mbar_wait_drain(bar(Q_DO_FULL), (it - 1) & 1, p.err);
      for (uint32_t i = (kc > kKStages ? kc - kKStages : 0); i < kc; ++i)
        mbar_wait_drain(bar(Q_K_FULL + i % kKStages), (i / kKStages) & 1, p.err);
      for (uint32_t i = (vc > kVStages ? vc - kVStages : 0); i < vc; ++i)
        mbar_wait_drain(bar(Q_V_FULL + i % kVStages), (i / kVStages) & 1, p.err);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer A: S, dQ
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(kBlk, kBlk, false);  // S (B = K K-major)
      constexpr uint32_t idQ = idesc_bf16_f32(kBlk, D, true);      // dQ (B = K MN-major)
      uint32_t kc = 0, bc = 0;  // K tiles, blocks (global counts)
      int it = 0;
      bool ok = true, issued = false;
      auto w = [&](uint32_t b_, uint32_t par) { return mbar_wait(b_, par, abort_flag, p.err); };
      // S of block c (K tile k): after the compute warps have read S of block c - 1
      auto issue_s = [&](uint32_t k, uint32_t c, bool last) -> bool {
        // the K tile first (it has almost always landed), then the compute warps' barrier
        const uint32_t st = k % kKStages;
        if (!w(bar(Q_K_FULL + st), (k / kKStages) & 1)) return false;
        if (c > 0 && !w(bar(Q_S_EMPTY), (c - 1) & 1)) return false;
        tc_fence_after();
        const uint32_t sk = base + C::kOffK + st * C::kTileBytes;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * C::kChunkBytes + (ks & 3) * 32;
          mma_ts(tbase + C::kTmemS, tbase + C::kTmemQ + 8 * ks,
                 smem_desc_sw128(sk + off, 16, 1024), idS, ks > 0 ? 1u : 0u);
        }
        issued = true;
        mma_commit(bar(Q_S_FULL));
        if (last) mma_commit(bar(Q_QR_EMPTY));  // the item's last read of its Q rows
        return true;
      };
      // dQ += dS_c K_c (K tile k), once the compute warps have written dS_c
      auto issue_dq = [&](uint32_t k, uint32_t c, bool first, bool last) -> bool {
        if (!w(bar(Q_DS_FULL), c & 1)) return false;
        if (first && it > 0 && !w(bar(Q_DQ_EMPTY), (it - 1) & 1)) return false;
        tc_fence_after();
        const uint32_t st = k % kKStages;
        const uint32_t sk = base + C::kOffK + st * C::kTileBytes;
#pragma unroll
        for (int ks = 0; ks < kBlk / 16; ++ks)
          mma_ts(tbase + C::kTmemDQ, tbase + C::kTmemDS + 8 * ks,
                 smem_desc_sw128(sk + ks * 2048, C::kChunkBytes, 1024), idQ,
                 (!first || ks > 0) ? 1u : 0u);
        mma_commit(bar(Q_K_EMPTY + st));  // K_c: read by S_c and dQ_c, both issued here
        mma_commit(bar(Q_DS_FREE));
        if (last) mma_commit(bar(Q_DQ_FULL));
        return true;
      };
      // Per item: S_0, then for each block j: S_{j+1} and dQ_{j-1}; dQ_{J-1} at the end.
      // The compute warps write dS_{j-1} only after computing P_j, so dQ lags S by two
      // blocks and its completion overlaps a whole block of their work.
      for (int idx = blockIdx.x; idx < p.items && ok; idx += gridDim.x, ++it) {
        int bh, mt, J;
        dq_item(idx, p, bh, mt, J);
        ok = w(bar(Q_QR_FULL), it & 1) && issue_s(kc, bc, J == 1);
        for (int j = 0; j < J && ok; ++j) {
          if (j + 1 < J && !(ok = issue_s(kc + j + 1, bc + j + 1, j + 2 == J))) break;
          if (j >= 1 && !(ok = issue_dq(kc + j - 1, bc + j - 1, j == 1, false))) break;
        }
        if (ok) ok = issue_dq(kc + J - 1, bc + J - 1, J == 1, true);
        kc += J;
        bc += J;
      }
      if (issued) {
        mma_commit(bar(Q_DRAIN_A));
        mbar_wait_drain(bar(Q_DRAIN_A), 0, p.err);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ MMA issuer B: dP
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(kBlk, kBlk, false);
      uint32_t vc = 0, bc = 0;
      int it = 0;
      bool ok = true, issued = false;
      auto w = [&](uint32_t b_, uint32_t par) { return mbar_wait(b_, par, abort_flag, p.err); };
      const uint32_t sdo = base + C::kOffDO;
      for (int idx = blockIdx.x; idx < p.items && ok; idx += gridDim.x, ++it) {
        int bh, mt, J;
        dq_item(idx, p, bh, mt, J);
        ok = w(bar(Q_DO_FULL), it & 1);
        for (int j = 0; j < J && ok; ++j, ++vc, ++bc) {
          // dP overwrites dP of block bc - 1: wait until the compute warps have read it
          const uint32_t st = vc % kVStages;
          if (!(ok = w(bar(Q_V_FULL + st), (vc / kVStages) & 1))) break;
          if (bc > 0 && !(ok = w(bar(Q_DP_EMPTY), (bc - 1) & 1))) break;
          tc_fence_after();
          const uint32_t sv = base + C::kOffV + st * C::kTileBytes;
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = (ks >> 2) * C::kChunkBytes + (ks & 3) * 32;
            mma_ss(tbase + C::kTmemDP, smem_desc_sw128(sdo + off, 16, 1024),
                   smem_desc_sw128(sv + off, 16, 1024), idS, ks > 0 ? 1u : 0u);
          }
          issued = true;
          mma_commit(bar(Q_V_EMPTY + st));
          mma_commit(bar(Q_DP_FULL));
          if (j + 1 == J) mma_commit(bar(Q_DO_EMPTY));
        }
      }
      if (issued) {
        mma_commit(bar(Q_DRAIN_B));
        mbar_wait_drain(bar(Q_DRAIN_B), 0, p.err);
      }
    }
  } else {
    // ------------------------------------------------------------ compute warpgroups
    const int h = (warp - 3) >> 2;
    const int quarter = warp & 3;                    // TMEM lane quarter of this warp
    const int r = 32 * quarter + lane;               // query row of the block (TMEM lane)
    const uint32_t lrow = (32u * quarter) << 16;
    const float qk = p.a.qk_scale;
    float* rsx = reinterpret_cast<float*>(gbase + C::kOffRs);  // [2 groups][128 rows]
    auto wwait = [&](uint32_t b_, uint32_t par) {
      const bool okw = mbar_wait(b_, par, abort_flag, p.err);
      return __all_sync(0xffffffffu, okw) != 0;
    };
    // half h of this thread's Q row into TMEM as bf16 pairs (D / 4 columns); rows past Nq
    // are zero (their lse is +inf, so P = 0 there).  Each thread reads a different row,
    // so one load instruction touches 32 lines; with a 32-byte aligned q the rows are
    // read 32 bytes at a time.
    const bool q32 = (reinterpret_cast<uintptr_t>(p.a.q) & 31u) == 0;
    auto load_q = [&](int bh, int mt) {
      constexpr int kCols = D / 4;
      const int row = mt * kBlk + r;
      const uint16_t* src = p.a.q + (static_cast<size_t>(bh) * p.a.Nq + row) * D + (D / 2) * h;
      uint32_t v[kCols];
#pragma unroll
      for (int u = 0; u < kCols; ++u) v[u] = 0u;
      if (row < p.a.Nq) {
        if (q32) {  // 32-byte loads: half the L1 wavefronts of 16-byte ones for these rows
#pragma unroll
          for (int u = 0; u < kCols / 8; ++u) load32(src + 16 * u, &v[8 * u]);
        } else {
#pragma unroll
          for (int u = 0; u < kCols / 4; ++u) {
            const uint4 x = *reinterpret_cast<const uint4*>(src + 8 * u);
            v[4 * u] = x.x;
            v[4 * u + 1] = x.y;
            v[4 * u + 2] = x.z;
            v[4 * u + 3] = x.w;
          }
        }
      }
      const uint32_t dst = tbase + lrow + C::kTmemQ + kCols * h;
      if constexpr (kCols == 32)
        tmem_st32(dst, v);
      else
        tmem_st16(dst, v);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(Q_QR_FULL));
    };
    uint32_t bc = 0;
    int it = 0;
    bool ok = true;
    // lse and Delta of this thread's row in the next item, read with its Q rows
    float lse_n = 0.f, delta_n = 0.f;
    auto load_next = [&](int bh, int mt) {
      load_q(bh, mt);
      const size_t prow = static_cast<size_t>(bh) * p.nq_pad + mt * kBlk + r;
      lse_n = p.a.lse_pad[prow];
      delta_n = p.a.delta[prow];
    };
    if (static_cast<int>(blockIdx.x) < p.items) {
      int bh, mt, J;
      dq_item(blockIdx.x, p, bh, mt, J);
      load_next(bh, mt);
    }
    for (int idx = blockIdx.x; idx < p.items && ok; idx += gridDim.x, ++it) {
      int bh, mt, J;
      dq_item(idx, p, bh, mt, J);
      const int row = mt * kBlk + r;
      const float lse_r = lse_n;
      const float delta_r = delta_n;
      const int nidx = idx + static_cast<int>(gridDim.x);
      {  // the next item's Q half-row, lse and Delta, read during this item, into L2 now
        if (nidx < p.items) {
          int nbh, nmt, nJ;
          dq_item(nidx, p, nbh, nmt, nJ);
          const int nrow = nmt * kBlk + r;
          const size_t nprow = static_cast<size_t>(nbh) * p.nq_pad + nrow;
          if (nrow < p.a.Nq)
            prefetch_l2(p.a.q + (static_cast<size_t>(nbh) * p.a.Nq + nrow) * D + (D / 2) * h);
          prefetch_l2(p.a.lse_pad + nprow);
          prefetch_l2(p.a.delta + nprow);
        }
      }
      // dS of block c (keys [64h, 64h + 64)) -> TMEM dS columns [32h, 32h + 32), once dQ
      // of block c - 1 has read the buffer.  dS_c is held in registers and written after
      // P of block c + 1 has been computed, so dQ_{c-1} has a block's time to complete.
      uint32_t pk[32];
      float rs = 0.f;                                  // sum of this thread's fp32 dS
      auto write_ds = [&](uint32_t c) -> bool {
        if (c > 0 && !wwait(bar(Q_DS_FREE), (c - 1) & 1)) return false;
        tc_fence_after();
        tmem_st32(tbase + lrow + C::kTmemDS + 32 * h, pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(Q_DS_FULL));
        return true;
      };
      for (int j = 0; j < J && ok; ++j, ++bc) {
        if (!(ok = wwait(bar(Q_S_FULL), bc & 1))) break;
        tc_fence_after();
        uint32_t pr[64];                               // S, then P, of this row's 64 keys
        tmem_ld32(tbase + lrow + C::kTmemS + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&pr[0]));
        tmem_ld32(tbase + lrow + C::kTmemS + 64 * h + 32,
                  *reinterpret_cast<uint32_t(*)[32]>(&pr[32]));
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bar(Q_S_EMPTY));
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          const float2 x = fma_rn_f32x2(make_float2(__uint_as_float(pr[i]), __uint_as_float(pr[i + 1])),
                                        make_float2(qk, qk), make_float2(-lse_r, -lse_r));
          pr[i] = __float_as_uint(ex2f(x.x));
          pr[i + 1] = __float_as_uint(ex2f(x.y));
        }
        // keys past Nkv, and keys after the row on the causal diagonal: P = 0 (a
        // warp-uniform pass over the few blocks that have such keys)
        const int key0 = j * kBlk + 64 * h;
        if (key0 + 64 > p.a.Nkv || (p.a.causal && j == mt)) {
          const int lim = p.a.causal ? min(p.a.Nkv - 1, row) : p.a.Nkv - 1;
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (key0 + i > lim) pr[i] = 0u;
        }
        if (j > 0 && !(ok = write_ds(bc - 1))) break;
        if (!(ok = wwait(bar(Q_DP_FULL), bc & 1))) break;
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t dr[32];
          tmem_ld32(tbase + lrow + C::kTmemDP + 64 * h + 32 * cc, dr);
          tmem_wait_ld();
          if (cc == 1) {                               // every read of this dP is done
            tc_fence_before();
            mbar_arrive(bar(Q_DP_EMPTY));
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 d = mul_rn_f32x2(
                make_float2(__uint_as_float(pr[32 * cc + 2 * i]), __uint_as_float(pr[32 * cc + 2 * i + 1])),
                add_rn_f32x2(make_float2(__uint_as_float(dr[2 * i]), __uint_as_float(dr[2 * i + 1])),
                             make_float2(-delta_r, -delta_r)));
            pk[16 * cc + i] = pack_bf16x2(d.x, d.y);
            if constexpr (kSmooth) rs += d.x + d.y;
          }
        }
      }
      if (ok) ok = write_ds(bc - 1);   // the item's last dS
      if (!ok) break;
      // the next item's Q rows go in once this item's last S has read the current ones
      if (nidx < p.items) {
        if (!(ok = wwait(bar(Q_QR_EMPTY), it & 1))) break;
        tc_fence_after();
        int nbh, nmt, nJ;
        dq_item(nidx, p, nbh, nmt, nJ);
        load_next(nbh, nmt);
      }
      // ---- epilogue: group h stores dQ columns [hD/2, (h+1)D/2) of its row
      if (!(ok = wwait(bar(Q_DQ_FULL), it & 1))) break;
      tc_fence_after();
      // SMOOTH_K: the row's dS sum over both groups' keys.  Written only after Q_DQ_FULL,
      // which needs both groups' last dS of this item, so the other group has read the
      // previous item's value by then.
      float rowsum = 0.f;
      if constexpr (kSmooth) {
        rsx[h * 128 + r] = rs;
        mbar_arrive(bar(Q_RS));
        if (!(ok = wwait(bar(Q_RS), it & 1))) break;
        rowsum = rsx[r] + rsx[128 + r];
      }
      uint32_t o[D / 2];
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tmem_ld32(tbase + lrow + C::kTmemDQ + (D / 2) * h + 32 * c,
                  *reinterpret_cast<uint32_t(*)[32]>(&o[32 * c]));
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar(Q_DQ_EMPTY));
      if constexpr (kSmooth) {
        const float4* km = reinterpret_cast<const float4*>(p.a.k_mean + (D / 2) * h);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          const float4 m = km[c];
          o[4 * c] = __float_as_uint(fmaf(rowsum, m.x, __uint_as_float(o[4 * c])));
          o[4 * c + 1] = __float_as_uint(fmaf(rowsum, m.y, __uint_as_float(o[4 * c + 1])));
          o[4 * c + 2] = __float_as_uint(fmaf(rowsum, m.z, __uint_as_float(o[4 * c + 2])));
          o[4 * c + 3] = __float_as_uint(fmaf(rowsum, m.w, __uint_as_float(o[4 * c + 3])));
        }
      }
      if (row < p.a.Nq) {
        const float sc = p.a.sm_scale;
        uint4* dst = reinterpret_cast<uint4*>(p.a.dq + (static_cast<size_t>(bh) * p.a.Nq + row) * D +
                                              (D / 2) * h);
#pragma unroll
        for (int v = 0; v < D / 16; ++v)
          dst[v] = make_uint4(
              pack_bf16x2(__uint_as_float(o[8 * v]) * sc, __uint_as_float(o[8 * v + 1]) * sc),
              pack_bf16x2(__uint_as_float(o[8 * v + 2]) * sc, __uint_as_float(o[8 * v + 3]) * sc),
              pack_bf16x2(__uint_as_float(o[8 * v + 4]) * sc, __uint_as_float(o[8 * v + 5]) * sc),
              pack_bf16x2(__uint_as_float(o[8 * v + 6]) * sc, __uint_as_float(o[8 * v + 7]) * sc));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

template <int D>
cudaError_t launch_bwd_dq_d(const BwdArgs& a, unsigned int* err, int num_sms, cudaStream_t s) {
  using C = BwdDq<D>;
  const int BH = a.B * a.H;
  DqParams p;
  p.a = a;
  p.err = err;
  p.mtiles = (a.Nq + kBlk - 1) / kBlk;
  p.ntiles = (a.Nkv + kBlk - 1) / kBlk;
  p.items = BH * p.mtiles;
  p.nq_pad = p.mtiles * kBlk;
  // a causal item streams its head's K and V blocks
  p.hgroup = causal_head_group(4ll * a.Nkv * D, BH);
  CUtensorMap mk, mv, mdo;
  if (!make_bf16_map_3d(&mk, a.k, D, a.Nkv, BH) || !make_bf16_map_3d(&mv, a.v, D, a.Nkv, BH) ||
      !make_bf16_map_3d(&mdo, a.dO, D, a.Nq, BH))
    return cudaErrorInvalidValue;
  auto kern = a.k_mean != nullptr ? attn_bwd_dq_kernel<D, true> : attn_bwd_dq_kernel<D, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(C::kSmemBytes));
  if (e != cudaSuccess) return e;
  const int grid = p.items < num_sms ? p.items : num_sms;
  kern<<<grid, kThreads, C::kSmemBytes, s>>>(mk, mv, mdo, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq(const BwdArgs& a, unsigned int* err, int num_sms, cudaStream_t s) {
  return a.D == 64 ? launch_bwd_dq_d<64>(a, err, num_sms, s)
                   : launch_bwd_dq_d<128>(a, err, num_sms, s);
}

}  // namespace qat
