// attn_fwd_sm100.cu -- QAT attention forward on the Blackwell tensor core (tcgen05 +
// TMEM + TMA), warp-specialized and persistent.
//
// Method ("attn_qat_train.py", _attn_fwd / _attn_fwd_inner), per query row i and KV
// tile j:  S = Q K_j^T;  x = S * qk_scale (masked keys -inf);  running max m;
//   p = exp2(x - m);  l = alpha l + rowsum p (unquantized);  per 64-key quant tile
//   amax = max p, Pq = quant(p) (qat_quant.cuh);  O_q = alpha O_q + Pq V_j;
//   O_hp = alpha O_hp + P V_j;  epilogue O / l, lse = m + log2 l.
//
// CTA layout (352 threads, one CTA per SM, persistent over (head, 128-row q tile)):
//   warp 0      TMA producer: Q tile once per work item, K tiles (3-stage ring) and
//               V tiles (2-stage ring), 128 keys x D, 128-byte swizzled boxes.
//   warp 1      TMEM allocator; lane 0 issues the score MMAs:
//                 S_j = Q K_j^T            (SS, M=128, N=128 keys, K=D) -> TMEM S[j%2]
//   warp 2      lane 0 issues the value MMAs:
//                 O_q += Pq_j V_j          (TS: A = Pq in TMEM, B = V MN-major in smem)
//                 O_hp += P_j V_j          (TS, same V descriptors: the two P tiles share V)
//               The two streams progress independently: scores run ahead while the value
//               MMAs wait for P.  S_{j+2} reuses the buffer that holds P_j, so warp 1
//               waits for warp 2's commit of PV_j before issuing it.
//   warps 3-10  softmax + quantization in two warpgroups: warps 3-6 take keys 0-63 and
//               warps 7-10 keys 64-127 of each S row (one 64-key quantization tile per
//               thread), exchanging the row max through shared memory.  P is written
//               back into the S buffer it came from as two bf16 tiles (Pq in columns
//               0-63, P in 64-127), consumed by the TS MMAs.  Epilogue: warps 3-6 store
//               O_q and lse, warps 7-10 O_hp; at the end of the item, or (short items,
//               the kDefer instance) after the next item's first block of P.
// TMEM (512 columns): S0 [0,128), S1 [128,256), O_q [256,256+D), O_hp [256+D,256+2D).
//
// The running max is updated only when it grows by more than 8 (base-2 units), so P
// may reach 2^8 and the O rescale is rare.  The FP8 code depends only on p / amax, so
// this leaves the quantization unchanged in exact arithmetic (the max element of every
// tile still maps to 448) and l, O_q and O_hp stay consistent.
#include "qat_internal.h"
#include "qat_quant.cuh"
#include "sm100.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

namespace qat {
namespace {

using namespace sm100;

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kThreads = 352;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: p <= 2^8 between rescales

template <int D>
struct FwdTc {
  static constexpr int kChunks = D / 64;                 // 128-byte column chunks per row
  static constexpr uint32_t kChunkBytes = kBM * 128;     // one 128-row x 64-col box: 16 KB
  static constexpr uint32_t kTileBytes = kChunks * kChunkBytes;
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffK = kOffQ + kTileBytes;
  static constexpr uint32_t kOffV = kOffK + kKStages * kTileBytes;
  static constexpr uint32_t kOffBar = kOffV + kVStages * kTileBytes;
  static constexpr uint32_t kOffMisc = kOffBar + 256;
  static constexpr uint32_t kOffX = kOffMisc + 64;     // row-max / row-sum exchange, 3 KB
  static constexpr uint32_t kOffStage = kOffX + 3072;  // epilogue staging, 2 KB per softmax warp
  static constexpr uint32_t kUsed = kOffStage + 8 * 2048;
  // at least 116 KB so that no two CTAs share an SM (each holds all 512 TMEM columns)
  static constexpr uint32_t kSmemBytes = (kUsed + 1024 > 118784u ? kUsed + 1024 : 118784u);
  static constexpr uint32_t kTmemOq = 256;
  static constexpr uint32_t kTmemOhp = 256 + D;
};

// barrier indices (8 bytes each) in the barrier block
enum : uint32_t {
  BAR_Q_FULL = 0, BAR_Q_EMPTY = 1, BAR_K_FULL = 2, BAR_K_EMPTY = 5, BAR_V_FULL = 8,
  BAR_V_EMPTY = 10, BAR_S_FULL = 12, BAR_P_FULL = 14, BAR_O_DONE = 16, BAR_O_EMPTY = 17,
  BAR_DRAIN = 18, BAR_S_FREE = 20, BAR_DRAIN_B = 22, BAR_O_FINAL = 23,
  BAR_XQ = 24,  // 4 row-exchange barriers, one per TMEM lane quarter
  BAR_COUNT = 28
};
static_assert(BAR_COUNT * 8 <= 256, "barrier block");

struct TcParams {
  FwdArgs a;
  unsigned int* err;
  int mtiles;   // ceil(Nq / 128)
  int items;    // B * H * mtiles
  int hgroup;   // heads per group of the causal order (causal_head_group)
};

__device__ __forceinline__ void item_coords(int idx, const TcParams& p, int& bh, int& mt) {
  const int BH = p.a.B * p.a.H;
  if (p.a.causal) {  // longest rows first, heads in L2-sized groups
    int cls;
    causal_item(idx, BH, p.mtiles, p.hgroup, bh, cls);
    mt = p.mtiles - 1 - cls;
  } else {           // head-major: CTAs running together share one head's K/V in L2
    bh = idx / p.mtiles;
    mt = idx % p.mtiles;
  }
}

__device__ __forceinline__ int kv_tiles(const TcParams& p, int mt) {
  const int n = (p.a.Nkv + kBN - 1) / kBN;
  return p.a.causal ? min(n, mt + 1) : n;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Bounds of 384 threads cap registers at 168 per thread: with 11 warps, three share a
// sub-partition's 16K registers, so a 352-thread CTA cannot launch with more.
// kDefer: each item's epilogue waits for the next item's first block of P (short items,
// see the softmax warps); a separate instance, since with the epilogue inside the block
// loop long items ran 2-4% slower.
template <int D, bool kDefer>
__global__ void __launch_bounds__(384, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const TcParams p) {
  using C = FwdTc<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + C::kOffBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kOffMisc);
  volatile WaitCtl* abort_flag = reinterpret_cast<volatile WaitCtl*>(gbase + C::kOffMisc + 8);
  auto bar = [&](uint32_t i) { return bars + 8u * i; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    wait_ctl_init(abort_flag, p.err);
    mbar_init(bar(BAR_Q_FULL), 1);
    mbar_init(bar(BAR_Q_EMPTY), 1);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(bar(BAR_K_FULL + s), 1);
      mbar_init(bar(BAR_K_EMPTY + s), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(bar(BAR_V_FULL + s), 1);
      mbar_init(bar(BAR_V_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(BAR_S_FULL + b), 1);
      mbar_init(bar(BAR_P_FULL + b), 256);
      mbar_init(bar(BAR_S_FREE + b), 1);
    }
    mbar_init(bar(BAR_O_DONE), 1);
    mbar_init(bar(BAR_O_EMPTY), 256);
    mbar_init(bar(BAR_DRAIN), 1);
    mbar_init(bar(BAR_DRAIN_B), 1);
    mbar_init(bar(BAR_O_FINAL), 1);
    for (int q = 0; q < 4; ++q) mbar_init(bar(BAR_XQ + q), 64);
    fence_barrier_init();
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
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
      uint32_t kc = 0, vc = 0, qn = 0;  // K, V and Q loads issued
      int it = 0;
      bool ok = true;
      for (int idx = blockIdx.x; idx < p.items && ok; idx += gridDim.x, ++it) {
        int bh, mt;
        item_coords(idx, p, bh, mt);
        const int J = kv_tiles(p, mt);
        ok = mbar_wait(bar(BAR_Q_EMPTY), (it & 1) ^ 1, abort_flag, p.err);
        if (!ok) break;
        ++qn;
        mbar_arrive_expect_tx(bar(BAR_Q_FULL), C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(base + C::kOffQ + c * C::kChunkBytes, &tmQ, bar(BAR_Q_FULL), 64 * c,
                      mt * kBM, bh);
        // the next item's Q tile into L2 (each Q tile is read once, so from DRAM): its
        // load then waits only for the L2 when the Q buffer frees up
        if (idx + static_cast<int>(gridDim.x) < p.items) {
          int nbh, nmt;
          item_coords(idx + gridDim.x, p, nbh, nmt);
          for (int c = 0; c < C::kChunks; ++c) tma_prefetch_l2_3d(&tmQ, 64 * c, nmt * kBM, nbh);
        }
        for (int j = 0; j <= J && ok; ++j) {
          if (j < J) {  // K_j
            const uint32_t st = kc % kKStages, use = kc / kKStages;
            ok = mbar_wait(bar(BAR_K_EMPTY + st), (use & 1) ^ 1, abort_flag, p.err);
            if (!ok) break;
            mbar_arrive_expect_tx(bar(BAR_K_FULL + st), C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_3d(base + C::kOffK + st * C::kTileBytes + c * C::kChunkBytes, &tmK,
                          bar(BAR_K_FULL + st), 64 * c, j * kBN, bh);
            ++kc;
          }
          if (j >= 1) {  // V_{j-1}: one tile behind K, matching the MMA issue order
            const uint32_t st = vc % kVStages, use = vc / kVStages;
            ok = mbar_wait(bar(BAR_V_EMPTY + st), (use & 1) ^ 1, abort_flag, p.err);
            if (!ok) break;
            mbar_arrive_expect_tx(bar(BAR_V_FULL + st), C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_3d(base + C::kOffV + st * C::kTileBytes + c * C::kChunkBytes, &tmV,
                          bar(BAR_V_FULL + st), 64 * c, (j - 1) * kBN, bh);
            ++vc;
          }
        }
      }
      // drain: every issued load must land before the CTA can exit (after an abort the
      // score MMAs may not have waited for the last Q tile)
      if (qn > 0) mbar_wait_drain(bar(BAR_Q_FULL), (qn - 1) & 1, p.err);
      for (uint32_t i = (kc > kKStages ? kc - kKStages : 0); i < kc; ++i)
        mbar_wait_drain(bar(BAR_K_FULL + i % kKStages), (i / kKStages) & 1, p.err);
      for (uint32_t i = (vc > kVStages ? vc - kVStages : 0); i < vc; ++i)
        mbar_wait_drain(bar(BAR_V_FULL + i % kVStages), (i / kVStages) & 1, p.err);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ score MMAs (S = Q K^T)
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(kBM, kBN, false);
      uint32_t kc = 0, sc = 0;
      int it = 0;
      bool ok = true, issued = false;
      for (int idx = blockIdx.x; idx < p.items && ok; idx += gridDim.x, ++it) {
        int bh, mt;
        item_coords(idx, p, bh, mt);
        const int J = kv_tiles(p, mt);
        ok = mbar_wait(bar(BAR_Q_FULL), it & 1, abort_flag, p.err);
        for (int j = 0; j < J && ok; ++j, ++kc, ++sc) {
          const uint32_t st = kc % kKStages;
          const uint32_t b = sc & 1;
          ok = mbar_wait(bar(BAR_K_FULL + st), (kc / kKStages) & 1, abort_flag, p.err);
          // buffer b holds P of tile sc - 2 until its value MMAs have completed
          if (ok && sc >= 2)
            ok = mbar_wait(bar(BAR_S_FREE + b), ((sc - 2) >> 1) & 1, abort_flag, p.err);
          if (!ok) break;
          tc_fence_after();
          const uint32_t qb = base + C::kOffQ;
          const uint32_t kb = base + C::kOffK + st * C::kTileBytes;
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = (ks >> 2) * C::kChunkBytes + (ks & 3) * 32;
            mma_ss(tbase + b * 128, smem_desc_sw128(qb + off, 16, 1024),
                   smem_desc_sw128(kb + off, 16, 1024), idS, ks > 0 ? 1u : 0u);
          }
          issued = true;
          mma_commit(bar(BAR_K_EMPTY + st));
          mma_commit(bar(BAR_S_FULL + b));
          if (j == J - 1) mma_commit(bar(BAR_Q_EMPTY));
        }
      }
      if (issued) {  // drain: wait until every MMA this thread issued has completed
        mma_commit(bar(BAR_DRAIN));
        mbar_wait_drain(bar(BAR_DRAIN), 0, p.err);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ value MMAs (P V)
    if (lane == 0) {
      constexpr uint32_t idPV = idesc_bf16_f32(kBM, D, true);
      uint32_t vc = 0, pc = 0;
      int it = 0;
      bool ok = true, issued = false;
      for (int idx = blockIdx.x; idx < p.items && ok; idx += gridDim.x, ++it) {
        int bh, mt;
        item_coords(idx, p, bh, mt);
        const int J = kv_tiles(p, mt);
        for (int j = 0; j < J && ok; ++j, ++vc, ++pc) {
          const uint32_t b = pc & 1;
          // V first (it has almost always landed), then P from the softmax warps
          const uint32_t st = vc % kVStages;
          ok = mbar_wait(bar(BAR_V_FULL + st), (vc / kVStages) & 1, abort_flag, p.err);
          if (ok) ok = mbar_wait(bar(BAR_P_FULL + b), (pc >> 1) & 1, abort_flag, p.err);
          if (ok && j == 0) ok = mbar_wait(bar(BAR_O_EMPTY), (it & 1) ^ 1, abort_flag, p.err);
          if (!ok) break;
          tc_fence_after();
          const uint32_t vbase = base + C::kOffV + st * C::kTileBytes;
          const uint32_t sP = tbase + b * 128;
#pragma unroll
          for (int ks = 0; ks < kBN / 16; ++ks) {
            const uint64_t dv = smem_desc_sw128(vbase + ks * 2048, C::kChunkBytes, 1024);
            mma_ts(tbase + C::kTmemOq, sP + 8 * ks, dv, idPV, (j > 0 || ks > 0) ? 1u : 0u);
          }
#pragma unroll
          for (int ks = 0; ks < kBN / 16; ++ks) {
            const uint64_t dv = smem_desc_sw128(vbase + ks * 2048, C::kChunkBytes, 1024);
            mma_ts(tbase + C::kTmemOhp, sP + 64 + 8 * ks, dv, idPV, (j > 0 || ks > 0) ? 1u : 0u);
          }
          issued = true;
          mma_commit(bar(BAR_V_EMPTY + st));
          mma_commit(bar(BAR_O_DONE));
          mma_commit(bar(BAR_S_FREE + b));
          if (j + 1 == J) mma_commit(bar(BAR_O_FINAL));  // the item's O is complete
        }
      }
      if (issued) {
        mma_commit(bar(BAR_DRAIN_B));
        mbar_wait_drain(bar(BAR_DRAIN_B), 0, p.err);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    // Two warpgroups: h = 0 (warps 3-6) owns keys 0-63 of every S row, h = 1 (warps
    // 7-10) keys 64-127 -- each thread one row of one 64-key quantization tile.
    const int h = (warp - 3) >> 2;
    const int quarter = warp & 3;                 // TMEM lane quarter of this warp
    const int r = 32 * quarter + lane;            // row of the 128-row tile
    const uint32_t lrow = (32u * quarter) << 16;  // TMEM lane offset
    const float qk = p.a.qk_scale;
    float* xmax = reinterpret_cast<float*>(gbase + C::kOffX);        // [2 parity][2 h][128]
    float* xsum = reinterpret_cast<float*>(gbase + C::kOffX + 2048); // [2 h][128]
    // Epilogue stores: 64 bytes of each of the warp's 32 rows (this thread's row is its
    // lane) go through the warp's 2 KB of shared memory, with the 16-byte chunks XOR-
    // swizzled by row so that the row-wise writes and the column-wise reads are both free
    // of bank conflicts.  Read back, one store instruction writes 8 rows x 64 bytes (16
    // full sectors) instead of 32 rows x 16 bytes (32 half sectors).
    uint4* stg = reinterpret_cast<uint4*>(gbase + C::kOffStage) + (warp - 3) * 128;
    auto store_rows64 = [&](const uint4 (&v)[4], char* row0, size_t row_bytes, int rows_valid) {
#pragma unroll
      for (int i = 0; i < 4; ++i) stg[lane * 4 + (i ^ ((lane >> 1) & 3))] = v[i];
      __syncwarp();
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int rr = 8 * k + (lane >> 2), cc = lane & 3;
        const uint4 x = stg[rr * 4 + (cc ^ ((rr >> 1) & 3))];
        if (rr < rows_valid) *reinterpret_cast<uint4*>(row0 + rr * row_bytes + 16 * cc) = x;
      }
      __syncwarp();  // the next call overwrites the staging
    };
    // tcgen05.ld/st are warp-collective: every wait result is made warp-uniform
    auto wwait = [&](uint32_t b_, uint32_t par) {
      const bool w = mbar_wait(b_, par, abort_flag, p.err);
      return __all_sync(0xffffffffu, w) != 0;
    };
    // exchange between the two groups: a row's two halves live in the two warps of one
    // TMEM lane quarter (warps w and w + 4, which share warp & 3), so each pair
    // synchronises on its own barrier: every thread arrives after writing its value and
    // waits (bounded) for the phase before reading its partner's.  The barrier also
    // orders the pair's TMEM reads of S before either writes P over it, and a pair waits
    // only for itself, not for the slowest of all eight warps (-0.7% at c4).
    uint32_t xc = 0;
    auto exchange = [&]() {
      tc_fence_before();
      mbar_arrive(bar(BAR_XQ + quarter));
      const bool w = wwait(bar(BAR_XQ + quarter), xc & 1);
      ++xc;
      tc_fence_after();
      return w;
    };
    // With kDefer an item's epilogue runs after the next item's first block of P, so that
    // the wait for its last PV products and the next item's first score product overlap
    // the softmax of that block instead of following the epilogue (at B1 H40 Nq16384
    // Nkv512, 4 blocks per item: 0.272 -> 0.252 ms).  O stays in TMEM until then: the
    // next item's first PV waits for O_EMPTY, and a rescale needs j > 0.
    int e_bh = 0, e_mt = 0, e_it = -1;  // the item whose epilogue is pending (e_it >= 0)
    float e_m = 0.f, e_l = 1.f;         // its running max and row sum
    auto epilogue = [&]() -> bool {
      // O_DONE cannot be used here: it completes once per block, and at the end of an
      // item the PV products of the last two blocks may both still be running (S of
      // the last block only waited for PV two blocks back).  A parity wait on a barrier
      // two phases behind passes at once, so the epilogue waits on O_FINAL, committed
      // after the item's last PV: one phase per item.
      if (!wwait(bar(BAR_O_FINAL), e_it & 1)) return false;
      tc_fence_after();
      const float inv_l = 1.0f / e_l;
      const int row = e_mt * kBM + r;
      const bool in = row < p.a.Nq;
      // the warp's first row, and how many of its 32 rows exist
      const int wrow = e_mt * kBM + 32 * quarter;
      const int wvalid = min(32, p.a.Nq - wrow);
      const size_t orow0 = static_cast<size_t>(e_bh) * p.a.Nq + wrow;
      const uint32_t tO = tbase + lrow + (h ? C::kTmemOhp : C::kTmemOq);
      uint16_t* out = h ? p.a.o_hp : p.a.o_q;
      float* out32 = h ? p.a.o_hp_f32 : p.a.o_q_f32;  // partial results stay fp32
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + 32 * c, o);
        tmem_wait_ld();
        if (out32 != nullptr) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint4 v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t* x = o + 16 * half + 4 * i;
              v[i] = make_uint4(__float_as_uint(__uint_as_float(x[0]) * inv_l),
                                __float_as_uint(__uint_as_float(x[1]) * inv_l),
                                __float_as_uint(__uint_as_float(x[2]) * inv_l),
                                __float_as_uint(__uint_as_float(x[3]) * inv_l));
            }
            store_rows64(v, reinterpret_cast<char*>(out32 + orow0 * D + 32 * c + 16 * half),
                         D * sizeof(float), wvalid);
          }
          continue;
        }
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack_bf16(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
        const uint4 v[4] = {make_uint4(w[0], w[1], w[2], w[3]), make_uint4(w[4], w[5], w[6], w[7]),
                            make_uint4(w[8], w[9], w[10], w[11]), make_uint4(w[12], w[13], w[14], w[15])};
        store_rows64(v, reinterpret_cast<char*>(out + orow0 * D + 32 * c), D * sizeof(uint16_t), wvalid);
      }
      tc_fence_before();
      mbar_arrive(bar(BAR_O_EMPTY));
      if (in && h == 0) p.a.lse[static_cast<size_t>(e_bh) * p.a.Nq + row] = e_m + log2f(e_l);
      e_it = -1;
      return true;
    };
    uint32_t sc = 0, pvc = 0;                     // S tiles consumed, PV groups done
    int it = 0;
    bool ok = true;
    for (int idx = blockIdx.x; idx < p.items && ok; idx += gridDim.x, ++it) {
      int bh, mt;
      item_coords(idx, p, bh, mt);
      const int J = kv_tiles(p, mt);
      const int row = mt * kBM + r;
      float m_used = -INFINITY, l = 0.f;
      for (int j = 0; j < J && ok; ++j) {
        const uint32_t b = sc & 1;
        ok = wwait(bar(BAR_S_FULL + b), (sc >> 1) & 1);
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[64];
        const uint32_t tS = tbase + lrow + b * 128;
        tmem_ld32(tS + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        tmem_ld32(tS + 64 * h + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        tmem_wait_ld();
        float* s = reinterpret_cast<float*>(sr);
        const int key0 = j * kBN + 64 * h;
        if (j * kBN + kBN > p.a.Nkv || (p.a.causal && j == mt)) {
          const int lim = p.a.causal ? min(p.a.Nkv - 1, row) : p.a.Nkv - 1;
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (key0 + i > lim) s[i] = -INFINITY;
        }
        float t = fmax3(s[0], s[1], s[2]);
#pragma unroll
        for (int i = 3; i < 63; i += 2) t = fmax3(t, s[i], s[i + 1]);
        t = fmaxf(t, s[63]);
        // exchange the tile maxima of the row; the barrier also orders both groups'
        // TMEM reads of S before either writes P over it
        xmax[(j & 1) * 256 + h * 128 + r] = t;
        if (!(ok = exchange())) break;
        const float t_other = xmax[(j & 1) * 256 + (h ^ 1) * 128 + r];
        const float tmax = fmaxf(t, t_other) * qk;
        float alpha = 1.f;
        bool resc = false;
        if (tmax > m_used + kRescaleThreshold) {
          if (j > 0) {
            resc = true;
            alpha = ex2(m_used - tmax);
          }
          m_used = tmax;
        }
        const float negm = -m_used;
        const TileScale ts = tile_scale(ex2(fmaf(t, qk, negm)));
        l *= alpha;
        float2 lsum = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t pq[16], ph[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 x = fma_rn_f32x2(make_float2(s[32 * c + 2 * i], s[32 * c + 2 * i + 1]),
                                          make_float2(qk, qk), make_float2(negm, negm));
            const float p0 = ex2(x.x), p1 = ex2(x.y);
            lsum = add_rn_f32x2(lsum, make_float2(p0, p1));
            ph[i] = pack_bf16(p0, p1);
            if (p.a.quant) {
              uint16_t cd;
              __nv_bfloat162 qv = quant_pair(p0, p1, ts, &cd);
              pq[i] = *reinterpret_cast<uint32_t*>(&qv);
            } else {
              pq[i] = ph[i];
            }
          }
          tmem_st16(tS + 32 * h + 16 * c, pq);
          tmem_st16(tS + 64 + 32 * h + 16 * c, ph);
        }
        l += lsum.x + lsum.y;
        tmem_wait_st();
        if (__any_sync(0xffffffffu, resc)) {
          // O must hold every PV issued so far before it is rescaled; group h rescales
          // O_q (h = 0) or O_hp (h = 1)
          ok = wwait(bar(BAR_O_DONE), (pvc - 1) & 1);
          if (!ok) break;
          tc_fence_after();
          const uint32_t tO = tbase + lrow + (h ? C::kTmemOhp : C::kTmemOq);
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + 32 * c, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tO + 32 * c, o);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(bar(BAR_P_FULL + b));
        ++sc;
        ++pvc;  // PV_j will be issued once every row has arrived
        if (kDefer && j == 0 && e_it >= 0 && !(ok = epilogue())) break;  // the previous item's
      }
      if (!ok) break;
      // ---------------------------------------------------------- end of item
      // the row sum over both groups; the epilogue now, or (kDefer) after the next
      // item's first P
      xsum[h * 128 + r] = l;
      if (!(ok = exchange())) break;
      e_l = xsum[r] + xsum[128 + r];
      e_m = m_used;
      e_bh = bh;
      e_mt = mt;
      e_it = it;
      if (!kDefer && !(ok = epilogue())) break;
    }
    if constexpr (kDefer) {
      if (ok && e_it >= 0) ok = epilogue();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

// ------------------------------------------------------------------ host side

template <int D>
cudaError_t launch_fwd_tc_d(const FwdArgs& a, unsigned int* err, int num_sms, cudaStream_t s) {
  using C = FwdTc<D>;
  const int BH = a.B * a.H;
  CUtensorMap mq, mk, mv;
  if (!make_bf16_map_3d(&mq, a.q, D, a.Nq, BH) ||
      !make_bf16_map_3d(&mk, a.k, D, a.Nkv, BH, a.kv_head_rows) ||
      !make_bf16_map_3d(&mv, a.v, D, a.Nkv, BH, a.kv_head_rows))
    return cudaErrorInvalidValue;
  TcParams p;
  p.a = a;
  p.err = err;
  p.mtiles = (a.Nq + kBM - 1) / kBM;
  p.items = BH * p.mtiles;
  // a causal item streams its head's K and V blocks
  p.hgroup = causal_head_group(4ll * a.Nkv * D, BH);
  // deferred epilogues for items of at most 8 key blocks (non-causal)
  const bool defer = !a.causal && a.Nkv <= 8 * kBN;
  auto kern = defer ? attn_fwd_tc_kernel<D, true> : attn_fwd_tc_kernel<D, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(C::kSmemBytes));
  if (e != cudaSuccess) return e;
  const int grid = p.items < num_sms ? p.items : num_sms;
  kern<<<grid, kThreads, C::kSmemBytes, s>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

}  // namespace

bool make_bf16_map_3d(CUtensorMap* m, const void* ptr, int D, int N, int BH, int head_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  if (head_rows < 0) head_rows = N;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(head_rows) * D * 2};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_ext_map_3d(CUtensorMap* m, const void* ptr, int N, int BH) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {16, static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {32, static_cast<cuuint64_t>(N) * 32};
  const cuuint32_t box[3] = {16, 128, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_fwd_tc(const FwdArgs& a, unsigned int* err, int num_sms, cudaStream_t s) {
  return a.D == 64 ? launch_fwd_tc_d<64>(a, err, num_sms, s)
                   : launch_fwd_tc_d<128>(a, err, num_sms, s);
}

}  // namespace qat
