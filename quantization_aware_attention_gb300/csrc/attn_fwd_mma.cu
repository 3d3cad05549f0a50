// attn_fwd_mma.cu -- QAT attention forward on warp-level mma.sync tensor-core ops.
//
// One CTA = 4 warps = 64 query rows of one (b, h); each warp owns 16 rows and streams
// 64-key tiles of K and V (one tile = one quantization tile, aligned at key 0).
// Per tile ("attn_qat_train.py", _attn_fwd_inner):
//   S = Q K^T; x = S * qk_scale (masked keys -> -inf); m' = max(m, rowmax x);
//   p = exp2(x - m'); alpha = exp2(m - m'); l = alpha l + rowsum p (unquantized p);
//   amax = rowmax p over the tile; Pq = quant(p) per the per-tile rule;
//   O_q = alpha O_q + Pq V;  O_hp = alpha O_hp + bf16(p) V.
// Epilogue (_attn_fwd): O_q / l, O_hp / l stored as bf16, lse = m + log2 l.
// The quantized code depends only on p / amax, so quantizing relative to the running
// max gives the same codes as relative to the final max, up to fp32 rounding.
#include "qat_internal.h"
#include "qat_mma.cuh"
#include "qat_quant.cuh"

#include <math.h>

namespace qat {
namespace {

constexpr int kBM = 64;   // query rows per CTA
constexpr int kBN = 64;   // keys per tile (= quantization tile)
constexpr int kThreads = 128;

template <int D>
struct FwdSmem {
  static constexpr int LD = D + 8;  // padded row stride, keeps fragment loads conflict-light
  static constexpr size_t bytes = sizeof(uint16_t) * (kBM + 2 * kBN) * LD;
};

template <int D>
__global__ void __launch_bounds__(kThreads) attn_fwd_mma_kernel(const FwdArgs a) {
  constexpr int LD = FwdSmem<D>::LD;
  constexpr int KS = D / 16;  // k-steps over the head dimension
  constexpr int DT = D / 8;   // 8-wide output column tiles
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint16_t* sQ = reinterpret_cast<uint16_t*>(smem_raw);
  uint16_t* sK = sQ + kBM * LD;
  uint16_t* sV = sK + kBN * LD;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int m0 = blockIdx.x * kBM;
  const size_t bh = blockIdx.y;
  const uint16_t* Qh = a.q + bh * a.Nq * D;
  const uint16_t* Kh = a.k + bh * a.Nkv * D;
  const uint16_t* Vh = a.v + bh * a.Nkv * D;

  load_rows<kBM, D, LD, kThreads>(sQ, Qh, m0, a.Nq, tid);

  const int lr = warp * 16 + g;             // local row of accumulator elements 0,1
  const int row_a = m0 + lr, row_b = row_a + 8;

  float oq[DT][4], oh[DT][4];
#pragma unroll
  for (int i = 0; i < DT; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) oq[i][e] = oh[i][e] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};

  const int n_end = a.causal ? min(a.Nkv, m0 + kBM) : a.Nkv;
  for (int n0 = 0; n0 < n_end; n0 += kBN) {
    __syncthreads();  // previous K/V tile fully consumed (and Q stored on entry)
    load_rows<kBN, D, LD, kThreads>(sK, Kh, n0, a.Nkv, tid);
    load_rows<kBN, D, LD, kThreads>(sV, Vh, n0, a.Nkv, tid);
    __syncthreads();

    // ---- S = Q K^T (16 rows x 64 keys per warp)
    float s[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t af[4];
      af[0] = ld_s32(sQ + lr * LD + ks * 16 + 2 * c);
      af[1] = ld_s32(sQ + (lr + 8) * LD + ks * 16 + 2 * c);
      af[2] = ld_s32(sQ + lr * LD + ks * 16 + 8 + 2 * c);
      af[3] = ld_s32(sQ + (lr + 8) * LD + ks * 16 + 8 + 2 * c);
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const uint16_t* kr = sK + (nt * 8 + g) * LD + ks * 16 + 2 * c;
        mma_16816(s[nt], af, ld_s32(kr), ld_s32(kr + 8));
      }
    }

    // ---- scale, mask, running max
    float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = n0 + nt * 8 + 2 * c + (e & 1);
        const int i = (e < 2) ? row_a : row_b;
        const bool ok = (j < a.Nkv) && (!a.causal || j <= i);
        const float x = ok ? s[nt][e] * a.qk_scale : -INFINITY;
        s[nt][e] = x;
        tmax[e >> 1] = fmaxf(tmax[e >> 1], x);
      }
    float alpha[2], m_use[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float m_new = fmaxf(m_run[r], quad_max(tmax[r]));
      m_use[r] = (m_new == -INFINITY) ? 0.f : m_new;
      alpha[r] = fast_exp2(m_run[r] - m_use[r]);
      m_run[r] = m_new;
    }

    // ---- p = exp2(x - m), row sums (unquantized) and per-tile amax
    float rsum[2] = {0.f, 0.f}, amax[2] = {0.f, 0.f};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p = fast_exp2(s[nt][e] - m_use[e >> 1]);
        s[nt][e] = p;
        rsum[e >> 1] += p;
        amax[e >> 1] = fmaxf(amax[e >> 1], p);
      }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      l_run[r] = l_run[r] * alpha[r] + quad_sum(rsum[r]);
      amax[r] = quad_max(amax[r]);
    }

    // ---- A fragments: quantized and high-precision P (k = 16 keys per fragment)
    uint32_t aq[4][4], ah[4][4];
    const TileScale ts0 = tile_scale(amax[0]);
    const TileScale ts1 = tile_scale(amax[1]);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const float* lo = s[2 * kk];
      const float* hi = s[2 * kk + 1];
      ah[kk][0] = pack_bf16_rn(lo[0], lo[1]);
      ah[kk][1] = pack_bf16_rn(lo[2], lo[3]);
      ah[kk][2] = pack_bf16_rn(hi[0], hi[1]);
      ah[kk][3] = pack_bf16_rn(hi[2], hi[3]);
      if (a.quant) {
        uint16_t cd;
        aq[kk][0] = bf162_bits(quant_pair(lo[0], lo[1], ts0, &cd));
        aq[kk][1] = bf162_bits(quant_pair(lo[2], lo[3], ts1, &cd));
        aq[kk][2] = bf162_bits(quant_pair(hi[0], hi[1], ts0, &cd));
        aq[kk][3] = bf162_bits(quant_pair(hi[2], hi[3], ts1, &cd));
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) aq[kk][e] = ah[kk][e];
      }
    }

    // ---- rescale and accumulate both outputs with the shared V tile
#pragma unroll
    for (int dt = 0; dt < DT; ++dt) {
      oq[dt][0] *= alpha[0]; oq[dt][1] *= alpha[0];
      oq[dt][2] *= alpha[1]; oq[dt][3] *= alpha[1];
      oh[dt][0] *= alpha[0]; oh[dt][1] *= alpha[0];
      oh[dt][2] *= alpha[1]; oh[dt][3] *= alpha[1];
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint16_t* v0 = sV + (kk * 16 + 2 * c) * LD + g;
#pragma unroll
      for (int dt = 0; dt < DT; ++dt) {
        const uint16_t* vp = v0 + dt * 8;
        const uint32_t b0 = pack_u16(vp[0], vp[LD]);
        const uint32_t b1 = pack_u16(vp[8 * LD], vp[9 * LD]);
        mma_16816(oq[dt], aq[kk], b0, b1);
        mma_16816(oh[dt], ah[kk], b0, b1);
      }
    }
  }

  // ---- epilogue
  const size_t obase = bh * static_cast<size_t>(a.Nq) * D;
  const float inv0 = l_run[0] > 0.f ? 1.0f / l_run[0] : 0.f;
  const float inv1 = l_run[1] > 0.f ? 1.0f / l_run[1] : 0.f;
#pragma unroll
  for (int dt = 0; dt < DT; ++dt) {
    const int col = dt * 8 + 2 * c;
    if (row_a < a.Nq) {
      *reinterpret_cast<uint32_t*>(a.o_q + obase + static_cast<size_t>(row_a) * D + col) =
          pack_bf16_rn(oq[dt][0] * inv0, oq[dt][1] * inv0);
      *reinterpret_cast<uint32_t*>(a.o_hp + obase + static_cast<size_t>(row_a) * D + col) =
          pack_bf16_rn(oh[dt][0] * inv0, oh[dt][1] * inv0);
    }
    if (row_b < a.Nq) {
      *reinterpret_cast<uint32_t*>(a.o_q + obase + static_cast<size_t>(row_b) * D + col) =
          pack_bf16_rn(oq[dt][2] * inv1, oq[dt][3] * inv1);
      *reinterpret_cast<uint32_t*>(a.o_hp + obase + static_cast<size_t>(row_b) * D + col) =
          pack_bf16_rn(oh[dt][2] * inv1, oh[dt][3] * inv1);
    }
  }
  if (c == 0) {
    if (row_a < a.Nq) a.lse[bh * a.Nq + row_a] = m_run[0] + log2f(l_run[0]);
    if (row_b < a.Nq) a.lse[bh * a.Nq + row_b] = m_run[1] + log2f(l_run[1]);
  }
}

template <int D>
cudaError_t launch_fwd_mma_d(const FwdArgs& a, cudaStream_t s) {
  const size_t smem = FwdSmem<D>::bytes;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_mma_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const dim3 grid((a.Nq + kBM - 1) / kBM, a.B * a.H);
  attn_fwd_mma_kernel<D><<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_mma(const FwdArgs& a, cudaStream_t s) {
  return a.D == 64 ? launch_fwd_mma_d<64>(a, s) : launch_fwd_mma_d<128>(a, s);
}

}  // namespace qat
