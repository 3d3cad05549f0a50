// attn_bwd_mma.cu -- QAT attention backward (straight-through estimator) on warp-level
// mma.sync tensor-core ops.
//
// Gradients of L = <dO, O_hp>: quantization of P is the identity for the backward.
//   preprocess  ("attn_qat_train.py", _attn_bwd_preprocess): Delta_i = sum_d dO_id O_hp,id
//   dK/dV kernel (_attn_bwd_dkdv, _attn_bwd_dkdv_cross): one CTA per 64-key block,
//     looping over 64-row query blocks: S^T = K Q^T, P^T = exp2(S^T qk_scale - lse),
//     dP^T = V dO^T, dS^T = P^T o (dP^T - Delta); dV += P^T dO; dK += dS^T Q;
//     dK *= sm_scale at the end.
//   dQ kernel (_attn_bwd_dq, _attn_bwd_dq_cross): one CTA per 64-row query block,
//     looping over key blocks: dQ += dS K, dQ *= sm_scale at the end.
// P is rematerialized from Q, K and the saved base-2 lse ("support for pytorch
// autograd": the rematerialization trick of FlashAttention).
#include "qat_internal.h"
#include "qat_mma.cuh"

#include <math.h>

namespace qat {
namespace {

constexpr int kBlk = 64;
constexpr int kThreads = 128;

// ------------------------------------------------------------------ preprocess

template <int D>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const uint16_t* __restrict__ o,
                                                             const uint16_t* __restrict__ dO,
                                                             float* __restrict__ delta,
                                                             long long rows) {
  constexpr int PER = D / 32;  // elements per lane
  const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long r = warp; r < rows; r += nwarps) {
    const uint16_t* op = o + r * D + lane * PER;
    const uint16_t* dp = dO + r * D + lane * PER;
    float acc = 0.f;
    if constexpr (PER == 4) {
      const uint2 ov = *reinterpret_cast<const uint2*>(op);
      const uint2 dv = *reinterpret_cast<const uint2*>(dp);
      const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
      const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&dv);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float2 of = __bfloat1622float2(o2[i]);
        const float2 df = __bfloat1622float2(d2[i]);
        acc = fmaf(of.x, df.x, acc);
        acc = fmaf(of.y, df.y, acc);
      }
    } else {
      const uint32_t ov = *reinterpret_cast<const uint32_t*>(op);
      const uint32_t dv = *reinterpret_cast<const uint32_t*>(dp);
      const float2 of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ov));
      const float2 df = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&dv));
      acc = fmaf(of.x, df.x, of.y * df.y);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) delta[r] = acc;
  }
}

// ------------------------------------------------------------------ dK / dV

template <int D>
struct BwdSmem {
  static constexpr int LD = D + 8;
  static constexpr size_t bytes = sizeof(uint16_t) * 4 * kBlk * LD + sizeof(float) * 2 * kBlk;
};

template <int D>
__global__ void __launch_bounds__(kThreads) attn_bwd_dkdv_mma_kernel(const BwdArgs a) {
  constexpr int LD = BwdSmem<D>::LD;
  constexpr int KS = D / 16;
  constexpr int DT = D / 8;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint16_t* sK = reinterpret_cast<uint16_t*>(smem_raw);
  uint16_t* sV = sK + kBlk * LD;
  uint16_t* sQ = sV + kBlk * LD;
  uint16_t* sdO = sQ + kBlk * LD;
  float* sLse = reinterpret_cast<float*>(sdO + kBlk * LD);
  float* sDelta = sLse + kBlk;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int n0 = blockIdx.x * kBlk;
  const size_t bh = blockIdx.y;
  const uint16_t* Qh = a.q + bh * a.Nq * D;
  const uint16_t* dOh = a.dO + bh * a.Nq * D;
  const float* lse_h = a.lse + bh * a.Nq;
  const float* delta_h = a.delta + bh * a.Nq;

  load_rows<kBlk, D, LD, kThreads>(sK, a.k + bh * a.Nkv * D, n0, a.Nkv, tid);
  load_rows<kBlk, D, LD, kThreads>(sV, a.v + bh * a.Nkv * D, n0, a.Nkv, tid);

  const int lr = warp * 16 + g;               // local key row of elements 0,1
  const int key_a = n0 + lr, key_b = key_a + 8;

  float dk[DT][4], dv[DT][4];
#pragma unroll
  for (int i = 0; i < DT; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) dk[i][e] = dv[i][e] = 0.f;

  const int m_start = a.causal ? n0 : 0;  // causal: queries i >= key j only
  for (int m0 = m_start; m0 < a.Nq; m0 += kBlk) {
    __syncthreads();
    load_rows<kBlk, D, LD, kThreads>(sQ, Qh, m0, a.Nq, tid);
    load_rows<kBlk, D, LD, kThreads>(sdO, dOh, m0, a.Nq, tid);
    if (tid < kBlk) {
      const bool in = m0 + tid < a.Nq;
      sLse[tid] = in ? lse_h[m0 + tid] : 0.f;
      sDelta[tid] = in ? delta_h[m0 + tid] : 0.f;
    }
    __syncthreads();

    // S^T = K Q^T and dP^T = V dO^T (16 keys x 64 queries per warp)
    float st[8][4], dpt[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) st[nt][e] = dpt[nt][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t kf[4], vf[4];
      kf[0] = ld_s32(sK + lr * LD + ks * 16 + 2 * c);
      kf[1] = ld_s32(sK + (lr + 8) * LD + ks * 16 + 2 * c);
      kf[2] = ld_s32(sK + lr * LD + ks * 16 + 8 + 2 * c);
      kf[3] = ld_s32(sK + (lr + 8) * LD + ks * 16 + 8 + 2 * c);
      vf[0] = ld_s32(sV + lr * LD + ks * 16 + 2 * c);
      vf[1] = ld_s32(sV + (lr + 8) * LD + ks * 16 + 2 * c);
      vf[2] = ld_s32(sV + lr * LD + ks * 16 + 8 + 2 * c);
      vf[3] = ld_s32(sV + (lr + 8) * LD + ks * 16 + 8 + 2 * c);
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const uint16_t* qr = sQ + (nt * 8 + g) * LD + ks * 16 + 2 * c;
        mma_16816(st[nt], kf, ld_s32(qr), ld_s32(qr + 8));
        const uint16_t* dr = sdO + (nt * 8 + g) * LD + ks * 16 + 2 * c;
        mma_16816(dpt[nt], vf, ld_s32(dr), ld_s32(dr + 8));
      }
    }

    // P^T and dS^T
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int ql = nt * 8 + 2 * c + (e & 1);
        const int i = m0 + ql;
        const int j = (e < 2) ? key_a : key_b;
        const bool ok = (i < a.Nq) && (j < a.Nkv) && (!a.causal || j <= i);
        const float p = ok ? fast_exp2(st[nt][e] * a.qk_scale - sLse[ql]) : 0.f;
        st[nt][e] = p;
        dpt[nt][e] = p * (dpt[nt][e] - sDelta[ql]);
      }

    // dV += P^T dO ; dK += dS^T Q   (k = 16 queries per step)
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4], sa[4];
      pa[0] = pack_bf16_rn(st[2 * kk][0], st[2 * kk][1]);
      pa[1] = pack_bf16_rn(st[2 * kk][2], st[2 * kk][3]);
      pa[2] = pack_bf16_rn(st[2 * kk + 1][0], st[2 * kk + 1][1]);
      pa[3] = pack_bf16_rn(st[2 * kk + 1][2], st[2 * kk + 1][3]);
      sa[0] = pack_bf16_rn(dpt[2 * kk][0], dpt[2 * kk][1]);
      sa[1] = pack_bf16_rn(dpt[2 * kk][2], dpt[2 * kk][3]);
      sa[2] = pack_bf16_rn(dpt[2 * kk + 1][0], dpt[2 * kk + 1][1]);
      sa[3] = pack_bf16_rn(dpt[2 * kk + 1][2], dpt[2 * kk + 1][3]);
      const uint16_t* do0 = sdO + (kk * 16 + 2 * c) * LD + g;
      const uint16_t* q0 = sQ + (kk * 16 + 2 * c) * LD + g;
#pragma unroll
      for (int dt = 0; dt < DT; ++dt) {
        const uint16_t* dp = do0 + dt * 8;
        mma_16816(dv[dt], pa, pack_u16(dp[0], dp[LD]), pack_u16(dp[8 * LD], dp[9 * LD]));
        const uint16_t* qp = q0 + dt * 8;
        mma_16816(dk[dt], sa, pack_u16(qp[0], qp[LD]), pack_u16(qp[8 * LD], qp[9 * LD]));
      }
    }
  }

  const size_t kvbase = bh * static_cast<size_t>(a.Nkv) * D;
#pragma unroll
  for (int dt = 0; dt < DT; ++dt) {
    const int col = dt * 8 + 2 * c;
    if (key_a < a.Nkv) {
      *reinterpret_cast<uint32_t*>(a.dv + kvbase + static_cast<size_t>(key_a) * D + col) =
          pack_bf16_rn(dv[dt][0], dv[dt][1]);
      *reinterpret_cast<uint32_t*>(a.dk + kvbase + static_cast<size_t>(key_a) * D + col) =
          pack_bf16_rn(dk[dt][0] * a.sm_scale, dk[dt][1] * a.sm_scale);
    }
    if (key_b < a.Nkv) {
      *reinterpret_cast<uint32_t*>(a.dv + kvbase + static_cast<size_t>(key_b) * D + col) =
          pack_bf16_rn(dv[dt][2], dv[dt][3]);
      *reinterpret_cast<uint32_t*>(a.dk + kvbase + static_cast<size_t>(key_b) * D + col) =
          pack_bf16_rn(dk[dt][2] * a.sm_scale, dk[dt][3] * a.sm_scale);
    }
  }
}

// ------------------------------------------------------------------ dQ

template <int D>
__global__ void __launch_bounds__(kThreads) attn_bwd_dq_mma_kernel(const BwdArgs a) {
  constexpr int LD = BwdSmem<D>::LD;
  constexpr int KS = D / 16;
  constexpr int DT = D / 8;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint16_t* sQ = reinterpret_cast<uint16_t*>(smem_raw);
  uint16_t* sdO = sQ + kBlk * LD;
  uint16_t* sK = sdO + kBlk * LD;
  uint16_t* sV = sK + kBlk * LD;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int m0 = blockIdx.x * kBlk;
  const size_t bh = blockIdx.y;
  const uint16_t* Kh = a.k + bh * a.Nkv * D;
  const uint16_t* Vh = a.v + bh * a.Nkv * D;

  load_rows<kBlk, D, LD, kThreads>(sQ, a.q + bh * a.Nq * D, m0, a.Nq, tid);
  load_rows<kBlk, D, LD, kThreads>(sdO, a.dO + bh * a.Nq * D, m0, a.Nq, tid);

  const int lr = warp * 16 + g;
  const int row_a = m0 + lr, row_b = row_a + 8;
  const float lse_a = row_a < a.Nq ? a.lse[bh * a.Nq + row_a] : 0.f;
  const float lse_b = row_b < a.Nq ? a.lse[bh * a.Nq + row_b] : 0.f;
  const float del_a = row_a < a.Nq ? a.delta[bh * a.Nq + row_a] : 0.f;
  const float del_b = row_b < a.Nq ? a.delta[bh * a.Nq + row_b] : 0.f;

  float dq[DT][4];
#pragma unroll
  for (int i = 0; i < DT; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) dq[i][e] = 0.f;

  const int n_end = a.causal ? min(a.Nkv, m0 + kBlk) : a.Nkv;
  for (int n0 = 0; n0 < n_end; n0 += kBlk) {
    __syncthreads();
    load_rows<kBlk, D, LD, kThreads>(sK, Kh, n0, a.Nkv, tid);
    load_rows<kBlk, D, LD, kThreads>(sV, Vh, n0, a.Nkv, tid);
    __syncthreads();

    float s[8][4], dp[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[nt][e] = dp[nt][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t qf[4], df[4];
      qf[0] = ld_s32(sQ + lr * LD + ks * 16 + 2 * c);
      qf[1] = ld_s32(sQ + (lr + 8) * LD + ks * 16 + 2 * c);
      qf[2] = ld_s32(sQ + lr * LD + ks * 16 + 8 + 2 * c);
      qf[3] = ld_s32(sQ + (lr + 8) * LD + ks * 16 + 8 + 2 * c);
      df[0] = ld_s32(sdO + lr * LD + ks * 16 + 2 * c);
      df[1] = ld_s32(sdO + (lr + 8) * LD + ks * 16 + 2 * c);
      df[2] = ld_s32(sdO + lr * LD + ks * 16 + 8 + 2 * c);
      df[3] = ld_s32(sdO + (lr + 8) * LD + ks * 16 + 8 + 2 * c);
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const uint16_t* kr = sK + (nt * 8 + g) * LD + ks * 16 + 2 * c;
        mma_16816(s[nt], qf, ld_s32(kr), ld_s32(kr + 8));
        const uint16_t* vr = sV + (nt * 8 + g) * LD + ks * 16 + 2 * c;
        mma_16816(dp[nt], df, ld_s32(vr), ld_s32(vr + 8));
      }
    }

#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = n0 + nt * 8 + 2 * c + (e & 1);
        const int i = (e < 2) ? row_a : row_b;
        const bool ok = (j < a.Nkv) && (i < a.Nq) && (!a.causal || j <= i);
        const float p = ok ? fast_exp2(s[nt][e] * a.qk_scale - ((e < 2) ? lse_a : lse_b)) : 0.f;
        s[nt][e] = p * (dp[nt][e] - ((e < 2) ? del_a : del_b));  // dS
      }

#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t sa[4];
      sa[0] = pack_bf16_rn(s[2 * kk][0], s[2 * kk][1]);
      sa[1] = pack_bf16_rn(s[2 * kk][2], s[2 * kk][3]);
      sa[2] = pack_bf16_rn(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      sa[3] = pack_bf16_rn(s[2 * kk + 1][2], s[2 * kk + 1][3]);
      const uint16_t* k0 = sK + (kk * 16 + 2 * c) * LD + g;
#pragma unroll
      for (int dt = 0; dt < DT; ++dt) {
        const uint16_t* kp = k0 + dt * 8;
        mma_16816(dq[dt], sa, pack_u16(kp[0], kp[LD]), pack_u16(kp[8 * LD], kp[9 * LD]));
      }
    }
  }

  const size_t qbase = bh * static_cast<size_t>(a.Nq) * D;
#pragma unroll
  for (int dt = 0; dt < DT; ++dt) {
    const int col = dt * 8 + 2 * c;
    if (row_a < a.Nq)
      *reinterpret_cast<uint32_t*>(a.dq + qbase + static_cast<size_t>(row_a) * D + col) =
          pack_bf16_rn(dq[dt][0] * a.sm_scale, dq[dt][1] * a.sm_scale);
    if (row_b < a.Nq)
      *reinterpret_cast<uint32_t*>(a.dq + qbase + static_cast<size_t>(row_b) * D + col) =
          pack_bf16_rn(dq[dt][2] * a.sm_scale, dq[dt][3] * a.sm_scale);
  }
}

template <int D>
cudaError_t launch_bwd_mma_d(const BwdArgs& a, cudaStream_t s) {
  const size_t smem = BwdSmem<D>::bytes;
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_dkdv_mma_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_bwd_dq_mma_kernel<D>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const dim3 grid_kv((a.Nkv + kBlk - 1) / kBlk, a.B * a.H);
  attn_bwd_dkdv_mma_kernel<D><<<grid_kv, kThreads, smem, s>>>(a);
  if (a.Nq > 0) {
    const dim3 grid_q((a.Nq + kBlk - 1) / kBlk, a.B * a.H);
    attn_bwd_dq_mma_kernel<D><<<grid_q, kThreads, smem, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_preprocess(const BwdArgs& a, cudaStream_t s) {
  const long long rows = static_cast<long long>(a.B) * a.H * a.Nq;
  if (rows == 0) return cudaSuccess;
  long long blocks = (rows + 7) / 8;
  if (blocks > 152 * 64) blocks = 152 * 64;
  if (a.D == 64)
    bwd_preprocess_kernel<64><<<static_cast<unsigned>(blocks), 256, 0, s>>>(a.o_hp, a.dO, a.delta, rows);
  else
    bwd_preprocess_kernel<128><<<static_cast<unsigned>(blocks), 256, 0, s>>>(a.o_hp, a.dO, a.delta, rows);
  return cudaGetLastError();
}

cudaError_t launch_bwd_mma(const BwdArgs& a, cudaStream_t s) {
  return a.D == 64 ? launch_bwd_mma_d<64>(a, s) : launch_bwd_mma_d<128>(a, s);
}

}  // namespace qat
