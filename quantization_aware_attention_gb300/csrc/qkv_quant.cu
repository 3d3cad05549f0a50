// qkv_quant.cu -- the page's IS_QAT input path: fake quantization of Q, K and V per
// (head, 32-token block) to FP8 E4M3 with an absmax scale, and smooth_k's per-channel
// mean of K over batch, heads and tokens, and that mean's subtraction alone.
//
// Sources ("attn_qat_train.py", _attention.forward): fake_quantize_q / fake_quantize_kv
// run one program per 32-token block of one (batch, head); smooth_k subtracts
// k.mean(dim=(0, 1, 2)) first.  quant_utils is not on the pages; the rule implemented
// is the library's per-tile rule (qat_quant.cuh) applied to each 32-token x D block:
//   x' = fl32(x - mean_c)  (when a mean is given),  amax = max |x'| over the block,
//   code = E4M3_RNE_SATFINITE(fl32(x' * fl32(448 / amax))),
//   out = bf16_RN(fl32(decode(code) * fl32(amax / 448))).
// Both kernels are HBM-bound elementwise passes.
#include "qat_internal.h"
#include "qat_quant.cuh"

#include <cuda_bf16.h>

namespace qat {
namespace {

constexpr int kTokBlk = 32;
constexpr int kThreads = 128;

// Sum over rows of a [rows, D] bf16 matrix into fp32 sums[D] (atomics; zeroed by the
// launcher).  16 threads cover one row (8 channels each for D = 128, 4 for D = 64).
template <int D>
__global__ void __launch_bounds__(256) channel_sum_kernel(const uint16_t* __restrict__ x,
                                                          float* __restrict__ sums,
                                                          long long rows) {
  constexpr int PER = D / 16;          // channels per thread
  __shared__ float part[16][D];
  const int t = threadIdx.x & 15;      // channel group
  const int rsub = threadIdx.x >> 4;   // row within the 16 rows of one step
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  for (long long r = static_cast<long long>(blockIdx.x) * 16 + rsub; r < rows;
       r += static_cast<long long>(gridDim.x) * 16) {
    const uint16_t* src = x + r * D + t * PER;
    if constexpr (PER == 8) {
      const uint4 v = *reinterpret_cast<const uint4*>(src);
      const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(b[i]);
        acc[2 * i] += f.x;
        acc[2 * i + 1] += f.y;
      }
    } else {
      const uint2 v = *reinterpret_cast<const uint2*>(src);
      const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float2 f = __bfloat1622float2(b[i]);
        acc[2 * i] += f.x;
        acc[2 * i + 1] += f.y;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < PER; ++i) part[rsub][t * PER + i] = acc[i];
  __syncthreads();
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float s = 0.f;
#pragma unroll
    for (int rr = 0; rr < 16; ++rr) s += part[rr][c];
    atomicAdd(sums + c, s);
  }
}

__global__ void scale_kernel(float* v, int n, float s) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) v[i] *= s;
}

// One CTA per (head, 32-token block): amax over the block, then every element coded.
template <int D>
__global__ void __launch_bounds__(kThreads) fake_quant_tokens_kernel(
    const uint16_t* __restrict__ x, const float* __restrict__ mean, uint16_t* __restrict__ out,
    float* __restrict__ scales, int N, int nblk) {
  constexpr int CH = kTokBlk * D / 8;        // 16-byte chunks per block
  constexpr int PERT = CH / kThreads;        // chunks per thread (4 for D=128, 2 for D=64)
  __shared__ float red[kThreads / 32];
  const long long bh = blockIdx.x / nblk;
  const int blk = blockIdx.x % nblk;
  const int tok0 = blk * kTokBlk;
  const size_t base = (static_cast<size_t>(bh) * N + tok0) * D;
  float v[PERT][8];
  bool in[PERT];
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < PERT; ++k) {
    const int ch = threadIdx.x + k * kThreads;
    const int tok = ch / (D / 8), col = (ch % (D / 8)) * 8;
    in[k] = tok0 + tok < N;
    uint4 raw = make_uint4(0u, 0u, 0u, 0u);
    if (in[k]) raw = *reinterpret_cast<const uint4*>(x + base + static_cast<size_t>(tok) * D + col);
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(b[i]);
      v[k][2 * i] = f.x;
      v[k][2 * i + 1] = f.y;
    }
    if (mean != nullptr) {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[k][i] = __fsub_rn(v[k][i], mean[col + i]);
    }
    if (in[k]) {
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[k][i]));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) amax = fmaxf(amax, red[w]);
  const TileScale ts = tile_scale(amax);
  if (scales != nullptr && threadIdx.x == 0) scales[blockIdx.x] = ts.scale;
#pragma unroll
  for (int k = 0; k < PERT; ++k) {
    if (!in[k]) continue;
    const int ch = threadIdx.x + k * kThreads;
    const int tok = ch / (D / 8), col = (ch % (D / 8)) * 8;
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint16_t cd;
      __nv_bfloat162 q = quant_pair(v[k][2 * i], v[k][2 * i + 1], ts, &cd);
      w[i] = *reinterpret_cast<uint32_t*>(&q);
    }
    *reinterpret_cast<uint4*>(out + base + static_cast<size_t>(tok) * D + col) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// out = bf16_RN(fl32(x - mean_c)) for every element of a [rows, D] bf16 matrix: smooth_k's
// subtraction without the quantization, for the page's backward on unquantized inputs
// (use_qat_qkv_backward = False).  One thread per 8 elements (16-byte loads and stores).
template <int D>
__global__ void __launch_bounds__(256) subtract_mean_kernel(const uint16_t* __restrict__ x,
                                                            const float* __restrict__ mean,
                                                            uint16_t* __restrict__ out,
                                                            long long n8) {
  for (long long i = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x; i < n8;
       i += static_cast<long long>(gridDim.x) * 256) {
    const int col = static_cast<int>(i % (D / 8)) * 8;
    const uint4 raw = *reinterpret_cast<const uint4*>(x + i * 8);
    const float4 m0 = *reinterpret_cast<const float4*>(mean + col);
    const float4 m1 = *reinterpret_cast<const float4*>(mean + col + 4);
    const float mm[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&raw);
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(b[k]);
      __nv_bfloat162 r = __floats2bfloat162_rn(__fsub_rn(f.x, mm[2 * k]), __fsub_rn(f.y, mm[2 * k + 1]));
      w[k] = *reinterpret_cast<uint32_t*>(&r);
    }
    *reinterpret_cast<uint4*>(out + i * 8) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace

cudaError_t launch_subtract_mean(const uint16_t* x, const float* mean, uint16_t* out,
                                 long long rows, int D, int num_sms, cudaStream_t s) {
  const long long n8 = rows * D / 8;
  long long blocks = (n8 + 255) / 256;
  if (blocks > static_cast<long long>(num_sms) * 32) blocks = static_cast<long long>(num_sms) * 32;
  if (blocks == 0) return cudaSuccess;
  if (D == 64)
    subtract_mean_kernel<64><<<static_cast<unsigned>(blocks), 256, 0, s>>>(x, mean, out, n8);
  else
    subtract_mean_kernel<128><<<static_cast<unsigned>(blocks), 256, 0, s>>>(x, mean, out, n8);
  return cudaGetLastError();
}

cudaError_t launch_channel_mean(const uint16_t* x, float* mean, long long rows, int D,
                                int num_sms, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(mean, 0, sizeof(float) * D, s);
  if (e != cudaSuccess || rows == 0) return e;
  long long blocks = (rows + 15) / 16;
  if (blocks > static_cast<long long>(num_sms) * 8) blocks = static_cast<long long>(num_sms) * 8;
  if (D == 64)
    channel_sum_kernel<64><<<static_cast<unsigned>(blocks), 256, 0, s>>>(x, mean, rows);
  else
    channel_sum_kernel<128><<<static_cast<unsigned>(blocks), 256, 0, s>>>(x, mean, rows);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  scale_kernel<<<1, 128, 0, s>>>(mean, D, static_cast<float>(1.0 / static_cast<double>(rows)));
  return cudaGetLastError();
}

cudaError_t launch_fake_quant_tokens(const uint16_t* x, const float* mean, uint16_t* out,
                                     float* scales, int BH, int N, int D, cudaStream_t s) {
  const int nblk = (N + kTokBlk - 1) / kTokBlk;
  const long long grid = static_cast<long long>(BH) * nblk;
  if (grid == 0) return cudaSuccess;
  if (D == 64)
    fake_quant_tokens_kernel<64><<<static_cast<unsigned>(grid), kThreads, 0, s>>>(x, mean, out,
                                                                                  scales, N, nblk);
  else
    fake_quant_tokens_kernel<128><<<static_cast<unsigned>(grid), kThreads, 0, s>>>(x, mean, out,
                                                                                   scales, N, nblk);
  return cudaGetLastError();
}

}  // namespace qat
