// attn_merge.cu -- merge of two partial attention results over disjoint key sets:
//   lse = log2(2^lse_a + 2^lse_b),   O = 2^(lse_a - lse) O_a + 2^(lse_b - lse) O_b
// for both O_q and O_hp (exact for O_q when every key chunk starts at a multiple of 64,
// so that no quantization tile is split).  The accumulator (a) is updated in place; the
// merged outputs can also be written as bf16.  One warp per query row; HBM-bound.
#include "qat_internal.h"

#include <cuda_bf16.h>
#include <math.h>

namespace qat {
namespace {

template <int D>
__global__ void __launch_bounds__(256) merge_kernel(float* __restrict__ oq_a, float* __restrict__ oh_a,
                                                    float* __restrict__ lse_a,
                                                    const float* __restrict__ oq_b,
                                                    const float* __restrict__ oh_b,
                                                    const float* __restrict__ lse_b,
                                                    uint16_t* __restrict__ oq_out,
                                                    uint16_t* __restrict__ oh_out, long long rows) {
  constexpr int PER = D / 32;
  const long long w0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const int lane = threadIdx.x & 31;
  for (long long r = w0; r < rows; r += nw) {
    const float la = lse_a[r], lb = lse_b[r];
    float hi = fmaxf(la, lb);
    if (hi == -INFINITY) hi = 0.f;  // both empty: weights 0, output left as 0
    const float wa = exp2f(la - hi), wb = exp2f(lb - hi);
    const float tot = wa + wb;
    const float ca = tot > 0.f ? wa / tot : 0.f, cb = tot > 0.f ? wb / tot : 0.f;
    const size_t off = static_cast<size_t>(r) * D + lane * PER;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      float* a = t ? oh_a : oq_a;
      const float* b = t ? oh_b : oq_b;
      uint16_t* out = t ? oh_out : oq_out;
      float m[PER];
      if constexpr (PER == 4) {
        const float4 x = *reinterpret_cast<const float4*>(a + off);
        const float4 y = *reinterpret_cast<const float4*>(b + off);
        m[0] = ca * x.x + cb * y.x;
        m[1] = ca * x.y + cb * y.y;
        m[2] = ca * x.z + cb * y.z;
        m[3] = ca * x.w + cb * y.w;
        *reinterpret_cast<float4*>(a + off) = make_float4(m[0], m[1], m[2], m[3]);
      } else {
        const float2 x = *reinterpret_cast<const float2*>(a + off);
        const float2 y = *reinterpret_cast<const float2*>(b + off);
        m[0] = ca * x.x + cb * y.x;
        m[1] = ca * x.y + cb * y.y;
        *reinterpret_cast<float2*>(a + off) = make_float2(m[0], m[1]);
      }
      if (out != nullptr) {
#pragma unroll
        for (int i = 0; i < PER; i += 2) {
          __nv_bfloat162 v = __floats2bfloat162_rn(m[i], m[i + 1]);
          *reinterpret_cast<__nv_bfloat162*>(out + off + i) = v;
        }
      }
    }
    if (lane == 0) lse_a[r] = (tot > 0.f) ? hi + log2f(tot) : -INFINITY;
  }
}

}  // namespace

cudaError_t launch_merge(float* o_q_acc, float* o_hp_acc, float* lse_acc, const float* o_q_part,
                         const float* o_hp_part, const float* lse_part, uint16_t* o_q_out,
                         uint16_t* o_hp_out, long long rows, int D, int num_sms, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  long long blocks = (rows + 7) / 8;
  if (blocks > static_cast<long long>(num_sms) * 64) blocks = static_cast<long long>(num_sms) * 64;
  if (D == 64)
    merge_kernel<64><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        o_q_acc, o_hp_acc, lse_acc, o_q_part, o_hp_part, lse_part, o_q_out, o_hp_out, rows);
  else
    merge_kernel<128><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        o_q_acc, o_hp_acc, lse_acc, o_q_part, o_hp_part, lse_part, o_q_out, o_hp_out, rows);
  return cudaGetLastError();
}

}  // namespace qat
