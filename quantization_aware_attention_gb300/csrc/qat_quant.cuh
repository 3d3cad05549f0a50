// qat_quant.cuh -- the per-tile FP8 E4M3 fake-quantization rule applied to softmax
// probabilities, shared by every kernel of the library and its debug entry point.
//
// Rule for one query row x one 64-key tile of fp32 probabilities p (all >= 0):
//   amax = max_j p_j;  if amax == 0 the tile quantizes to zeros with scale 0;
//   inv = RN(448 / amax), scale = RN(amax / 448)            (IEEE division)
//   code_j = E4M3 round-to-nearest-even, saturating (RN(p_j * inv))
//   value_j = bf16_RN(RN(decode(code_j) * scale))
// Source: "attn_qat_train.py", the fake_quantize call of _attn_fwd_inner (P quantized
// per query rows x KV tile with the row sum taken from unquantized P); the page does
// not show quant_utils, so FP8 E4M3 with an absmax / 448 scale per row x 64 keys is the
// reading this library implements.  Division and multiplication use the explicit
// round-to-nearest intrinsics so no contraction or fast-math changes the result.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace qat {

constexpr float kE4M3Max = 448.0f;
constexpr int kQuantTile = 64;

struct TileScale {
  float inv;    // 448 / amax   (0 when amax == 0)
  float scale;  // amax / 448   (0 when amax == 0)
};

__device__ __forceinline__ TileScale tile_scale(float amax) {
  TileScale t;
  if (amax > 0.0f) {
    t.inv = __fdiv_rn(kE4M3Max, amax);
    t.scale = __fdiv_rn(amax, kE4M3Max);
  } else {
    t.inv = 0.0f;
    t.scale = 0.0f;
  }
  return t;
}

// Two fp32 values -> two E4M3 codes, `lo` in bits 0..7 and `hi` in bits 8..15.
__device__ __forceinline__ uint16_t e4m3x2_rn_satfinite(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two E4M3 codes -> their exact values as fp32 (lo = bits 0..7).
__device__ __forceinline__ float2 e4m3x2_decode(uint16_t codes) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(codes));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

// Quantize a pair of probabilities of one tile: returns the bf16 pair of quantized
// values (lo in the low half), and the two code bytes through `codes`.
__device__ __forceinline__ __nv_bfloat162 quant_pair(float p0, float p1, TileScale t,
                                                     uint16_t* codes) {
  const uint16_t c = e4m3x2_rn_satfinite(__fmul_rn(p0, t.inv), __fmul_rn(p1, t.inv));
  *codes = c;
  const float2 d = e4m3x2_decode(c);
  return __floats2bfloat162_rn(__fmul_rn(d.x, t.scale), __fmul_rn(d.y, t.scale));
}

}  // namespace qat
