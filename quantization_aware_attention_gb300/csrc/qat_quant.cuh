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

// Packed fp32 pair helpers (two IEEE round-to-nearest operations per instruction).
__device__ __forceinline__ unsigned long long f2_pack(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ float2 f2_unpack(unsigned long long v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}

__device__ __forceinline__ float2 mul_rn_f32x2(float2 a, float2 b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_pack(a.x, a.y)), "l"(f2_pack(b.x, b.y)));
  return f2_unpack(d);
}

__device__ __forceinline__ float2 fma_rn_f32x2(float2 a, float2 b, float2 c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(f2_pack(a.x, a.y)), "l"(f2_pack(b.x, b.y)), "l"(f2_pack(c.x, c.y)));
  return f2_unpack(d);
}

__device__ __forceinline__ float2 add_rn_f32x2(float2 a, float2 b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_pack(a.x, a.y)), "l"(f2_pack(b.x, b.y)));
  return f2_unpack(d);
}

// Quantize a pair of probabilities of one tile: returns the bf16 pair of quantized
// values (p0 in the low half), and the two code bytes through `codes`.
__device__ __forceinline__ __nv_bfloat162 quant_pair(float p0, float p1, TileScale t,
                                                     uint16_t* codes) {
  const float2 x = mul_rn_f32x2(make_float2(p0, p1), make_float2(t.inv, t.inv));
  const uint16_t c = e4m3x2_rn_satfinite(x.x, x.y);
  *codes = c;
  const float2 d = mul_rn_f32x2(e4m3x2_decode(c), make_float2(t.scale, t.scale));
  return __floats2bfloat162_rn(d.x, d.y);
}

}  // namespace qat
