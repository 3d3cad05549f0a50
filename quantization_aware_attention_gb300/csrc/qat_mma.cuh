// qat_mma.cuh -- warp-level helpers of the mma.sync (m16n8k16, bf16 -> fp32) kernels:
// fragment loads from padded shared-memory tiles, the MMA itself, fast exp2 and
// quad (4-lane) reductions.
//
// Fragment layouts of mma.m16n8k16 (g = lane / 4, c = lane % 4):
//   A (16x16, row-major): reg0 = A[g][2c..2c+1],   reg1 = A[g+8][2c..2c+1],
//                         reg2 = A[g][2c+8..+9],   reg3 = A[g+8][2c+8..+9]
//   B (16x8, k x n):      reg0 = B[2c..2c+1][g],   reg1 = B[2c+8..+9][g]
//   C (16x8 fp32):        c0,c1 = C[g][2c..2c+1],  c2,c3 = C[g+8][2c..2c+1]
// so two adjacent C tiles (n = 8 each) of a 16-row strip re-pack directly into one
// A fragment of k = 16 -- the probabilities never leave registers.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace qat {

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4],
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t ld_s32(const uint16_t* p) {
  return *reinterpret_cast<const uint32_t*>(p);
}

// Two bf16 elements that are not adjacent in memory, packed lo | hi << 16.
__device__ __forceinline__ uint32_t pack_u16(uint16_t lo, uint16_t hi) {
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

__device__ __forceinline__ uint32_t bf162_bits(__nv_bfloat162 v) {
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_bf16_rn(float lo, float hi) {
  return bf162_bits(__floats2bfloat162_rn(lo, hi));
}

__device__ __forceinline__ float quad_max(float x) {
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 1));
  return fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 2));
}

__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  return x + __shfl_xor_sync(0xffffffffu, x, 2);
}

// Copy rows [row0, row0 + ROWS) of a [N, D] bf16 matrix into a shared tile with row
// stride LD elements; rows at or beyond N are zero-filled.  16-byte accesses.
template <int ROWS, int D, int LD, int NTHREADS>
__device__ __forceinline__ void load_rows(uint16_t* dst, const uint16_t* src, int row0,
                                          int N, int tid) {
  constexpr int CH = D / 8;
#pragma unroll 4
  for (int idx = tid; idx < ROWS * CH; idx += NTHREADS) {
    const int r = idx / CH, ch = idx % CH;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (row0 + r < N)
      val = *reinterpret_cast<const uint4*>(src + static_cast<size_t>(row0 + r) * D + ch * 8);
    *reinterpret_cast<uint4*>(dst + r * LD + ch * 8) = val;
  }
}

}  // namespace qat
