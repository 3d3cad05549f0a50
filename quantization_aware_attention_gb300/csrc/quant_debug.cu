// quant_debug.cu -- test entry kernel: applies the per-tile FP8 rule of qat_quant.cuh
// to caller-supplied fp32 tiles so the rule can be compared bit for bit with the
// specification (one warp per row x 64-column tile, two columns per lane).
#include "qat_internal.h"
#include "qat_quant.cuh"

namespace qat {
namespace {

__global__ void __launch_bounds__(256) debug_quant_kernel(const float* __restrict__ p, int rows,
                                                          int cols, float* __restrict__ deq,
                                                          float* __restrict__ scales,
                                                          uint8_t* __restrict__ codes) {
  const int tiles = (cols + kQuantTile - 1) / kQuantTile;
  const long long total = static_cast<long long>(rows) * tiles;
  const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const int lane = threadIdx.x & 31;
  for (long long w = warp; w < total; w += nwarps) {
    const long long r = w / tiles;
    const int t = static_cast<int>(w % tiles);
    const int j0 = t * kQuantTile + 2 * lane;
    const float* pr = p + r * cols;
    const float x0 = (j0 < cols) ? pr[j0] : 0.f;
    const float x1 = (j0 + 1 < cols) ? pr[j0 + 1] : 0.f;
    float amax = fmaxf(x0, x1);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const TileScale ts = tile_scale(amax);
    uint16_t cd;
    const __nv_bfloat162 v = quant_pair(x0, x1, ts, &cd);
    const float2 vf = __bfloat1622float2(v);
    if (j0 < cols) {
      deq[r * cols + j0] = vf.x;
      codes[r * cols + j0] = static_cast<uint8_t>(cd & 0xFF);
    }
    if (j0 + 1 < cols) {
      deq[r * cols + j0 + 1] = vf.y;
      codes[r * cols + j0 + 1] = static_cast<uint8_t>(cd >> 8);
    }
    if (lane == 0) scales[r * tiles + t] = ts.scale;
  }
}

}  // namespace

cudaError_t launch_debug_quant(const float* p, int rows, int cols, float* deq, float* scales,
                               uint8_t* codes, cudaStream_t s) {
  const long long tiles = static_cast<long long>(rows) * ((cols + kQuantTile - 1) / kQuantTile);
  if (tiles == 0) return cudaSuccess;
  long long blocks = (tiles + 7) / 8;
  if (blocks > 152 * 32) blocks = 152 * 32;
  debug_quant_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(p, rows, cols, deq, scales,
                                                                   codes);
  return cudaGetLastError();
}

}  // namespace qat
