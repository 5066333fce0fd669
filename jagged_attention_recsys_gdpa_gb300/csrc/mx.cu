// MXFP8 quantization of a jagged bf16 tensor: FP8 E4M3 codes at the same
// (unpadded) positions plus one E8M0 scale per block of 32 sequence-local rows
// x 32 head columns. One warp per block: lane i holds row i of the block (32
// values, 64 bytes), the block's largest magnitude comes from one warp-wide
// max, the scale exponent from its bits, and the codes from the hardware's
// round-to-nearest-even, saturating conversion.
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace jattn {
namespace {

constexpr int kMxWarps = 8;

__device__ __forceinline__ uint32_t e4m3_code(float x) {
  // both halves take x, so the code sits in either byte whatever the packing order
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(d) : "f"(x));
  return d & 0xffu;
}

__global__ void __launch_bounds__(kMxWarps * 32)
    mx_quant_kernel(const int64_t* __restrict__ off, int B, int H, int D, const uint4* __restrict__ x,
                    uint4* __restrict__ codes, uint8_t* __restrict__ scales, const int* __restrict__ block_start,
                    const int* __restrict__ n_blocks, int64_t max_blocks) {
  const int lane = threadIdx.x & 31;
  const int64_t w = static_cast<int64_t>(blockIdx.x) * kMxWarps + (threadIdx.x >> 5);
  const int cols = D / 32;
  const int64_t g = w / (static_cast<int64_t>(H) * cols);  // row block
  if (g >= max_blocks || g >= *n_blocks) return;
  const int hc = static_cast<int>(w % (static_cast<int64_t>(H) * cols));
  const int h = hc / cols, c = hc % cols;
  // sequence of row block g: the last b in [0, B) with block_start[b] <= g
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (block_start[mid] <= g) lo = mid;
    else hi = mid - 1;
  }
  const int64_t row = off[lo] + 32 * (g - block_start[lo]) + lane;
  const bool valid = row < off[lo + 1];
  // this lane's 32 values: 64 bytes at (row, h, 32c)
  const int64_t e0 = (row * H + h) * D + 32 * c;  // element index
  uint32_t v[16];
  if (valid) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 p = x[e0 / 8 + q];
      v[4 * q] = p.x; v[4 * q + 1] = p.y; v[4 * q + 2] = p.z; v[4 * q + 3] = p.w;
    }
  } else {
#pragma unroll
    for (int q = 0; q < 16; ++q) v[q] = 0u;
  }
  // block amax: magnitudes as bit patterns order like their values
  uint32_t m = 0;
#pragma unroll
  for (int q = 0; q < 16; ++q) m = max(m, max((v[q] << 16) & 0x7fffffffu, v[q] & 0x7fff0000u));
  m = __reduce_max_sync(0xffffffffu, m);
  // E - 127 = floor(log2(amax)) - 8, clamped at E >= 0 (zero and tiny blocks: E = 0)
  const int efield = static_cast<int>(m >> 23);
  const int E = efield > 8 ? efield - 8 : 0;
  const float inv_x = __uint_as_float(static_cast<uint32_t>(254 - E) << 23);  // 2^(127 - E)
  if (valid) {
    uint32_t out[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      uint32_t word = 0;
#pragma unroll
      for (int k = 0; k < 2; ++k) {  // bf16 pair 2q + k -> bytes 4q + 2k, 4q + 2k + 1
        const uint32_t pair = v[2 * q + k];
        const uint32_t b0 = e4m3_code(__uint_as_float(pair << 16) * inv_x);
        const uint32_t b1 = e4m3_code(__uint_as_float(pair & 0xffff0000u) * inv_x);
        word |= (b0 | (b1 << 8)) << (16 * k);
      }
      out[q] = word;
    }
    uint4* dst = codes + e0 / 16;
    dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
    dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
  }
  if (lane == 0) scales[(g * H + h) * cols + c] = static_cast<uint8_t>(E);
}

}  // namespace

cudaError_t launch_mx_quant(const int64_t* off, int B, int H, int D, int64_t max_blocks, const void* x, void* codes,
                            uint8_t* scales, const int* block_start, const int* n_blocks, cudaStream_t stream) {
  const int64_t warps = max_blocks * H * (D / 32);
  if (warps == 0) return cudaSuccess;
  const int64_t grid = (warps + kMxWarps - 1) / kMxWarps;
  mx_quant_kernel<<<static_cast<unsigned>(grid), kMxWarps * 32, 0, stream>>>(
      off, B, H, D, static_cast<const uint4*>(x), static_cast<uint4*>(codes), scales, block_start, n_blocks,
      max_blocks);
  return cudaGetLastError();
}

}  // namespace jattn
