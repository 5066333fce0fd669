// Rotary position embedding on a jagged tensor: y = R(pos) x (or R(pos)^T x),
// the forward-side pass for attention whose backward rotates dQ and dK back in
// its epilogues. Pairs (2m, 2m+1) of each head turn by the angle whose cos /
// sin the caller's tables hold at row pos (positions as in jattn.h). One
// thread per 16-byte piece (4 pairs): a bandwidth-bound pass.
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace jattn {
namespace {

constexpr int kRopeBlock = 256;

// One thread per (row, 16-byte piece of a head): it finds the row's sequence,
// reads the piece's 4 cos / sin values once and rotates that piece in every
// head.
__global__ void __launch_bounds__(kRopeBlock)
    rope_kernel(const int64_t* __restrict__ own_off, const int64_t* __restrict__ other_off, int B, int keys,
                int inverse, int H, int D, int64_t total, const uint4* __restrict__ x, uint4* y,
                const float* __restrict__ cos_t, const float* __restrict__ sin_t, int rows, DevStatus* status) {
  const int per_head = D / 8;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kRopeBlock + threadIdx.x;
  if (t >= total * per_head) return;
  const int64_t r = t / per_head;
  const int piece = static_cast<int>(t % per_head);
  const int m0 = piece * 4;  // first pair of this piece within its head
  // sequence of row r: the last b in [0, B) with own_off[b] <= r
  int64_t lo = 0, hi = B - 1;
  while (lo < hi) {
    const int64_t mid = (lo + hi + 1) >> 1;
    if (own_off[mid] <= r) lo = mid;
    else hi = mid - 1;
  }
  const int64_t l_own = own_off[lo + 1] - own_off[lo];
  const int64_t l_other = other_off[lo + 1] - other_off[lo];
  const int64_t i = r - own_off[lo];
  const int64_t delta = keys ? l_own - l_other : l_other - l_own;  // Lkv - Lq
  const int64_t pos = keys ? i + (delta < 0 ? -delta : 0) : i + (delta > 0 ? delta : 0);
  const bool ok = pos >= 0 && pos < rows && i >= 0 && i < l_own;  // also guards offsets that are not a prefix sum
  if (!ok) record_error(status, JATTN_ERR_ROPE, 71, static_cast<int>(pos < 0 ? -1 : (pos > rows ? rows : pos)));
  float cs[4] = {1.0f, 1.0f, 1.0f, 1.0f}, sn[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  if (ok) {
    const float4 c4 = *reinterpret_cast<const float4*>(cos_t + pos * (D / 2) + m0);
    const float4 s4 = *reinterpret_cast<const float4*>(sin_t + pos * (D / 2) + m0);
    const float sg = inverse ? -1.0f : 1.0f;
    cs[0] = c4.x; cs[1] = c4.y; cs[2] = c4.z; cs[3] = c4.w;
    sn[0] = sg * s4.x; sn[1] = sg * s4.y; sn[2] = sg * s4.z; sn[3] = sg * s4.w;
  }
  for (int h = 0; h < H; ++h) {
    const int64_t idx = (r * H + h) * per_head + piece;
    const uint4 w = x[idx];
    const uint32_t in[4] = {w.x, w.y, w.z, w.w};
    uint32_t out[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {  // word e holds pair m0 + e: element 2m in the low half
      const float x0 = __uint_as_float(in[e] << 16), x1 = __uint_as_float(in[e] & 0xffff0000u);
      out[e] = pack_bf16x2(fmaf(x0, cs[e], -x1 * sn[e]), fmaf(x0, sn[e], x1 * cs[e]));
    }
    y[idx] = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

// out[m * rows + p] = in[p * half + m]: row-major [rows, half] tables to the
// pair-major layout the backward epilogues read (consecutive positions, i.e.
// consecutive rows of a warp, at consecutive addresses). 32 x 32 tiles.
__global__ void __launch_bounds__(1024)
    rope_transpose_kernel(const float* __restrict__ in_c, const float* __restrict__ in_s, int rows, int half,
                          float* __restrict__ out_c, float* __restrict__ out_s) {
  __shared__ float tile[2][32][33];
  const int p0 = blockIdx.x * 32, m0 = blockIdx.y * 32;
  const int tx = threadIdx.x, ty = threadIdx.y;
  if (p0 + ty < rows && m0 + tx < half) {
    tile[0][ty][tx] = in_c[static_cast<int64_t>(p0 + ty) * half + m0 + tx];
    tile[1][ty][tx] = in_s[static_cast<int64_t>(p0 + ty) * half + m0 + tx];
  }
  __syncthreads();
  if (m0 + ty < half && p0 + tx < rows) {
    out_c[static_cast<int64_t>(m0 + ty) * rows + p0 + tx] = tile[0][tx][ty];
    out_s[static_cast<int64_t>(m0 + ty) * rows + p0 + tx] = tile[1][tx][ty];
  }
}

}  // namespace

cudaError_t launch_rope(const int64_t* own_off, const int64_t* other_off, int B, int keys, int inverse, int H,
                        int D, int64_t total, const void* x, void* y, const float* cos_t, const float* sin_t,
                        int rows, DevStatus* status, cudaStream_t stream) {
  const int64_t n = total * (D / 8);
  if (n == 0) return cudaSuccess;
  const int64_t blocks = (n + kRopeBlock - 1) / kRopeBlock;
  rope_kernel<<<static_cast<unsigned>(blocks), kRopeBlock, 0, stream>>>(
      own_off, other_off, B, keys, inverse, H, D, total, static_cast<const uint4*>(x), static_cast<uint4*>(y), cos_t,
      sin_t, rows, status);
  return cudaGetLastError();
}

cudaError_t launch_rope_transpose(const float* cos_t, const float* sin_t, int rows, int half, float* cos_pm,
                                  float* sin_pm, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>((rows + 31) / 32), static_cast<unsigned>((half + 31) / 32));
  rope_transpose_kernel<<<grid, dim3(32, 32), 0, stream>>>(cos_t, sin_t, rows, half, cos_pm, sin_pm);
  return cudaGetLastError();
}

}  // namespace jattn
