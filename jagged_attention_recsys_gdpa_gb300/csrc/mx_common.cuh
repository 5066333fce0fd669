// Helpers shared by the MXFP8 attention kernels (fwd_mx.cu, bwd_mx.cu): work
// items, block-scale words and their layouts in tensor memory.
#pragma once
#include <cstdint>

#include "common.cuh"

namespace jattn {
namespace mx {

struct Item {
  int b, qt, lo, hi, h, lq, lkv;
  int64_t q0, k0;
};

__device__ __forceinline__ bool load_item(const AttnArgs& a, long long round, Item& it) {
  const long long n_items = static_cast<long long>(*a.n_tiles) * a.H;
  const long long k = zigzag_item(round, blockIdx.x, gridDim.x);
  if (k >= n_items) return false;
  const int4 t = a.tiles[k / a.H];
  it.h = static_cast<int>(k % a.H);
  it.b = t.x;
  it.qt = t.y;
  it.lo = t.z;
  it.hi = t.w;
  it.q0 = a.q_off[it.b];
  it.k0 = a.kv_off[it.b];
  it.lq = static_cast<int>(a.q_off[it.b + 1] - it.q0);
  it.lkv = static_cast<int>(a.kv_off[it.b + 1] - it.k0);
  return true;
}

// The 4 scale bytes of row block g (head h, D / 32 = 4 column blocks) as one word.
__device__ __forceinline__ uint32_t sf_word(const uint8_t* sf, int g, int H, int h) {
  return __ldg(reinterpret_cast<const uint32_t*>(sf + (static_cast<int64_t>(g) * H + h) * 4));
}

// Row block r of sequence b, clamped to the sequence's blocks (tile rows past
// the sequence read some finite scale; their scores are masked).
__device__ __forceinline__ int row_block(const int* bs, int b, int r) {
  const int first = bs[b], last = bs[b + 1] - 1;
  return min(first + r, max(last, first));
}

// The 4 scale words of row blocks 4j .. 4j + 3 (key tile j) of one head, the
// block indices clamped to the sequence's [first, last] (loads only; they are
// issued a step before their use).
__device__ __forceinline__ void kv_scale_load(const uint8_t* sf, int first, int last, int j, int H, int h,
                                              uint32_t (&r)[4]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) r[c] = sf_word(sf, min(first + 4 * j + c, last), H, h);
}
// In the replicated layout (lane l of every quarter, column c = index 32c + l)
// a K tile's words are the row blocks' words as they are (4 column blocks in
// the bytes); a V tile's column block c takes byte c of each row block's word.
__device__ __forceinline__ void v_scale_words(const uint32_t (&r)[4], uint32_t (&w)[4]) {
#pragma unroll
  for (int c = 0; c < 4; ++c)
    w[c] = ((r[0] >> (8 * c)) & 0xffu) | (((r[1] >> (8 * c)) & 0xffu) << 8) | (((r[2] >> (8 * c)) & 0xffu) << 16) |
           (((r[3] >> (8 * c)) & 0xffu) << 24);
}

// Bounded wait of a role's last step (its copies or MMAs in flight landing
// before the CTA exits): gives up silently after timeout_ns.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > timeout_ns) return;
  }
}

// Scale exponent of a 32-element block of P = 2^x whose largest exponent
// argument is xmax: e = ceil(xmax) - 8, so the block's P / 2^e lie in (0, 256]
// with the largest in (128, 256]; clamped to keep 2^e a normal float (a block
// with no allowed entry takes any scale, its codes are 0).
__device__ __forceinline__ int p_block_exp(float xmax) {
  return (xmax == -INFINITY) ? -8 : max(-100, min(100, static_cast<int>(ceilf(xmax)) - 8));
}

// Words of row blocks r0 .. r0 + N - 1 of one sequence and head, the indices
// clamped to the sequence's blocks [first, last] (rows past the sequence read
// some finite scale; their entries are masked).
template <int N>
__device__ __forceinline__ void block_words(const uint8_t* sf, int first, int last, int r0, int H, int h,
                                            uint32_t (&w)[N]) {
#pragma unroll
  for (int c = 0; c < N; ++c) w[c] = sf_word(sf, min(first + r0 + c, last), H, h);
}

// E8M0 exponent of a [32, 32] block from its largest magnitude's bit pattern
// (OCP Microscaling rule): E - 127 = floor(log2 amax) - 8, E >= 0; zero and
// tiny blocks get E = 0.
__device__ __forceinline__ int block_exponent(uint32_t amax_bits) {
  const int efield = static_cast<int>(amax_bits >> 23);
  return efield > 8 ? efield - 8 : 0;
}

}  // namespace mx
}  // namespace jattn
