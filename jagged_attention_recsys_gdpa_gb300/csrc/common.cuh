// Shared device-side definitions for the jagged attention kernels.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/jattn.h"
#include "ptx.cuh"

namespace jattn {

constexpr int kTile = 128;        // rows of a Q tile, rows of a K/V tile
constexpr int kCostBuckets = 1024;  // schedule cost is capped at kCostBuckets - 1
constexpr int kSchedBlock = 256;    // tiles per block in the schedule kernels

// Status words in the first 256 bytes of the workspace.
struct DevStatus {
  int code;    // first error recorded (JATTN_OK when clean)
  int where;   // which wait / check set it
  int detail;  // sequence index or other detail
  int pad;
};

// Everything a persistent attention kernel needs besides its tensor maps.
struct AttnArgs {
  const int64_t* q_off;
  const int64_t* kv_off;
  const int4* tiles;       // sorted schedule: (b, row tile, col tile lo, col tile hi)
  const int* n_tiles;      // device count of tiles
  int H;
  int mask;
  int window;
  float scale;             // softmax scale applied to q.k
  float scale_log2;        // scale * log2(e)
  int norm_by_lkv;
  // outputs / extra inputs (meaning depends on the kernel)
  __nv_bfloat16* out0;
  __nv_bfloat16* out1;
  float* f0;               // lse (fwd) / lse (bwd)
  float* f1;               // Di (bwd): written by the dQ pass, read by the dK/dV pass
  const __nv_bfloat16* in0;
  const __nv_bfloat16* in1;
  DevStatus* status;
  uint64_t timeout_ns;
  int debug_flags;
  int out_v8;              // output rows may be written with 32-byte stores (bases 32-byte aligned)
  // rotary tables, pair-major [D/2][rope_rows] (dQ / dK epilogues rotate back
  // by R(pos)^T; consecutive rows of a warp read consecutive words); nullptr: none
  const float* rope_cos;
  const float* rope_sin;
  int rope_rows;
  // dQ pass of softmax attention whose every item holds a single key tile
  // (self-attention with blocks that divide the tile): the row maximum, sum
  // and Di come from the tile itself, no O or LSE is read, and the pass writes
  // LSE (a.f0) and Di (a.f1) for the dK/dV pass.
  int in_tile_stats;
  // MXFP8 passes: E8M0 scales [row blocks, H, D/32] of Q and of K / V, and
  // the first row block of each sequence (int32 [B+1]) of the two sides
  const uint8_t* sf_q;
  const uint8_t* sf_k;
  const uint8_t* sf_v;
  const int* bs_q;
  const int* bs_kv;
  // MXFP8 backward: E8M0 scales of dO (row blocks of the query side)
  const uint8_t* sf_do;
  // third output of the fused short-query backward (dK; out0 = dQ, out1 = dV)
  __nv_bfloat16* out2;
};

// The bf16 pair of what the bf16 pair `hi` of (x0, x1) leaves out.
__device__ __forceinline__ uint32_t bf16x2_lo(float x0, float x1, uint32_t hi) {
  const float2 hf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hi));
  return pack_bf16x2(x0 - hf.x, x1 - hf.y);
}

// Store 16 packed words (32 bf16 values, 64 bytes) of one output row: two
// 32-byte stores when the output base is 32-byte aligned, else four 16-byte
// stores. Every row start and column offset used with it is a multiple of
// 32 bytes, so the base alone decides.
__device__ __forceinline__ void store_words16(void* dst, const uint32_t (&w)[16], int v8) {
  if (v8) {
    uint32_t* p = reinterpret_cast<uint32_t*>(dst);
#pragma unroll
    for (int h = 0; h < 2; ++h)
      asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p + 8 * h), "r"(w[8 * h]),
                   "r"(w[8 * h + 1]), "r"(w[8 * h + 2]), "r"(w[8 * h + 3]), "r"(w[8 * h + 4]), "r"(w[8 * h + 5]),
                   "r"(w[8 * h + 6]), "r"(w[8 * h + 7])
                   : "memory");
  } else {
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int e = 0; e < 4; ++e) d[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
  }
}

// tanh-GELU's Taylor polynomial at 0 through x^6 and its derivative, on the
// FMA pipe only. With c = sqrt(2/pi), a = 0.044715 and u = c (x + a x^3),
// tanh u = u - u^3/3 + 2u^5/15 - ..., so x/2 (1 + tanh u) = x/2 + g2 x^2 +
// g4 x^4 + g6 x^6 + O(x^8) with the coefficients below (odd powers above 1
// cancel: x tanh u is even).
struct GeluPoly {
  static constexpr double c = 0.7978845608028654;  // sqrt(2/pi)
  static constexpr double a = 0.044715;
  static constexpr float g2 = static_cast<float>(c / 2);
  static constexpr float g4 = static_cast<float>((c * a - c * c * c / 3) / 2);
  static constexpr float g6 = static_cast<float>((2 * c * c * c * c * c / 15 - c * c * c * a) / 2);
};
__device__ __forceinline__ float gelu_poly(float x) {
  const float x2 = x * x;
  return fmaf(x2, fmaf(x2, fmaf(x2, GeluPoly::g6, GeluPoly::g4), GeluPoly::g2), 0.5f * x);
}
__device__ __forceinline__ float gelu_poly_grad(float x) {
  const float x2 = x * x;
  return fmaf(x, fmaf(x2, fmaf(x2, 6.0f * GeluPoly::g6, 4.0f * GeluPoly::g4), 2.0f * GeluPoly::g2), 0.5f);
}

// Rotary positions of sequence-local query row i and key row j: both sides end
// at the same position and the longer one starts at 0 (delta = Lkv - Lq).
__device__ __forceinline__ int rope_pos_q(int i, int delta) { return i + max(delta, 0); }
__device__ __forceinline__ int rope_pos_k(int j, int delta) { return j + max(-delta, 0); }

// x = R(pos)^T y in place on 16 pairs of fp32 values (bit patterns in v):
// pair e is turned back by the angle whose cos / sin are c[e * stride] /
// s[e * stride] (pair-major tables: c and s point at the first pair's entry
// for this row's position).
__device__ __forceinline__ void rope_back16(uint32_t* v, const float* c, const float* s, int stride) {
  float ca[16], sa[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    ca[e] = __ldg(c + static_cast<int64_t>(e) * stride);
    sa[e] = __ldg(s + static_cast<int64_t>(e) * stride);
  }
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const float y0 = __uint_as_float(v[2 * e]), y1 = __uint_as_float(v[2 * e + 1]);
    v[2 * e] = __float_as_uint(fmaf(y0, ca[e], y1 * sa[e]));
    v[2 * e + 1] = __float_as_uint(fmaf(y1, ca[e], -y0 * sa[e]));
  }
}

// floor(x / w) for w >= 1 and any sign of x
__device__ __forceinline__ int floor_div(int x, int w) { return x >= 0 ? x / w : -((w - 1 - x) / w); }

// Visible key interval [lo, hi) of sequence-local query row i
// (bottom-right aligned, delta = Lkv - Lq). Window implies causal; a block
// mask of width W keeps the keys of the block that holds position i + delta.
__device__ __forceinline__ void key_interval(int i, int delta, int lkv, int mask, int window, int& lo, int& hi) {
  lo = 0;
  hi = lkv;
  if (mask & (JATTN_MASK_CAUSAL | JATTN_MASK_WINDOW)) hi = min(hi, i + delta + 1);
  if (mask & JATTN_MASK_WINDOW) lo = max(lo, i + delta - window + 1);
  if (mask & JATTN_MASK_BLOCK) {
    const int b0 = floor_div(i + delta, window) * window;
    lo = max(lo, b0);
    hi = min(hi, b0 + window);
  }
}

// Visible query interval [lo, hi) of sequence-local key row j.
__device__ __forceinline__ void query_interval(int j, int delta, int lq, int mask, int window, int& lo, int& hi) {
  lo = 0;
  hi = lq;
  if (mask & (JATTN_MASK_CAUSAL | JATTN_MASK_WINDOW)) lo = max(lo, j - delta);
  if (mask & JATTN_MASK_WINDOW) hi = min(hi, j - delta + window);
  if (mask & JATTN_MASK_BLOCK) {
    const int b0 = (j / window) * window;  // j >= 0
    lo = max(lo, b0 - delta);
    hi = min(hi, b0 + window - delta);
  }
}

// Column-tile range of row tile rt (of row_tile rows) of one sequence (see the interval rules in
// key_interval / query_interval; both ends are monotone in the row index, so
// the union over the non-empty rows of a tile is [lo(first), hi(last))).
__device__ __forceinline__ void tile_range(int lq, int lkv, int rt, int row_tile, int col_tile, int mask,
                                           int window, int transposed, int& c_lo, int& c_hi) {
  const int delta = lkv - lq;
  const bool causal = mask & (JATTN_MASK_CAUSAL | JATTN_MASK_WINDOW);
  const bool win = mask & JATTN_MASK_WINDOW;
  const bool blk = mask & JATTN_MASK_BLOCK;
  const int nrows = transposed ? lkv : lq;
  const int ncols = transposed ? lq : lkv;
  int first = rt * row_tile;
  int last = min((rt + 1) * row_tile, nrows) - 1;
  c_lo = c_hi = 0;
  if (ncols == 0 || first > last) return;
  int lo, hi, lo2, hi2;
  if (!transposed) {
    // query rows before key position 0 see nothing under causal and block masks
    if (causal || blk) first = max(first, -delta);
    if (win) last = min(last, lkv - 1 - delta + window - 1);
    if (first > last) return;
    key_interval(first, delta, lkv, mask, window, lo, hi);
    key_interval(last, delta, lkv, mask, window, lo2, hi2);
  } else {
    if (win) first = max(first, delta - window + 1);
    // key blocks that end before the first query position (delta) see no query
    if (blk) first = max(first, floor_div(delta, window) * window);
    if (causal) last = min(last, lq + delta - 1);
    if (first > last) return;
    query_interval(first, delta, lq, mask, window, lo, hi);
    query_interval(last, delta, lq, mask, window, lo2, hi2);
  }
  c_lo = lo / col_tile;
  c_hi = (hi2 + col_tile - 1) / col_tile;
}

__device__ __forceinline__ void record_error(DevStatus* st, int code, int where, int detail) {
  if (atomicCAS(&st->code, 0, code) == 0) {
    st->where = where;
    st->detail = detail;
  }
}

// Pair-0 entries of position pos in the pair-major tables (pair m is m *
// rope_rows further on): nullptr when no rotation is asked for, or (after
// recording JATTN_ERR_ROPE) when pos is past the tables.
__device__ __forceinline__ void rope_rows_at(const AttnArgs& a, int pos, const float*& c, const float*& s) {
  c = s = nullptr;
  if (a.rope_cos == nullptr) return;
  if (pos < 0 || pos >= a.rope_rows) {
    record_error(a.status, JATTN_ERR_ROPE, 70, pos);
    return;
  }
  c = a.rope_cos + pos;
  s = a.rope_sin + pos;
}

// Bounded mbarrier wait. Returns false (and raises the CTA abort flag and the
// device status) once `timeout_ns` elapses or another role has aborted.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         const AttnArgs& a, int where) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > a.timeout_ns) {
      *abort_flag = 1;
      record_error(a.status, JATTN_ERR_TIMEOUT, where, blockIdx.x);
      return false;
    }
  }
}

// Persistent-grid zigzag: the k-th item (k = round * G + pos) processed by CTA g.
__device__ __forceinline__ long long zigzag_item(long long round, int g, int G) {
  return round * G + ((round & 1) ? (G - 1 - g) : g);
}

}  // namespace jattn
