// Backward pass of jagged softmax attention on MXFP8 operands, sm_103a.
//
// "GEM Training" post, section "Low Precision Flash Attention": the backward
// runs every product as a block-scaled FP8 MMA. Q, K, V and dO arrive as E4M3
// codes with one E8M0 scale per 32 x 32 block (jattn_mxfp8_quantize), and the
// intermediates are quantized online: P for dV = P~^T dO inside the softmax
// warps, and dS for dQ = scale dS~ K and dK = scale dS~^T Q with one scale per
// 32 x 32 block of (query, key) pairs from a warp-wide maximum (the post's
// [32, 32] square blocks: the same blocks serve dS and dS^T). Three kernels:
//   mx_di    D_i = <dO_i, O_i> per query row and head, dO dequantized
//   dq_mx    one item = (sequence, 128-query tile, head) walking its key
//            tiles: S = Q K^T, dP = dO V^T, dS = P (dP - D), dQ += dS~ K
//   dkdv_mx  one item = (sequence, 128-key tile, head) walking its queries
//            96 at a time: S^T = K Q^T, dP^T = V dO^T, dV += P~^T dO,
//            dK += dS~^T Q
// Both MMA kernels are persistent and warp-specialised like the bf16
// backward: a TMA producer warp, an MMA-issuing warp, and activation warps
// that own one TMEM lane (a query row, or a key row) each. The activation
// warps write the FP8 codes of P and dS into the TMEM columns of the scores
// they have read (4 codes per column, the A operand of the next MMA) and
// every scale factor the MMAs read, before the barrier that releases them.
//
// Tensor memory (512 columns) sets the dK/dV pass's shape: four 128-column
// accumulators (S^T, dP^T, dV, dK) would leave no column for scale factors,
// so the pass walks queries in steps of 96 (three 32-query blocks): S^T and
// dP^T take 96 columns each, and three activation warpgroups own one query
// block each, so every P~ scale (per key row and 32-query block) and every
// dS~ block maximum (32 key rows of a warp x 32 queries) is local to a warp.
#include <cstdint>

#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"
#include "mx_common.cuh"

namespace jattn {

namespace {

constexpr int kD = 128;                 // head dimension (one head row of codes = 128 bytes)
constexpr int kTileBytes = kTile * kD;  // 128 rows of E4M3 codes
constexpr float kLog2e = 1.4426950408889634f;

// 2^e as a float, e in [-126, 127]
__device__ __forceinline__ float pow2i(int e) { return __uint_as_float(static_cast<uint32_t>(127 + e) << 23); }

// Largest magnitude of 32 values (three-input maxima of magnitudes, four
// chains), as its bit pattern: non-negative floats order like their bits.
__device__ __forceinline__ uint32_t amax_bits32(const float* x) {
  float m[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int c = 0; c < 32; c += 8)
#pragma unroll
    for (int e = 0; e < 4; ++e) m[e] = fmax3(m[e], fabsf(x[c + 2 * e]), fabsf(x[c + 2 * e + 1]));
  return __float_as_uint(fmax3(m[0], m[1], fmaxf(m[2], m[3])));
}

// 32 values times 2^(127 - E) as E4M3 codes, 4 per word (value 4w + b in byte b).
__device__ __forceinline__ void codes32(const float* x, int E, uint32_t (&pk)[8]) {
  const float inv = __uint_as_float(static_cast<uint32_t>(254 - E) << 23);
  const uint64_t inv2 = f2(inv, inv);
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    float a0, a1, a2, a3;
    f2_split(fmul2(f2(x[4 * w], x[4 * w + 1]), inv2), a0, a1);
    f2_split(fmul2(f2(x[4 * w + 2], x[4 * w + 3]), inv2), a2, a3);
    pk[w] = pack_e4m3x2(a0, a1) | (pack_e4m3x2(a2, a3) << 16);
  }
}

// MN-major B-operand scale words of a tile whose K dimension runs over row
// blocks (3 or 4 of them, words r): column c (head columns 32c ..) takes byte
// c of each row block's word, the K block in the byte.
template <int N>
__device__ __forceinline__ void mn_words(const uint32_t (&r)[N], uint32_t (&w)[4]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t x = 0;
#pragma unroll
    for (int k = 0; k < N; ++k) x |= ((r[k] >> (8 * c)) & 0xffu) << (8 * k);
    w[c] = x;
  }
}

// ============================================================================ D_i
// D_i = sum_d dO~_id O_id per query row and head: one warp per (row block,
// head), lane l on row l of the block; dO from its codes and its block's 4
// scales, O from the forward's bf16 output.
constexpr int kDiWarps = 8;

__device__ __forceinline__ float e4m3_value(uint32_t code) {
  // the code in both bytes: either half of the result is its value
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(code | (code << 8))));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xffffu)));
}

__global__ void __launch_bounds__(kDiWarps * 32)
    mx_di_kernel(const int64_t* __restrict__ off, int B, int H, const uint8_t* __restrict__ dout,
                 const uint8_t* __restrict__ sf, const int* __restrict__ bs, const __nv_bfloat16* __restrict__ o,
                 float* __restrict__ di, int64_t max_blocks) {
  const int lane = threadIdx.x & 31;
  const int64_t w = static_cast<int64_t>(blockIdx.x) * kDiWarps + (threadIdx.x >> 5);
  const int64_t g = w / H;  // row block
  if (g >= max_blocks || g >= bs[B]) return;
  const int h = static_cast<int>(w % H);
  int lo = 0, hi = B - 1;  // sequence of row block g: the last b with bs[b] <= g
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (bs[mid] <= g) lo = mid;
    else hi = mid - 1;
  }
  const int64_t row = off[lo] + 32 * (g - bs[lo]) + lane;
  if (row >= off[lo + 1]) return;
  const uint32_t sw = __ldg(reinterpret_cast<const uint32_t*>(sf + (g * H + h) * 4));
  const uint4* cp = reinterpret_cast<const uint4*>(dout + (row * H + h) * kD);
  const uint4* op = reinterpret_cast<const uint4*>(o + (row * H + h) * kD);
  float acc = 0.0f;
#pragma unroll
  for (int blk = 0; blk < 4; ++blk) {  // 32 columns per scale
    float part = 0.0f;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint4 c4 = cp[2 * blk + q];
      const uint32_t cw[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const uint4 o4 = op[4 * blk + 2 * q + half];
        const uint32_t ow[4] = {o4.x, o4.y, o4.z, o4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {  // bf16 pair e: columns 2e, 2e + 1 of these 8
          const float2 of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[e]));
          const uint32_t word = cw[2 * half + (e >> 1)];
          const int sh = 16 * (e & 1);
          part = fmaf(e4m3_value((word >> sh) & 0xffu), of.x, part);
          part = fmaf(e4m3_value((word >> (sh + 8)) & 0xffu), of.y, part);
        }
      }
    }
    acc = fmaf(part, ldexpf(1.0f, static_cast<int>((sw >> (8 * blk)) & 0xffu) - 127), acc);
  }
  di[row * H + h] = acc;
}

// ============================================================================ dQ
namespace dqc {
constexpr int kThreads = 384;  // warp 0 TMA, warp 1 MMA, warps 2-3 idle, warps 4-11 two activation warpgroups
constexpr int kStages = 4;
constexpr int kQOff = 0, kDOOff = kTileBytes, kKVOff = 2 * kTileBytes;  // stage s: K, then V
constexpr int kBarOff = kKVOff + kStages * 2 * kTileBytes;
constexpr int kSmemBytes = kBarOff + 512;
constexpr uint32_t kSCol = 0, kDPCol = 128, kDQCol = 256;
// scale factors: Q, dO (A of S, dP), K, V (B of S, dP), K as the MN-major B of
// dQ, dS (A of dQ: [2 warpgroups][4 lane quarters])
constexpr uint32_t kSfQ = 384, kSfDO = 388, kSfK = 392, kSfV = 396, kSfKmn = 400, kSfDS = 404;
constexpr int kCtlRegs = 104;  // 384 x 168 at launch = 128 x 104 + 256 x 200
constexpr int kActRegs = 200;
struct Bars {
  uint64_t qd_full, qd_empty;
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t sf_ready, s_full, s_free, dp_full, ds_ready, acc_full, acc_empty, drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Bars) <= 512, "barrier block overflows its slot");
static_assert(kSmemBytes <= 227 * 1024, "shared memory");
}  // namespace dqc

__global__ void __launch_bounds__(dqc::kThreads, 1)
    dq_mx_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                 const AttnArgs a) {
  using namespace dqc;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) record_error(a.status, JATTN_ERR_UNSUPPORTED, 19, blockIdx.x);
    return;
  }
  uint8_t* sm = smem_raw;
  Bars* bars = reinterpret_cast<Bars*>(sm + kBarOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &bars->abort_flag;

  if (threadIdx.x == 0) {
    mbar_init(&bars->qd_full, 1);
    mbar_init(&bars->qd_empty, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    mbar_init(&bars->sf_ready, 2 * kTile);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, 2 * kTile);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->ds_ready, 2 * kTile);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, 2 * kTile);
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtlRegs));
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        uint32_t q_cnt = 0, kv_it = 0;
        bool ok = true;
        mx::Item it;
        for (long long r = 0; ok && mx::load_item(a, r, it); ++r) {
          if (it.hi <= it.lo) continue;
          if (!(ok = wait_bar(&bars->qd_empty, (q_cnt & 1) ^ 1, abort_flag, a, 140))) break;
          const int yq = static_cast<int>(it.q0) + it.qt * kTile;
          if (!(a.debug_flags & 1)) {
            mbar_arrive_expect_tx(&bars->qd_full, 2 * kTileBytes);
            tma_load_2d(sm + kQOff, &tmQ, &bars->qd_full, it.h * kD, yq);
            tma_load_2d(sm + kDOOff, &tmDO, &bars->qd_full, it.h * kD, yq);
          }
          ++q_cnt;
          for (int j = it.lo; j < it.hi && ok; ++j, ++kv_it) {
            const int s = kv_it % kStages;
            if (!(ok = wait_bar(&bars->kv_empty[s], ((kv_it / kStages) & 1) ^ 1, abort_flag, a, 141))) break;
            const int yk = static_cast<int>(it.k0) + j * kTile;
            mbar_arrive_expect_tx(&bars->kv_full[s], 2 * kTileBytes);
            tma_load_2d(sm + kKVOff + s * 2 * kTileBytes, &tmK, &bars->kv_full[s], it.h * kD, yk);
            tma_load_2d(sm + kKVOff + s * 2 * kTileBytes + kTileBytes, &tmV, &bars->kv_full[s], it.h * kD, yk);
          }
        }
        if (q_cnt > 0 && !(a.debug_flags & 1)) mx::drain_wait(&bars->qd_full, (q_cnt - 1) & 1, a.timeout_ns);
        for (uint32_t i = (kv_it > kStages ? kv_it - kStages : 0); i < kv_it; ++i)
          mx::drain_wait(&bars->kv_full[i % kStages], (i / kStages) & 1, a.timeout_ns);
      }
      __syncwarp();
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        const uint32_t sKV = smem_u32(sm + kKVOff);
        // K-major descriptors advance 32 bytes (2 units) per K block; the
        // MN-major K tile (B of dQ) 32 rows of 128 bytes per K block
        const uint64_t dQ = sdesc_sw128(smem_u32(sm + kQOff), 16, 1024);
        const uint64_t dDO = sdesc_sw128(smem_u32(sm + kDOOff), 16, 1024);
        const uint64_t dK0 = sdesc_sw128(sKV, 16, 1024);
        const uint64_t dV0 = sdesc_sw128(sKV + kTileBytes, 16, 1024);
        const uint64_t dKmn0 = sdesc_sw128(sKV, kTile * 128, 1024);
        constexpr uint64_t kStageUnits = (2 * kTileBytes) >> 4;
        uint32_t q_cnt = 0, kv_it = 0, sf_cnt = 0, acc_cnt = 0, g = 0;  // g: key tiles so far
        bool ok = true;
        auto issue_s = [&](int ks) {
#pragma unroll
          for (int kb = 0; kb < 4; ++kb)
            mma_mx_ss(tmem + kSCol, dQ + 2 * kb, dK0 + ks * kStageUnits + 2 * kb,
                      idesc_mx_e4m3(kTile, kTile, false, false, kb, kb), tmem + kSfQ, tmem + kSfK, kb > 0);
          mma_commit(&bars->s_full);
        };
        auto issue_dp = [&](int ks) {
#pragma unroll
          for (int kb = 0; kb < 4; ++kb)
            mma_mx_ss(tmem + kDPCol, dDO + 2 * kb, dV0 + ks * kStageUnits + 2 * kb,
                      idesc_mx_e4m3(kTile, kTile, false, false, kb, kb), tmem + kSfDO, tmem + kSfV, kb > 0);
          mma_commit(&bars->dp_full);
        };
        mx::Item it;
        for (long long r = 0; ok && mx::load_item(a, r, it); ++r) {
          if (it.hi <= it.lo) continue;
          const int n = it.hi - it.lo;
          if (!(ok = wait_bar(&bars->qd_full, q_cnt & 1, abort_flag, a, 150))) break;
          // the activation warps have written the scales of Q, dO and of the first K / V tile
          if (!(ok = wait_bar(&bars->sf_ready, sf_cnt & 1, abort_flag, a, 151))) break;
          ++sf_cnt;
          if (!(ok = wait_bar(&bars->kv_full[kv_it % kStages], (kv_it / kStages) & 1, abort_flag, a, 152))) break;
          tc_fence_after();
          issue_s(kv_it % kStages);
          issue_dp(kv_it % kStages);
          for (int t = 0; t < n && ok; ++t) {
            const uint32_t ki = kv_it + t;
            const int s = ki % kStages;
            if (t + 1 < n) {  // S(t + 1) once the scores of tile t are read (single S buffer)
              if (!(ok = wait_bar(&bars->s_free, (g + t) & 1, abort_flag, a, 153))) break;
              if (!(ok = wait_bar(&bars->kv_full[(ki + 1) % kStages], ((ki + 1) / kStages) & 1, abort_flag, a, 154)))
                break;
              tc_fence_after();
              issue_s((ki + 1) % kStages);
            }
            if (t == 0 && !(ok = wait_bar(&bars->acc_empty, (acc_cnt & 1) ^ 1, abort_flag, a, 155))) break;
            if (!(ok = wait_bar(&bars->ds_ready, (g + t) & 1, abort_flag, a, 156))) break;
            tc_fence_after();
#pragma unroll
            for (int kb = 0; kb < 4; ++kb)  // keys 32kb ..: dS of warpgroup kb / 2 at dP columns 64 (kb / 2) + 8 (kb % 2)
              mma_mx_ts(tmem + kDQCol, tmem + kDPCol + 64 * (kb >> 1) + 8 * (kb & 1),
                        dKmn0 + s * kStageUnits + kb * (32 * 128 / 16), idesc_mx_e4m3(kTile, kD, false, true, kb, kb),
                        tmem + kSfDS + 4 * (kb >> 1), tmem + kSfKmn, (kb > 0 || t > 0) ? 1u : 0u);
            mma_commit(&bars->kv_empty[s]);  // K(t) read by S(t) and dQ(t), V(t) by dP(t)
            if (t + 1 < n) issue_dp((ki + 1) % kStages);
          }
          if (!ok) break;
          mma_commit(&bars->acc_full);
          ++acc_cnt;
          mma_commit(&bars->qd_empty);
          ++q_cnt;
          kv_it += n;
          g += n;
        }
        mma_commit(&bars->drain);
        mx::drain_wait(&bars->drain, 0, a.timeout_ns);
      }
      __syncwarp();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kActRegs));
    // ------------------------------------------------------------ activation warpgroups
    const int half = (warp - 4) >> 2;  // key columns [64 half, 64 half + 64) of every tile
    const int quarter = warp & 3;
    const int row = 32 * quarter + lane;  // TMEM lane == query row of the tile
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    uint32_t g = 0, acc_cnt = 0;
    bool ok = true;
    mx::Item it;
    for (long long r = 0; ok && mx::load_item(a, r, it); ++r) {
      const int il = it.qt * kTile + row;
      const bool valid = il < it.lq;
      const int64_t gi = (it.q0 + il) * a.H + it.h;
      __nv_bfloat16* dq_row = a.out0 + gi * kD + 64 * half;
      if (it.hi <= it.lo) {  // no key tile: dQ rows are zero
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(dq_row);
          for (int e = 0; e < 8; ++e) dst[e] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      const int n = it.hi - it.lo;
      int klo, khi;
      key_interval(il, it.lkv - it.lq, it.lkv, a.mask, a.window, klo, khi);
      if (!valid) khi = klo;
      const bool any = khi > klo;
      const float lse2 = any ? a.f0[gi] * kLog2e : 0.0f;
      const float di = any ? a.f1[gi] : 0.0f;
      const int kv_first = a.bs_kv[it.b], kv_last = max(a.bs_kv[it.b + 1] - 1, kv_first);
      const int q_first = a.bs_q[it.b], q_last = max(a.bs_q[it.b + 1] - 1, q_first);
      {  // scales of Q (warpgroup 0) / dO (1) and of the first K / V tile
        uint32_t w[4], wk[4];
        mx::block_words(half == 0 ? a.sf_q : a.sf_do, q_first, q_last, 4 * it.qt, a.H, it.h, w);
        mx::kv_scale_load(half == 0 ? a.sf_k : a.sf_v, kv_first, kv_last, it.lo, a.H, it.h, wk);
        tmem_st4(tmem + lane_base + (half == 0 ? kSfQ : kSfDO), w[0], w[1], w[2], w[3]);
        tmem_st4(tmem + lane_base + (half == 0 ? kSfK : kSfV), wk[0], wk[1], wk[2], wk[3]);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->sf_ready);
      }
      const uint64_t c2 = f2(a.scale_log2, a.scale_log2), nl2 = f2(-lse2, -lse2), ndi = f2(-di, -di);
      for (int t = 0; t < n; ++t) {
        const int j = it.lo + t;
        const uint32_t gt = g + t;
        // scale words this step hands over, loaded before the waits: the next
        // K (warpgroup 0) / V (1) tile, and this K tile as dQ's B (0)
        uint32_t w_next[4] = {0, 0, 0, 0}, w_k[4] = {0, 0, 0, 0};
        if (t + 1 < n) mx::kv_scale_load(half == 0 ? a.sf_k : a.sf_v, kv_first, kv_last, j + 1, a.H, it.h, w_next);
        if (half == 0) mx::kv_scale_load(a.sf_k, kv_first, kv_last, j, a.H, it.h, w_k);
        ok = __all_sync(0xffffffffu, wait_bar(&bars->s_full, gt & 1, abort_flag, a, 160));
        if (!ok) break;
        tc_fence_after();
        float p[64];
        {
          uint32_t* pu = reinterpret_cast<uint32_t*>(p);
          const uint32_t tS = tmem + lane_base + kSCol + 64 * half;
          tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(pu));
          tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(pu + 32));
          tmem_ld_wait();
        }
        // S is read: the next tile's K scales (read by S(t + 1)), then release S
        if (half == 0 && t + 1 < n) {
          tmem_st4(tmem + lane_base + kSfK, w_next[0], w_next[1], w_next[2], w_next[3]);
          tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(&bars->s_free);
        const int clo = klo - j * kTile - 64 * half, chi = khi - j * kTile - 64 * half;
        if (clo > 0 || chi < 64) {
#pragma unroll
          for (int c = 0; c < 64; ++c) p[c] = (c >= clo && c < chi) ? p[c] : -INFINITY;
        }
#pragma unroll
        for (int c = 0; c < 64; c += 2) {  // P = 2^(s scale log2e - LSE log2e)
          float x0, x1;
          f2_split(ffma2(f2(p[c], p[c + 1]), c2, nl2), x0, x1);
          p[c] = ex2_approx(x0);
          p[c + 1] = ex2_approx(x1);
        }
        ok = __all_sync(0xffffffffu, wait_bar(&bars->dp_full, gt & 1, abort_flag, a, 161));
        if (!ok) break;
        tc_fence_after();
        {
          uint32_t dp[64];
          const uint32_t tDP = tmem + lane_base + kDPCol + 64 * half;
          tmem_ld32(tDP, *reinterpret_cast<uint32_t(*)[32]>(dp));
          tmem_ld32(tDP + 32, *reinterpret_cast<uint32_t(*)[32]>(dp + 32));
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 64; c += 2) {  // dS = P (dP - D), in place of P
            float d0, d1;
            f2_split(fmul2(f2(p[c], p[c + 1]), fadd2(f2(__uint_as_float(dp[c]), __uint_as_float(dp[c + 1])), ndi)),
                     d0, d1);
            p[c] = d0;
            p[c + 1] = d1;
          }
        }
        // [32, 32] blocks: 32 query rows of this warp x 32 keys; the block's
        // scale from the warp-wide largest magnitude
        uint32_t pk[16], sfw = 0;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int E = mx::block_exponent(__reduce_max_sync(0xffffffffu, amax_bits32(p + 32 * k)));
          uint32_t c8[8];
          codes32(p + 32 * k, E, c8);
#pragma unroll
          for (int w = 0; w < 8; ++w) pk[8 * k + w] = c8[w];
          sfw |= static_cast<uint32_t>(E) << (8 * (2 * half + k));
        }
        tmem_st16(tmem + lane_base + kDPCol + 64 * half, pk);
        tmem_st1(tmem + lane_base + kSfDS + 4 * half + quarter, sfw);
        if (half == 0) {  // this K tile as dQ's MN-major B
          uint32_t w[4];
          mn_words(w_k, w);
          tmem_st4(tmem + lane_base + kSfKmn, w[0], w[1], w[2], w[3]);
        } else if (t + 1 < n) {  // the next V tile (read by dP(t + 1))
          tmem_st4(tmem + lane_base + kSfV, w_next[0], w_next[1], w_next[2], w_next[3]);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->ds_ready);
      }
      if (!ok) break;
      g += n;
      ok = __all_sync(0xffffffffu, wait_bar(&bars->acc_full, acc_cnt & 1, abort_flag, a, 162));
      if (!ok) break;
      ++acc_cnt;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + kDQCol + 64 * half + 32 * c, v);
        tmem_ld_wait();
        if (valid) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * a.scale, __uint_as_float(v[2 * e + 1]) * a.scale);
          store_words16(dq_row + 32 * c, w, a.out_v8);
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->acc_empty);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ============================================================================ dK / dV
namespace kvc {
constexpr int kThreads = 512;  // warp 0 TMA, warp 1 MMA, warps 2-3 LSE / D staging, warps 4-15 three warpgroups
constexpr int kStep = 96;      // queries per step: three 32-query blocks
constexpr int kStepBytes = kStep * kD;
constexpr int kStages = 4;
constexpr int kKOff = 0, kVOff = kTileBytes, kQOff = 2 * kTileBytes;  // stage s: Q, then dO
constexpr int kLdOff = kQOff + kStages * 2 * kStepBytes;               // [2 slots][-LSE log2e, -D][96] fp32
constexpr int kBarOff = kLdOff + 2 * 2 * kStep * 4;
constexpr int kSmemBytes = kBarOff + 512;
constexpr uint32_t kSCol = 0, kDPCol = 128, kDVCol = 256, kDKCol = 384;
// scale factors in the columns the 96-wide S^T / dP^T leave free: K, V (A of
// S^T, dP^T), Q, dO (B of S^T, dP^T), dO and Q as the MN-major B of dV and dK,
// then P~^T and dS~^T (A of dV, dK: [3 query blocks][4 lane quarters])
constexpr uint32_t kSfK = 96, kSfV = 100, kSfQ = 104, kSfDO = 108, kSfDOmn = 112, kSfQmn = 116;
constexpr uint32_t kSfP = 224, kSfDS = 236;
// Register split (setmaxnreg): 512 threads x 128 at launch = 65536 >=
// 128 x 72 (control warpgroup) + 384 x 144 (activation warpgroups) = 64512.
constexpr int kCtlRegs = 72;
constexpr int kActRegs = 144;
struct Bars {
  uint64_t kv_full, kv_empty;
  uint64_t qd_full[kStages], qd_empty[kStages];
  uint64_t sf_ready, s_full, p_ready, dp_full, ds_ready, acc_full, acc_empty;
  uint64_t ld_full[2], ld_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Bars) <= 512, "barrier block overflows its slot");
static_assert(kSmemBytes <= 227 * 1024, "shared memory");
static_assert(kStepBytes % 1024 == 0, "stage tiles stay 1024-byte aligned");
static_assert(kCtlRegs * 128 + kActRegs * 384 <= 65536, "register split");
}  // namespace kvc

// 96-query steps [st0, st1) of a key-tile item whose query tiles are [lo, hi).
__device__ __forceinline__ void step_range(const mx::Item& it, int& st0, int& st1) {
  const int q_end = min(it.hi * kTile, it.lq);
  st0 = (it.lo * kTile) / kvc::kStep;
  st1 = (q_end + kvc::kStep - 1) / kvc::kStep;
}

__global__ void __launch_bounds__(kvc::kThreads, 1)
    dkdv_mx_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                   const AttnArgs a) {
  using namespace kvc;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) record_error(a.status, JATTN_ERR_UNSUPPORTED, 19, blockIdx.x);
    return;
  }
  uint8_t* sm = smem_raw;
  Bars* bars = reinterpret_cast<Bars*>(sm + kBarOff);
  float* ld = reinterpret_cast<float*>(sm + kLdOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &bars->abort_flag;

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    mbar_init(&bars->kv_empty, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->qd_full[s], 1);
      mbar_init(&bars->qd_empty[s], 1);
    }
    mbar_init(&bars->sf_ready, kTile);  // warpgroup 2 writes an item's first scales
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->p_ready, 3 * kTile);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->ds_ready, 3 * kTile);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, 3 * kTile);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars->ld_full[x], 64);
      mbar_init(&bars->ld_empty[x], 3 * kTile);
    }
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtlRegs));
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        uint32_t kv_cnt = 0, qd_it = 0;
        bool ok = true;
        mx::Item it;
        for (long long r = 0; ok && mx::load_item(a, r, it); ++r) {
          if (it.hi <= it.lo) continue;
          if (!(ok = wait_bar(&bars->kv_empty, (kv_cnt & 1) ^ 1, abort_flag, a, 170))) break;
          ++kv_cnt;
          const int yk = static_cast<int>(it.k0) + it.qt * kTile;  // qt: the key tile of a transposed item
          if (!(a.debug_flags & 1)) {
            mbar_arrive_expect_tx(&bars->kv_full, 2 * kTileBytes);
            tma_load_2d(sm + kKOff, &tmK, &bars->kv_full, it.h * kD, yk);
            tma_load_2d(sm + kVOff, &tmV, &bars->kv_full, it.h * kD, yk);
          }
          int st0, st1;
          step_range(it, st0, st1);
          for (int st = st0; st < st1 && ok; ++st, ++qd_it) {
            const int s = qd_it % kStages;
            if (!(ok = wait_bar(&bars->qd_empty[s], ((qd_it / kStages) & 1) ^ 1, abort_flag, a, 171))) break;
            const int yq = static_cast<int>(it.q0) + st * kStep;
            mbar_arrive_expect_tx(&bars->qd_full[s], 2 * kStepBytes);
            tma_load_2d(sm + kQOff + s * 2 * kStepBytes, &tmQ, &bars->qd_full[s], it.h * kD, yq);
            tma_load_2d(sm + kQOff + s * 2 * kStepBytes + kStepBytes, &tmDO, &bars->qd_full[s], it.h * kD, yq);
          }
        }
        if (kv_cnt > 0 && !(a.debug_flags & 1)) mx::drain_wait(&bars->kv_full, (kv_cnt - 1) & 1, a.timeout_ns);
        for (uint32_t i = (qd_it > kStages ? qd_it - kStages : 0); i < qd_it; ++i)
          mx::drain_wait(&bars->qd_full[i % kStages], (i / kStages) & 1, a.timeout_ns);
      }
      __syncwarp();
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        const uint32_t sQ0 = smem_u32(sm + kQOff);
        const uint64_t dK = sdesc_sw128(smem_u32(sm + kKOff), 16, 1024);
        const uint64_t dV = sdesc_sw128(smem_u32(sm + kVOff), 16, 1024);
        const uint64_t dQ0 = sdesc_sw128(sQ0, 16, 1024), dDO0 = sdesc_sw128(sQ0 + kStepBytes, 16, 1024);
        // Q and dO as MN-major B operands (N = the head columns, K = queries):
        // K block kb is 32 rows of 128 bytes further
        const uint64_t dQmn0 = sdesc_sw128(sQ0, kTile * 128, 1024);
        const uint64_t dDOmn0 = sdesc_sw128(sQ0 + kStepBytes, kTile * 128, 1024);
        constexpr uint64_t kStageUnits = (2 * kStepBytes) >> 4;
        uint32_t kv_cnt = 0, qd_it = 0, sf_cnt = 0, acc_cnt = 0, g = 0;  // g: steps so far
        bool ok = true;
        auto issue_s = [&](int s) {
#pragma unroll
          for (int kb = 0; kb < 4; ++kb)
            mma_mx_ss(tmem + kSCol, dK + 2 * kb, dQ0 + s * kStageUnits + 2 * kb,
                      idesc_mx_e4m3(kTile, kStep, false, false, kb, kb), tmem + kSfK, tmem + kSfQ, kb > 0);
          mma_commit(&bars->s_full);
        };
        auto issue_dp = [&](int s) {
#pragma unroll
          for (int kb = 0; kb < 4; ++kb)
            mma_mx_ss(tmem + kDPCol, dV + 2 * kb, dDO0 + s * kStageUnits + 2 * kb,
                      idesc_mx_e4m3(kTile, kStep, false, false, kb, kb), tmem + kSfV, tmem + kSfDO, kb > 0);
          mma_commit(&bars->dp_full);
        };
        mx::Item it;
        for (long long r = 0; ok && mx::load_item(a, r, it); ++r) {
          if (it.hi <= it.lo) continue;
          int st0, st1;
          step_range(it, st0, st1);
          const int n = st1 - st0;
          if (!(ok = wait_bar(&bars->kv_full, kv_cnt & 1, abort_flag, a, 180))) break;
          ++kv_cnt;
          if (!(ok = wait_bar(&bars->sf_ready, sf_cnt & 1, abort_flag, a, 181))) break;
          ++sf_cnt;
          if (!(ok = wait_bar(&bars->qd_full[qd_it % kStages], (qd_it / kStages) & 1, abort_flag, a, 182))) break;
          tc_fence_after();
          issue_s(qd_it % kStages);
          issue_dp(qd_it % kStages);
          // K and V feed only S^T and dP^T: released once the item's last pair of them has completed
          if (n == 1) mma_commit(&bars->kv_empty);
          for (int i = 0; i < n && ok; ++i) {
            const uint32_t qi = qd_it + i;
            const int s = qi % kStages, s1 = (qi + 1) % kStages;
            const bool more = i + 1 < n;
            if (i == 0 && !(ok = wait_bar(&bars->acc_empty, (acc_cnt & 1) ^ 1, abort_flag, a, 183))) break;
            if (!(ok = wait_bar(&bars->p_ready, (g + i) & 1, abort_flag, a, 184))) break;
            tc_fence_after();
#pragma unroll
            for (int kb = 0; kb < 3; ++kb)  // queries 32kb ..: P~^T of warpgroup kb at S^T columns 32kb
              mma_mx_ts(tmem + kDVCol, tmem + kSCol + 32 * kb, dDOmn0 + s * kStageUnits + kb * (32 * 128 / 16),
                        idesc_mx_e4m3(kTile, kD, false, true, 0, kb), tmem + kSfP + 4 * kb, tmem + kSfDOmn,
                        (kb > 0 || i > 0) ? 1u : 0u);
            if (more) {
              if (!(ok = wait_bar(&bars->qd_full[s1], ((qi + 1) / kStages) & 1, abort_flag, a, 185))) break;
              tc_fence_after();
              issue_s(s1);
            }
            if (!(ok = wait_bar(&bars->ds_ready, (g + i) & 1, abort_flag, a, 186))) break;
            tc_fence_after();
#pragma unroll
            for (int kb = 0; kb < 3; ++kb)
              mma_mx_ts(tmem + kDKCol, tmem + kDPCol + 32 * kb, dQmn0 + s * kStageUnits + kb * (32 * 128 / 16),
                        idesc_mx_e4m3(kTile, kD, false, true, 0, kb), tmem + kSfDS + 4 * kb, tmem + kSfQmn,
                        (kb > 0 || i > 0) ? 1u : 0u);
            mma_commit(&bars->qd_empty[s]);
            if (more) issue_dp(s1);
            if (i + 2 == n) mma_commit(&bars->kv_empty);
          }
          if (!ok) break;
          mma_commit(&bars->acc_full);
          ++acc_cnt;
          qd_it += n;
          g += n;
        }
        mma_commit(&bars->drain);
        mx::drain_wait(&bars->drain, 0, a.timeout_ns);
      }
      __syncwarp();
    } else {
      // ------------------------------------------------------------ LSE / D staging (warps 2, 3)
      // Per step: -LSE log2(e) and -D of the step's 96 queries into one of two
      // shared slots (0 for queries past the sequence or that see no key).
      const int t = threadIdx.x - 64;  // 0 .. 63
      uint32_t gs = 0;
      bool ok = true;
      mx::Item it;
      for (long long r = 0; ok && mx::load_item(a, r, it); ++r) {
        if (it.hi <= it.lo) continue;
        int st0, st1;
        step_range(it, st0, st1);
        for (int st = st0; st < st1; ++st, ++gs) {
          const int slot = gs & 1;
          ok = __all_sync(0xffffffffu, wait_bar(&bars->ld_empty[slot], ((gs >> 1) & 1) ^ 1, abort_flag, a, 175));
          if (!ok) break;
          for (int k = t; k < kStep; k += 64) {
            const int iq = st * kStep + k;
            float l2 = 0.0f, d = 0.0f;
            if (iq < it.lq) {
              const int64_t gi = (it.q0 + iq) * a.H + it.h;
              const float lse = a.f0[gi];
              if (lse > -INFINITY) {
                l2 = lse * kLog2e;
                d = a.f1[gi];
              }
            }
            ld[(slot * 2) * kStep + k] = -l2;
            ld[(slot * 2 + 1) * kStep + k] = -d;
          }
          mbar_arrive(&bars->ld_full[slot]);
        }
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kActRegs));
    // ------------------------------------------------------------ activation warpgroups
    const int grp = (warp - 4) >> 2;  // query block of every step: S^T / dP^T columns [32 grp, 32 grp + 32)
    const int quarter = warp & 3;
    const int row = 32 * quarter + lane;  // TMEM lane == key row of the tile
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    uint32_t g = 0, acc_cnt = 0;
    bool ok = true;
    mx::Item it;
    for (long long r = 0; ok && mx::load_item(a, r, it); ++r) {
      const int jl = it.qt * kTile + row;  // sequence-local key row
      const bool valid = jl < it.lkv;
      const int64_t gk = (it.k0 + jl) * a.H + it.h;
      if (it.hi <= it.lo) {  // no query sees these keys: dV (warpgroup 0) and dK (1) rows are zero
        if (valid && grp < 2) {
          uint4* dst = reinterpret_cast<uint4*>((grp == 0 ? a.out1 : a.out0) + gk * kD);
          for (int e = 0; e < kD / 8; ++e) dst[e] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      int st0, st1;
      step_range(it, st0, st1);
      const int n = st1 - st0;
      int ilo, ihi;
      query_interval(jl, it.lkv - it.lq, it.lq, a.mask, a.window, ilo, ihi);
      if (!valid) ihi = ilo;
      const int kv_first = a.bs_kv[it.b], kv_last = max(a.bs_kv[it.b + 1] - 1, kv_first);
      const int q_first = a.bs_q[it.b], q_last = max(a.bs_q[it.b + 1] - 1, q_first);
      if (grp == 2) {  // scales of K, V and of the first step's Q, dO
        uint32_t w[4], w3[3];
        mx::kv_scale_load(a.sf_k, kv_first, kv_last, it.qt, a.H, it.h, w);
        tmem_st4(tmem + lane_base + kSfK, w[0], w[1], w[2], w[3]);
        mx::kv_scale_load(a.sf_v, kv_first, kv_last, it.qt, a.H, it.h, w);
        tmem_st4(tmem + lane_base + kSfV, w[0], w[1], w[2], w[3]);
        mx::block_words(a.sf_q, q_first, q_last, 3 * st0, a.H, it.h, w3);
        tmem_st4(tmem + lane_base + kSfQ, w3[0], w3[1], w3[2], 0u);
        mx::block_words(a.sf_do, q_first, q_last, 3 * st0, a.H, it.h, w3);
        tmem_st4(tmem + lane_base + kSfDO, w3[0], w3[1], w3[2], 0u);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->sf_ready);
      }
      const uint64_t c2 = f2(a.scale_log2, a.scale_log2);
      for (int i = 0; i < n; ++i) {
        const int st = st0 + i;
        const uint32_t gt = g + i;
        const int slot = gt & 1;
        const bool more = i + 1 < n;
        // scale words this step hands over, loaded before the waits:
        // warpgroup 0 this step's dO and Q (the MN-major B of dV, dK),
        // warpgroup 1 the next step's Q and dO (B of S^T, dP^T)
        uint32_t wa[3] = {0, 0, 0}, wb[3] = {0, 0, 0};
        if (grp == 0) {
          mx::block_words(a.sf_do, q_first, q_last, 3 * st, a.H, it.h, wa);
          mx::block_words(a.sf_q, q_first, q_last, 3 * st, a.H, it.h, wb);
        } else if (grp == 1 && more) {
          mx::block_words(a.sf_q, q_first, q_last, 3 * (st + 1), a.H, it.h, wa);
          mx::block_words(a.sf_do, q_first, q_last, 3 * (st + 1), a.H, it.h, wb);
        }
        ok = __all_sync(0xffffffffu, wait_bar(&bars->ld_full[slot], (gt >> 1) & 1, abort_flag, a, 190));
        ok = ok && __all_sync(0xffffffffu, wait_bar(&bars->s_full, gt & 1, abort_flag, a, 191));
        if (!ok) break;
        tc_fence_after();
        float p[32];
        tmem_ld32(tmem + lane_base + kSCol + 32 * grp, *reinterpret_cast<uint32_t(*)[32]>(p));
        tmem_ld_wait();
        const int c0 = st * kStep + 32 * grp;  // sequence-local query of column 0
        const int clo = ilo - c0, chi = ihi - c0;
        const ulonglong2* nl = reinterpret_cast<const ulonglong2*>(ld + (slot * 2) * kStep + 32 * grp);
        float xmax = -INFINITY;
#pragma unroll
        for (int c = 0; c < 32; c += 4) {  // exponent arguments s scale log2e - LSE log2e
          const ulonglong2 l4 = nl[c / 4];
          float x0, x1, x2, x3;
          f2_split(ffma2(f2(p[c], p[c + 1]), c2, l4.x), x0, x1);
          f2_split(ffma2(f2(p[c + 2], p[c + 3]), c2, l4.y), x2, x3);
          p[c] = x0;
          p[c + 1] = x1;
          p[c + 2] = x2;
          p[c + 3] = x3;
        }
        if (clo > 0 || chi < 32) {
#pragma unroll
          for (int c = 0; c < 32; ++c) p[c] = (c >= clo && c < chi) ? p[c] : -INFINITY;
        }
        {  // three-input maxima, four chains
          float mp[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int c = 0; c < 32; c += 8)
#pragma unroll
            for (int e = 0; e < 4; ++e) mp[e] = fmax3(mp[e], p[c + 2 * e], p[c + 2 * e + 1]);
          xmax = fmax3(mp[0], mp[1], fmaxf(mp[2], mp[3]));
        }
        // P~ of this key row's 32 queries: one scale 2^e from the largest P,
        // codes of P / 2^e; P itself (for dS) is the scaled value times 2^e
        const int e = mx::p_block_exp(xmax);
        const uint64_t ne2 = f2(-static_cast<float>(e), -static_cast<float>(e)), pe2 = f2(pow2i(e), pow2i(e));
        uint32_t pk[8];
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          float y[4];
#pragma unroll
          for (int b = 0; b < 4; b += 2) {
            float x0, x1;
            f2_split(fadd2(f2(p[4 * w + b], p[4 * w + b + 1]), ne2), x0, x1);
            y[b] = ex2_approx(x0);
            y[b + 1] = ex2_approx(x1);
          }
          pk[w] = pack_e4m3x2(y[0], y[1]) | (pack_e4m3x2(y[2], y[3]) << 16);
#pragma unroll
          for (int b = 0; b < 4; b += 2) f2_split(fmul2(f2(y[b], y[b + 1]), pe2), p[4 * w + b], p[4 * w + b + 1]);
        }
        tmem_st8(tmem + lane_base + kSCol + 32 * grp, pk);
        tmem_st1(tmem + lane_base + kSfP + 4 * grp + quarter, static_cast<uint32_t>(127 + e));
        if (grp == 0) {  // dO as dV's MN-major B
          uint32_t w[4];
          mn_words(wa, w);
          tmem_st4(tmem + lane_base + kSfDOmn, w[0], w[1], w[2], w[3]);
        } else if (grp == 1 && more) {  // next step's Q (B of S^T(i + 1))
          tmem_st4(tmem + lane_base + kSfQ, wa[0], wa[1], wa[2], 0u);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->p_ready);

        ok = __all_sync(0xffffffffu, wait_bar(&bars->dp_full, gt & 1, abort_flag, a, 192));
        if (!ok) break;
        tc_fence_after();
        {
          uint32_t dp[32];
          tmem_ld32(tmem + lane_base + kDPCol + 32 * grp, dp);
          tmem_ld_wait();
          const ulonglong2* nd = reinterpret_cast<const ulonglong2*>(ld + (slot * 2 + 1) * kStep + 32 * grp);
#pragma unroll
          for (int c = 0; c < 32; c += 4) {  // dS = P (dP - D), in place of P
            const ulonglong2 d4 = nd[c / 4];
            float d0, d1, d2, d3;
            f2_split(fmul2(f2(p[c], p[c + 1]), fadd2(f2(__uint_as_float(dp[c]), __uint_as_float(dp[c + 1])), d4.x)),
                     d0, d1);
            f2_split(fmul2(f2(p[c + 2], p[c + 3]),
                           fadd2(f2(__uint_as_float(dp[c + 2]), __uint_as_float(dp[c + 3])), d4.y)),
                     d2, d3);
            p[c] = d0;
            p[c + 1] = d1;
            p[c + 2] = d2;
            p[c + 3] = d3;
          }
        }
        // the [32, 32] block: this warp's 32 key rows x the warpgroup's 32 queries
        const int E = mx::block_exponent(__reduce_max_sync(0xffffffffu, amax_bits32(p)));
        codes32(p, E, pk);
        tmem_st8(tmem + lane_base + kDPCol + 32 * grp, pk);
        tmem_st1(tmem + lane_base + kSfDS + 4 * grp + quarter, static_cast<uint32_t>(E));
        if (grp == 0) {  // Q as dK's MN-major B
          uint32_t w[4];
          mn_words(wb, w);
          tmem_st4(tmem + lane_base + kSfQmn, w[0], w[1], w[2], w[3]);
        } else if (grp == 1 && more) {  // next step's dO (B of dP^T(i + 1))
          tmem_st4(tmem + lane_base + kSfDO, wb[0], wb[1], wb[2], 0u);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->ds_ready);
        mbar_arrive(&bars->ld_empty[slot]);
      }
      if (!ok) break;
      g += n;
      // ---------------- epilogue: 8 chunks of 32 columns (dV 0-3, dK 4-7), 3 / 3 / 2 per warpgroup
      ok = __all_sync(0xffffffffu, wait_bar(&bars->acc_full, acc_cnt & 1, abort_flag, a, 193));
      if (!ok) break;
      ++acc_cnt;
      tc_fence_after();
      const int ch0 = 3 * grp, ch1 = min(3 * grp + 3, 8);
      for (int ch = ch0; ch < ch1; ++ch) {
        uint32_t v[32];
        const bool is_dk = ch >= 4;
        tmem_ld32(tmem + lane_base + (is_dk ? kDKCol : kDVCol) + 32 * (ch & 3), v);
        tmem_ld_wait();
        if (valid) {
          const float mul = is_dk ? a.scale : 1.0f;
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
          store_words16((is_dk ? a.out0 : a.out1) + gk * kD + 32 * (ch & 3), w, a.out_v8);
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->acc_empty);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_mx_di(const int64_t* q_off, int B, int H, int64_t max_blocks, const uint8_t* dout,
                         const uint8_t* dout_scales, const int* block_start, const void* o, float* di,
                         cudaStream_t stream) {
  const int64_t warps = max_blocks * H;
  if (warps == 0) return cudaSuccess;
  const int64_t grid = (warps + kDiWarps - 1) / kDiWarps;
  mx_di_kernel<<<static_cast<unsigned>(grid), kDiWarps * 32, 0, stream>>>(
      q_off, B, H, dout, dout_scales, block_start, static_cast<const __nv_bfloat16*>(o), di, max_blocks);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq_mx(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                             const CUtensorMap& dout, const AttnArgs& a, int grid, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(dq_mx_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dqc::kSmemBytes);
  if (e != cudaSuccess) return e;
  dq_mx_kernel<<<grid, dqc::kThreads, dqc::kSmemBytes, stream>>>(q, k, v, dout, a);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv_mx(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                               const CUtensorMap& dout, const AttnArgs& a, int grid, cudaStream_t stream) {
  cudaError_t e =
      cudaFuncSetAttribute(dkdv_mx_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kvc::kSmemBytes);
  if (e != cudaSuccess) return e;
  dkdv_mx_kernel<<<grid, kvc::kThreads, kvc::kSmemBytes, stream>>>(q, k, v, dout, a);
  return cudaGetLastError();
}

}  // namespace jattn
