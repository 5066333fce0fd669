// Forward pass of jagged softmax attention on MXFP8 operands, sm_103a.
//
// "GEM Training" post, section "Low Precision Flash Attention": FlashAttention
// with block-scaled FP8 operands, the scale factors kept in tensor memory next
// to the accumulators, and the softmax output P quantized to FP8 inside the
// softmax with the scale its row maximum fixes. Q, K and V arrive as E4M3
// codes with one E8M0 scale per 32 x 32 block (jattn_mxfp8_quantize); the two
// products run as block-scaled tcgen05 MMAs (kind::mxf8f6f4, K = 32 per
// instruction) with fp32 accumulation.
//
// One persistent CTA per SM walks the longest-first schedule of 128-row query
// tiles. Roles (8 warps):
//   warp 0      TMA producer: the item's Q codes (two stages), K and V codes
//               (four stages each), 16 KB per 128 x 128 tile
//   warp 1      MMA issuer: S = Q K^T (4 MMAs), then O += P V (4 MMAs, P read
//               from TMEM)
//   warps 4-7   softmax, one query row per thread; they also write the scale
//               factors into TMEM before the MMAs that read them
// TMEM columns: S [0, 128), O [128, 256), scales of Q, K, P, V at 256, 260,
// 264, 268 (4 columns each). The running maximum moves whenever a row's
// maximum grows (O is rescaled then), so every P is at most 1 and its scale is
// the constant 2^-8 (E4M3's largest power of two is 2^8): P codes are
// E4M3(P * 2^8). The row sum l uses the unquantized P, in fp32.
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace jattn {

namespace {

constexpr int kThreads = 256;
constexpr int kD = 128;                 // head dimension (the codes of one head row fill 128 bytes)
constexpr int kTileBytes = kTile * kD;  // one 128-row tile of E4M3 codes
constexpr int kQStages = 2, kKVStages = 4;
constexpr int kQOff = 0;
constexpr int kKOff = kQOff + kQStages * kTileBytes;
constexpr int kVOff = kKOff + kKVStages * kTileBytes;
constexpr int kBarOff = kVOff + kKVStages * kTileBytes;
constexpr int kSmemBytes = kBarOff + 256;
constexpr uint32_t kSCol = 0, kOCol = 128, kSfQ = 256, kSfK = 260, kSfP = 264, kSfV = 268;
constexpr uint32_t kPScaleWord = 0x77777777u;  // E8M0 119 = 2^-8 in every byte

struct MxBars {
  uint64_t q_full[kQStages], q_empty[kQStages];
  uint64_t k_full[kKVStages], k_empty[kKVStages], v_full[kKVStages], v_empty[kKVStages];
  uint64_t sf_ready, s_full, p_full, o_full, o_empty, drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(MxBars) <= 256, "barrier block overflows its slot");
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > timeout_ns) return;
  }
}

struct MxItem {
  int b, qt, lo, hi, h, lq, lkv;
  int64_t q0, k0;
};

__device__ __forceinline__ bool load_mx_item(const AttnArgs& a, long long round, MxItem& it) {
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

__global__ void __launch_bounds__(kThreads, 1)
    fwd_mx_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const AttnArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) record_error(a.status, JATTN_ERR_UNSUPPORTED, 19, blockIdx.x);
    return;
  }
  uint8_t* sm = smem_raw;
  MxBars* bars = reinterpret_cast<MxBars*>(sm + kBarOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &bars->abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(&bars->q_full[s], 1);
      mbar_init(&bars->q_empty[s], 1);
    }
    for (int s = 0; s < kKVStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    mbar_init(&bars->sf_ready, kTile);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->p_full, kTile);
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->o_empty, kTile);
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      uint32_t q_it = 0, kv_it = 0;
      bool ok = true;
      MxItem it;
      for (long long r = 0; ok && load_mx_item(a, r, it); ++r) {
        if (it.hi <= it.lo) continue;
        const int qs = q_it % kQStages;
        if (!(ok = wait_bar(&bars->q_empty[qs], ((q_it / kQStages) & 1) ^ 1, abort_flag, a, 110))) break;
        if (!(a.debug_flags & 1)) {
          mbar_arrive_expect_tx(&bars->q_full[qs], kTileBytes);
          tma_load_2d(sm + kQOff + qs * kTileBytes, &tmQ, &bars->q_full[qs], it.h * kD,
                      static_cast<int>(it.q0) + it.qt * kTile);
        }
        ++q_it;
        for (int j = it.lo; j < it.hi && ok; ++j, ++kv_it) {
          const int s = kv_it % kKVStages;
          const uint32_t par = ((kv_it / kKVStages) & 1) ^ 1;
          const int y = static_cast<int>(it.k0) + j * kTile;
          if (!(ok = wait_bar(&bars->k_empty[s], par, abort_flag, a, 111))) break;
          mbar_arrive_expect_tx(&bars->k_full[s], kTileBytes);
          tma_load_2d(sm + kKOff + s * kTileBytes, &tmK, &bars->k_full[s], it.h * kD, y);
          if (!(ok = wait_bar(&bars->v_empty[s], par, abort_flag, a, 112))) break;
          mbar_arrive_expect_tx(&bars->v_full[s], kTileBytes);
          tma_load_2d(sm + kVOff + s * kTileBytes, &tmV, &bars->v_full[s], it.h * kD, y);
        }
      }
      // let every copy this thread started land before the CTA can exit
      for (uint32_t i = (q_it > kQStages ? q_it - kQStages : 0); i < q_it; ++i)
        if (!(a.debug_flags & 1)) drain_wait(&bars->q_full[i % kQStages], (i / kQStages) & 1, a.timeout_ns);
      for (uint32_t i = (kv_it > kKVStages ? kv_it - kKVStages : 0); i < kv_it; ++i) {
        drain_wait(&bars->k_full[i % kKVStages], (i / kKVStages) & 1, a.timeout_ns);
        drain_wait(&bars->v_full[i % kKVStages], (i / kKVStages) & 1, a.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t sQ = smem_u32(sm + kQOff), sK = smem_u32(sm + kKOff), sV = smem_u32(sm + kVOff);
      // descriptors of the tile bases; K block kb of a K-major tile is 32 bytes
      // further (2 units), of the MN-major V tile 32 rows of 128 bytes further
      const uint64_t dQ = sdesc_sw128(sQ, 16, 1024), dK = sdesc_sw128(sK, 16, 1024);
      const uint64_t dV = sdesc_sw128(sV, kTile * 128, 1024);
      constexpr uint64_t kTileUnits = kTileBytes >> 4;
      uint32_t q_it = 0, kv_it = 0, sf_cnt = 0, p_cnt = 0, o_cnt = 0;
      bool ok = true;
      MxItem it;
      auto issue_s = [&](int qs, int ks) {
#pragma unroll
        for (int kb = 0; kb < 4; ++kb)
          mma_mx_ss(tmem + kSCol, dQ + qs * kTileUnits + 2 * kb, dK + ks * kTileUnits + 2 * kb,
                    idesc_mx_e4m3(kTile, kTile, false, false, kb, kb), tmem + kSfQ, tmem + kSfK, kb > 0);
        mma_commit(&bars->s_full);
      };
      for (long long r = 0; ok && load_mx_item(a, r, it); ++r) {
        if (it.hi <= it.lo) continue;
        const int qs = q_it % kQStages;
        if (!(ok = wait_bar(&bars->q_full[qs], (q_it / kQStages) & 1, abort_flag, a, 120))) break;
        // the softmax warps have written the scales of Q and of the first K tile
        if (!(ok = wait_bar(&bars->sf_ready, sf_cnt & 1, abort_flag, a, 121))) break;
        ++sf_cnt;
        const int s0 = kv_it % kKVStages;
        if (!(ok = wait_bar(&bars->k_full[s0], (kv_it / kKVStages) & 1, abort_flag, a, 122))) break;
        tc_fence_after();
        issue_s(qs, s0);
        mma_commit(&bars->k_empty[s0]);
        for (int j = it.lo; j < it.hi && ok; ++j) {
          const uint32_t ki = kv_it + (j - it.lo);
          const int s = ki % kKVStages;
          if (!(ok = wait_bar(&bars->v_full[s], (ki / kKVStages) & 1, abort_flag, a, 123))) break;
          if (j == it.lo && !(ok = wait_bar(&bars->o_empty, (o_cnt & 1) ^ 1, abort_flag, a, 124))) break;
          // P of this tile, the scales of V and of the next K tile are in TMEM
          if (!(ok = wait_bar(&bars->p_full, p_cnt & 1, abort_flag, a, 125))) break;
          ++p_cnt;
          tc_fence_after();
#pragma unroll
          for (int kb = 0; kb < 4; ++kb)
            mma_mx_ts(tmem + kOCol, tmem + kSCol + 8 * kb, dV + s * kTileUnits + kb * (32 * 128 / 16),
                      idesc_mx_e4m3(kTile, kD, false, true, kb, kb), tmem + kSfP, tmem + kSfV,
                      (kb > 0 || j > it.lo) ? 1u : 0u);
          mma_commit(&bars->v_empty[s]);
          if (j + 1 < it.hi) {
            const int s1 = (ki + 1) % kKVStages;
            if (!(ok = wait_bar(&bars->k_full[s1], ((ki + 1) / kKVStages) & 1, abort_flag, a, 126))) break;
            tc_fence_after();
            issue_s(qs, s1);
            mma_commit(&bars->k_empty[s1]);
          }
        }
        if (!ok) break;
        mma_commit(&bars->o_full);
        ++o_cnt;
        mma_commit(&bars->q_empty[qs]);
        ++q_it;
        kv_it += it.hi - it.lo;
      }
      mma_commit(&bars->drain);
      drain_wait(&bars->drain, 0, a.timeout_ns);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax warps
    const int quarter = warp & 3;
    const int row = 32 * quarter + lane;  // TMEM lane == query row of the tile
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    const uint32_t tS = tmem + lane_base + kSCol, tO = tmem + lane_base + kOCol;
    uint32_t s_cnt = 0, o_cnt = 0;
    // P's scale is 2^-8 for every row and K block
    tmem_st4(tmem + lane_base + kSfP, kPScaleWord, kPScaleWord, kPScaleWord, kPScaleWord);
    tmem_st_wait();
    bool ok = true;
    MxItem it;
    for (long long r = 0; ok && load_mx_item(a, r, it); ++r) {
      const int il = it.qt * kTile + row;
      const bool valid = il < it.lq;
      const int64_t grow = it.q0 + il;
      __nv_bfloat16* orow = a.out0 + (grow * a.H + it.h) * kD;
      if (it.hi <= it.lo) {  // no key tile: rows see nothing
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow);
          for (int e = 0; e < kD / 8; ++e) dst[e] = make_uint4(0, 0, 0, 0);
          a.f0[grow * a.H + it.h] = -INFINITY;
        }
        continue;
      }
      const int delta = it.lkv - it.lq;
      int klo, khi;
      key_interval(il, delta, it.lkv, a.mask, a.window, klo, khi);
      if (!valid) khi = klo;
      // Scales in the replicated layout: lane l of every quarter, column c
      // holds index 32c + l (query row / key row / V column); Q and K carry
      // their 4 column blocks in the word's bytes, V its 4 key blocks.
      {
        uint32_t wq[4], wk[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          wq[c] = sf_word(a.sf_q, row_block(a.bs_q, it.b, 4 * it.qt + c), a.H, it.h);
          wk[c] = sf_word(a.sf_k, row_block(a.bs_kv, it.b, 4 * it.lo + c), a.H, it.h);
        }
        tmem_st4(tmem + lane_base + kSfQ, wq[0], wq[1], wq[2], wq[3]);
        tmem_st4(tmem + lane_base + kSfK, wk[0], wk[1], wk[2], wk[3]);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->sf_ready);
      }
      float m_run = -INFINITY, l_run = 0.0f;
      for (int j = it.lo; j < it.hi; ++j) {
        ok = __all_sync(0xffffffffu, wait_bar(&bars->s_full, s_cnt & 1, abort_flag, a, 130));
        if (!ok) break;
        ++s_cnt;
        tc_fence_after();
        float s[kTile];
        {
          uint32_t* su = reinterpret_cast<uint32_t*>(s);
#pragma unroll
          for (int c = 0; c < kTile / 32; ++c) tmem_ld32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(su + c * 32));
          tmem_ld_wait();
        }
        const int clo = klo - j * kTile, chi = khi - j * kTile;
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < kTile; ++c) {
          s[c] = (c >= clo && c < chi) ? s[c] : -INFINITY;
          mx = fmaxf(mx, s[c]);
        }
        const float m_new = fmaxf(m_run, mx * a.scale_log2);
        float alpha = 1.0f;
        if (m_new > m_run) {  // the running maximum moves whenever it grows: P <= 1
          alpha = (m_run == -INFINITY) ? 0.0f : ex2_approx(m_run - m_new);
          l_run *= alpha;
          m_run = m_new;
        }
        // O holds the products of the earlier tiles (complete: this S tile was
        // issued after them); scale it to the new maximum
        if (j > it.lo && __any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll
          for (int c = 0; c < kD / 16; ++c) {
            uint32_t o[16];
            tmem_ld16(tO + c * 16, o);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st16(tO + c * 16, o);
          }
        }
        const float mref = (m_run == -INFINITY) ? 0.0f : m_run;
        float lsum = 0.0f;
#pragma unroll
        for (int c0 = 0; c0 < kTile; c0 += 64) {
          uint32_t pk[16];
#pragma unroll
          for (int w = 0; w < 16; ++w) {  // word w: keys c0 + 4w .. c0 + 4w + 3, byte = key % 4
            float p[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              p[e] = ex2_approx(fmaf(s[c0 + 4 * w + e], a.scale_log2, -mref));
              lsum += p[e];
            }
            pk[w] = pack_e4m3x2(p[0] * 256.0f, p[1] * 256.0f) | (pack_e4m3x2(p[2] * 256.0f, p[3] * 256.0f) << 16);
          }
          // P codes of 64 keys in 16 columns, over the S columns already read
          tmem_st16(tS + c0 / 4, pk);
        }
        l_run += lsum;
        // scales of this V tile (its 4 key blocks in the bytes of each D-column
        // block's word) and of the next K tile, for the MMAs this handover
        // releases; the MMAs that read the previous ones have completed
        {
          const int g0 = row_block(a.bs_kv, it.b, 4 * j), g1 = row_block(a.bs_kv, it.b, 4 * j + 1);
          const int g2 = row_block(a.bs_kv, it.b, 4 * j + 2), g3 = row_block(a.bs_kv, it.b, 4 * j + 3);
          const uint32_t v0 = sf_word(a.sf_v, g0, a.H, it.h), v1 = sf_word(a.sf_v, g1, a.H, it.h);
          const uint32_t v2 = sf_word(a.sf_v, g2, a.H, it.h), v3 = sf_word(a.sf_v, g3, a.H, it.h);
          uint32_t wv[4];
#pragma unroll
          for (int c = 0; c < 4; ++c)  // column block c: byte kb = key block kb's scale
            wv[c] = ((v0 >> (8 * c)) & 0xffu) | (((v1 >> (8 * c)) & 0xffu) << 8) |
                    (((v2 >> (8 * c)) & 0xffu) << 16) | (((v3 >> (8 * c)) & 0xffu) << 24);
          tmem_st4(tmem + lane_base + kSfV, wv[0], wv[1], wv[2], wv[3]);
          if (j + 1 < it.hi) {
            uint32_t wk[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) wk[c] = sf_word(a.sf_k, row_block(a.bs_kv, it.b, 4 * (j + 1) + c), a.H, it.h);
            tmem_st4(tmem + lane_base + kSfK, wk[0], wk[1], wk[2], wk[3]);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->p_full);
      }
      if (!ok) break;
      // ---------------- epilogue
      ok = __all_sync(0xffffffffu, wait_bar(&bars->o_full, o_cnt & 1, abort_flag, a, 131));
      if (!ok) break;
      ++o_cnt;
      tc_fence_after();
      const float oscale = (l_run > 0.0f) ? 1.0f / l_run : 0.0f;
#pragma unroll
      for (int c = 0; c < kD / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + c * 32, o);
        tmem_ld_wait();
        if (valid) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * oscale, __uint_as_float(o[2 * e + 1]) * oscale);
          store_words16(orow + c * 32, w, a.out_v8);
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->o_empty);
      if (valid)
        a.f0[grow * a.H + it.h] = (l_run > 0.0f) ? (m_run + __log2f(l_run)) * 0.6931471805599453f : -INFINITY;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_fwd_mx(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const AttnArgs& a,
                          int grid, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(fwd_mx_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  fwd_mx_kernel<<<grid, kThreads, kSmemBytes, stream>>>(q, k, v, a);
  return cudaGetLastError();
}

}  // namespace jattn
