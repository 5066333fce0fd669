// Forward pass of jagged softmax attention on MXFP8 operands, sm_103a.
//
// "GEM Training" post, section "Low Precision Flash Attention": FlashAttention
// with block-scaled FP8 operands, the scale factors kept in tensor memory next
// to the accumulators, and the softmax output P quantized to FP8 inside the
// softmax, with scales its maxima fix. Q, K and V arrive as E4M3 codes with one
// E8M0 scale per 32 x 32 block (jattn_mxfp8_quantize); both products run as
// block-scaled tcgen05 MMAs (kind::mxf8f6f4, K = 32 per instruction) with fp32
// accumulation.
//
// One persistent CTA per SM walks the longest-first schedule of 128-row query
// tiles. Roles (12 warps):
//   warp 0      TMA producer: the item's Q codes (two stages), K and V codes of
//               one key tile per ring stage (four stages), 16 KB per tile
//   warp 1      MMA issuer: S(j) = Q K(j)^T into one of two S buffers, two key
//               tiles ahead of the softmax, and O += P(j) V(j) with P read
//               from TMEM
//   warps 4-11  two softmax warpgroups; warpgroup h owns key columns
//               [64h, 64h + 64) of every S tile and O columns [64h, 64h + 64);
//               warps w and w + 4 hold the same rows and combine row maxima and
//               sums through shared memory
// One thread issues a tcgen05 operation (MMA or commit) about every 60
// cycles at best, and every barrier wait adds more, so each key tile costs it
// 8 MMAs, three commits and two waits: K and V share a ring stage, one barrier
// and one release, and the S buffers make the MMAs of tile j + 2 independent
// of the softmax of tile j.
// TMEM columns: S0 [0, 128), S1 [128, 256), O [256, 384), scale factors from
// 384. P of warpgroup h overwrites columns [64h, 64h + 16) of its S buffer as
// E4M3 codes, 4 per column; every 32-key block of a row has its own scale,
// 2^(ceil(log2 max) - 8) of that block's largest P, so P / scale is at most
// 2^8 and small values keep their precision. The running maximum is lazy
// (it moves when a row's maximum grows by more than 2^8); the row sum l
// uses the unquantized P in fp32.
#include <cstdint>

#include "common.cuh"
#include "kernels.h"
#include "mx_common.cuh"

namespace jattn {

namespace {

constexpr int kThreads = 384;
constexpr int kD = 128;                 // head dimension (the codes of one head row fill 128 bytes)
constexpr int kTileBytes = kTile * kD;  // one 128-row tile of E4M3 codes
constexpr int kQStages = 2, kKVStages = 4;
constexpr int kQOff = 0;
constexpr int kKOff = kQOff + kQStages * kTileBytes;
constexpr int kVOff = kKOff + kKVStages * kTileBytes;
constexpr int kBarOff = kVOff + kKVStages * kTileBytes;
constexpr int kXchOff = kBarOff + 512;                 // [2 slots][2 halves][128 rows] fp32
constexpr int kSmemBytes = kXchOff + 2 * 2 * kTile * 4;
constexpr uint32_t kSCol = 0, kOCol = 256;
constexpr uint32_t kSfQ = 384, kSfK = 388, kSfV = 396, kSfP = 404;  // K, V: [2 buffers][4]; P: [2 buffers][2 halves][4]
constexpr float kRescaleLog2 = 8.0f;
// Register split (setmaxnreg): 384 threads x 168 at launch = 64512 =
// 128 x 104 (control warpgroup) + 256 x 200 (softmax warpgroups).
constexpr int kCtlRegs = 104;
constexpr int kActRegs = 200;

struct MxBars {
  uint64_t q_full[kQStages], q_empty[kQStages];
  uint64_t kv_full[kKVStages], kv_empty[kKVStages];
  // p_full is per S buffer: warps of different lane quarters may be a key tile
  // apart (the S buffers let them run one tile ahead of a slower quarter), and
  // one barrier would mix the arrivals of two tiles
  uint64_t sf_ready, s_full[2], p_full[2], pv_done, o_full, o_empty, drain;
  uint64_t xbar[2][4];  // row exchange per (slot, lane quarter), 64 arrivals
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(MxBars) <= 512, "barrier block overflows its slot");
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

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
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    mbar_init(&bars->sf_ready, kTile);  // warpgroup 0 writes the Q and K scales
    mbar_init(&bars->s_full[0], 1);
    mbar_init(&bars->s_full[1], 1);
    mbar_init(&bars->p_full[0], 2 * kTile);
    mbar_init(&bars->p_full[1], 2 * kTile);
    mbar_init(&bars->pv_done, 1);
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->o_empty, 2 * kTile);
    mbar_init(&bars->drain, 1);
    for (int x = 0; x < 2; ++x)
      for (int qq = 0; qq < 4; ++qq) mbar_init(&bars->xbar[x][qq], 64);
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
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        uint32_t q_it = 0, kv_it = 0;
        bool ok = true;
        mx::Item it;
        for (long long r = 0; ok && mx::load_item(a, r, it); ++r) {
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
            if (!(ok = wait_bar(&bars->kv_empty[s], ((kv_it / kKVStages) & 1) ^ 1, abort_flag, a, 111))) break;
            const int y = static_cast<int>(it.k0) + j * kTile;
            mbar_arrive_expect_tx(&bars->kv_full[s], 2 * kTileBytes);
            tma_load_2d(sm + kKOff + s * kTileBytes, &tmK, &bars->kv_full[s], it.h * kD, y);
            tma_load_2d(sm + kVOff + s * kTileBytes, &tmV, &bars->kv_full[s], it.h * kD, y);
          }
        }
        // let every copy this thread started land before the CTA can exit
        if (!(a.debug_flags & 1))
          for (uint32_t i = (q_it > kQStages ? q_it - kQStages : 0); i < q_it; ++i)
            mx::drain_wait(&bars->q_full[i % kQStages], (i / kQStages) & 1, a.timeout_ns);
        for (uint32_t i = (kv_it > kKVStages ? kv_it - kKVStages : 0); i < kv_it; ++i)
          mx::drain_wait(&bars->kv_full[i % kKVStages], (i / kKVStages) & 1, a.timeout_ns);
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
        uint32_t q_it = 0, kv_it = 0, sf_cnt = 0, o_cnt = 0, g = 0;  // g: key tiles so far
        bool ok = true;
        mx::Item it;
        // S(t) of global key tile t into buffer t & 1 from ring stage ks
        auto issue_s = [&](int qs, uint32_t t, int ks) {
          const uint32_t b = t & 1;
#pragma unroll
          for (int kb = 0; kb < 4; ++kb)
            mma_mx_ss(tmem + kSCol + b * kTile, dQ + qs * kTileUnits + 2 * kb, dK + ks * kTileUnits + 2 * kb,
                      idesc_mx_e4m3(kTile, kTile, false, false, kb, kb), tmem + kSfQ, tmem + kSfK + 4 * b, kb > 0);
          mma_commit(&bars->s_full[b]);
        };
        for (long long r = 0; ok && mx::load_item(a, r, it); ++r) {
          if (it.hi <= it.lo) continue;
          const int qs = q_it % kQStages;
          const int n = it.hi - it.lo;
          if (!(ok = wait_bar(&bars->q_full[qs], (q_it / kQStages) & 1, abort_flag, a, 120))) break;
          // warpgroup 0 has written the scales of Q and of the first two K tiles
          if (!(ok = wait_bar(&bars->sf_ready, sf_cnt & 1, abort_flag, a, 121))) break;
          ++sf_cnt;
          for (int t = 0; t < 2 && t < n && ok; ++t) {
            const uint32_t ki = kv_it + t;
            if (!(ok = wait_bar(&bars->kv_full[ki % kKVStages], (ki / kKVStages) & 1, abort_flag, a, 122))) break;
            tc_fence_after();
            issue_s(qs, g + t, ki % kKVStages);
          }
          for (int t = 0; t < n && ok; ++t) {
            const uint32_t ki = kv_it + t, b = (g + t) & 1;
            const int s = ki % kKVStages;
            if (t == 0 && !(ok = wait_bar(&bars->o_empty, (o_cnt & 1) ^ 1, abort_flag, a, 123))) break;
            // P of this tile and the scales of its V are in TMEM
            if (!(ok = wait_bar(&bars->p_full[b], ((g + t) >> 1) & 1, abort_flag, a, 124))) break;
            tc_fence_after();
#pragma unroll
            for (int kb = 0; kb < 4; ++kb)  // keys 32kb.. : P of warpgroup kb / 2 at S columns 64 (kb / 2) + 8 (kb % 2)
              mma_mx_ts(tmem + kOCol, tmem + kSCol + b * kTile + 64 * (kb >> 1) + 8 * (kb & 1),
                        dV + s * kTileUnits + kb * (32 * 128 / 16), idesc_mx_e4m3(kTile, kD, false, true, kb, kb),
                        tmem + kSfP + 8 * b + 4 * (kb >> 1), tmem + kSfV + 4 * b, (kb > 0 || t > 0) ? 1u : 0u);
            mma_commit(&bars->pv_done);
            mma_commit(&bars->kv_empty[s]);  // K(t) was read two tiles ago, V(t) just now
            if (t + 2 < n) {
              const uint32_t k2 = ki + 2;
              if (!(ok = wait_bar(&bars->kv_full[k2 % kKVStages], (k2 / kKVStages) & 1, abort_flag, a, 125))) break;
              tc_fence_after();
              issue_s(qs, g + t + 2, k2 % kKVStages);
            }
          }
          if (!ok) break;
          mma_commit(&bars->o_full);
          ++o_cnt;
          mma_commit(&bars->q_empty[qs]);
          ++q_it;
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
    // ------------------------------------------------------------ softmax warpgroups
    const int half = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int row = 32 * quarter + lane;  // TMEM lane == query row of the tile
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    float* xch = reinterpret_cast<float*>(sm + kXchOff);
    uint32_t x_cnt = 0, o_cnt = 0, g = 0;  // g: key tiles so far (both warpgroups see the same)
    // Row exchange with the partner warp (the other warpgroup, same lanes):
    // both write, meet on the (slot, quarter) mbarrier with a bounded wait,
    // and read the partner's value; two alternating slots.
    auto exchange = [&](float v, bool& okr) -> float {
      const int slot = x_cnt & 1;
      const uint32_t par = (x_cnt >> 1) & 1;
      ++x_cnt;
      xch[(slot * 2 + half) * kTile + row] = v;
      mbar_arrive(&bars->xbar[slot][quarter]);
      okr = __all_sync(0xffffffffu, wait_bar(&bars->xbar[slot][quarter], par, abort_flag, a, 132)) && okr;
      return xch[(slot * 2 + (half ^ 1)) * kTile + row];
    };
    bool ok = true;
    mx::Item it;
    for (long long r = 0; ok && mx::load_item(a, r, it); ++r) {
      const int il = it.qt * kTile + row;
      const bool valid = il < it.lq;
      const int64_t grow = it.q0 + il;
      __nv_bfloat16* orow = a.out0 + (grow * a.H + it.h) * kD + 64 * half;
      if (it.hi <= it.lo) {  // no key tile: rows see nothing
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow);
          for (int e = 0; e < 8; ++e) dst[e] = make_uint4(0, 0, 0, 0);
          if (half == 0) a.f0[grow * a.H + it.h] = -INFINITY;
        }
        continue;
      }
      const int n = it.hi - it.lo;
      const int delta = it.lkv - it.lq;
      int klo, khi;
      key_interval(il, delta, it.lkv, a.mask, a.window, klo, khi);
      if (!valid) khi = klo;
      // the key side's row blocks of this sequence (scale rows clamp to them)
      const int kv_first = a.bs_kv[it.b], kv_last = max(a.bs_kv[it.b + 1] - 1, kv_first);
      if (half == 0) {  // scales of Q and of the item's first two K tiles
        uint32_t w[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) w[c] = mx::sf_word(a.sf_q, mx::row_block(a.bs_q, it.b, 4 * it.qt + c), a.H, it.h);
        tmem_st4(tmem + lane_base + kSfQ, w[0], w[1], w[2], w[3]);
        for (int t = 0; t < 2 && t < n; ++t) {
          mx::kv_scale_load(a.sf_k, kv_first, kv_last, it.lo + t, a.H, it.h, w);
          tmem_st4(tmem + lane_base + kSfK + 4 * ((g + t) & 1), w[0], w[1], w[2], w[3]);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->sf_ready);
      }
      float m_run = -INFINITY, l_run = 0.0f;
      for (int t = 0; t < n; ++t) {
        const int j = it.lo + t;
        const uint32_t gt = g + t, b = gt & 1;
        // scale words this step hands over (warpgroup 1: V tile j; warpgroup 0:
        // K tile j + 2), loaded before the wait so their latency is hidden
        uint32_t sw[4] = {0, 0, 0, 0};
        if (half == 1) mx::kv_scale_load(a.sf_v, kv_first, kv_last, j, a.H, it.h, sw);
        else if (t + 2 < n) mx::kv_scale_load(a.sf_k, kv_first, kv_last, j + 2, a.H, it.h, sw);
        ok = __all_sync(0xffffffffu, wait_bar(&bars->s_full[b], (gt >> 1) & 1, abort_flag, a, 130));
        if (!ok) break;
        tc_fence_after();
        const uint32_t tS = tmem + lane_base + kSCol + b * kTile + 64 * half;
        float s[64];
        {
          uint32_t* su = reinterpret_cast<uint32_t*>(s);
          tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(su));
          tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(su + 32));
          tmem_ld_wait();
        }
        const int clo = klo - j * kTile - 64 * half, chi = khi - j * kTile - 64 * half;
        if (clo > 0 || chi < 64) {  // edge tile: keys outside the row's range drop out
#pragma unroll
          for (int c = 0; c < 64; ++c) s[c] = (c >= clo && c < chi) ? s[c] : -INFINITY;
        }
        // maxima of the two 32-key blocks (three-input maxima, four chains each)
        float bm[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          float mp[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int c = 32 * k; c < 32 * k + 32; c += 8)
#pragma unroll
            for (int e = 0; e < 4; ++e) mp[e] = fmax3(mp[e], s[c + 2 * e], s[c + 2 * e + 1]);
          bm[k] = fmax3(mp[0], mp[1], fmaxf(mp[2], mp[3]));
        }
        const float mx = fmaxf(fmaxf(bm[0], bm[1]), exchange(fmaxf(bm[0], bm[1]), ok));
        if (!ok) break;
        const float m_new = mx * a.scale_log2;
        bool rescale = false;
        float alpha = 1.0f;
        if (m_run == -INFINITY) {
          m_run = m_new;  // O and l hold nothing yet for this row
        } else if (m_new > m_run + kRescaleLog2) {
          alpha = ex2_approx(m_run - m_new);
          rescale = true;
          m_run = m_new;
          l_run *= alpha;
        }
        if (__any_sync(0xffffffffu, rescale)) {
          // O holds the products of the earlier tiles: the last of them must be done
          ok = __all_sync(0xffffffffu, wait_bar(&bars->pv_done, (gt - 1) & 1, abort_flag, a, 133));
          if (!ok) break;
          tc_fence_after();
          const uint32_t tO = tmem + lane_base + kOCol + 64 * half;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t o[16];
            tmem_ld16(tO + c * 16, o);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st16(tO + c * 16, o);
          }
        }
        const float mref = (m_run == -INFINITY) ? 0.0f : m_run;
        // P / 2^e of each 32-key block, e from the block's largest argument:
        // 2^(s c - m - e), the scale folded into the exponent; l gets the
        // block's sum times 2^e (unquantized P)
        uint32_t pk[16], sfb = 0;
        float lsum = 0.0f;
        const uint64_t c2 = f2(a.scale_log2, a.scale_log2);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int e = mx::p_block_exp(fmaf(bm[k], a.scale_log2, -mref));
          sfb |= static_cast<uint32_t>(127 + e) << (8 * (2 * half + k));
          const float off = mref + static_cast<float>(e);
          const uint64_t no2 = f2(-off, -off);
          uint64_t bs2[2] = {0, 0};
#pragma unroll
          for (int w = 0; w < 8; ++w) {  // word 8k + w: keys 32k + 4w .. + 3, byte = key % 4
            const int c = 32 * k + 4 * w;
            float x0, x1, x2, x3;
            f2_split(ffma2(f2(s[c], s[c + 1]), c2, no2), x0, x1);
            f2_split(ffma2(f2(s[c + 2], s[c + 3]), c2, no2), x2, x3);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1), p2 = ex2_approx(x2), p3 = ex2_approx(x3);
            bs2[0] = fadd2(bs2[0], f2(p0, p1));
            bs2[1] = fadd2(bs2[1], f2(p2, p3));
            pk[8 * k + w] = pack_e4m3x2(p0, p1) | (pack_e4m3x2(p2, p3) << 16);
          }
          float l0, l1;
          f2_split(fadd2(bs2[0], bs2[1]), l0, l1);
          lsum = fmaf(l0 + l1, __uint_as_float(static_cast<uint32_t>(127 + e) << 23), lsum);
        }
        l_run += lsum;
        // P codes over the first 16 of this warpgroup's S columns (already read),
        // this row's two block scales at column (quarter) of the warpgroup's word
        tmem_st16(tS, pk);
        tmem_st1(tmem + lane_base + kSfP + 8 * b + 4 * half + quarter, sfb);
        // scales of this V tile (warpgroup 1) and of K tile j + 2 (warpgroup 0),
        // for the MMAs this handover releases; the MMAs that read the buffers'
        // previous contents have completed (S(t) was issued after them)
        if (half == 1) {
          uint32_t w[4];
          mx::v_scale_words(sw, w);
          tmem_st4(tmem + lane_base + kSfV + 4 * b, w[0], w[1], w[2], w[3]);
        } else if (t + 2 < n) {
          tmem_st4(tmem + lane_base + kSfK + 4 * b, sw[0], sw[1], sw[2], sw[3]);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->p_full[b]);
      }
      if (!ok) break;
      g += n;
      // ---------------- epilogue: each warpgroup stores its 64 O columns
      const float l_tot = l_run + exchange(l_run, ok);
      if (!ok) break;
      ok = __all_sync(0xffffffffu, wait_bar(&bars->o_full, o_cnt & 1, abort_flag, a, 131));
      if (!ok) break;
      ++o_cnt;
      tc_fence_after();
      const float oscale = (l_tot > 0.0f) ? 1.0f / l_tot : 0.0f;
      const uint32_t tO = tmem + lane_base + kOCol + 64 * half;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
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
      if (valid && half == 0)
        a.f0[grow * a.H + it.h] = (l_tot > 0.0f) ? (m_run + __log2f(l_tot)) * 0.6931471805599453f : -INFINITY;
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
